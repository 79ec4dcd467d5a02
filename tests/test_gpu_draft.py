"""GPU parity for the parallel draft pass (pe_draft) against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from speculative_drafting_pe_gb300 import binding, synth

from parity import (GAP_MIN, LOGIT_RTOL, assert_drafts_match, assert_kv_close, assert_logits_close, oracle_batch,
                    oracle_request, read_new_kv, weights_to)

pytestmark = pytest.mark.gpu

# Small shapes that still span several GEMM tiles, split-K, ragged tails,
# both head sizes and several KV pages per request.
MINI_HD64 = synth.DrafterShape("mini-hd64", 512, 8, 2, 64, 1536, 5000)
MINI_HD128 = synth.DrafterShape("mini-hd128", 384, 4, 1, 128, 960, 3001)


def _draft(shape, W, inp, K, k_max=None, logits=True, stream=None):
    dev = torch.device("cuda")
    Wd = weights_to(W, dev)
    B = inp.last_token.shape[0]
    dr = binding.Drafter(shape, Wd, max_batch=B, k_max=k_max or K)
    kc, vc = inp.k_cache.to(dev).clone(), inp.v_cache.to(dev).clone()
    lg = torch.full((B, K, shape.vocab), float("nan"), device=dev) if logits else None
    d, st = dr.draft(inp.last_token.to(dev), inp.target_hidden.to(dev), inp.positions.to(dev),
                     inp.seq_lens.to(dev), inp.page_table.to(dev), inp.num_pages, kc, vc, K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    return dr, d.cpu().numpy(), st.cpu().numpy(), (lg.cpu().numpy() if logits else None), kc, vc


def _full_check(shape, W, inp, K, ref, d, st, lg, kc, vc):
    assert (st == binding.PE_REQ_OK).all()
    assert_logits_close(lg, ref["logits"])
    assert_drafts_match(d, ref)
    for b in range(inp.last_token.shape[0]):
        k_got, v_got = read_new_kv(inp, kc, vc, b, K)
        assert_kv_close(k_got, ref["k_new"][:, b], "k rows")
        assert_kv_close(v_got, ref["v_new"][:, b], "v rows")


def test_tiny_fp32_parity():
    wl = synth.WORKLOADS["tiny-fp32-b1-k3"]
    W = synth.make_weights(wl.shape, wl.seed)
    inp = synth.make_step_inputs(wl)
    ref = oracle_batch(wl.shape, synth.weights_to_numpy(W), inp, wl.K)
    dr, d, st, lg, kc, vc = _draft(wl.shape, W, inp, wl.K)
    _full_check(wl.shape, W, inp, wl.K, ref, d, st, lg, kc, vc)


@pytest.mark.parametrize("shape", [MINI_HD64, MINI_HD128], ids=lambda s: s.name)
@pytest.mark.parametrize("B,K", [(3, 5), (1, 1), (2, 16)])
def test_mini_bf16_parity(shape, B, K):
    wl = synth.Workload("mini", shape, B, K, (1, 300), (0.7, 0.7), 21)
    W = synth.make_weights(shape, 21)
    inp = synth.make_step_inputs(wl)
    ref = oracle_batch(shape, synth.weights_to_numpy(W), inp, K)
    dr, d, st, lg, kc, vc = _draft(shape, W, inp, K)
    _full_check(shape, W, inp, K, ref, d, st, lg, kc, vc)


def test_prefix_row_entries_untouched():
    # The pass writes only entries S_b .. S_b+K-1; committed prefix entries stay.
    shape = MINI_HD64
    wl = synth.Workload("mini", shape, 2, 4, (20, 60), (0.7, 0.7), 22)
    W = synth.make_weights(shape, 22)
    inp = synth.make_step_inputs(wl)
    _, d, st, lg, kc, vc = _draft(shape, W, inp, 4, logits=False)
    before_k, after_k = inp.k_cache, kc.cpu()
    mask = torch.ones(before_k.shape[1], dtype=torch.bool)
    for b in range(2):
        S = int(inp.seq_lens[b])
        for j in range(4):
            e = S + j
            page = int(inp.page_table[b, e // 16])
            after_k[:, page, :, e % 16, :] = before_k[:, page, :, e % 16, :]
    assert torch.equal(after_k, before_k)


def test_status_errors_skip_request():
    shape = MINI_HD64
    wl = synth.Workload("mini", shape, 3, 4, (20, 60), (0.7, 0.7), 23)
    W = synth.make_weights(shape, 23)
    inp = synth.make_step_inputs(wl)
    inp.seq_lens[1] = inp.page_table.shape[1] * 16 - 2       # S + K exceeds capacity
    inp.page_table[2, 0] = inp.num_pages + 5                  # bad page index
    ref0 = oracle_request(shape, synth.weights_to_numpy(W), inp, 0, 4)
    _, d, st, lg, kc, vc = _draft(shape, W, inp, 4)
    assert list(st) == [binding.PE_REQ_OK, binding.PE_REQ_CAPACITY, binding.PE_REQ_BAD_PAGE]
    assert (d[1:] == -1).all()
    assert_logits_close(lg[:1], ref0["logits"])
    assert_drafts_match(d[:1], ref0)
    # no cache writes for the failed requests: only request 0's new entries differ
    changed = (kc.cpu() != inp.k_cache).any(dim=(0, 2, 3, 4)).nonzero().flatten().tolist()
    S0 = int(inp.seq_lens[0])
    own = {int(inp.page_table[0, (S0 + j) // 16]) for j in range(4)}
    assert set(changed) <= own


def test_deterministic_across_runs():
    shape = MINI_HD64
    wl = synth.Workload("mini", shape, 4, 7, (100, 400), (0.7, 0.7), 24)
    W = synth.make_weights(shape, 24)
    inp = synth.make_step_inputs(wl)
    _, d1, _, l1, _, _ = _draft(shape, W, inp, 7)
    _, d2, _, l2, _, _ = _draft(shape, W, inp, 7)
    np.testing.assert_array_equal(d1, d2)
    np.testing.assert_array_equal(l1, l2)


def test_draft_then_verify_next_step_writes_at_slot_mapping():
    shape = MINI_HD64
    K = 5
    wl = synth.Workload("mini", shape, 3, K, (30, 90), (0.7, 0.7), 25)
    W = synth.make_weights(shape, 25)
    inp = synth.make_step_inputs(wl)
    dev = torch.device("cuda")
    dr, d, st, _, kc, vc = _draft(shape, W, inp, K, logits=False)
    g = synth.plant_targets(d, inp.alpha, shape.vocab, 25)
    out = binding.verify_rebuild(torch.as_tensor(d, device=dev), torch.as_tensor(g, device=dev),
                                 inp.page_table.to(dev), inp.num_pages, inp.positions.to(dev),
                                 inp.seq_lens.to(dev))
    torch.cuda.synchronize()
    a, bonus = oracle.verify(d, g)
    np.testing.assert_array_equal(out["accepted"].cpu().numpy(), a)
    # next step: last token = bonus, new positions / seq_lens
    before = kc.clone()
    d2, st2 = dr.draft(out["bonus"], inp.target_hidden.to(dev), out["positions"], out["seq_lens"],
                       inp.page_table.to(dev), inp.num_pages, kc, vc, K)
    torch.cuda.synchronize()
    assert (st2.cpu().numpy() == 0).all()
    slots = out["slot_mapping"].cpu().numpy()
    diff = (kc != before).any(dim=(0, 2, 4))        # [pages, 16]
    written = set((diff.nonzero()[:, 0] * 16 + diff.nonzero()[:, 1]).cpu().tolist())
    assert written <= set(slots.flatten().tolist())
    rb = out["rollback_slots"].cpu().numpy()
    assert set(rb[rb >= 0].tolist()) <= set(slots.flatten().tolist())


@pytest.mark.parametrize("K", [3, 7, 11])
def test_qwen_b1_full_size(K):
    wl = synth.WORKLOADS[f"qwen-b1-k{K}"]
    dev = torch.device("cuda")
    W = synth.make_weights(wl.shape, wl.seed, device=dev)
    inp = synth.make_step_inputs(wl, device=dev)
    Wn = synth.weights_to_numpy(W)
    ref = oracle_request(wl.shape, Wn, inp, 0, K)
    dr = binding.Drafter(wl.shape, W, max_batch=1, k_max=K)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.empty(1, K, wl.shape.vocab, device=dev)
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    assert int(st[0]) == 0
    assert_logits_close(lg.cpu().numpy(), ref["logits"])
    assert_drafts_match(d.cpu().numpy(), ref)
    k_got, v_got = read_new_kv(inp, kc, vc, 0, K)
    assert_kv_close(k_got, ref["k_new"][:, 0], "k rows")
    assert_kv_close(v_got, ref["v_new"][:, 0], "v rows")


_FULL = {}


def _full_size_setup(wl):
    """Device weights and their host copy for a workload's drafter, shared by
    the full-size tests of the same shape and seed."""
    key = (wl.shape.name, wl.seed)
    if key not in _FULL:
        _FULL.clear()
        dev = torch.device("cuda")
        W = synth.make_weights(wl.shape, wl.seed, device=dev)
        _FULL[key] = (W, synth.weights_to_numpy(W))
    return _FULL[key]


def _sample_requests(seq_lens):
    """The longest-prefix request (the one cut into the most attention
    pieces when pieces are used), the shortest, and the median one."""
    order = np.argsort(seq_lens, kind="stable")
    return sorted({int(order[-1]), int(order[0]), int(order[len(order) // 2])})


C3_PAIRS = [f"qwen-b{B}-k{K}" for B in (4, 8, 32, 128) for K in (3, 7, 11)]


@pytest.mark.parametrize("name", C3_PAIRS + ["gptoss-b64-k10"])
def test_batched_full_size_sampled(name):
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    W, Wn = _full_size_setup(wl)
    inp = synth.make_step_inputs(wl, device=dev)
    dr = binding.Drafter(wl.shape, W, max_batch=wl.B, k_max=wl.K)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.empty(wl.B, wl.K, wl.shape.vocab, device=dev)
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, wl.K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    assert (st.cpu().numpy() == 0).all()
    dn = d.cpu().numpy()
    assert ((dn >= 0) & (dn < wl.shape.vocab)).all()
    for b in _sample_requests(inp.seq_lens.cpu().numpy()):
        ref = oracle_request(wl.shape, Wn, inp, b, wl.K)
        assert_logits_close(lg[b:b + 1].cpu().numpy(), ref["logits"])
        assert_drafts_match(dn[b:b + 1], ref)
        k_got, v_got = read_new_kv(inp, kc, vc, b, wl.K)
        assert_kv_close(k_got, ref["k_new"][:, 0], "k rows")
        assert_kv_close(v_got, ref["v_new"][:, 0], "v rows")
    dr.close()


@pytest.mark.parametrize("name", ["qwen-b32-k11", "qwen-b128-k7", "qwen-b128-k11", "gptoss-b64-k10"])
def test_batched_every_request_matches_the_request_alone(name):
    # Every request of a full-size batch (not a sample) against the same
    # request drafted alone at B=1, whose path the full-size B=1 tests pin
    # to the oracle: the batched launches (other token tiles, split-K,
    # epilogue warp groups, attention pieces) may change rounding only.
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    W = synth.make_weights(wl.shape, wl.seed, device=dev)
    inp = synth.make_step_inputs(wl, device=dev)
    V = wl.shape.vocab
    dr = binding.Drafter(wl.shape, W, max_batch=wl.B, k_max=wl.K)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.empty(wl.B, wl.K, V, device=dev)
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, wl.K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    assert (st.cpu().numpy() == 0).all()
    dr.close()
    one = binding.Drafter(wl.shape, W, max_batch=1, k_max=wl.K)
    kc1, vc1 = inp.k_cache.clone(), inp.v_cache.clone()   # each request writes only its own pages
    lg1 = torch.empty(1, wl.K, V, device=dev)
    bad_logits, bad_drafts = [], []
    for b in range(wl.B):
        s = slice(b, b + 1)
        d1, st1 = one.draft(inp.last_token[s], inp.target_hidden[s], inp.positions[s], inp.seq_lens[s],
                            inp.page_table[s], inp.num_pages, kc1, vc1, wl.K, logits=lg1)
        err = (lg[b] - lg1[0]).abs().amax(dim=-1)
        scale = lg1[0].abs().amax(dim=-1)
        if bool((err > LOGIT_RTOL * scale).any()):
            bad_logits.append(b)
        top2 = lg1[0].topk(2, dim=-1).values
        sure = (top2[:, 0] - top2[:, 1]) > GAP_MIN
        if bool(((d[b] != d1[0]) & sure).any()):
            bad_drafts.append(b)
    torch.cuda.synchronize()
    assert one.device_errors() == 0
    assert not bad_logits, f"requests whose batched logits differ from the request alone: {bad_logits}"
    assert not bad_drafts, f"requests whose batched drafts differ where the gap is clear: {bad_drafts}"
    for b in range(wl.B):
        k_b, v_b = read_new_kv(inp, kc, vc, b, wl.K)
        k_1, v_1 = read_new_kv(inp, kc1, vc1, b, wl.K)
        assert_kv_close(k_b, k_1, f"k rows of request {b}")
        assert_kv_close(v_b, v_1, f"v rows of request {b}")
    one.close()


@pytest.mark.parametrize("name", ["qwen-b32-k7", "qwen-b128-k11", "gptoss-b64-k10"])
def test_full_size_batches_are_deterministic(name):
    # The same batch drafted twice (two epilogue warp groups, attention
    # pieces, split-K clusters): every logit, draft and cache row must repeat
    # bit for bit; a read racing with an earlier kernel's writes would not.
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    W = synth.make_weights(wl.shape, wl.seed, device=dev)
    inp = synth.make_step_inputs(wl, device=dev)
    dr = binding.Drafter(wl.shape, W, max_batch=wl.B, k_max=wl.K)
    runs = []
    for _ in range(2):
        kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
        lg = torch.empty(wl.B, wl.K, wl.shape.vocab, device=dev)
        d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                         inp.num_pages, kc, vc, wl.K, logits=lg)
        torch.cuda.synchronize()
        runs.append((lg, d, kc, vc))
    assert dr.device_errors() == 0
    (l1, d1, k1, v1), (l2, d2, k2, v2) = runs
    assert torch.equal(d1, d2)
    assert torch.equal(l1, l2)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    dr.close()


@pytest.mark.parametrize("name", ["qwen-b1-k7", "qwen-b128-k11"])
def test_step_graph_without_logits_matches_oracle(name):
    # The exact call the benchmark times: draft (no logits output) + verify
    # replayed from the step graph. Drafts under the gap rule, the verify
    # outputs bit-exact against the oracle's verify of those drafts.
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    W, Wn = _full_size_setup(wl)
    inp = synth.make_step_inputs(wl, device=dev)
    dr = binding.Drafter(wl.shape, W, max_batch=wl.B, k_max=wl.K)
    g = torch.as_tensor(synth.plant_targets(np.zeros((wl.B, wl.K), np.int64), inp.alpha, wl.shape.vocab, wl.seed),
                        device=dev)
    sg = dr.step_graph(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                       inp.num_pages, inp.k_cache, inp.v_cache, wl.K, g)
    sg.launch()
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    dn = sg.out["drafts"].cpu().numpy()
    assert (sg.out["draft_status"].cpu().numpy() == 0).all()
    for b in _sample_requests(inp.seq_lens.cpu().numpy()):
        ref = oracle_request(wl.shape, Wn, inp, b, wl.K)
        assert_drafts_match(dn[b:b + 1], ref)
    a, bonus = oracle.verify(dn, g.cpu().numpy())
    meta = oracle.rebuild_metadata(a, wl.K, inp.seq_lens.cpu().numpy(), inp.positions.cpu().numpy(),
                                   inp.page_table.cpu().numpy(), inp.num_pages)
    np.testing.assert_array_equal(sg.out["accepted"].cpu().numpy(), a)
    np.testing.assert_array_equal(sg.out["bonus"].cpu().numpy(), bonus)
    for k in ("slot_mapping", "rollback_slots", "status", "positions", "seq_lens"):
        np.testing.assert_array_equal(sg.out[k].cpu().numpy(), meta[k], err_msg=k)
    sg.close()
    dr.close()
