"""GPU parity for the parallel draft pass with re-fed real rows
(pe_draft_refeed) and its verify/rebuild (pe_verify_rebuild_refeed) against
the oracle's draft_pass_refeed and rebuild_metadata_refeed."""

import numpy as np
import pytest
import torch

import oracle
from speculative_drafting_pe_gb300 import binding, synth

from parity import (assert_drafts_match, assert_kv_close, assert_logits_close, read_new_kv, request_subproblem,
                    weights_to)

pytestmark = pytest.mark.gpu

MINI_HD64 = synth.DrafterShape("mini-hd64", 512, 8, 2, 64, 1536, 5000)
MINI_HD128 = synth.DrafterShape("mini-hd128", 384, 4, 1, 128, 960, 3001)


def _setup(shape, B, K, n_max, seed, dev, prefix=(1, 300), W=None):
    wl = synth.Workload("refeed", shape, B, K, prefix, (0.7, 0.7), seed)
    if W is None:
        W = weights_to(synth.make_weights(shape, seed), dev)
    inp = synth.make_step_inputs(wl, device=dev, K=K + n_max)
    tokens, n_real, th = synth.make_refeed_inputs(wl, n_max, device=dev)
    return wl, W, inp, tokens, n_real, th


def _gpu(dr, inp, tokens, n_real, th, K, logits=True):
    B = tokens.shape[0]
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.full((B, K, dr.shape.vocab), float("nan"), device=dr.device) if logits else None
    d, st = dr.draft_refeed(tokens, n_real, th, inp.positions, inp.seq_lens, inp.page_table, inp.num_pages, kc, vc,
                            K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    return d.cpu().numpy(), st.cpu().numpy(), (lg.cpu().numpy() if logits else None), kc, vc


def _oracle_req(shape, Wn, inp, b, tokens, n_real, th, K):
    sp = request_subproblem(inp, b)
    return oracle.draft_pass_refeed(shape, Wn, tokens[b:b + 1].cpu().numpy(), n_real[b:b + 1].cpu().numpy(),
                                    th[b:b + 1].cpu().double().numpy(), sp["positions"], sp["seq_lens"],
                                    sp["page_table"], sp["k_cache"], sp["v_cache"], K)


def _check_req(shape, Wn, inp, b, tokens, n_real, th, K, d, lg, kc, vc):
    ref = _oracle_req(shape, Wn, inp, b, tokens, n_real, th, K)
    assert_logits_close(lg[b:b + 1], ref["logits"])
    assert_drafts_match(d[b:b + 1], ref)
    T = int(n_real[b]) + K - 1
    k_got, v_got = read_new_kv(inp, kc, vc, b, T)
    assert_kv_close(k_got, ref["k_new"][:, 0, :T], "k rows")
    assert_kv_close(v_got, ref["v_new"][:, 0, :T], "v rows")


@pytest.mark.parametrize("shape", [MINI_HD64, MINI_HD128], ids=lambda s: s.name)
@pytest.mark.parametrize("B,K,n_max", [(3, 5, 4), (1, 1, 2), (2, 7, 8), (4, 3, 1)])
def test_refeed_mini_parity(shape, B, K, n_max):
    dev = torch.device("cuda")
    wl, W, inp, tokens, n_real, th = _setup(shape, B, K, n_max, 71, dev)
    Wn = synth.weights_to_numpy(W)
    dr = binding.Drafter(shape, W, max_batch=B, k_max=max(K, n_max))
    d, st, lg, kc, vc = _gpu(dr, inp, tokens, n_real, th, K)
    assert (st == binding.PE_REQ_OK).all()
    for b in range(B):
        _check_req(shape, Wn, inp, b, tokens, n_real, th, K, d, lg, kc, vc)


def test_refeed_one_real_row_equals_parallel_pass():
    dev = torch.device("cuda")
    shape, B, K = MINI_HD64, 3, 5
    wl, W, inp, tokens, n_real, th = _setup(shape, B, K, 1, 72, dev)
    dr = binding.Drafter(shape, W, max_batch=B, k_max=K)
    d1, st1, lg1, kc1, vc1 = _gpu(dr, inp, tokens, n_real, th, K)
    kc2, vc2 = inp.k_cache.clone(), inp.v_cache.clone()
    lg2 = torch.empty(B, K, shape.vocab, device=dev)
    d2, st2 = dr.draft(tokens[:, 0].contiguous(), th[:, 0].contiguous(), inp.positions, inp.seq_lens,
                       inp.page_table, inp.num_pages, kc2, vc2, K, logits=lg2)
    torch.cuda.synchronize()
    assert np.array_equal(d1, d2.cpu().numpy())
    assert np.array_equal(lg1, lg2.cpu().numpy())
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)


def test_refeed_status_errors_skip_request():
    dev = torch.device("cuda")
    shape, B, K, n_max = MINI_HD64, 4, 4, 3
    wl, W, inp, tokens, n_real, th = _setup(shape, B, K, n_max, 73, dev, prefix=(20, 60))
    n_real[1] = n_max + 1                                    # out of range
    tokens[2, 0] = shape.vocab                               # bad token among the real rows
    n_real[2] = max(int(n_real[2]), 1)
    inp.seq_lens[3] = inp.page_table.shape[1] * 16 - n_max   # entries past the page table
    Wn = synth.weights_to_numpy(W)
    dr = binding.Drafter(shape, W, max_batch=B, k_max=K)
    d, st, lg, kc, vc = _gpu(dr, inp, tokens, n_real, th, K)
    assert list(st) == [binding.PE_REQ_OK, binding.PE_REQ_BAD_INPUT, binding.PE_REQ_BAD_INPUT,
                        binding.PE_REQ_CAPACITY]
    assert (d[1:] == -1).all()
    _check_req(shape, Wn, inp, 0, tokens, n_real, th, K, d, lg, kc, vc)
    changed = (kc.cpu() != inp.k_cache.cpu()).any(dim=(0, 2, 3, 4)).nonzero().flatten().tolist()
    S0 = int(inp.seq_lens[0])
    own = {int(inp.page_table[0, (S0 + j) // 16]) for j in range(int(n_real[0]) + K - 1)}
    assert set(changed) <= own


def _verify_case(B, K, seed):
    rng = np.random.default_rng(seed)
    v = synth.make_verify_inputs(B, K, 1000, (0, 400), 0.6, seed=seed)
    v["n_real"] = rng.integers(1, K + 2, size=B).astype(np.int32)
    # pages for the next pass's n' + K - 1 entries beyond S + n
    v["page_table"], v["num_pages"] = synth.page_pool(v["seq_lens"], 2 * K + 2, 16, rng)
    return v


@pytest.mark.parametrize("K", [1, 3, 11, 16])
def test_verify_refeed_bit_exact(lib, K):
    dev = torch.device("cuda")
    v = _verify_case(97, K, 80 + K)
    t = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device=dev)
    out = binding.verify_rebuild_refeed(t(v["drafts"]), t(v["targets"]), t(v["page_table"]), v["num_pages"],
                                        t(v["n_real"]), t(v["positions"]), t(v["seq_lens"]))
    torch.cuda.synchronize()
    a, bonus = oracle.verify(v["drafts"], v["targets"])
    meta = oracle.rebuild_metadata_refeed(a, K, v["n_real"], v["seq_lens"], v["positions"], v["page_table"],
                                          v["num_pages"])
    np.testing.assert_array_equal(out["accepted"].cpu().numpy(), a)
    np.testing.assert_array_equal(out["bonus"].cpu().numpy(), bonus)
    np.testing.assert_array_equal(out["emitted"].cpu().numpy(), oracle.emitted_tokens(v["drafts"], a, bonus))
    for k in ("seq_lens", "positions", "n_real", "slot_mapping", "rollback_slots", "status"):
        np.testing.assert_array_equal(out[k].cpu().numpy(), meta[k], err_msg=k)


def test_verify_refeed_status_cases(lib):
    dev = torch.device("cuda")
    K = 3
    pt = np.array([[0, 1], [2, 3], [4, -1], [5, 6]])
    v = dict(drafts=np.array([[1, 2, 3]] * 4), targets=np.array([[1, 2, 3, 9], [5, 5, 5, 5], [1, 2, 3, 9],
                                                                  [5, 5, 5, 5]]),
             seq_lens=np.array([20, 5, 10, -2]), positions=np.array([30, 30, 12, 4]), n_real=np.array([4, 1, 2, 1]))
    t = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device=dev)
    out = binding.verify_rebuild_refeed(t(v["drafts"]), t(v["targets"]), t(pt), 7, t(v["n_real"]),
                                        t(v["positions"]), t(v["seq_lens"]))
    torch.cuda.synchronize()
    a, _ = oracle.verify(v["drafts"], v["targets"])
    meta = oracle.rebuild_metadata_refeed(a, K, v["n_real"], v["seq_lens"], v["positions"], pt, 7)
    for k in ("seq_lens", "positions", "n_real", "slot_mapping", "rollback_slots", "status"):
        np.testing.assert_array_equal(out[k].cpu().numpy(), meta[k], err_msg=k)


def test_refeed_two_steps_write_where_the_rebuild_says():
    # step 1 drafts with re-fed rows, the verify rebuilds the metadata, and
    # step 2 (re-feeding the emitted tokens) writes exactly the slots the
    # rebuild listed
    dev = torch.device("cuda")
    shape, B, K, n_max = MINI_HD128, 3, 4, 3
    wl, W, inp, tokens, n_real, th = _setup(shape, B, K, n_max, 74, dev, prefix=(30, 90))
    # pages for two steps of up to K+1 real rows and K-1 placeholders
    inp = synth.make_step_inputs(wl, device=dev, K=3 * K + 2)
    dr = binding.Drafter(shape, W, max_batch=B, k_max=K + 1)
    d, st, _, kc, vc = _gpu(dr, inp, tokens, n_real, th, K, logits=False)
    g = torch.as_tensor(synth.plant_targets(d, inp.alpha, shape.vocab, 74), device=dev)
    out = binding.verify_rebuild_refeed(torch.as_tensor(d, device=dev), g, inp.page_table, inp.num_pages, n_real,
                                        inp.positions, inp.seq_lens)
    torch.cuda.synchronize()
    assert (out["status"].cpu().numpy() == 0).all()
    n2 = out["n_real"]
    n2_max = int(n2.max())
    tok2 = out["emitted"][:, :n2_max].contiguous()
    th2 = torch.randn(B, n2_max, 3 * shape.hidden, device=dev).to(torch.bfloat16)
    before = kc.clone()
    d2, st2 = dr.draft_refeed(tok2, n2, th2, out["positions"], out["seq_lens"], inp.page_table, inp.num_pages, kc,
                              vc, K)
    torch.cuda.synchronize()
    assert (st2.cpu().numpy() == 0).all()
    slots = out["slot_mapping"].cpu().numpy()
    diff = (kc != before).any(dim=(0, 2, 4))
    written = set((diff.nonzero()[:, 0] * 16 + diff.nonzero()[:, 1]).cpu().tolist())
    assert written <= set(slots[slots >= 0].tolist())
    assert dr.device_errors() == 0


@pytest.mark.parametrize("name,n_max", [("qwen-b1-k7", 8), ("qwen-b8-k7", 8), ("qwen-b32-k3", 4)])
def test_refeed_full_size(name, n_max):
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    W = synth.make_weights(wl.shape, wl.seed, device=dev)
    Wn = synth.weights_to_numpy(W)
    wl2, _, inp, tokens, n_real, th = _setup(wl.shape, wl.B, wl.K, n_max, wl.seed, dev, prefix=wl.prefix, W=W)
    dr = binding.Drafter(wl.shape, W, max_batch=wl.B, k_max=max(wl.K, n_max))
    d, st, lg, kc, vc = _gpu(dr, inp, tokens, n_real, th, wl.K)
    assert (st == binding.PE_REQ_OK).all()
    seq = inp.seq_lens.cpu().numpy()
    for b in sorted({int(np.argmax(seq)), int(np.argmin(seq))}):
        _check_req(wl.shape, Wn, inp, b, tokens, n_real, th, wl.K, d, lg, kc, vc)
