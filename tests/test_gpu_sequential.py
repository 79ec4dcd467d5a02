"""GPU parity for sequential (EAGLE-style) drafting, pe_draft_sequential:
K one-row passes on the same kernels, against the oracle's
draft_sequential. The oracle is given the GPU's drafts as the input tokens
of passes 1..K-1, so that a near-tie decided differently in one pass cannot
make the two implementations draft different sequences afterwards; every
row's logits, the drafts under the gap rule and every pass's cache rows are
then compared."""

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


def _oracle_seq(shape, Wn, inp, b, K, tokens):
    sp = request_subproblem(inp, b)
    return oracle.draft_sequential(shape, Wn, sp["last_token"], sp["target_hidden"], sp["positions"],
                                   sp["seq_lens"], sp["page_table"], sp["k_cache"], sp["v_cache"], K,
                                   tokens=tokens[None, :])


def _gpu_seq(shape, W, inp, K, logits=True):
    dev = torch.device("cuda")
    B = inp.last_token.shape[0]
    dr = binding.Drafter(shape, W, max_batch=B, k_max=K)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.full((B, K, shape.vocab), float("nan"), device=dev) if logits else None
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, K, logits=lg, sequential=True)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    return dr, d.cpu().numpy(), st.cpu().numpy(), (lg.cpu().numpy() if logits else None), kc, vc


def _check_request(shape, Wn, inp, b, K, d, lg, kc, vc):
    ref = _oracle_seq(shape, Wn, inp, b, K, d[b])
    assert_logits_close(lg[b:b + 1], ref["logits"])
    assert_drafts_match(d[b:b + 1], ref)
    k_got, v_got = read_new_kv(inp, kc, vc, b, K)
    assert_kv_close(k_got, ref["k_new"][:, 0], "k rows")
    assert_kv_close(v_got, ref["v_new"][:, 0], "v rows")


@pytest.mark.parametrize("shape", [MINI_HD64, MINI_HD128], ids=lambda s: s.name)
@pytest.mark.parametrize("B,K", [(3, 5), (1, 1), (2, 16)])
def test_sequential_mini_parity(shape, B, K):
    dev = torch.device("cuda")
    wl = synth.Workload("mini-seq", shape, B, K, (1, 300), (0.7, 0.7), 41)
    W = weights_to(synth.make_weights(shape, 41), dev)
    inp = synth.make_step_inputs(wl, device=dev)
    Wn = synth.weights_to_numpy(W)
    _, d, st, lg, kc, vc = _gpu_seq(shape, W, inp, K)
    assert (st == binding.PE_REQ_OK).all()
    for b in range(B):
        _check_request(shape, Wn, inp, b, K, d, lg, kc, vc)


def test_sequential_k1_equals_parallel_k1():
    # one sequential pass runs the parallel pass's kernels on the same rows
    dev = torch.device("cuda")
    shape = MINI_HD64
    wl = synth.Workload("mini-seq", shape, 4, 1, (20, 200), (0.7, 0.7), 42)
    W = weights_to(synth.make_weights(shape, 42), dev)
    inp = synth.make_step_inputs(wl, device=dev)
    dr = binding.Drafter(shape, W, max_batch=4, k_max=1)
    out = []
    for seq in (False, True):
        kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
        lg = torch.empty(4, 1, shape.vocab, device=dev)
        d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                         inp.num_pages, kc, vc, 1, logits=lg, sequential=seq)
        torch.cuda.synchronize()
        out.append((d.clone(), lg.clone(), kc))
    assert torch.equal(out[0][0], out[1][0])
    assert torch.equal(out[0][1], out[1][1])
    assert torch.equal(out[0][2], out[1][2])


def test_sequential_status_errors_skip_request():
    dev = torch.device("cuda")
    shape = MINI_HD64
    K = 4
    wl = synth.Workload("mini-seq", shape, 3, K, (20, 60), (0.7, 0.7), 43)
    W = weights_to(synth.make_weights(shape, 43), dev)
    inp = synth.make_step_inputs(wl, device=dev)
    inp.seq_lens[1] = inp.page_table.shape[1] * 16 - 2       # S + K exceeds capacity
    inp.page_table[2, 0] = inp.num_pages + 5                  # bad page index
    Wn = synth.weights_to_numpy(W)
    _, d, st, lg, kc, vc = _gpu_seq(shape, W, inp, K)
    assert list(st) == [binding.PE_REQ_OK, binding.PE_REQ_CAPACITY, binding.PE_REQ_BAD_PAGE]
    assert (d[1:] == -1).all()
    _check_request(shape, Wn, inp, 0, K, d, lg, kc, vc)
    changed = (kc.cpu() != inp.k_cache.cpu()).any(dim=(0, 2, 3, 4)).nonzero().flatten().tolist()
    S0 = int(inp.seq_lens[0])
    own = {int(inp.page_table[0, (S0 + j) // 16]) for j in range(K)}
    assert set(changed) <= own


def test_sequential_step_graph_matches_direct_calls():
    dev = torch.device("cuda")
    shape = MINI_HD128
    K = 5
    wl = synth.Workload("mini-seq", shape, 3, K, (40, 300), (0.7, 0.7), 44)
    W = weights_to(synth.make_weights(shape, 44), dev)
    inp = synth.make_step_inputs(wl, device=dev)
    dr, d, st, _, kc, vc = _gpu_seq(shape, W, inp, K, logits=False)
    g = torch.as_tensor(synth.plant_targets(d, inp.alpha, shape.vocab, 44), device=dev)
    ref = binding.verify_rebuild(torch.as_tensor(d, device=dev), g, inp.page_table, inp.num_pages, inp.positions,
                                 inp.seq_lens)
    torch.cuda.synchronize()
    kc2, vc2 = inp.k_cache.clone(), inp.v_cache.clone()
    sg = dr.step_graph(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                       inp.num_pages, kc2, vc2, K, g, sequential=True)
    for _ in range(2):
        sg.launch()
    torch.cuda.synchronize()
    assert np.array_equal(sg.out["drafts"].cpu().numpy(), d)
    for k in ("accepted", "bonus", "slot_mapping", "rollback_slots", "status", "positions", "seq_lens"):
        assert torch.equal(sg.out[k], ref[k]), k
    assert torch.equal(kc2, kc) and torch.equal(vc2, vc)
    assert dr.device_errors() == 0


@pytest.mark.parametrize("name,K", [("qwen-b1-k3", 3), ("qwen-b4-k3", 3)])
def test_sequential_full_size(name, K):
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    W = synth.make_weights(wl.shape, wl.seed, device=dev)
    Wn = synth.weights_to_numpy(W)
    inp = synth.make_step_inputs(wl, device=dev)
    _, d, st, lg, kc, vc = _gpu_seq(wl.shape, W, inp, K)
    assert (st == binding.PE_REQ_OK).all()
    seq = inp.seq_lens.cpu().numpy()
    for b in sorted({int(np.argmax(seq)), int(np.argmin(seq))}):
        _check_request(wl.shape, Wn, inp, b, K, d, lg, kc, vc)
