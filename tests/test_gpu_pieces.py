"""Length-aware attention pieces (used from 16 (request, kv head) pairs on):
each request's cache entries cut into pieces of about the same tile count,
the partials of a request with several pieces combined by the merge kernel.
Checked against the oracle on mini shapes that switch the mode on, with
failed requests among the batch."""

import numpy as np
import pytest
import torch

from speculative_drafting_pe_gb300 import binding, synth

from parity import (assert_drafts_match, assert_kv_close, assert_logits_close, oracle_batch, oracle_request,
                    read_new_kv, weights_to)

pytestmark = pytest.mark.gpu

MINI_HD64 = synth.DrafterShape("mini-hd64", 512, 8, 2, 64, 1536, 5000)     # G = 4
MINI_HD128 = synth.DrafterShape("mini-hd128", 384, 4, 1, 128, 960, 3001)   # G = 4
MINI_MHA = synth.DrafterShape("mini-mha", 256, 2, 2, 128, 512, 3000)       # G = 1: odd query-row counts

# per-GEMM pass with logits: FC, row build, 4 x (QKV, attention, O, gate/up,
# down), LM head, logits scaling, argmax; pieces add one merge per layer
LAUNCHES_WITH_LOGITS = 25
MERGES = 4


def _draft(shape, W, inp, K):
    dev = torch.device("cuda")
    B = inp.last_token.shape[0]
    dr = binding.Drafter(shape, weights_to(W, dev), max_batch=B, k_max=K)
    kc, vc = inp.k_cache.to(dev).clone(), inp.v_cache.to(dev).clone()
    lg = torch.full((B, K, shape.vocab), float("nan"), device=dev)
    d, st = dr.draft(inp.last_token.to(dev), inp.target_hidden.to(dev), inp.positions.to(dev),
                     inp.seq_lens.to(dev), inp.page_table.to(dev), inp.num_pages, kc, vc, K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    n = dr.launch_count()
    dr.close()
    return d.cpu().numpy(), st.cpu().numpy(), lg.cpu().numpy(), kc, vc, n


@pytest.mark.parametrize("shape,B,K", [(MINI_HD64, 9, 5), (MINI_HD128, 16, 7), (MINI_MHA, 16, 5)],
                         ids=["hd64-b9k5", "hd128-b16k7", "mha-b16k5"])
def test_pieces_oracle_parity(shape, B, K):
    # prefixes up to 1100 entries: requests longer than four 64-entry tiles
    # are cut into several pieces, short ones stay whole
    wl = synth.Workload("pieces", shape, B, K, (1, 1100), (0.7, 0.7), 31 + B)
    W = synth.make_weights(shape, wl.seed)
    inp = synth.make_step_inputs(wl)
    ref = oracle_batch(shape, synth.weights_to_numpy(W), inp, K)
    d, st, lg, kc, vc, n = _draft(shape, W, inp, K)
    assert n == LAUNCHES_WITH_LOGITS + MERGES, n
    assert (st == binding.PE_REQ_OK).all()
    assert_logits_close(lg, ref["logits"])
    assert_drafts_match(d, ref)
    for b in range(B):
        k_got, v_got = read_new_kv(inp, kc, vc, b, K)
        assert_kv_close(k_got, ref["k_new"][:, b], "k rows")
        assert_kv_close(v_got, ref["v_new"][:, b], "v rows")


def test_pieces_failed_requests_write_nothing():
    shape, B, K = MINI_HD64, 10, 4
    wl = synth.Workload("pieces-status", shape, B, K, (300, 1000), (0.7, 0.7), 47)
    W = synth.make_weights(shape, wl.seed)
    inp = synth.make_step_inputs(wl)
    inp.seq_lens[1] = inp.page_table.shape[1] * 16 - 2       # S + K exceeds capacity
    inp.page_table[2, 3] = inp.num_pages + 5                  # bad page index inside a long request
    d, st, lg, kc, vc, n = _draft(shape, W, inp, K)
    assert n == LAUNCHES_WITH_LOGITS + MERGES, n
    assert st[1] == binding.PE_REQ_CAPACITY and st[2] == binding.PE_REQ_BAD_PAGE
    assert (np.delete(st, [1, 2]) == binding.PE_REQ_OK).all()
    assert (d[1:3] == -1).all()
    Wn = synth.weights_to_numpy(W)
    for b in (0, 5, 9):
        ref = oracle_request(shape, Wn, inp, b, K)
        assert_logits_close(lg[b:b + 1], ref["logits"])
        assert_drafts_match(d[b:b + 1], ref)
    changed = (kc.cpu() != inp.k_cache).any(dim=(0, 2, 3, 4)).nonzero().flatten().tolist()
    mine = set()
    for b in range(B):
        if b in (1, 2):
            continue
        S = int(inp.seq_lens[b])
        mine |= {int(inp.page_table[b, (S + j) // 16]) for j in range(K)}
    assert set(changed) <= mine


def test_pieces_deterministic():
    shape, B, K = MINI_HD64, 12, 6
    wl = synth.Workload("pieces-det", shape, B, K, (1, 1100), (0.5, 0.8), 53)
    W = synth.make_weights(shape, wl.seed)
    inp = synth.make_step_inputs(wl)
    d1, _, l1, _, _, _ = _draft(shape, W, inp, K)
    d2, _, l2, _, _, _ = _draft(shape, W, inp, K)
    np.testing.assert_array_equal(d1, d2)
    np.testing.assert_array_equal(l1, l2)
