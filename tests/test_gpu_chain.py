"""The persistent layer chain (O, gate/up, down and the next QKV or the LM
head in one cooperative launch per layer), selected by PE_LAYER_CHAIN=1 at
handle creation: against the oracle, and against the per-GEMM launches of
the same draft pass (the default)."""

import dataclasses

import numpy as np
import pytest
import torch

from speculative_drafting_pe_gb300 import binding, synth

import oracle  # noqa: F401  (the parity helpers call it)
from parity import (assert_drafts_match, assert_kv_close, assert_logits_close, oracle_batch, read_new_kv,
                    weights_to)

pytestmark = pytest.mark.gpu

MINI_HD64 = synth.DrafterShape("mini-hd64", 512, 8, 2, 64, 1536, 5000)
MINI_ODD_H = synth.DrafterShape("mini-h448", 448, 4, 2, 64, 1088, 2500)   # H not a multiple of 128


def _run(monkeypatch, chain, shape, W, inp, K, logits=True):
    monkeypatch.setenv("PE_LAYER_CHAIN", "1" if chain else "0")
    dev = torch.device("cuda")
    B = inp.last_token.shape[0]
    dr = binding.Drafter(shape, W, max_batch=B, k_max=K)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.empty(B, K, shape.vocab, device=dev) if logits else None
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    n = dr.launch_count()
    dr.close()
    return d.cpu().numpy(), st.cpu().numpy(), (lg.cpu().numpy() if logits else None), kc, vc, n


def _setup(shape, B, K, seed, prefix=(1, 700)):
    dev = torch.device("cuda")
    wl = synth.Workload("chain", shape, B, K, prefix, (0.7, 0.7), seed)
    W = weights_to(synth.make_weights(shape, seed), dev)
    inp = synth.make_step_inputs(wl, device=dev)
    return W, inp


def _compare(a, b, K):
    d1, st1, lg1, kc1, vc1, _ = a
    d2, st2, lg2, kc2, vc2, _ = b
    assert (st1 == binding.PE_REQ_OK).all() and (st2 == binding.PE_REQ_OK).all()
    # logits: the two paths sum in different orders and round different
    # intermediates to bf16; per row they agree far inside the oracle rule
    diff = np.abs(lg1 - lg2).max(axis=-1)
    scale = np.abs(lg2).max(axis=-1)
    assert (diff <= 1e-2 * scale).all(), float((diff / scale).max())
    # drafts: equal wherever the per-GEMM path's top-2 gap exceeds twice the
    # row's largest logit difference (the argmax cannot move there)
    top2 = np.sort(lg2, axis=-1)[..., -2:]
    gap = top2[..., 1] - top2[..., 0]
    firm = gap > 2 * diff
    assert firm.mean() > 0.5
    assert (d1[firm] == d2[firm]).all()
    # the new cache rows agree the same way (every other entry is untouched by both)
    for x, y in ((kc1, kc2), (vc1, vc2)):
        dx = (x.float() - y.float()).abs().max().item()
        assert dx <= 1e-2 * y.float().abs().max().item(), dx


@pytest.mark.parametrize("shape,B,K", [(MINI_HD64, 3, 5), (MINI_HD64, 4, 16), (MINI_ODD_H, 2, 7)],
                         ids=["mini-b3k5", "mini-b4k16", "oddH-b2k7"])
def test_chain_matches_per_gemm_path(monkeypatch, shape, B, K):
    W, inp = _setup(shape, B, K, seed=41 + B)
    a = _run(monkeypatch, True, shape, W, inp, K)
    b = _run(monkeypatch, False, shape, W, inp, K)
    _compare(a, b, K)
    # the chained pass: FC, row build, layer 0 QKV, 4 attentions, 4 chains,
    # logits scaling, argmax; the per-GEMM pass launches every GEMM alone
    assert a[5] == 13, a[5]
    assert b[5] == 25, b[5]


def test_chain_oracle_parity(monkeypatch):
    shape = MINI_HD64
    wl = synth.Workload("chain-oracle", shape, 3, 5, (1, 300), (0.7, 0.7), 23)
    W = synth.make_weights(shape, 23)
    inp = synth.make_step_inputs(wl)
    ref = oracle_batch(shape, synth.weights_to_numpy(W), inp, wl.K)
    dev = torch.device("cuda")
    # the oracle's own inputs, copied to the device
    inp_d = dataclasses.replace(inp, **{f.name: getattr(inp, f.name).to(dev) for f in dataclasses.fields(inp)
                                        if isinstance(getattr(inp, f.name), torch.Tensor)})
    d, st, lg, kc, vc, n = _run(monkeypatch, True, shape, weights_to(W, dev), inp_d, wl.K)
    assert n == 13
    assert (st == binding.PE_REQ_OK).all()
    assert_logits_close(lg, ref["logits"])
    assert_drafts_match(d, ref)
    for b in range(wl.B):
        k_got, v_got = read_new_kv(inp, kc, vc, b, wl.K)
        assert_kv_close(k_got, ref["k_new"][:, b], "k rows")
        assert_kv_close(v_got, ref["v_new"][:, b], "v rows")


@pytest.mark.parametrize("K", [3, 11])
def test_chain_qwen_shape_b1(monkeypatch, K):
    shape = synth.QWEN3_CODER_30B_A3B
    W, inp = _setup(shape, 1, K, seed=5, prefix=(2048, 2048))
    a = _run(monkeypatch, True, shape, W, inp, K)
    b = _run(monkeypatch, False, shape, W, inp, K)
    _compare(a, b, K)


def test_chain_repeatable_and_counters_reset(monkeypatch):
    """Two chained passes in a row give bit-identical results: the phase
    counters and tile tickets are back at zero after every launch."""
    W, inp = _setup(MINI_HD64, 2, 9, seed=77)
    a = _run(monkeypatch, True, MINI_HD64, W, inp, 9)
    monkeypatch.setenv("PE_LAYER_CHAIN", "1")
    dev = torch.device("cuda")
    dr = binding.Drafter(MINI_HD64, W, max_batch=2, k_max=9)
    outs = []
    for _ in range(3):
        kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
        lg = torch.empty(2, 9, MINI_HD64.vocab, device=dev)
        d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                         inp.num_pages, kc, vc, 9, logits=lg)
        torch.cuda.synchronize()
        outs.append((d.cpu().numpy(), lg.cpu().numpy()))
    assert dr.device_errors() == 0
    dr.close()
    for d, lg in outs:
        assert (d == a[0]).all()
        assert np.array_equal(lg, a[2])


def test_chain_wait_gives_up_and_the_handle_recovers(monkeypatch):
    # Host-side injection: the first phase's tickets are primed so that its
    # shared tiles never complete. The next phase's waits must give up after
    # their time limit, report PE_DEVERR_CHAIN_TIMEOUT and return; the next
    # draft pass on the same handle must then be oracle-correct.
    import time

    shape, B, K = MINI_HD64, 2, 5
    W, inp = _setup(shape, B, K, seed=61)
    ref = oracle_batch(shape, synth.weights_to_numpy(W), inp, K)
    monkeypatch.setenv("PE_LAYER_CHAIN", "1")
    dev = torch.device("cuda")
    dr = binding.Drafter(shape, W, max_batch=B, k_max=K)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    dr.test_stall_chain()
    t0 = time.time()
    dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table, inp.num_pages,
             kc, vc, K)
    torch.cuda.synchronize()
    waited = time.time() - t0
    bits = dr.device_errors()
    assert bits & binding.PE_DEVERR_CHAIN_TIMEOUT, bits
    assert waited < 30.0, waited
    assert dr.launch_count() < 27          # the chain ran (it replaces 13 per-GEMM launches)

    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.empty(B, K, shape.vocab, device=dev)
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    assert (st.cpu().numpy() == binding.PE_REQ_OK).all()
    assert_logits_close(lg.cpu().numpy(), ref["logits"])
    assert_drafts_match(d.cpu().numpy(), ref)
    for b in range(B):
        k_got, v_got = read_new_kv(inp, kc, vc, b, K)
        assert_kv_close(k_got, ref["k_new"][:, b], "k rows")
        assert_kv_close(v_got, ref["v_new"][:, b], "v rows")
    dr.close()
