"""FP8 (E4M3) drafter weights on the GPU: the FP8-weight GEMM engine against a
float64 product of the decoded weights, and the whole draft pass (parallel
and sequential) against the oracle run on the dequantised weights
(W = decode(q) * scale per output row)."""

import numpy as np
import pytest
import torch

import oracle
from speculative_drafting_pe_gb300 import binding, synth

from parity import (assert_drafts_match, assert_kv_close, assert_logits_close, oracle_batch, oracle_request,
                    read_new_kv)

pytestmark = pytest.mark.gpu

MINI_HD64 = synth.DrafterShape("mini-hd64", 512, 8, 2, 64, 1536, 5000)
MINI_HD128 = synth.DrafterShape("mini-hd128", 384, 4, 1, 128, 960, 3001)


def _codes(M, Kd, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = torch.randn(M, Kd, generator=g, device="cuda") * 0.05
    s = w.abs().amax(dim=1).clamp_min(1e-30) / 448.0
    q = (w / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return q, s.contiguous(), g


# split-K through scratch (few tiles), many tiles (persistent), token tiles
# of 128 and a ragged second one, ragged M and a K that is not a multiple of
# the 128-code stage
@pytest.mark.parametrize("M,N,Kd", [(2048, 7, 4096), (5120, 16, 2048), (1000, 33, 272), (640, 300, 1024),
                                    (151936 // 8, 11, 2048)])
def test_linear_fp8_matches_float64(M, N, Kd):
    q, s, g = _codes(M, Kd, M + N + Kd)
    x = torch.randn(N, Kd, generator=g, device="cuda").to(torch.bfloat16)
    y = binding.linear_fp8(q, s, x)
    torch.cuda.synchronize()
    w = oracle.dequant_rows(q.cpu().numpy(), s.cpu().numpy())
    ref = x.double().cpu().numpy() @ w.T
    err = np.abs(y.double().cpu().numpy() - ref).max()
    assert err <= 1e-4 * np.abs(ref).max(), (err, np.abs(ref).max())


def test_linear_fp8_every_finite_code_exactly():
    # every finite E4M3 code (subnormals, zeros, +-448 included) in every
    # position of a 16-byte chunk: with x = one-hot rows, y reads the decoded
    # weights back through the tensor cores exactly
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    M, Kd = 128, 256
    rng = np.random.default_rng(3)
    q = np.stack([np.roll(np.resize(codes, Kd), 17 * m) for m in range(M)]).astype(np.uint8)
    scale = rng.uniform(0.5, 2.0, size=M).astype(np.float32)
    w = torch.as_tensor(q, device="cuda")
    s = torch.as_tensor(scale, device="cuda")
    x = torch.eye(Kd, device="cuda", dtype=torch.bfloat16)[:64]
    y = binding.linear_fp8(w, s, x.contiguous())
    torch.cuda.synchronize()
    ref = oracle.dequant_rows(q, scale)[:, :64].T
    np.testing.assert_array_equal(y.cpu().numpy().astype(np.float64), ref.astype(np.float32).astype(np.float64))


def _fp8_setup(shape, seed, wl=None, device="cuda"):
    W = synth.make_weights(shape, seed, device=device)
    Wq, sc = synth.quantize_weights_fp8(W)
    Wn, Sn = synth.fp8_to_numpy(Wq, sc)
    return Wq, sc, oracle.dequant_weights(Wn, Sn)


def _full_check(inp, K, ref, d, st, lg, kc, vc):
    assert (st == binding.PE_REQ_OK).all()
    assert_logits_close(lg, ref["logits"])
    assert_drafts_match(d, ref)
    for b in range(inp.last_token.shape[0]):
        k_got, v_got = read_new_kv(inp, kc, vc, b, K)
        assert_kv_close(k_got, ref["k_new"][:, b], "k rows")
        assert_kv_close(v_got, ref["v_new"][:, b], "v rows")


@pytest.mark.parametrize("shape", [MINI_HD64, MINI_HD128], ids=lambda s: s.name)
@pytest.mark.parametrize("B,K", [(3, 5), (1, 1), (2, 16)])
def test_fp8_drafter_mini_parity(shape, B, K):
    dev = torch.device("cuda")
    wl = synth.Workload("mini-fp8", shape, B, K, (1, 300), (0.7, 0.7), 51)
    Wq, sc, Wd = _fp8_setup(shape, 51)
    inp = synth.make_step_inputs(wl, device=dev)
    ref = oracle_batch(shape, Wd, inp, K)
    dr = binding.Drafter(shape, Wq, max_batch=B, k_max=K, fp8_scales=sc)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.full((B, K, shape.vocab), float("nan"), device=dev)
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    _full_check(inp, K, ref, d.cpu().numpy(), st.cpu().numpy(), lg.cpu().numpy(), kc, vc)


def test_fp8_sequential_mini_parity():
    dev = torch.device("cuda")
    shape, B, K = MINI_HD128, 2, 4
    wl = synth.Workload("mini-fp8", shape, B, K, (10, 200), (0.7, 0.7), 52)
    Wq, sc, Wd = _fp8_setup(shape, 52)
    inp = synth.make_step_inputs(wl, device=dev)
    dr = binding.Drafter(shape, Wq, max_batch=B, k_max=K, fp8_scales=sc)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.empty(B, K, shape.vocab, device=dev)
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, K, logits=lg, sequential=True)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    dn = d.cpu().numpy()
    ref = oracle.draft_sequential(shape, Wd, inp.last_token.cpu().numpy(), inp.target_hidden.cpu().double().numpy(),
                                  inp.positions.cpu().numpy(), inp.seq_lens.cpu().numpy(),
                                  inp.page_table.cpu().numpy(), inp.k_cache.cpu().double().numpy(),
                                  inp.v_cache.cpu().double().numpy(), K, tokens=dn)
    _full_check(inp, K, ref, dn, st.cpu().numpy(), lg.cpu().numpy(), kc, vc)


@pytest.mark.parametrize("name", ["qwen-b1-k7", "qwen-b32-k11", "qwen-b128-k11", "gptoss-b64-k10"])
def test_fp8_full_size_sampled(name):
    wl = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    Wq, sc, Wd = _fp8_setup(wl.shape, wl.seed, device=dev)
    inp = synth.make_step_inputs(wl, device=dev)
    dr = binding.Drafter(wl.shape, Wq, max_batch=wl.B, k_max=wl.K, fp8_scales=sc)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    lg = torch.empty(wl.B, wl.K, wl.shape.vocab, device=dev)
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, wl.K, logits=lg)
    torch.cuda.synchronize()
    assert dr.device_errors() == 0
    assert (st.cpu().numpy() == 0).all()
    dn = d.cpu().numpy()
    seq = inp.seq_lens.cpu().numpy()
    for b in sorted({int(np.argmax(seq)), int(np.argmin(seq))}):
        ref = oracle_request(wl.shape, Wd, inp, b, wl.K)
        assert_logits_close(lg[b:b + 1].cpu().numpy(), ref["logits"])
        assert_drafts_match(dn[b:b + 1], ref)
        k_got, v_got = read_new_kv(inp, kc, vc, b, wl.K)
        assert_kv_close(k_got, ref["k_new"][:, 0], "k rows")
        assert_kv_close(v_got, ref["v_new"][:, 0], "v rows")
    # the step graph (no logits) gives the same drafts as the direct call
    g = torch.zeros(wl.B, wl.K + 1, dtype=torch.int32, device=dev)
    sg = dr.step_graph(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                       inp.num_pages, inp.k_cache.clone(), inp.v_cache.clone(), wl.K, g)
    sg.launch()
    torch.cuda.synchronize()
    assert np.array_equal(sg.out["drafts"].cpu().numpy(), dn)
    sg.close()
    dr.close()
