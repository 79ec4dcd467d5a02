"""pe_linear_noalloc, the GEMM entry point for callers that cannot allocate
device memory, checked against pe_linear on the same inputs, two calls in a
row. Collected last so that a failure here comes after every other test."""

import ctypes

import pytest
import torch

from speculative_drafting_pe_gb300 import binding

pytestmark = pytest.mark.gpu

SHAPES = [(2048, 7, 4096), (5120, 11, 2048), (1000, 33, 520), (384, 300, 256)]
WS_LIMIT_FLOATS = 2 << 20          # the entry point's built-in split-K scratch
TICKET_LIMIT = 4096


def _scratch_need(dtype_code, M, N, Kd):
    lib = binding.load()
    wsf, nt = ctypes.c_int64(0), ctypes.c_int32(0)
    assert lib.pe_linear_scratch(dtype_code, M, N, Kd, ctypes.byref(wsf), ctypes.byref(nt)) == 0
    return wsf.value, nt.value


def _inputs(M, N, Kd, dt, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = (torch.randn(M, Kd, generator=g, device="cuda") * 0.05).to(dt)
    x = torch.randn(N, Kd, generator=g, device="cuda").to(dt)
    return w, x


def _check_two_calls(w, x, dtype):
    ref = binding.linear(w, x)
    torch.cuda.synchronize()
    tol = 4e-3 if dtype == "fp32" else 1e-5       # the GEMM tests' tolerances
    scale = ref.double().abs().max().item()
    y = torch.empty(x.shape[0], w.shape[0], dtype=torch.float32, device="cuda")
    for _ in range(2):
        y.fill_(float("nan"))
        binding.linear_noalloc(w, x, y=y)
        torch.cuda.synchronize()
        err = (y.double() - ref.double()).abs().max().item()
        assert err <= tol * scale, (err, scale)


@pytest.mark.parametrize("M,N,Kd", SHAPES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noalloc_matches_linear_on_two_calls_in_a_row(M, N, Kd, dtype):
    binding.load()
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    w, x = _inputs(M, N, Kd, dt, M + 3 * N + 7 * Kd)
    _check_two_calls(w, x, dtype)


def test_noalloc_many_tiles_without_split_k():
    # An LM-head-sized GEMM has more tiles than the ticket array holds but
    # needs no split-K (and so no tickets): it must be accepted.
    M, N, Kd = 151936, 1408, 2048
    ws, tiles = _scratch_need(binding.PE_DTYPE_BF16, M, N, Kd)
    assert ws == 0 and tiles > TICKET_LIMIT
    w, x = _inputs(M, N, Kd, torch.bfloat16, 5)
    _check_two_calls(w, x, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noalloc_runs_while_another_stream_captures_in_global_mode(dtype):
    # While a stream of this process captures a CUDA graph in global mode,
    # cudaMalloc anywhere in the process fails; the entry point must still
    # run (on a stream that is not capturing) and give pe_linear's result.
    binding.load()
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    w, x = _inputs(2048, 9, 4096, dt, 11)
    ref = binding.linear(w, x)
    y = torch.empty(9, 2048, dtype=torch.float32, device="cuda")
    binding.linear_noalloc(w, x, y=y)          # first call on the device: address lookup, kernel load
    torch.cuda.synchronize()
    run = torch.cuda.Stream()
    cap = torch.cuda.Stream()
    z = torch.zeros(16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    y.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        graph.capture_begin(capture_error_mode="global")
        z.add_(1.0)
        try:
            binding.linear_noalloc(w, x, y=y, stream=run)
        finally:
            graph.capture_end()
    run.synchronize()
    torch.cuda.synchronize()
    tol = 4e-3 if dtype == "fp32" else 1e-5
    assert (y.double() - ref.double()).abs().max().item() <= tol * ref.double().abs().max().item()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = binding.load()
    M, N, Kd = 4096, 256, 16384
    ws, tiles = _scratch_need(binding.PE_DTYPE_BF16, M, N, Kd)
    assert ws > WS_LIMIT_FLOATS, (ws, tiles)
    # buffers of the full size, so that even a missed rejection would compute
    # in bounds
    w = torch.zeros(M, Kd, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(N, Kd, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(N, M, dtype=torch.float32, device="cuda")
    rc = lib.pe_linear_noalloc(binding.PE_DTYPE_BF16, M, N, Kd, binding._p(w), binding._p(x), binding._p(y), None)
    assert rc == -1
    assert b"maximum" in lib.pe_last_error()
