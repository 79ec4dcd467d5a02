"""pe_linear_noalloc, the GEMM entry point for callers that cannot allocate
device memory, checked against pe_linear on the same inputs, two calls in a
row. Collected last so that a failure here comes after every other test."""

import pytest
import torch

from speculative_drafting_pe_gb300 import binding

pytestmark = pytest.mark.gpu

SHAPES = [(2048, 7, 4096), (5120, 11, 2048), (1000, 33, 520), (384, 300, 256)]


@pytest.mark.parametrize("M,N,Kd", SHAPES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noalloc_matches_linear_on_two_calls_in_a_row(M, N, Kd, dtype):
    binding.load()
    g = torch.Generator(device="cuda").manual_seed(M + 3 * N + 7 * Kd)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    w = (torch.randn(M, Kd, generator=g, device="cuda") * 0.05).to(dt)
    x = torch.randn(N, Kd, generator=g, device="cuda").to(dt)
    ref = binding.linear(w, x)
    torch.cuda.synchronize()
    tol = 4e-3 if dtype == "fp32" else 1e-5       # the GEMM tests' tolerances
    scale = ref.double().abs().max().item()
    y = torch.empty(N, M, dtype=torch.float32, device="cuda")
    for _ in range(2):
        y.fill_(float("nan"))
        binding.linear_noalloc(w, x, y=y)
        torch.cuda.synchronize()
        err = (y.double() - ref.double()).abs().max().item()
        assert err <= tol * scale, (err, scale)


def test_noalloc_allocates_nothing_after_first_call():
    binding.load()
    g = torch.Generator(device="cuda").manual_seed(11)
    w = (torch.randn(2048, 4096, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    x = torch.randn(9, 4096, generator=g, device="cuda").to(torch.bfloat16)
    y = torch.empty(9, 2048, dtype=torch.float32, device="cuda")
    binding.linear_noalloc(w, x, y=y)          # first call on the device: address lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        binding.linear_noalloc(w, x, y=y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = binding.load()
    w = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(16, 16, dtype=torch.float32, device="cuda")
    # a shape with many split-K tiles: M = 4096 rows, N = 256 tokens, deep K
    rc = lib.pe_linear_noalloc(0, 4096, 256, 16384, binding._p(w), binding._p(x), binding._p(y), None)
    assert rc == -1
    assert b"maximum" in lib.pe_last_error()
