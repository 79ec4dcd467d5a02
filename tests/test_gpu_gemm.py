"""The tcgen05 GEMM engine alone (pe_linear) against a float64 matmul of the
same bf16 / fp32 inputs, over ragged shapes, split-K and several N tiles."""

import pytest
import torch

from speculative_drafting_pe_gb300 import binding

pytestmark = pytest.mark.gpu

SHAPES = [
    # M, N, Kd
    (128, 16, 64),        # one tile, one k-block
    (256, 3, 2048),       # split-K, ragged N
    (5120, 11, 2048),     # QKV-like at B=1
    (2048, 7, 4096),      # O-like, deep split-K
    (1000, 33, 520),      # ragged M, N and K tail
    (384, 300, 256),      # two N tiles
    (512, 1408, 128),     # six N tiles (B=128, K=11 rows)
    (151936, 7, 256),     # persistent: 1187 tiles over the resident CTAs (double-buffered accumulator)
    (20000, 300, 128),    # persistent with two N tiles per weight tile
]


@pytest.mark.parametrize("M,N,Kd", SHAPES)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_linear_matches_float64(lib, M, N, Kd, dtype):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + Kd)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    w = (torch.randn(M, Kd, generator=g, device="cuda") * 0.05).to(dt)
    x = torch.randn(N, Kd, generator=g, device="cuda").to(dt)
    y = binding.linear(w, x)
    torch.cuda.synchronize()
    if dtype == "fp32":
        # tensor cores read fp32 operands as tf32 (10-bit mantissa)
        ref = x.double() @ w.double().T
        tol = 4e-3
    else:
        ref = x.double() @ w.double().T
        tol = 1e-5
    err = (y.double() - ref).abs().max().item()
    scale = ref.abs().max().item()
    assert err <= tol * scale, (err, scale)


def test_linear_repeatable_and_tickets_reset(lib):
    g = torch.Generator(device="cuda").manual_seed(5)
    w = (torch.randn(2048, 4096, generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    x = torch.randn(5, 4096, generator=g, device="cuda").to(torch.bfloat16)
    y1 = binding.linear(w, x)
    y2 = binding.linear(w, x)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
