"""Host-side arithmetic of the measurement (CPU): the algorithmic bytes the
roofline divides by, the kernel-source hash that decides whether a profile's
DRAM counters still apply, and the benchmark's options."""

import dataclasses

import pytest

import bench
from speculative_drafting_pe_gb300 import synth


def _weight_params(s):
    """Parameter count of the drafter, matrix by matrix, without the token
    embedding (of which a step reads only the gathered rows)."""
    H, F, V, hd = s.hidden, s.ffn, s.vocab, s.head_dim
    qkv = (s.n_q_heads + 2 * s.n_kv_heads) * hd
    fc = H * 3 * H
    layer0 = qkv * 2 * H + H * s.n_q_heads * hd + 2 * F * H + F * H
    layer = qkv * H + H * s.n_q_heads * hd + 2 * F * H + F * H
    lm = V * H
    gains = 2 * H + 4 * 2 * H + H            # layer-0 input gains, two per layer, final
    return fc + layer0 + 3 * layer + lm + gains + H   # + the shared hidden vector h_shared


@pytest.mark.parametrize("shape,total_m", [(synth.QWEN3_CODER_30B_A3B, 560.7), (synth.GPT_OSS_20B, 1023.5)])
def test_weight_parameters_match_the_shape_totals(shape, total_m):
    # totals computed from the shapes: 560.7 M (FC 12.6 M, layer 0 67.1 M,
    # layers 1-3 56.6 M each, LM head 311.2 M) and 1023.5 M
    n = _weight_params(shape)
    assert abs(n / 1e6 - total_m) < 0.1, n
    assert shape.param_count() - shape.vocab * shape.hidden == pytest.approx(n, rel=1e-4)


def test_step_bytes_is_weights_plus_kv_read_and_write():
    wl = synth.WORKLOADS["qwen-b1-k7"]
    s = wl.shape
    seq = [2048]
    weights = (_weight_params(s) + wl.B * s.hidden) * 2          # + the B gathered embedding rows
    per_entry_per_layer = s.n_kv_heads * s.head_dim * 2 * 2      # K and V, bf16
    kv = (2048 + wl.K) * per_entry_per_layer * 4 + wl.K * per_entry_per_layer * 4
    assert bench.step_bytes(wl, seq) == pytest.approx(weights + kv, rel=2e-4)
    assert bench.step_bytes(wl, seq) / 1e9 == pytest.approx(1.138, abs=0.002)


def test_lm_head_work_per_launch():
    wl = synth.WORKLOADS["qwen-b1-k7"]
    s = wl.shape
    R = wl.B * wl.K
    b, f = bench.algorithmic_work("lm_head", wl, [2048])
    assert b == s.vocab * s.hidden * 2 + R * s.hidden * 2 + R * 8     # weights, B operand, argmax records
    assert f == 2 * R * s.vocab * s.hidden


def test_attention_work_counts_every_cache_entry_once_per_layer():
    wl = synth.WORKLOADS["qwen-b4-k11"]
    s = wl.shape
    seq = [512, 1000, 4096, 8000]
    b, _ = bench.algorithmic_work("attention", wl, seq)
    kv = sum(S + wl.K for S in seq) * s.n_kv_heads * s.head_dim * 2 * 2
    q_and_out = 2 * wl.B * wl.K * s.n_q_heads * s.head_dim * 2
    assert b == kv + q_and_out


def test_source_hash_ignores_comments_and_whitespace(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k(int* x) { x[0] = 1; }\n")
    h0 = bench.kernel_source_hash(str(tmp_path))
    src.write_text("// a kernel\n__global__ void k(int* x) {\n    /* store */ x[0] = 1;   // one\n}\n")
    assert bench.kernel_source_hash(str(tmp_path)) == h0
    src.write_text("__global__ void k(int* x) { x[0] = 2; }\n")
    assert bench.kernel_source_hash(str(tmp_path)) != h0


def test_max_prefix_option_caps_both_ends():
    a = bench.parse_args(["--workload", "qwen-b128-k11", "--max-prefix", "512"])
    assert a.max_prefix == 512
    assert bench.parse_args([]).max_prefix == 0
    wl = synth.WORKLOADS["qwen-b128-k11"]
    capped = dataclasses.replace(wl, prefix=(min(wl.prefix[0], 512), min(wl.prefix[1], 512)))
    assert capped.prefix == (512, 512) and capped.B == wl.B and capped.K == wl.K


def test_fp8_step_bytes_count_one_byte_per_gemm_weight_plus_row_scales():
    wl = synth.WORKLOADS["qwen-b1-k7"]
    s = wl.shape
    seq = [2048]
    full = bench.step_bytes(wl, seq)
    fp8 = bench.step_bytes(wl, seq, fp8=True)
    mats = bench.gemm_weight_shapes(s)
    assert len(mats) == 2 + 5 * 4
    params = sum(r * c for r, c in mats)
    rows = sum(r for r, _ in mats)
    assert full - fp8 == params * 2 - (params + 4 * rows)
    # the GEMM matrices are all weights but the embedding and the small vectors
    assert params == pytest.approx(s.param_count() - s.vocab * s.hidden, rel=1e-3)
    b, _ = bench.algorithmic_work("lm_head", wl, seq, fp8=True)
    R = wl.B * wl.K
    assert b == s.vocab * s.hidden + 4 * s.vocab + R * s.hidden * 2 + R * 8
