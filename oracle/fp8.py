"""FP8 (E4M3) drafter weights, decoded plainly.

TEST INFRASTRUCTURE ONLY: see the package docstring.

The pages' benchmarks run the target model in FP8 ([zh] "在 Amazon SageMaker
AI 上使用 P-EAGLE 并行化推测解码", section "基准测试"). For the drafter this
oracle reads "FP8 drafter weights" as (reading F1, also in the design notes):
every GEMM weight matrix (FC, QKV, O, gate, up, down, LM head) is stored as
E4M3 codes q[m, k] with one float32 scale per output row m, and stands for
W[m, k] = decode(q[m, k]) * scale[m]; embeddings, placeholders, norm gains,
activations and the KV cache keep their own precision.

E4M3 ("fn" variant, no infinities): bit 7 sign, bits 6..3 exponent with bias
7, bits 2..0 mantissa. Exponent field 0 encodes subnormals m/8 * 2^-6; the
code S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448.
"""

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(q):
    """Float64 values of E4M3 codes (uint8 array of any shape)."""
    q = np.asarray(q, dtype=np.uint8).astype(np.int64)
    sign = (q >> 7) & 1
    exp = (q >> 3) & 0xF
    man = q & 0x7
    normal = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    subnormal = (man / 8.0) * 2.0 ** -6
    mag = np.where(exp == 0, subnormal, normal)
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def dequant_rows(q, scale):
    """W[m, k] = decode(q[m, k]) * scale[m] in float64 (reading F1)."""
    return e4m3_decode(q) * np.asarray(scale, dtype=np.float64).reshape(-1, 1)


GEMM_MATRICES = ("fc", "lm_head")
LAYER_GEMM_MATRICES = ("w_qkv", "w_o", "w_gate", "w_up", "w_down")


def dequant_weights(Wq, scales):
    """A float64 weight dict for draft_pass / draft_sequential from FP8 codes.

    Wq: the weight dict with every GEMM matrix replaced by its uint8 codes;
    scales: {"fc": [H], "lm_head": [V], "layers": [{"w_qkv": ..., ...}]}.
    The other entries are passed through unchanged.
    """
    out = {k: v for k, v in Wq.items() if k != "layers"}
    for k in GEMM_MATRICES:
        out[k] = dequant_rows(Wq[k], scales[k])
    out["layers"] = []
    for L, S in zip(Wq["layers"], scales["layers"]):
        d = dict(L)
        for k in LAYER_GEMM_MATRICES:
            d[k] = dequant_rows(L[k], S[k])
        out["layers"].append(d)
    return out
