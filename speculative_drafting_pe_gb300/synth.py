"""Seeded synthetic inputs for the P-EAGLE drafter and verifier.

This module holds drafter shapes, workload definitions and random draws only;
it computes no step of the method. Tests and the benchmark hand the same
tensors to the CUDA path and to the CPU oracle.

Value recipe (random-init drafter, synthetic step inputs):
  * weight matrices and embeddings ~ N(0, 0.02); norm gains ~ 1 + N(0, 0.02);
    h_shared ~ N(0, 1); target hidden states ~ N(0, 1);
  * committed drafter-cache entries ~ N(0, 1);
  * token ids uniform in [0, V); prefix lengths uniform in the workload's
    range; the RoPE position of row 0 is the prefix length plus U[0, 16);
  * page tables: a random permutation of one shared page pool, each request
    owning enough 16-token pages for its prefix plus two steps of K rows;
  * planted agreement: target token g[b, j] equals the draft with
    probability alpha_b, independently per position, else another token.

Small metadata (lengths, token ids, page tables, masks) comes from numpy's
PCG64; float tensors come from a torch generator on the requested device.
"""

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class DrafterShape:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    dtype: str = "bf16"          # "bf16" or "fp32" (weights, activations, KV cache)
    n_layers: int = 4
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    page_size: int = 16

    @property
    def qkv_rows(self):
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def param_count(self):
        H, F, V = self.hidden, self.ffn, self.vocab
        qd = self.n_q_heads * self.head_dim
        per_layer = self.qkv_rows * H + H * qd + 3 * F * H + 2 * H
        layer0_extra = self.qkv_rows * H + H   # 2H-wide QKV input, two input gains
        return (3 * H * H + 2 * V * H + 3 * H
                + self.n_layers * per_layer + layer0_extra)


TINY_FP32 = DrafterShape("tiny-fp32", 256, 4, 2, 64, 512, 4096, dtype="fp32")
QWEN3_CODER_30B_A3B = DrafterShape("qwen3-coder-30b-a3b-shaped", 2048, 32, 4, 128, 6144, 151936)
GPT_OSS_20B = DrafterShape("gpt-oss-20b-shaped", 2880, 64, 8, 64, 8640, 201088)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: DrafterShape
    B: int
    K: int
    prefix: tuple          # (lo, hi) inclusive
    alpha: tuple           # (lo, hi) per-request uniform; lo == hi means fixed
    seed: int


def _workloads():
    w = {}
    w["tiny-fp32-b1-k3"] = Workload("tiny-fp32-b1-k3", TINY_FP32, 1, 3, (64, 64), (0.7, 0.7), 0)
    for K in (3, 7, 11):
        n = f"qwen-b1-k{K}"
        w[n] = Workload(n, QWEN3_CODER_30B_A3B, 1, K, (2048, 2048), (0.7, 0.7), 0)
    for B in (4, 8, 32, 128):
        for K in (3, 7, 11):
            n = f"qwen-b{B}-k{K}"
            w[n] = Workload(n, QWEN3_CODER_30B_A3B, B, K, (512, 8192), (0.5, 0.8), 1)
    w["gptoss-b64-k10"] = Workload("gptoss-b64-k10", GPT_OSS_20B, 64, 10, (1024, 4096), (0.6, 0.6), 2)
    return w


WORKLOADS = _workloads()

# Verify + metadata-rebuild stress: B=128, K=11, vocab 151936, ragged lengths.
VERIFY_STRESS = dict(B=128, K=11, vocab=151936, seq_lens=(512, 8192), alphas=(0.3, 0.55, 0.8), seed=3)


def _np_rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _torch_gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_weights(shape, seed, device="cpu"):
    """Random-init drafter weights (dict of tensors, [out, in] matrices)."""
    dt = shape.torch_dtype
    g = _torch_gen(seed, device)
    H, F, V = shape.hidden, shape.ffn, shape.vocab
    qd = shape.n_q_heads * shape.head_dim

    def normal(*size, std=0.02, mean=0.0):
        t = torch.randn(*size, generator=g, device=device, dtype=torch.float32)
        t.mul_(std).add_(mean)
        return t.to(dt)

    W = {
        "fc": normal(H, 3 * H),
        "embed": normal(V, H),
        "emb_mask": normal(H),
        "h_shared": normal(H, std=1.0),
        "final_norm": normal(H, mean=1.0),
        "lm_head": normal(V, H),
        "layers": [],
    }
    for layer in range(shape.n_layers):
        first = layer == 0
        W["layers"].append({
            "norm_e": normal(H, mean=1.0) if first else None,
            "norm_h": normal(H, mean=1.0) if first else None,
            "attn_norm": None if first else normal(H, mean=1.0),
            "w_qkv": normal(shape.qkv_rows, 2 * H if first else H),
            "w_o": normal(H, qd),
            "mlp_norm": normal(H, mean=1.0),
            "w_gate": normal(F, H),
            "w_up": normal(F, H),
            "w_down": normal(H, F),
        })
    return W


@dataclass
class StepInputs:
    last_token: torch.Tensor      # [B] int32
    target_hidden: torch.Tensor   # [B, 3H]
    positions: torch.Tensor       # [B] int32 (Q_b: RoPE position of row 0)
    seq_lens: torch.Tensor        # [B] int32 (S_b: committed drafter-cache entries)
    page_table: torch.Tensor      # [B, max_pages] int32, -1 where unused
    num_pages: int
    k_cache: torch.Tensor         # [L, num_pages, nkv, P, hd]
    v_cache: torch.Tensor
    alpha: np.ndarray             # [B] planted per-position agreement rate
    K: int


def page_pool(seq_lens, K, page_size, rng, spare=1):
    """Per-request page tables over one randomly permuted pool.

    Each request owns ceil((S_b + 2K) / P) pages (this step's rows and the
    next step's). Returns (page_table [B, max_pages] int32, num_pages).
    """
    need = [int(math.ceil((int(s) + 2 * K) / page_size)) for s in seq_lens]
    max_pages = max(need)
    num_pages = sum(need) + spare
    perm = rng.permutation(num_pages)
    pt = np.full((len(seq_lens), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[off:off + n]
        off += n
    return pt, num_pages


def make_step_inputs(wl, device="cpu", seed=None, B=None, K=None):
    """Seeded step inputs for a workload (optionally overriding B or K)."""
    shape = wl.shape
    B = wl.B if B is None else B
    K = wl.K if K is None else K
    seed = wl.seed if seed is None else seed
    rng = _np_rng(seed + 101)
    lo, hi = wl.prefix
    seq_lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    positions = (seq_lens + rng.integers(0, 16, size=B)).astype(np.int32)
    last_token = rng.integers(0, shape.vocab, size=B).astype(np.int32)
    a_lo, a_hi = wl.alpha
    alpha = np.full(B, a_lo) if a_lo == a_hi else rng.uniform(a_lo, a_hi, size=B)
    page_table, num_pages = page_pool(seq_lens, K, shape.page_size, rng)

    g = _torch_gen(seed + 202, device)
    dt = shape.torch_dtype
    th = torch.randn(B, 3 * shape.hidden, generator=g, device=device, dtype=torch.float32).to(dt)
    cache_shape = (shape.n_layers, num_pages, shape.n_kv_heads, shape.page_size, shape.head_dim)
    k_cache = torch.empty(cache_shape, dtype=dt, device=device)
    v_cache = torch.empty(cache_shape, dtype=dt, device=device)
    for layer in range(shape.n_layers):
        for c in (k_cache, v_cache):
            c[layer] = torch.randn(cache_shape[1:], generator=g, device=device,
                                   dtype=torch.float32).to(dt)

    def it(x):
        return torch.as_tensor(x, dtype=torch.int32).to(device)

    return StepInputs(it(last_token), th, it(positions), it(seq_lens), it(page_table),
                      num_pages, k_cache, v_cache, alpha, K)


def make_refeed_inputs(wl, n_max, device="cpu", seed=None):
    """Re-fed real rows for a workload: n_real [B] uniform in 1..n_max,
    tokens [B, n_max] uniform ids and target hidden states [B, n_max, 3H]
    ~ N(0, 1) (entries past n_real[b] are drawn too and left unused).
    Pair with make_step_inputs(wl, K=wl.K + n_max) so that the page tables
    cover every entry the pass writes."""
    shape = wl.shape
    seed = wl.seed if seed is None else seed
    rng = _np_rng(seed + 505)
    n_real = rng.integers(1, n_max + 1, size=wl.B).astype(np.int32)
    tokens = rng.integers(0, shape.vocab, size=(wl.B, n_max)).astype(np.int32)
    g = _torch_gen(seed + 606, device)
    th = torch.randn(wl.B, n_max, 3 * shape.hidden, generator=g, device=device, dtype=torch.float32)
    return (torch.as_tensor(tokens).to(device), torch.as_tensor(n_real).to(device), th.to(shape.torch_dtype))


def plant_targets(drafts, alpha, vocab, seed):
    """Target argmax tokens g [B, K+1] that agree with `drafts` [B, K]
    independently per position with probability alpha[b]; g[:, K] uniform."""
    rng = _np_rng(seed + 303)
    d = np.asarray(drafts, dtype=np.int64)
    B, K = d.shape
    alpha = np.broadcast_to(np.asarray(alpha, dtype=np.float64), (B,))
    agree = rng.random((B, K)) < alpha[:, None]
    shift = 1 + rng.integers(0, vocab - 1, size=(B, K))
    g = np.empty((B, K + 1), dtype=np.int64)
    g[:, :K] = np.where(agree, d, (d + shift) % vocab)
    g[:, K] = rng.integers(0, vocab, size=B)
    return g.astype(np.int32)


def make_verify_inputs(B, K, vocab, seq_range, alpha, seed, page_size=16):
    """Uniform drafts, planted targets, ragged lengths and page tables for the
    verify/rebuild stress case. Returns a dict of numpy int32 arrays."""
    rng = _np_rng(seed + 404)
    drafts = rng.integers(0, vocab, size=(B, K)).astype(np.int32)
    targets = plant_targets(drafts, np.full(B, alpha), vocab, seed + int(alpha * 1000))
    lo, hi = seq_range
    seq_lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    positions = (seq_lens + rng.integers(0, 16, size=B)).astype(np.int32)
    page_table, num_pages = page_pool(seq_lens, K, page_size, rng)
    return dict(drafts=drafts, targets=targets, seq_lens=seq_lens, positions=positions,
                page_table=page_table, num_pages=num_pages)


FP8_LAYER_MATRICES = ("w_qkv", "w_o", "w_gate", "w_up", "w_down")


def quantize_weights_fp8(W):
    """FP8 drafter weights from a random-init weight dict: every GEMM matrix
    (FC, QKV, O, gate, up, down, LM head) becomes E4M3 codes (uint8, same
    [out, in] layout, torch's round-to-nearest-even float8_e4m3fn conversion)
    with one float32 scale per output row, max|row| / 448; the other entries
    are kept. Returns (Wq, scales) with the same nesting as W."""
    def q(t):
        t32 = t.to(torch.float32)
        s = t32.abs().amax(dim=1).clamp_min(1e-30) / 448.0
        codes = (t32 / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        return codes.contiguous(), s.contiguous()

    Wq = {k: v for k, v in W.items() if k != "layers"}
    scales = {"layers": []}
    for k in ("fc", "lm_head"):
        Wq[k], scales[k] = q(W[k])
    Wq["layers"] = []
    for L in W["layers"]:
        Lq, Ls = dict(L), {}
        for k in FP8_LAYER_MATRICES:
            Lq[k], Ls[k] = q(L[k])
        Wq["layers"].append(Lq)
        scales["layers"].append(Ls)
    return Wq, scales


def fp8_to_numpy(Wq, scales):
    """Host copies for the oracle: uint8 codes and float32 scales as numpy,
    other tensors as float32 (exact for bf16)."""
    def cv(t):
        if t is None:
            return None
        t = t.detach().to("cpu")
        return t.numpy() if t.dtype == torch.uint8 else t.to(torch.float32).numpy()
    Wn = {k: cv(v) for k, v in Wq.items() if k != "layers"}
    Wn["layers"] = [{k: cv(v) for k, v in L.items()} for L in Wq["layers"]]
    Sn = {k: cv(v) for k, v in scales.items() if k != "layers"}
    Sn["layers"] = [{k: cv(v) for k, v in L.items()} for L in scales["layers"]]
    return Wn, Sn


def weights_to_numpy(W):
    """Host float32 copies of a weight dict for the oracle (exact for bf16 and
    fp32 values; the oracle widens to float64 as it computes)."""
    def cv(t):
        return None if t is None else t.detach().to("cpu", torch.float32).numpy()
    out = {k: cv(v) for k, v in W.items() if k != "layers"}
    out["layers"] = [{k: cv(v) for k, v in L.items()} for L in W["layers"]]
    return out
