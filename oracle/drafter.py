"""P-EAGLE parallel draft pass in float64, one plain step at a time.

TEST INFRASTRUCTURE ONLY: see the package docstring. Nothing in the product
path imports this module.

What the method computes comes from these pages (cited by title and section):

[zh] "在 Amazon SageMaker AI 上使用 P-EAGLE 并行化推测解码" (the Chinese
     translation of the AWS post), section "解决方案概述" (Solution overview):
     - "P-EAGLE 如何打破这个链": two learned parameters stand in for the
       unknown inputs of future positions: a mask-token embedding (emb_mask)
       and one hidden vector shared by every multi-token position (h_shared).
     - "逐步草稿过程" Step 1: hidden states from target layers 2, L/2 and L-1
       are concatenated to 3d.  Step 2: position 1 uses the real embedding of
       the token just produced together with the captured target hidden state;
       positions 2..K use emb_mask together with h_shared; all K positions go
       through the drafter's transformer layers (4 in practice) and then the
       LM head, which yields K draft tokens at once.
[ko] "Parallelize speculative decoding with P-EAGLE on Amazon SageMaker AI"
     (Korean summary), section 8: emb_mask and h_shared replace the unknown
     inputs of future positions.
[ja] "Amazon SageMaker AIにおけるP-EAGLEによる推論高速化", section
     "アーキテクチャの深化と今後の展望": the drafter is a light 4-layer model.

The pages leave the layer internals open. The readings taken here (each one
is also listed in the design notes):
 R1  FC fusion: h = W_fc [h_lo; h_mid; h_hi] maps 3H -> H; it is applied to
     the target hidden state of position 1 only.
 R2  Layer 0 attends over the 2H-wide concat
     [RMSNorm_e(embedding); RMSNorm_h(hidden)] and its residual stream starts
     at the hidden half (h for position 1, h_shared for the others).
     Layers 1..3 are standard pre-norm GQA + SwiGLU blocks.
 R3  RMSNorm x / sqrt(mean(x^2) + eps) * gain; no biases, no QK-norm; a final
     RMSNorm before an LM head that is not tied to the embedding.
 R4  RoPE in rotate-half form: pairs (i, i + hd/2),
     inv_freq_i = theta^(-2 i / hd), angle = position * inv_freq_i.
 R5  Attention: scale 1/sqrt(hd); query head h reads kv head
     floor(h * nkv / nq); softmax in full precision.
 R6  Row j of request b (j = 0 is position 1 above) sits at RoPE position
     Q_b + j and at drafter-cache entry S_b + j; it attends to cache entries
     0 .. S_b + j (the S_b committed entries plus new rows 0..j).
 R7  argmax ties go to the lowest vocabulary index.

Cache layout (a data layout shared with the CUDA path, not code):
k_cache / v_cache are [n_layers, num_pages, n_kv_heads, page_size, head_dim];
cache entry e of request b lives in page page_table[b, e // page_size] at
slot e % page_size.
"""

import numpy as np


def rms_norm(x, gain, eps):
    """RMSNorm over the last axis (reading R3)."""
    x = np.asarray(x, dtype=np.float64)
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + eps) * np.asarray(gain, dtype=np.float64)


def silu(x):
    """SiLU(x) = x * sigmoid(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def rope_neox(x, pos, theta):
    """Rotate-half RoPE (reading R4).

    x:   [..., hd] float64.
    pos: integer positions broadcastable to x.shape[:-1].
    """
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = float(theta) ** (-2.0 * i / hd)
    angle = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c = np.cos(angle)
    s = np.sin(angle)
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def linear(x, w, row_block=16384):
    """y = x @ W^T for a weight W stored [out, in].

    Every output element is one full dot product in float64. W is converted
    to float64 a block of rows at a time only to bound host memory.
    """
    x = np.asarray(x, dtype=np.float64)
    n_out = w.shape[0]
    y = np.empty(x.shape[:-1] + (n_out,), dtype=np.float64)
    for o0 in range(0, n_out, row_block):
        wb = np.asarray(w[o0:o0 + row_block], dtype=np.float64)
        y[..., o0:o0 + row_block] = x @ wb.T
    return y


def gather_prefix_kv(cache_l, page_table_b, n_entries, page_size):
    """Cache entries 0..n_entries-1 of one request -> [n_entries, nkv, hd]."""
    e = np.arange(n_entries)
    pages = np.asarray(page_table_b)[e // page_size]
    slots = e % page_size
    return np.asarray(cache_l[pages, :, slots, :], dtype=np.float64)


def causal_paged_attention(q, k_all, v_all, n_prefix):
    """Attention of the K new rows of one request (reading R5, R6).

    q:      [K, nq, hd]   rotated queries of the new rows.
    k_all:  [n_prefix + K, nkv, hd]  prefix entries followed by the new rows.
    v_all:  same shape as k_all.
    Row j sees entries 0 .. n_prefix + j.
    """
    n_rows, nq, hd = q.shape
    nkv = k_all.shape[1]
    out = np.zeros((n_rows, nq, hd), dtype=np.float64)
    scale = 1.0 / np.sqrt(hd)
    for h in range(nq):
        kvh = (h * nkv) // nq
        for j in range(n_rows):
            n_vis = n_prefix + j + 1
            scores = (k_all[:n_vis, kvh, :] @ q[j, h, :]) * scale
            p = np.exp(scores - scores.max())
            p = p / p.sum()
            out[j, h, :] = p @ v_all[:n_vis, kvh, :]
    return out


def build_rows(cfg, W, last_token, h, K):
    """Build the K input rows of every request (pages' Step 2; reading R2).

    Row 0: real embedding of the last accepted token + fused target hidden h.
    Rows 1..K-1: emb_mask + h_shared.
    Returns (u [B, K, 2H], resid [B, K, H]).
    """
    B = len(last_token)
    H = cfg.hidden
    emb = np.empty((B, K, H), dtype=np.float64)
    hid = np.empty((B, K, H), dtype=np.float64)
    emb[:, 0, :] = np.asarray(W["embed"], dtype=np.float64)[np.asarray(last_token)]
    hid[:, 0, :] = h
    if K > 1:
        emb[:, 1:, :] = np.asarray(W["emb_mask"], dtype=np.float64)
        hid[:, 1:, :] = np.asarray(W["h_shared"], dtype=np.float64)
    L0 = W["layers"][0]
    u = np.concatenate(
        [rms_norm(emb, L0["norm_e"], cfg.rms_eps), rms_norm(hid, L0["norm_h"], cfg.rms_eps)],
        axis=-1,
    )
    return u, hid.copy()


def argmax_lowest(logits):
    """argmax over the last axis; ties go to the lowest index (reading R7)."""
    return np.argmax(logits, axis=-1).astype(np.int64)


def top2_gap(logits):
    """Difference between the largest and second-largest logit per row."""
    part = np.partition(logits, -2, axis=-1)
    return part[..., -1] - part[..., -2]


def run_layers(cfg, W, u, resid, positions, seq_lens, page_table, k_cache, v_cache, perturb_rows=None):
    """The drafter's 4 layers over the new rows of every request (R2..R6).

    u [B, K, 2H] layer-0 input rows, resid [B, K, H] the residual stream they
    start from; row j of request b is at RoPE position positions[b] + j and
    cache entry seq_lens[b] + j, and attends to entries 0 .. seq_lens[b] + j
    (the committed ones read from the cache, then the new rows themselves).
    Returns (resid [B, K, H] after the last layer, k_new, v_new
    [L, B, K, nkv, hd]: the rows the pass writes to the cache).
    """
    B, K = u.shape[:2]
    nq, nkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    eps = cfg.rms_eps
    P = cfg.page_size
    positions = np.asarray(positions, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    if perturb_rows is not None:
        u = perturb_rows(u)

    pos = positions[:, None] + np.arange(K)[None, :]           # R6
    k_new = np.empty((cfg.n_layers, B, K, nkv, hd), dtype=np.float64)
    v_new = np.empty_like(k_new)

    for layer, Lw in enumerate(W["layers"]):
        x = u if layer == 0 else rms_norm(resid, Lw["attn_norm"], eps)
        qkv = linear(x, Lw["w_qkv"])
        q = qkv[..., : nq * hd].reshape(B, K, nq, hd)
        k = qkv[..., nq * hd: (nq + nkv) * hd].reshape(B, K, nkv, hd)
        v = qkv[..., (nq + nkv) * hd:].reshape(B, K, nkv, hd)
        q = rope_neox(q, pos[:, :, None], cfg.rope_theta)
        k = rope_neox(k, pos[:, :, None], cfg.rope_theta)
        k_new[layer] = k
        v_new[layer] = v

        attn = np.empty((B, K, nq, hd), dtype=np.float64)
        for b in range(B):
            kp = gather_prefix_kv(k_cache[layer], page_table[b], seq_lens[b], P)
            vp = gather_prefix_kv(v_cache[layer], page_table[b], seq_lens[b], P)
            k_all = np.concatenate([kp, k[b]], axis=0)
            v_all = np.concatenate([vp, v[b]], axis=0)
            attn[b] = causal_paged_attention(q[b], k_all, v_all, int(seq_lens[b]))

        resid = resid + linear(attn.reshape(B, K, nq * hd), Lw["w_o"])
        x = rms_norm(resid, Lw["mlp_norm"], eps)
        gate = linear(x, Lw["w_gate"])
        up = linear(x, Lw["w_up"])
        resid = resid + linear(silu(gate) * up, Lw["w_down"])
    return resid, k_new, v_new


def lm_head_logits(cfg, W, resid):
    """Final RMSNorm and LM head: fp64 logits of every row (pages' Step 2)."""
    return linear(rms_norm(resid, W["final_norm"], cfg.rms_eps), W["lm_head"])


def draft_pass(cfg, W, last_token, target_hidden, positions, seq_lens,
               page_table, k_cache, v_cache, K, perturb_rows=None):
    """One parallel draft pass for a batch of B requests.

    cfg: object with hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn,
         vocab, rms_eps, rope_theta, page_size.
    W:   dict of arrays: fc [H,3H], embed [V,H], emb_mask [H], h_shared [H],
         final_norm [H], lm_head [V,H], layers: list of dicts with norm_e,
         norm_h (layer 0), attn_norm (layers 1..), w_qkv, w_o, mlp_norm,
         w_gate, w_up, w_down (all [out, in]).
    last_token [B]; target_hidden [B, 3H]; positions Q [B]; seq_lens S [B];
    page_table [B, max_pages]; k_cache/v_cache [L, pages, nkv, P, hd] (read).
    perturb_rows: optional test hook applied to the [B, K, 2H] layer-0 input.

    Returns a dict: logits [B,K,V], drafts [B,K], gap [B,K] (top-2 logit gap),
    k_new / v_new [L, B, K, nkv, hd] (the rows the pass writes to the cache at
    entries S_b + j), h [B, H] (FC output).
    """
    # Step 1 input: the 3d concat of target hidden states, fused to H (R1).
    h = linear(target_hidden, W["fc"])

    # Step 2: K rows per request (R2), all through the layers in one pass.
    u, resid = build_rows(cfg, W, last_token, h, K)
    resid, k_new, v_new = run_layers(cfg, W, u, resid, positions, seq_lens, page_table, k_cache, v_cache,
                                     perturb_rows=perturb_rows)
    logits = lm_head_logits(cfg, W, resid)
    return {
        "logits": logits,
        "drafts": argmax_lowest(logits),
        "gap": top2_gap(logits),
        "k_new": k_new,
        "v_new": v_new,
        "h": h,
    }


def draft_sequential(cfg, W, last_token, target_hidden, positions, seq_lens,
                     page_table, k_cache, v_cache, K, tokens=None):
    """Sequential (EAGLE-style) drafting: K passes of one row per request.

    The chain P-EAGLE breaks ([zh] "P-EAGLE 如何打破这个链"): every draft
    needs the embedding of the token drafted just before it and the hidden
    state that produced it. Readings (also in the design notes):
     S1  Pass 0 is the parallel pass's row 0: embedding of the last accepted
         token and the FC-fused target hidden state. Pass j > 0 takes the
         embedding of draft j-1 and, as its hidden half and residual start,
         the drafter's own final residual stream of pass j-1 (the hidden
         state before the final RMSNorm, H-wide, where the parallel pass uses
         h_shared).
     S2  Pass j sits at RoPE position Q_b + j and cache entry S_b + j; its
         k/v rows are written there before pass j+1 attends over entries
         0 .. S_b + j + 1, so the cache holds real rows for every pass.
    tokens: optional [B, K] int array; when given, pass j > 0 takes
    tokens[:, j-1] as its input token instead of its own draft j-1 (to
    compare against another implementation whose drafts differ at a near
    tie). Returns the same dict as draft_pass (h is the FC output).
    """
    B = len(last_token)
    H = cfg.hidden
    eps = cfg.rms_eps
    P = cfg.page_size
    positions = np.asarray(positions, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    L0 = W["layers"][0]
    embed = np.asarray(W["embed"], dtype=np.float64)

    h = linear(target_hidden, W["fc"])
    tok = np.asarray(last_token, dtype=np.int64)
    hid = h
    logits = np.empty((B, K, cfg.vocab), dtype=np.float64)
    k_new = np.empty((cfg.n_layers, B, K, cfg.n_kv_heads, cfg.head_dim), dtype=np.float64)
    v_new = np.empty_like(k_new)
    for j in range(K):
        u = np.concatenate([rms_norm(embed[tok], L0["norm_e"], eps), rms_norm(hid, L0["norm_h"], eps)], axis=-1)
        resid, kj, vj = run_layers(cfg, W, u[:, None, :], hid[:, None, :].copy(), positions + j, seq_lens + j,
                                   page_table, kc, vc)
        logits[:, j] = lm_head_logits(cfg, W, resid)[:, 0]
        k_new[:, :, j], v_new[:, :, j] = kj[:, :, 0], vj[:, :, 0]
        for b in range(B):                                       # S2: the pass's rows join the cache
            e = int(seq_lens[b]) + j
            page = int(page_table[b][e // P])
            kc[:, page, :, e % P, :] = kj[:, b, 0]
            vc[:, page, :, e % P, :] = vj[:, b, 0]
        d = argmax_lowest(logits[:, j])
        tok = d if tokens is None or j + 1 >= K else np.asarray(tokens, dtype=np.int64)[:, j]
        hid = resid[:, 0]
    return {
        "logits": logits,
        "drafts": argmax_lowest(logits),
        "gap": top2_gap(logits),
        "k_new": k_new,
        "v_new": v_new,
        "h": h,
    }


def draft_pass_refeed(cfg, W, tokens, n_real, target_hidden, positions, seq_lens,
                      page_table, k_cache, v_cache, K):
    """Parallel draft pass with the accepted tokens re-fed as real rows.

    Reading F2 (the alternative to R6 where the pages are silent on the
    drafter's bookkeeping; also in the design notes): after a verify, the n_b
    tokens it emitted (the accepted drafts and the bonus token) come back
    with the target's hidden states at their positions as n_b REAL rows -
    each row the embedding of its token and the FC-fused hidden state, the
    pages' position-1 input - ahead of the K-1 placeholder rows (emb_mask,
    h_shared). Real row i sits at position Q_b + i and cache entry S_b + i;
    placeholder j (1..K-1) at position Q_b + n_b - 1 + j and entry
    S_b + n_b - 1 + j. Draft 0 is the argmax of the last real row, draft j
    that of placeholder j. Every row attends causally as in R6.

    tokens [B, n_max] (entries past n_real[b] unused), n_real [B] in
    1..n_max, target_hidden [B, n_max, 3H]. Each request runs as its own
    batch of n_b + K - 1 rows. Returns logits / drafts / gap [B, K, ...] and
    k_new / v_new [L, B, n_max + K - 1, nkv, hd] (rows past n_b + K - 1 of a
    request are NaN).
    """
    B = len(n_real)
    H = cfg.hidden
    eps = cfg.rms_eps
    n_max = int(np.max(n_real))
    T_max = n_max + K - 1
    L0 = W["layers"][0]
    embed = np.asarray(W["embed"], dtype=np.float64)
    logits = np.empty((B, K, cfg.vocab), dtype=np.float64)
    k_new = np.full((cfg.n_layers, B, T_max, cfg.n_kv_heads, cfg.head_dim), np.nan)
    v_new = np.full_like(k_new, np.nan)
    for b in range(B):
        n = int(n_real[b])
        h = linear(np.asarray(target_hidden[b, :n], dtype=np.float64), W["fc"])      # R1, per real row
        emb = embed[np.asarray(tokens[b, :n], dtype=np.int64)]
        if K > 1:
            emb = np.concatenate([emb, np.repeat(np.asarray(W["emb_mask"], np.float64)[None], K - 1, 0)])
            hid = np.concatenate([h, np.repeat(np.asarray(W["h_shared"], np.float64)[None], K - 1, 0)])
        else:
            hid = h
        u = np.concatenate([rms_norm(emb, L0["norm_e"], eps), rms_norm(hid, L0["norm_h"], eps)], axis=-1)
        resid, kb, vb = run_layers(cfg, W, u[None], hid[None].copy(), np.asarray(positions)[b:b + 1],
                                   np.asarray(seq_lens)[b:b + 1], np.asarray(page_table)[b:b + 1],
                                   k_cache, v_cache)
        logits[b] = lm_head_logits(cfg, W, resid[0, n - 1:])
        k_new[:, b, :n + K - 1] = kb[:, 0]
        v_new[:, b, :n + K - 1] = vb[:, 0]
    return {
        "logits": logits,
        "drafts": argmax_lowest(logits),
        "gap": top2_gap(logits),
        "k_new": k_new,
        "v_new": v_new,
    }
