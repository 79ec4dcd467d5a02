"""Sampled drafting and stochastic acceptance, plainly.

TEST INFRASTRUCTURE ONLY: see the package docstring.

[zh] "在 Amazon SageMaker AI 上使用 P-EAGLE 并行化推测解码", section "逐步草稿过程":
the target verifies the K drafts in one pass with the standard acceptance
rule, and the output is the target's own ("并行草稿的实际优势": no quality
loss); the deployment's request payload samples at temperature 0.3. With
sampling, the standard rule is speculative sampling (reading A1, also in the
design notes):
 - draft distributions q_j = softmax(l_j / T) from the drafter's logits of
   row j; P-EAGLE's rows all come from one pass, so each draft d_j is drawn
   from its own q_j, independently;
 - target distributions p_j = softmax(g_j / T), j = 0..K, from the target's
   logits at the K+1 verified positions;
 - for j = 0, 1, ...: draft d_j is accepted when u_j < p_j(d_j) / q_j(d_j);
   at the first rejection the step emits a token drawn from
   max(0, p_j - q_j) / sum(max(0, p_j - q_j)); if every draft is accepted it
   emits a bonus token drawn from p_K.
 - Every draw is inverse-CDF sampling with a uniform u in [0, 1) passed in:
   the smallest index i with cumsum(probs)[i] > u * sum(probs).
The emitted tokens are then distributed as sampling the target alone.
"""

import numpy as np


def softmax_t(logits, T):
    """softmax(logits / T) over the last axis, float64."""
    z = np.asarray(logits, dtype=np.float64) / float(T)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def sample_inverse_cdf(weights, u):
    """Smallest index i with sum(weights[:i+1]) > u * sum(weights) for one
    row of non-negative weights (not necessarily normalised); u in [0, 1).
    Also returns the margin: the distance of u * total from the nearest
    cumulative boundary, relative to the total (how far the draw is from
    going to a neighbouring index)."""
    w = np.asarray(weights, dtype=np.float64)
    c = np.cumsum(w)
    total = c[-1]
    x = float(u) * total
    i = int(np.searchsorted(c, x, side="right"))
    i = min(i, len(w) - 1)
    while w[i] == 0.0 and i > 0:         # never land on an index of weight 0
        i -= 1
    lo = c[i - 1] if i > 0 else 0.0
    margin = min(x - lo, c[i] - x) / total
    return i, margin


def sample_drafts(draft_logits, T, u):
    """Drafts d[b, j] ~ softmax(l[b, j] / T) by inverse CDF with u[b, j].
    Returns (drafts [B, K], margins [B, K])."""
    lg = np.asarray(draft_logits, dtype=np.float64)
    B, K = lg.shape[:2]
    d = np.empty((B, K), dtype=np.int64)
    m = np.empty((B, K))
    for b in range(B):
        for j in range(K):
            d[b, j], m[b, j] = sample_inverse_cdf(softmax_t(lg[b, j], T), u[b, j])
    return d, m


def verify_stochastic(drafts, draft_logits, target_logits, T, u_accept, u_final):
    """Speculative-sampling acceptance (reading A1) for a batch.

    drafts [B, K]; draft_logits [B, K, V]; target_logits [B, K+1, V];
    u_accept [B, K] and u_final [B] uniforms in [0, 1).
    Returns a dict: accepted [B] (a_b), final [B] (the resampled token at the
    first rejection, or the bonus from p_K), emitted [B, K+1] (d[:a], final,
    then -1), and margin [B]: the smallest decision margin of the request
    (|u_j - ratio_j| of every acceptance test made, and the final draw's
    inverse-CDF margin), for comparisons with another implementation.
    """
    d = np.asarray(drafts, dtype=np.int64)
    B, K = d.shape
    q = softmax_t(draft_logits, T)
    p = softmax_t(target_logits, T)
    accepted = np.empty(B, dtype=np.int64)
    final = np.empty(B, dtype=np.int64)
    margin = np.empty(B)
    emitted = np.full((B, K + 1), -1, dtype=np.int64)
    for b in range(B):
        a = 0
        mb = np.inf
        while a < K:
            ratio = p[b, a, d[b, a]] / q[b, a, d[b, a]]
            mb = min(mb, abs(float(u_accept[b, a]) - ratio))
            if float(u_accept[b, a]) < ratio:
                a += 1
            else:
                break
        if a < K:
            w = np.maximum(p[b, a] - q[b, a], 0.0)
        else:
            w = p[b, K]
        tok, m = sample_inverse_cdf(w, u_final[b])
        accepted[b], final[b], margin[b] = a, tok, min(mb, m)
        emitted[b, :a] = d[b, :a]
        emitted[b, a] = tok
    return {"accepted": accepted, "final": final, "emitted": emitted, "margin": margin}
