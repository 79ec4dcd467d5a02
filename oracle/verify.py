"""Greedy verification, bonus token and batch-metadata rebuild, plainly.

TEST INFRASTRUCTURE ONLY: see the package docstring.

Sources (page titles and sections):
[zh] "在 Amazon SageMaker AI 上使用 P-EAGLE 并行化推测解码", section
     "解决方案概述" / "逐步草稿过程": the target checks all K candidates in
     one verification pass with the standard acceptance rule; section
     "并行草稿的实际优势" ("无质量妥协"): the output equals what the target
     alone would produce, so with greedy decoding the emitted tokens are the
     target's own argmax tokens.
[ja] "Amazon SageMaker AIにおけるP-EAGLEによる推論高速化": a fused kernel
     rebuilds the batch metadata after verification (details not given).
[ko-lesson] "프로덕션의 EAGLE-3 추측 디코딩", section "개념" (Concept):
     expected tokens per target pass 1 + K*alpha and speedup
     (1 + K*alpha) / (1 + epsilon), worked example K=5, alpha=0.7,
     epsilon=0.1 -> 4.5 / 1.1; section "한 줄로 보는 손익분기 수식":
     break-even alpha = verify_overhead / K.

Readings where the pages are silent (also listed in the design notes):
 V1  Acceptance is greedy: a_b = length of the longest prefix on which the
     drafts d[b, :] equal the target's argmax tokens g[b, :K]; the bonus token
     is g[b, a_b]; emitted tokens are d[b, :a_b] followed by the bonus.
 V2  Drafter-cache bookkeeping: the pass wrote rows 0..K-1 at entries
     S_b .. S_b+K-1. Rows 0 .. min(a_b, K-1) are kept, so
     kept = min(a_b, K-1) + 1 and S_b' = S_b + kept. The position of the next
     step's row 0 is Q_b' = Q_b + a_b + 1.
 V3  The next step's slot mapping: entry S_b' + j lives at physical slot
     page_table[b, (S_b'+j) // P] * P + (S_b'+j) % P for j < K.
 V4  Rolled-back slots are those of entries S_b' .. S_b+K-1
     (K - kept of them), padded with -1 to K.
 V5  A request whose length or position is outside [0, 2^31 - 1 - 2K]
     (negative, or so large that the next step's entries or positions would
     not fit a signed 32-bit integer) gets status REQ_BAD_INPUT; one whose
     next K entries do not fit its page table (S_b' + K > max_pages * P)
     gets REQ_CAPACITY; one whose needed page index is outside
     [0, num_pages) gets REQ_BAD_PAGE. For such a request seq_lens /
     positions are returned unchanged and the slot and rollback rows are all
     -1; accepted length and bonus are still reported.
"""

import numpy as np

REQ_OK = 0
REQ_CAPACITY = 1
REQ_BAD_PAGE = 2
REQ_BAD_INPUT = 3
INT32_MAX = 2 ** 31 - 1


def accept_length(d_row, g_row):
    """Number of leading positions where the draft equals the target token (V1)."""
    a = 0
    while a < len(d_row) and int(d_row[a]) == int(g_row[a]):
        a += 1
    return a


def verify(drafts, target_tokens):
    """Greedy acceptance for a batch. drafts [B, K], target_tokens [B, K+1]."""
    drafts = np.asarray(drafts)
    target_tokens = np.asarray(target_tokens)
    B, K = drafts.shape
    accepted = np.array([accept_length(drafts[b], target_tokens[b, :K]) for b in range(B)],
                        dtype=np.int64)
    bonus = target_tokens[np.arange(B), accepted].astype(np.int64)
    return accepted, bonus


def emitted_tokens(drafts, accepted, bonus):
    """[B, K+1] tokens the step emits, -1 padded (V1)."""
    B, K = np.asarray(drafts).shape
    out = np.full((B, K + 1), -1, dtype=np.int64)
    for b in range(B):
        a = int(accepted[b])
        out[b, :a] = drafts[b, :a]
        out[b, a] = bonus[b]
    return out


def rebuild_metadata(accepted, K, seq_lens, positions, page_table, num_pages, page_size=16):
    """Batch metadata for the next step (V2..V5).

    Returns a dict with seq_lens, positions (both [B]), slot_mapping [B, K],
    rollback_slots [B, K] and status [B].
    """
    accepted = np.asarray(accepted, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    page_table = np.asarray(page_table, dtype=np.int64)
    B = len(accepted)
    max_pages = page_table.shape[1]

    new_S = seq_lens.copy()
    new_Q = positions.copy()
    slot_mapping = np.full((B, K), -1, dtype=np.int64)
    rollback = np.full((B, K), -1, dtype=np.int64)
    status = np.full(B, REQ_OK, dtype=np.int64)

    for b in range(B):
        a = int(accepted[b])
        S, Q = int(seq_lens[b]), int(positions[b])
        if not (0 <= S <= INT32_MAX - 2 * K and 0 <= Q <= INT32_MAX - 2 * K):
            status[b] = REQ_BAD_INPUT
            continue
        kept = min(a, K - 1) + 1
        S_next = S + kept
        Q_next = Q + a + 1
        if S_next + K > max_pages * page_size:
            status[b] = REQ_CAPACITY
            continue
        slots = []
        for j in range(K):
            e = S_next + j
            page = int(page_table[b, e // page_size])
            if page < 0 or page >= num_pages:
                status[b] = REQ_BAD_PAGE
                break
            slots.append(page * page_size + e % page_size)
        if status[b] != REQ_OK:
            continue
        new_S[b] = S_next
        new_Q[b] = Q_next
        slot_mapping[b, :] = slots
        n_rollback = K - kept
        rollback[b, :n_rollback] = slots[:n_rollback]

    return {
        "seq_lens": new_S,
        "positions": new_Q,
        "slot_mapping": slot_mapping,
        "rollback_slots": rollback,
        "status": status,
    }


def expected_tokens_iid(alpha, K):
    """Mean tokens per step when each position agrees independently with
    probability alpha: E[a + 1] = sum_{j=0..K} alpha^j."""
    alpha = float(alpha)
    if alpha == 1.0:
        return float(K + 1)
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha)


def tokens_per_pass_linear(alpha, K):
    """The lesson page's simple model of tokens per target pass: 1 + K*alpha."""
    return 1.0 + K * float(alpha)


def speedup_linear(alpha, K, overhead):
    """The lesson page's speedup model (1 + K*alpha) / (1 + overhead)."""
    return tokens_per_pass_linear(alpha, K) / (1.0 + float(overhead))


def breakeven_alpha(overhead, K):
    """alpha at which speedup_linear equals 1: overhead / K."""
    return float(overhead) / K


def rebuild_metadata_refeed(accepted, K, n_real, seq_lens, positions, page_table, num_pages, page_size=16):
    """Batch metadata after a verify when the next pass re-feeds the emitted
    tokens as real rows (reading F2 of the drafter).

    The pass just verified wrote n_b real rows at entries S_b .. S_b+n_b-1
    and K-1 placeholder rows after them. The real rows stay committed and the
    placeholders are rolled back: S_b' = S_b + n_b, Q_b' = Q_b + n_b, and the
    next pass has n_b' = a_b + 1 real rows (the accepted drafts and the bonus
    token). Returns seq_lens, positions, n_real (next step), slot_mapping
    [B, 2K] (slots of the next pass's entries S_b' .. S_b'+n_b'+K-2, then -1),
    rollback_slots [B, K] (slots of entries S_b+n_b .. S_b+n_b+K-2, then -1)
    and status, with the input checks of V5 (a request whose next pass does
    not fit its page table, or whose page is out of range, keeps its
    metadata, n_real' = n_real, and gets -1 rows).
    """
    accepted = np.asarray(accepted, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    n_real = np.asarray(n_real, dtype=np.int64)
    page_table = np.asarray(page_table, dtype=np.int64)
    B = len(accepted)
    max_pages = page_table.shape[1]
    new_S, new_Q, new_n = seq_lens.copy(), positions.copy(), n_real.copy()
    slot_mapping = np.full((B, 2 * K), -1, dtype=np.int64)
    rollback = np.full((B, K), -1, dtype=np.int64)
    status = np.full(B, REQ_OK, dtype=np.int64)

    def slot(b, e):
        page = int(page_table[b, e // page_size])
        return None if page < 0 or page >= num_pages else page * page_size + e % page_size

    for b in range(B):
        S, Q, n, a = int(seq_lens[b]), int(positions[b]), int(n_real[b]), int(accepted[b])
        if not (0 <= S <= INT32_MAX - 4 * K and 0 <= Q <= INT32_MAX - 4 * K and 1 <= n <= K + 1):
            status[b] = REQ_BAD_INPUT
            continue
        S2, Q2, n2 = S + n, Q + n, a + 1
        if S2 + n2 + K - 1 > max_pages * page_size:
            status[b] = REQ_CAPACITY
            continue
        nxt = [slot(b, S2 + j) for j in range(n2 + K - 1)]
        rb = [slot(b, S + n + j) for j in range(K - 1)]
        if any(x is None for x in nxt + rb):
            status[b] = REQ_BAD_PAGE
            continue
        new_S[b], new_Q[b], new_n[b] = S2, Q2, n2
        slot_mapping[b, :len(nxt)] = nxt
        rollback[b, :len(rb)] = rb
    return {"seq_lens": new_S, "positions": new_Q, "n_real": new_n, "slot_mapping": slot_mapping,
            "rollback_slots": rollback, "status": status}
