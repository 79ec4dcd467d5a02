"""Pins for the CPU oracle: each test checks it against something other than
itself (library routines, closed forms, brute force, invariants the pages
state). CPU only."""

import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from speculative_drafting_pe_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# A tiny drafter for whole-pass pins: several heads, GQA group 2, 3 pages.
TINY = synth.DrafterShape("oracle-pin", hidden=32, n_q_heads=4, n_kv_heads=2, head_dim=8,
                          ffn=64, vocab=97, dtype="fp32")


def _tiny_case(K, B=2, seed=5, prefix=(20, 41)):
    wl = synth.Workload("pin", TINY, B, K, prefix, (0.7, 0.7), seed)
    W = synth.make_weights(TINY, seed)
    inp = synth.make_step_inputs(wl, K=K)
    return W, inp


def _run_oracle(W, inp, K, **kw):
    Wn = synth.weights_to_numpy(W)
    return oracle.draft_pass(
        TINY, Wn, inp.last_token.numpy(), inp.target_hidden.double().numpy(),
        inp.positions.numpy(), inp.seq_lens.numpy(), inp.page_table.numpy(),
        inp.k_cache.double().numpy(), inp.v_cache.double().numpy(), K, **kw)


# --------------------------------------------------------------- building blocks

def test_rms_norm_matches_torch_library():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(5, 7, 33)) * 3.0
    g = 1.0 + 0.1 * rng.normal(size=33)
    ref = F.rms_norm(torch.tensor(x), (33,), weight=torch.tensor(g), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, g, 1e-6), ref, rtol=1e-13, atol=1e-13)


def test_silu_matches_torch_library():
    x = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(oracle.silu(x), F.silu(torch.tensor(x)).numpy(), rtol=1e-13, atol=1e-15)


def test_rope_equals_complex_rotation():
    # Rotate-half RoPE is multiplication of z = x1 + i x2 by exp(i * pos * inv_freq).
    rng = np.random.default_rng(1)
    hd, theta = 16, 1e4
    x = rng.normal(size=(6, hd))
    pos = np.array([0, 1, 7, 100, 2047, 8191])
    half = hd // 2
    inv = theta ** (-(np.arange(half) * 2.0) / hd)
    z = (x[:, :half] + 1j * x[:, half:]) * np.exp(1j * pos[:, None] * inv[None, :])
    ref = np.concatenate([z.real, z.imag], axis=1)
    np.testing.assert_allclose(oracle.rope_neox(x, pos, theta), ref, rtol=1e-12, atol=1e-12)


def test_rope_special_cases():
    # position 0 is the identity; hd=2 rotates by exactly `pos` radians.
    x = np.random.default_rng(2).normal(size=(3, 8))
    np.testing.assert_array_equal(oracle.rope_neox(x, np.zeros(3), 1e4), x)
    out = oracle.rope_neox(np.array([[1.0, 0.0]]), np.array([0.5]), 1e4)
    np.testing.assert_allclose(out, [[np.cos(0.5), np.sin(0.5)]], rtol=1e-15)


def test_rope_relative_position_property():
    # <rope(q, p1), rope(k, p2)> depends only on p1 - p2.
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=64), rng.normal(size=64)
    d1 = oracle.rope_neox(q, np.array(10), 1e4) @ oracle.rope_neox(k, np.array(3), 1e4)
    d2 = oracle.rope_neox(q, np.array(1007), 1e4) @ oracle.rope_neox(k, np.array(1000), 1e4)
    assert abs(d1 - d2) < 1e-9


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(4)
    K, nq, nkv, hd, S = 5, 8, 2, 16, 37
    q = rng.normal(size=(K, nq, hd))
    k_all = rng.normal(size=(S + K, nkv, hd))
    v_all = rng.normal(size=(S + K, nkv, hd))
    out = oracle.causal_paged_attention(q, k_all, v_all, S)
    G = nq // nkv
    qt = torch.tensor(q).permute(1, 0, 2)[None]                       # [1, nq, K, hd]
    kt = torch.tensor(k_all).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    vt = torch.tensor(v_all).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    mask = torch.arange(S + K)[None, :] <= (S + torch.arange(K))[:, None]
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_gather_prefix_kv_follows_page_table():
    # Encode (page, head, slot, dim) in the value and read entries back.
    P, npg, nkv, hd = 16, 9, 2, 3
    cache = np.zeros((npg, nkv, P, hd))
    for p, h, s, d in itertools.product(range(npg), range(nkv), range(P), range(hd)):
        cache[p, h, s, d] = p * 1000 + h * 100 + s + d / 10
    pt = np.array([7, 2, 5, 0])
    out = oracle.gather_prefix_kv(cache, pt, 50, P)
    for e in range(50):
        page = pt[e // P]
        for h in range(nkv):
            assert out[e, h, 0] == page * 1000 + h * 100 + e % P


def test_linear_is_x_times_w_transposed():
    rng = np.random.default_rng(6)
    x = rng.normal(size=(3, 11))
    w = rng.normal(size=(40000, 11)).astype(np.float32)
    ref = F.linear(torch.tensor(x), torch.tensor(w, dtype=torch.float64)).numpy()
    np.testing.assert_allclose(oracle.linear(x, w), ref, rtol=1e-12, atol=1e-12)


def test_argmax_ties_go_to_lowest_index_and_gap():
    logits = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0], [0.0, -1.0, 2.5, 2.0]])
    np.testing.assert_array_equal(oracle.argmax_lowest(logits), [1, 0, 2])
    np.testing.assert_allclose(oracle.top2_gap(logits), [0.0, 0.0, 0.5])


def test_build_rows_row0_real_rest_placeholders():
    W, inp = _tiny_case(K=4)
    Wn = synth.weights_to_numpy(W)
    h = np.random.default_rng(7).normal(size=(2, TINY.hidden))
    u, resid = oracle.build_rows(TINY, Wn, inp.last_token.numpy(), h, 4)
    H = TINY.hidden
    for b in range(2):
        e0 = Wn["embed"][inp.last_token[b]].astype(np.float64)
        ge = Wn["layers"][0]["norm_e"].astype(np.float64)
        np.testing.assert_allclose(u[b, 0, :H], e0 / np.sqrt(np.mean(e0 ** 2) + 1e-6) * ge)
        np.testing.assert_allclose(resid[b, 0], h[b])
        for j in range(1, 4):
            m = Wn["emb_mask"].astype(np.float64)
            np.testing.assert_allclose(u[b, j, :H], m / np.sqrt(np.mean(m ** 2) + 1e-6) * ge)
            np.testing.assert_allclose(resid[b, j], Wn["h_shared"])


# --------------------------------------------------------------- whole draft pass

def _torch_reference_pass(W, inp, K, full=False):
    """Independent float64 restatement with torch library routines
    (F.linear, F.rms_norm, F.silu, SDPA, complex-number RoPE) and an explicit
    per-entry walk of the page table. With full=True also returns, per layer,
    the layer's input rows x [L, B, K, in], the rotated new k rows and the
    raw new v rows [L, B, K, nkv, hd] that the pass writes to the cache."""
    cfg = TINY
    d = torch.float64
    t = lambda a: a.to(d)
    B = inp.last_token.shape[0]
    H, nq, nkv, hd = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    eps = cfg.rms_eps
    nl = len(W["layers"])

    def norm(x, g):
        return F.rms_norm(x, (x.shape[-1],), weight=t(g), eps=eps)

    def rope(x, pos):
        half = hd // 2
        inv = cfg.rope_theta ** (-(torch.arange(half, dtype=d) * 2.0) / hd)
        ang = pos.to(d)[..., None] * inv
        z = torch.complex(x[..., :half], x[..., half:]) * torch.polar(torch.ones_like(ang), ang)
        return torch.cat([z.real, z.imag], dim=-1)

    h = F.linear(t(inp.target_hidden), t(W["fc"]))
    emb = torch.stack([t(W["embed"][int(tok)]) for tok in inp.last_token])
    L0 = W["layers"][0]
    logits = torch.empty(B, K, cfg.vocab, dtype=d)
    xs = [[None] * B for _ in range(nl)]
    k_rows = torch.empty(nl, B, K, nkv, hd, dtype=d)
    v_rows = torch.empty(nl, B, K, nkv, hd, dtype=d)
    for b in range(B):
        rows_e = [emb[b]] + [t(W["emb_mask"])] * (K - 1)
        rows_h = [h[b]] + [t(W["h_shared"])] * (K - 1)
        x = torch.cat([norm(torch.stack(rows_e), L0["norm_e"]), norm(torch.stack(rows_h), L0["norm_h"])], -1)
        r = torch.stack(rows_h).clone()
        S = int(inp.seq_lens[b])
        pos = int(inp.positions[b]) + torch.arange(K)
        for li, Lw in enumerate(W["layers"]):
            if li > 0:
                x = norm(r, Lw["attn_norm"])
            xs[li][b] = x
            qkv = F.linear(x, t(Lw["w_qkv"]))
            q = rope(qkv[:, : nq * hd].reshape(K, nq, hd), pos[:, None])
            k = rope(qkv[:, nq * hd:(nq + nkv) * hd].reshape(K, nkv, hd), pos[:, None])
            v = qkv[:, (nq + nkv) * hd:].reshape(K, nkv, hd)
            k_rows[li, b], v_rows[li, b] = k, v
            ks, vs = [], []
            for e in range(S):
                page = int(inp.page_table[b, e // cfg.page_size])
                ks.append(t(inp.k_cache[li, page, :, e % cfg.page_size, :]))
                vs.append(t(inp.v_cache[li, page, :, e % cfg.page_size, :]))
            k_all = torch.cat([torch.stack(ks), k]) if S else k
            v_all = torch.cat([torch.stack(vs), v]) if S else v
            G = nq // nkv
            mask = torch.arange(S + K)[None, :] <= (S + torch.arange(K))[:, None]
            a = F.scaled_dot_product_attention(
                q.permute(1, 0, 2)[None],
                k_all.permute(1, 0, 2).repeat_interleave(G, 0)[None],
                v_all.permute(1, 0, 2).repeat_interleave(G, 0)[None], attn_mask=mask)
            r = r + F.linear(a[0].permute(1, 0, 2).reshape(K, nq * hd), t(Lw["w_o"]))
            x = norm(r, Lw["mlp_norm"])
            r = r + F.linear(F.silu(F.linear(x, t(Lw["w_gate"]))) * F.linear(x, t(Lw["w_up"])), t(Lw["w_down"]))
        logits[b] = F.linear(norm(r, W["final_norm"]), t(W["lm_head"]))
    if not full:
        return logits.numpy()
    return dict(logits=logits.numpy(), x=[torch.stack(xs[li]) for li in range(nl)], k_new=k_rows.numpy(),
                v_new=v_rows.numpy())


@pytest.mark.parametrize("K", [1, 4])
def test_draft_pass_matches_independent_torch_restatement(K):
    # K=1 is one ordinary (sequential) EAGLE step: row 0 only.
    W, inp = _tiny_case(K)
    out = _run_oracle(W, inp, K)
    ref = _torch_reference_pass(W, inp, K)
    np.testing.assert_allclose(out["logits"], ref, rtol=1e-10, atol=1e-10)
    ok = out["gap"] > 1e-9
    np.testing.assert_array_equal(out["drafts"][ok], ref.argmax(-1)[ok])


def test_prefix_consistency_and_row0_independent_of_K():
    # Rows are causal: drafts for K' < K equal the first K' drafts for K.
    W, inp = _tiny_case(K=6)
    full = _run_oracle(W, inp, 6)
    for Kp in (1, 2, 5):
        part = _run_oracle(W, inp, Kp)
        np.testing.assert_allclose(part["logits"], full["logits"][:, :Kp], rtol=1e-10, atol=1e-11)
        ok = part["gap"] > 1e-9
        np.testing.assert_array_equal(part["drafts"][ok], full["drafts"][:, :Kp][ok])


def test_perturbing_later_rows_leaves_earlier_rows_unchanged():
    W, inp = _tiny_case(K=5)
    base = _run_oracle(W, inp, 5)

    def hook(u):
        u = u.copy()
        u[:, 3:, :] += 0.5
        return u

    pert = _run_oracle(W, inp, 5, perturb_rows=hook)
    np.testing.assert_array_equal(pert["logits"][:, :3], base["logits"][:, :3])
    assert np.abs(pert["logits"][:, 3:] - base["logits"][:, 3:]).max() > 1e-5


def test_draft_argmax_exhaustive_on_tiny_vocab():
    W, inp = _tiny_case(K=3)
    out = _run_oracle(W, inp, 3)
    V = TINY.vocab
    for b, j in itertools.product(range(2), range(3)):
        row = out["logits"][b, j]
        best = 0
        for v in range(V):
            if row[v] > row[best]:
                best = v
        assert out["drafts"][b, j] == best


def test_new_kv_rows_match_independent_torch_restatement():
    # The rows the pass writes to the cache (k after RoPE, v as projected)
    # equal the torch restatement's own k and v rows, layer by layer.
    W, inp = _tiny_case(K=4)
    out = _run_oracle(W, inp, 4)
    ref = _torch_reference_pass(W, inp, 4, full=True)
    assert out["k_new"].shape == (4, 2, 4, TINY.n_kv_heads, TINY.head_dim)
    np.testing.assert_allclose(out["k_new"], ref["k_new"], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["v_new"], ref["v_new"], rtol=1e-10, atol=1e-10)


def _unrotate(k, pos):
    """Inverse rotate-half RoPE by complex division: k [..., hd], pos [...]."""
    hd = k.shape[-1]
    half = hd // 2
    inv = TINY.rope_theta ** (-(np.arange(half) * 2.0) / hd)
    z = (k[..., :half] + 1j * k[..., half:]) * np.exp(-1j * np.asarray(pos, dtype=np.float64)[..., None] * inv)
    return np.concatenate([z.real, z.imag], axis=-1)


def _kv_rows_violations(k_new, v_new, x, W, positions, K):
    """Checks k_new / v_new [L, B, K, nkv, hd] against the layer inputs x
    (list of [B, K, in] float64 tensors): un-rotating row j of request b by
    the angle of position Q_b + j must give W_k x exactly, v must be W_v x
    unrotated. Returns the list of failed checks (empty when all hold)."""
    nq, nkv, hd = TINY.n_q_heads, TINY.n_kv_heads, TINY.head_dim
    bad = []
    B = k_new.shape[1]
    pos = np.asarray(positions, dtype=np.int64)[:, None] + np.arange(K)[None, :]      # [B, K]
    for li, Lw in enumerate(W["layers"]):
        wq = torch.as_tensor(Lw["w_qkv"]).double()
        k_raw = F.linear(x[li], wq[nq * hd:(nq + nkv) * hd]).numpy().reshape(B, K, nkv, hd)
        v_raw = F.linear(x[li], wq[(nq + nkv) * hd:]).numpy().reshape(B, K, nkv, hd)
        un = _unrotate(k_new[li], pos[:, :, None])
        if not np.allclose(un, k_raw, rtol=1e-9, atol=1e-10):
            bad.append(f"layer {li}: k does not un-rotate to W_k x at positions Q+j")
        if not np.allclose(v_new[li], v_raw, rtol=1e-9, atol=1e-10):
            bad.append(f"layer {li}: v is not W_v x")
    return bad


def test_new_kv_rows_are_rotated_with_row_positions():
    # k of row j un-rotates (angle of position Q_b + j) to an independent
    # F.linear of that layer's input; v is that layer's raw projection.
    W, inp = _tiny_case(K=3)
    out = _run_oracle(W, inp, 3)
    ref = _torch_reference_pass(W, inp, 3, full=True)
    assert _kv_rows_violations(out["k_new"], out["v_new"], ref["x"], W, inp.positions.numpy(), 3) == []
    # rotating by Q_b + j + 1 instead is caught
    pos1 = inp.positions.numpy() + 1
    assert _kv_rows_violations(out["k_new"], out["v_new"], ref["x"], W, pos1, 3) != []


@pytest.mark.parametrize("mistake", ["unrotated_k", "position_off_by_one", "k_v_swapped"])
def test_kv_row_check_fails_on_planted_oracle_mistakes(mistake):
    # Each plausible mistake in how the oracle forms its new cache rows leaves
    # the logits unchanged; the row check above must still reject it.
    W, inp = _tiny_case(K=3)
    out = _run_oracle(W, inp, 3)
    ref = _torch_reference_pass(W, inp, 3, full=True)
    k, v = out["k_new"].copy(), out["v_new"].copy()
    pos = inp.positions.numpy()[:, None] + np.arange(3)[None, :]
    if mistake == "unrotated_k":
        k = _unrotate(k, pos[None, :, :, None])
    elif mistake == "position_off_by_one":
        k = oracle.rope_neox(_unrotate(k, pos[None, :, :, None]), (pos + 1)[None, :, :, None], TINY.rope_theta)
    else:
        k, v = v, k
    assert _kv_rows_violations(k, v, ref["x"], W, inp.positions.numpy(), 3) != []


# --------------------------------------------------------------- sequential drafting

def _torch_sequential(W, inp, K):
    """Independent float64 restatement of sequential EAGLE drafting: per
    request, K one-row passes; each layer's cache is a Python list of the
    committed rows (walked through the page table) to which every pass
    appends its own k/v row; the single query attends to the whole list."""
    cfg = TINY
    d = torch.float64
    t = lambda a: a.to(d)
    H, nq, nkv, hd = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    eps = cfg.rms_eps
    G = nq // nkv

    def norm(x, g):
        return F.rms_norm(x, (x.shape[-1],), weight=t(g), eps=eps)

    def rope(x, pos):
        half = hd // 2
        inv = cfg.rope_theta ** (-(torch.arange(half, dtype=d) * 2.0) / hd)
        ang = torch.tensor(float(pos), dtype=d) * inv
        z = torch.complex(x[..., :half], x[..., half:]) * torch.polar(torch.ones_like(ang), ang)
        return torch.cat([z.real, z.imag], dim=-1)

    B = inp.last_token.shape[0]
    h = F.linear(t(inp.target_hidden), t(W["fc"]))
    logits = torch.empty(B, K, cfg.vocab, dtype=d)
    k_rows = torch.empty(4, B, K, nkv, hd, dtype=d)
    v_rows = torch.empty(4, B, K, nkv, hd, dtype=d)
    L0 = W["layers"][0]
    for b in range(B):
        S, Q = int(inp.seq_lens[b]), int(inp.positions[b])
        ks = [[t(inp.k_cache[li, int(inp.page_table[b, e // 16]), :, e % 16, :]) for e in range(S)]
              for li in range(4)]
        vs = [[t(inp.v_cache[li, int(inp.page_table[b, e // 16]), :, e % 16, :]) for e in range(S)]
              for li in range(4)]
        tok, hid = int(inp.last_token[b]), h[b]
        for j in range(K):
            x = torch.cat([norm(t(W["embed"][tok])[None], L0["norm_e"]), norm(hid[None], L0["norm_h"])], -1)
            r = hid[None].clone()
            for li, Lw in enumerate(W["layers"]):
                if li > 0:
                    x = norm(r, Lw["attn_norm"])
                qkv = F.linear(x, t(Lw["w_qkv"]))[0]
                q = rope(qkv[: nq * hd].reshape(nq, hd), Q + j)
                ks[li].append(rope(qkv[nq * hd:(nq + nkv) * hd].reshape(nkv, hd), Q + j))
                vs[li].append(qkv[(nq + nkv) * hd:].reshape(nkv, hd))
                k_rows[li, b, j], v_rows[li, b, j] = ks[li][-1], vs[li][-1]
                k_all = torch.stack(ks[li]).permute(1, 0, 2).repeat_interleave(G, 0)
                v_all = torch.stack(vs[li]).permute(1, 0, 2).repeat_interleave(G, 0)
                a = F.scaled_dot_product_attention(q[:, None, :], k_all, v_all)[:, 0, :]
                r = r + F.linear(a.reshape(1, nq * hd), t(Lw["w_o"]))
                x = norm(r, Lw["mlp_norm"])
                r = r + F.linear(F.silu(F.linear(x, t(Lw["w_gate"]))) * F.linear(x, t(Lw["w_up"])),
                                 t(Lw["w_down"]))
            logits[b, j] = F.linear(norm(r, W["final_norm"]), t(W["lm_head"]))[0]
            tok, hid = int(torch.argmax(logits[b, j])), r[0]
    return dict(logits=logits.numpy(), k_new=k_rows.numpy(), v_new=v_rows.numpy())


def _run_sequential(W, inp, K, **kw):
    Wn = synth.weights_to_numpy(W)
    return oracle.draft_sequential(
        TINY, Wn, inp.last_token.numpy(), inp.target_hidden.double().numpy(),
        inp.positions.numpy(), inp.seq_lens.numpy(), inp.page_table.numpy(),
        inp.k_cache.double().numpy(), inp.v_cache.double().numpy(), K, **kw)


def test_sequential_matches_independent_torch_restatement():
    W, inp = _tiny_case(K=4)
    out = _run_sequential(W, inp, 4)
    ref = _torch_sequential(W, inp, 4)
    np.testing.assert_allclose(out["logits"], ref["logits"], rtol=1e-10, atol=1e-10)
    ok = out["gap"] > 1e-9
    np.testing.assert_array_equal(out["drafts"][ok], ref["logits"].argmax(-1)[ok])
    # every pass's cache rows, the last pass's included
    np.testing.assert_allclose(out["k_new"], ref["k_new"], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["v_new"], ref["v_new"], rtol=1e-10, atol=1e-10)


def test_sequential_k1_is_the_parallel_pass_k1():
    # one sequential step and a one-row parallel pass are the same computation
    W, inp = _tiny_case(K=1)
    seq = _run_sequential(W, inp, 1)
    par = _run_oracle(W, inp, 1)
    for k in ("logits", "k_new", "v_new"):
        np.testing.assert_allclose(seq[k], par[k], rtol=1e-12, atol=1e-12)


def test_sequential_row0_equals_parallel_row0_and_later_rows_differ():
    W, inp = _tiny_case(K=4)
    seq = _run_sequential(W, inp, 4)
    par = _run_oracle(W, inp, 4)
    np.testing.assert_allclose(seq["logits"][:, 0], par["logits"][:, 0], rtol=1e-12, atol=1e-12)
    assert np.abs(seq["logits"][:, 1:] - par["logits"][:, 1:]).max() > 1e-3


def test_sequential_prefix_consistency_and_forced_tokens():
    W, inp = _tiny_case(K=5)
    full = _run_sequential(W, inp, 5)
    part = _run_sequential(W, inp, 2)
    np.testing.assert_allclose(part["logits"], full["logits"][:, :2], rtol=1e-12, atol=1e-12)
    # forcing the oracle's own drafts changes nothing
    same = _run_sequential(W, inp, 5, tokens=full["drafts"])
    np.testing.assert_array_equal(same["logits"], full["logits"])
    # forcing another token at pass 1 leaves passes 0 and 1 unchanged and moves pass 2
    forced = full["drafts"].copy()
    forced[:, 1] = (forced[:, 1] + 1) % TINY.vocab
    other = _run_sequential(W, inp, 5, tokens=forced)
    np.testing.assert_array_equal(other["logits"][:, :2], full["logits"][:, :2])
    assert np.abs(other["logits"][:, 2] - full["logits"][:, 2]).max() > 1e-6


def test_sequential_cache_rows_are_the_passes_own_rows():
    # the k/v rows pass j writes are those the torch restatement appends: check
    # through the next pass, which must see them (perturbing one changes it)
    W, inp = _tiny_case(K=3)
    out = _run_sequential(W, inp, 3)
    assert out["k_new"].shape == (4, 2, 3, TINY.n_kv_heads, TINY.head_dim)
    # pass 0's rows equal the parallel pass's row 0
    par = _run_oracle(W, inp, 3)
    np.testing.assert_allclose(out["k_new"][:, :, 0], par["k_new"][:, :, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["v_new"][:, :, 0], par["v_new"][:, :, 0], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------- FP8 weights

def test_e4m3_decode_matches_torch_float8_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert nan.sum() == 2                                    # 0x7F and 0xFF


def test_e4m3_decode_special_values():
    d = oracle.e4m3_decode(np.array([0x00, 0x80, 0x01, 0x07, 0x08, 0x38, 0x7E, 0xFE, 0x7F], dtype=np.uint8))
    np.testing.assert_array_equal(d[:8], [0.0, -0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 448.0, -448.0])
    assert np.signbit(d[1]) and np.isnan(d[8])
    assert oracle.E4M3_MAX == 448.0


def test_dequant_rows_scales_each_output_row():
    rng = np.random.default_rng(12)
    q = rng.integers(0, 256, size=(5, 9), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C                             # no NaN codes
    sc = rng.uniform(0.001, 2.0, size=5)
    ref = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy() * sc[:, None]
    np.testing.assert_array_equal(oracle.dequant_rows(q, sc), ref)


def test_fp8_weight_recipe_round_trips_within_e4m3_precision():
    # the synthetic FP8 weights decode to within half an E4M3 step of the
    # bf16 weights they were made from, and each row's largest magnitude maps
    # to 448 exactly
    W = synth.make_weights(TINY, 3)
    Wq, sc = synth.quantize_weights_fp8(W)
    Wn, Sn = synth.fp8_to_numpy(Wq, sc)
    Wd = oracle.dequant_weights(Wn, Sn)
    for name, w0, wd, s in [("fc", W["fc"], Wd["fc"], Sn["fc"]),
                            ("w_down", W["layers"][2]["w_down"], Wd["layers"][2]["w_down"],
                             Sn["layers"][2]["w_down"])]:
        w0 = w0.double().numpy()
        rel = np.abs(wd - w0) / np.maximum(np.abs(w0), 2.0 ** -6 * s[:, None])
        assert rel.max() <= 2.0 ** -4 + 1e-12, name
        np.testing.assert_allclose(np.abs(wd).max(axis=1), np.abs(w0).max(axis=1), rtol=1e-6)
    assert Wq["embed"] is W["embed"] and Wq["layers"][0]["norm_e"] is W["layers"][0]["norm_e"]


def test_fp8_draft_pass_is_the_draft_pass_on_dequantised_weights():
    # the oracle's FP8 drafter is its ordinary drafter on W = decode(q) * s;
    # the K=1 torch restatement confirms it on those weights
    W, inp = _tiny_case(K=3)
    Wq, sc = synth.quantize_weights_fp8(W)
    Wn, Sn = synth.fp8_to_numpy(Wq, sc)
    Wd = oracle.dequant_weights(Wn, Sn)
    out = oracle.draft_pass(TINY, Wd, inp.last_token.numpy(), inp.target_hidden.double().numpy(),
                            inp.positions.numpy(), inp.seq_lens.numpy(), inp.page_table.numpy(),
                            inp.k_cache.double().numpy(), inp.v_cache.double().numpy(), 3)
    Wt = {k: (torch.from_numpy(np.asarray(v)) if v is not None and k != "layers" else v) for k, v in Wd.items()}
    Wt["layers"] = [{k: (torch.from_numpy(np.asarray(v)) if v is not None else None) for k, v in L.items()}
                    for L in Wd["layers"]]
    ref = _torch_reference_pass(Wt, inp, 3)
    np.testing.assert_allclose(out["logits"], ref, rtol=1e-10, atol=1e-10)
    base = _run_oracle(W, inp, 3)
    assert np.abs(out["logits"] - base["logits"]).max() > 1e-6    # quantisation moved the logits


# --------------------------------------------------------------- re-fed real rows

def _torch_refeed(W, tokens, n_real, th, positions, seq_lens, page_table, kc, vc, K):
    """Independent float64 restatement of the re-fed pass: per request a list
    of n_b real rows (token embedding, FC of its target hidden state) and K-1
    placeholder rows, causal SDPA over the page-table walk of the committed
    entries followed by the rows, logits of the last real row and of every
    placeholder."""
    cfg = TINY
    d = torch.float64
    t = lambda a: torch.as_tensor(a).to(d)
    H, nq, nkv, hd = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    G = nq // nkv

    def norm(x, g):
        return F.rms_norm(x, (x.shape[-1],), weight=t(g), eps=cfg.rms_eps)

    def rope(x, pos):
        half = hd // 2
        inv = cfg.rope_theta ** (-(torch.arange(half, dtype=d) * 2.0) / hd)
        ang = pos.to(d)[..., None] * inv
        z = torch.complex(x[..., :half], x[..., half:]) * torch.polar(torch.ones_like(ang), ang)
        return torch.cat([z.real, z.imag], dim=-1)

    B = len(n_real)
    L0 = W["layers"][0]
    logits = torch.empty(B, K, cfg.vocab, dtype=d)
    T_max = int(max(n_real)) + K - 1
    k_rows = torch.full((4, B, T_max, nkv, hd), float("nan"), dtype=d)
    v_rows = torch.full((4, B, T_max, nkv, hd), float("nan"), dtype=d)
    for b in range(B):
        n = int(n_real[b])
        T = n + K - 1
        rows_e = [t(W["embed"][int(tokens[b, i])]) for i in range(n)] + [t(W["emb_mask"])] * (K - 1)
        rows_h = [F.linear(t(th[b, i]), t(W["fc"])) for i in range(n)] + [t(W["h_shared"])] * (K - 1)
        x = torch.cat([norm(torch.stack(rows_e), L0["norm_e"]), norm(torch.stack(rows_h), L0["norm_h"])], -1)
        r = torch.stack(rows_h).clone()
        S = int(seq_lens[b])
        pos = int(positions[b]) + torch.arange(T)
        for li, Lw in enumerate(W["layers"]):
            if li > 0:
                x = norm(r, Lw["attn_norm"])
            qkv = F.linear(x, t(Lw["w_qkv"]))
            q = rope(qkv[:, : nq * hd].reshape(T, nq, hd), pos[:, None])
            k = rope(qkv[:, nq * hd:(nq + nkv) * hd].reshape(T, nkv, hd), pos[:, None])
            v = qkv[:, (nq + nkv) * hd:].reshape(T, nkv, hd)
            k_rows[li, b, :T], v_rows[li, b, :T] = k, v
            ks = [t(kc[li, int(page_table[b, e // 16]), :, e % 16, :]) for e in range(S)]
            vs = [t(vc[li, int(page_table[b, e // 16]), :, e % 16, :]) for e in range(S)]
            k_all = torch.cat([torch.stack(ks), k]) if S else k
            v_all = torch.cat([torch.stack(vs), v]) if S else v
            mask = torch.arange(S + T)[None, :] <= (S + torch.arange(T))[:, None]
            a = F.scaled_dot_product_attention(
                q.permute(1, 0, 2)[None], k_all.permute(1, 0, 2).repeat_interleave(G, 0)[None],
                v_all.permute(1, 0, 2).repeat_interleave(G, 0)[None], attn_mask=mask)
            r = r + F.linear(a[0].permute(1, 0, 2).reshape(T, nq * hd), t(Lw["w_o"]))
            x = norm(r, Lw["mlp_norm"])
            r = r + F.linear(F.silu(F.linear(x, t(Lw["w_gate"]))) * F.linear(x, t(Lw["w_up"])), t(Lw["w_down"]))
        logits[b] = F.linear(norm(r[n - 1:], W["final_norm"]), t(W["lm_head"]))
    return dict(logits=logits.numpy(), k_new=k_rows.numpy(), v_new=v_rows.numpy())


def _refeed_case(K, n_real, seed=14):
    B = len(n_real)
    n_max = max(n_real)
    wl = synth.Workload("pin-refeed", TINY, B, K, (10, 40), (0.7, 0.7), seed)
    W = synth.make_weights(TINY, seed)
    inp = synth.make_step_inputs(wl, K=n_max + K)      # pages for the real rows and the placeholders
    rng = np.random.default_rng(seed)
    tokens = rng.integers(0, TINY.vocab, size=(B, n_max))
    th = torch.randn(B, n_max, 3 * TINY.hidden, generator=torch.Generator().manual_seed(seed), dtype=torch.float64)
    return W, inp, tokens, np.asarray(n_real), th


def _run_refeed(W, inp, tokens, n_real, th, K):
    return oracle.draft_pass_refeed(TINY, synth.weights_to_numpy(W), tokens, n_real, th.numpy(),
                                    inp.positions.numpy(), inp.seq_lens.numpy(), inp.page_table.numpy(),
                                    inp.k_cache.double().numpy(), inp.v_cache.double().numpy(), K)


def test_refeed_matches_independent_torch_restatement():
    K = 3
    W, inp, tokens, n_real, th = _refeed_case(K, [3, 1, 4])
    out = _run_refeed(W, inp, tokens, n_real, th, K)
    ref = _torch_refeed(W, tokens, n_real, th.numpy(), inp.positions.numpy(), inp.seq_lens.numpy(),
                        inp.page_table.numpy(), inp.k_cache.double().numpy(), inp.v_cache.double().numpy(), K)
    np.testing.assert_allclose(out["logits"], ref["logits"], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["k_new"], ref["k_new"], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(out["v_new"], ref["v_new"], rtol=1e-10, atol=1e-10)
    assert np.isnan(out["k_new"][:, 1, 1 + K - 1:]).all() and not np.isnan(out["k_new"][:, 2]).any()


def test_refeed_with_one_real_row_is_the_parallel_pass():
    K = 4
    W, inp, tokens, n_real, th = _refeed_case(K, [1, 1])
    out = _run_refeed(W, inp, tokens, n_real, th, K)
    par = oracle.draft_pass(TINY, synth.weights_to_numpy(W), tokens[:, 0], th[:, 0].numpy(), inp.positions.numpy(),
                            inp.seq_lens.numpy(), inp.page_table.numpy(), inp.k_cache.double().numpy(),
                            inp.v_cache.double().numpy(), K)
    np.testing.assert_allclose(out["logits"], par["logits"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["k_new"], par["k_new"], rtol=1e-12, atol=1e-12)


def test_refeed_real_rows_are_causal_and_placeholders_see_them():
    K = 3
    W, inp, tokens, n_real, th = _refeed_case(K, [3, 2])
    base = _run_refeed(W, inp, tokens, n_real, th, K)
    # another first real token moves every draft; another last real token
    # moves the drafts but not the first real row's cache rows
    t2 = tokens.copy()
    t2[:, 0] = (t2[:, 0] + 1) % TINY.vocab
    moved = _run_refeed(W, inp, t2, n_real, th, K)
    assert (np.abs(moved["logits"] - base["logits"]).max(axis=-1) > 1e-6).all()
    t3 = tokens.copy()
    t3[0, 2] = (t3[0, 2] + 1) % TINY.vocab
    moved3 = _run_refeed(W, inp, t3, n_real, th, K)
    np.testing.assert_array_equal(moved3["k_new"][:, 0, :2], base["k_new"][:, 0, :2])
    np.testing.assert_array_equal(moved3["logits"][1], base["logits"][1])     # other request untouched


def test_refeed_rebuild_against_explicit_slot_lists():
    rng = np.random.default_rng(15)
    P = 16
    for trial in range(200):
        B, K = 4, int(rng.integers(1, 12))
        S = rng.integers(0, 100, size=B)
        Q = S + rng.integers(0, 30, size=B)
        n = rng.integers(1, K + 2, size=B)
        max_pages = int(np.ceil((S.max() + 4 * K + 2) / P)) + int(rng.integers(0, 2))
        num_pages = B * max_pages + 3
        pt = rng.permutation(num_pages)[: B * max_pages].reshape(B, max_pages)
        a = rng.integers(0, K + 1, size=B)
        out = oracle.rebuild_metadata_refeed(a, K, n, S, Q, pt, num_pages, P)
        for b in range(B):
            slots = np.concatenate([p * P + np.arange(P) for p in pt[b]])
            assert out["status"][b] == oracle.REQ_OK
            assert out["seq_lens"][b] == S[b] + n[b] and out["positions"][b] == Q[b] + n[b]
            assert out["n_real"][b] == a[b] + 1
            m = a[b] + K
            np.testing.assert_array_equal(out["slot_mapping"][b, :m], slots[S[b] + n[b]: S[b] + n[b] + m])
            assert (out["slot_mapping"][b, m:] == -1).all()
            np.testing.assert_array_equal(out["rollback_slots"][b, :K - 1], slots[S[b] + n[b]: S[b] + n[b] + K - 1])
            assert (out["rollback_slots"][b, K - 1:] == -1).all()


def test_refeed_rebuild_status_cases():
    P, K = 16, 3
    pt = np.array([[0, 1], [2, 3], [4, -1], [5, 6]])
    S = np.array([20, 5, 10, -2])
    Q = np.array([30, 30, 12, 4])
    n = np.array([4, 1, 2, 1])
    a = np.array([3, 0, 3, 0])
    out = oracle.rebuild_metadata_refeed(a, K, n, S, Q, pt, num_pages=7, page_size=P)
    # 0: S'=24, next rows 4 + 2 = 6 -> 30 <= 32 fits; 1: fits; 2: S'=12, 4 + 2 rows reach entry 17 -> page -1
    np.testing.assert_array_equal(out["status"], [oracle.REQ_OK, oracle.REQ_OK, oracle.REQ_BAD_PAGE,
                                                  oracle.REQ_BAD_INPUT])
    out2 = oracle.rebuild_metadata_refeed(np.array([3]), K, np.array([4]), np.array([25]), np.array([30]),
                                          pt[:1], 7, P)
    assert out2["status"][0] == oracle.REQ_CAPACITY                   # 29 + 4 + 2 = 35 > 32
    np.testing.assert_array_equal(out["n_real"][2:], n[2:])


# --------------------------------------------------------------- sampling and stochastic acceptance

def test_inverse_cdf_on_a_grid_of_uniforms():
    w = np.array([0.2, 0.0, 0.5, 0.3])
    for u, want in [(0.0, 0), (0.1999, 0), (0.2001, 2), (0.6999, 2), (0.7001, 3), (0.9999, 3)]:
        i, m = oracle.sample_inverse_cdf(w, u)
        assert i == want, (u, i)
        assert m >= 0.0
    i, m = oracle.sample_inverse_cdf(w * 7.0, 0.45)          # weights need not be normalised
    assert i == 2 and abs(m - 0.25) < 1e-12                  # 0.45 is 0.25 from both 0.2 and 0.7


def test_sampled_drafts_follow_the_tempered_softmax():
    rng = np.random.default_rng(16)
    logits = rng.normal(size=(1, 1, 6)) * 2.0
    T = 0.7
    n = 100_000
    u = rng.random(n)
    d = np.array([oracle.sample_inverse_cdf(oracle.softmax_t(logits[0, 0], T), x)[0] for x in u])
    p = oracle.softmax_t(logits[0, 0], T)
    freq = np.bincount(d, minlength=6) / n
    assert (np.abs(freq - p) < 4 * np.sqrt(p * (1 - p) / n) + 1e-12).all()
    ref = torch.softmax(torch.tensor(logits[0, 0]) / T, dim=0).numpy()
    np.testing.assert_allclose(p, ref, rtol=1e-13)


def _spec_case(rng, K, V, B):
    dl = rng.normal(size=(B, K, V)) * 1.5
    tl = rng.normal(size=(B, K + 1, V)) * 1.5
    return dl, tl


def test_speculative_sampling_emits_the_target_distribution():
    # The first emitted token (the accepted draft d_0 or the draw at the
    # first rejection) is distributed as p_0, whatever q_0 is; the acceptance
    # rate of position 0 is sum_x min(p_0(x), q_0(x)).
    rng = np.random.default_rng(17)
    K, V, n = 3, 6, 100_000
    dl, tl = _spec_case(rng, K, V, 1)
    T = 0.9
    dl_b, tl_b = np.repeat(dl, n, 0), np.repeat(tl, n, 0)
    d, _ = oracle.sample_drafts(dl_b, T, rng.random((n, K)))
    out = oracle.verify_stochastic(d, dl_b, tl_b, T, rng.random((n, K)), rng.random(n))
    first = out["emitted"][:, 0]
    p0 = oracle.softmax_t(tl[0, 0], T)
    q0 = oracle.softmax_t(dl[0, 0], T)
    freq = np.bincount(first, minlength=V) / n
    assert (np.abs(freq - p0) < 4 * np.sqrt(p0 * (1 - p0) / n) + 1e-12).all(), (freq, p0)
    acc = (out["accepted"] >= 1).mean()
    want = np.minimum(p0, q0).sum()
    assert abs(acc - want) < 4 * np.sqrt(want * (1 - want) / n)
    assert ((out["accepted"] >= 0) & (out["accepted"] <= K)).all()


def test_stochastic_acceptance_with_q_equal_p_accepts_everything():
    rng = np.random.default_rng(18)
    K, V, B = 4, 9, 500
    dl, _ = _spec_case(rng, K, V, B)
    tl = np.concatenate([dl, rng.normal(size=(B, 1, V))], axis=1)
    d, _ = oracle.sample_drafts(dl, 1.3, rng.random((B, K)))
    out = oracle.verify_stochastic(d, dl, tl, 1.3, rng.random((B, K)), rng.random(B))
    assert (out["accepted"] == K).all()
    np.testing.assert_array_equal(out["emitted"][:, :K], d)


def test_stochastic_acceptance_at_low_temperature_is_greedy_acceptance():
    # T -> 0: every softmax becomes the one-hot of its argmax, the sampled
    # drafts are the argmax drafts and the rule reduces to the greedy one:
    # longest prefix with d == g, then the target's argmax token.
    rng = np.random.default_rng(19)
    K, V, B = 5, 40, 300
    dl, tl = _spec_case(rng, K, V, B)
    # every row's argmax leads its runner-up by at least 1 (one-hot at T = 1e-3)
    for arr in (dl, tl):
        flat = arr.reshape(-1, V)
        flat[np.arange(len(flat)), flat.argmax(-1)] += 1.0
    agree = rng.random((B, K)) < 0.6                          # plant agreement on the argmax
    for b in range(B):
        for j in range(K):
            if agree[b, j]:
                tl[b, j, np.argmax(dl[b, j])] = tl[b, j].max() + 1.0
    T = 1e-3
    d, _ = oracle.sample_drafts(dl, T, rng.random((B, K)))
    np.testing.assert_array_equal(d, dl.argmax(-1))
    out = oracle.verify_stochastic(d, dl, tl, T, rng.random((B, K)), rng.random(B))
    g = tl.argmax(-1)
    a, bonus = oracle.verify(d, g)
    np.testing.assert_array_equal(out["accepted"], a)
    np.testing.assert_array_equal(out["final"], bonus)


# --------------------------------------------------------------- verify / rebuild

def _brute_accept(d, g):
    K = len(d)
    return max(n for n in range(K + 1) if all(d[i] == g[i] for i in range(n)))


def test_verify_brute_force_tiny_vocab():
    V, K = 3, 3
    ds = np.array(list(itertools.product(range(V), repeat=K)))
    gs = np.array(list(itertools.product(range(V), repeat=K + 1)))
    D = np.repeat(ds, len(gs), axis=0)
    G = np.tile(gs, (len(ds), 1))
    a, bonus = oracle.verify(D, G)
    for i in range(len(D)):
        ai = _brute_accept(D[i], G[i])
        assert a[i] == ai and bonus[i] == G[i, ai]
        assert 0 <= a[i] <= K


def test_full_acceptance_gives_bonus_and_k_plus_1_tokens():
    d = np.array([[4, 8, 15, 16]])
    g = np.array([[4, 8, 15, 16, 23]])
    a, bonus = oracle.verify(d, g)
    assert a[0] == 4 and bonus[0] == 23
    em = oracle.emitted_tokens(d, a, bonus)
    np.testing.assert_array_equal(em[0], [4, 8, 15, 16, 23])
    a0, b0 = oracle.verify(d, np.array([[5, 8, 15, 16, 23]]))
    assert a0[0] == 0 and b0[0] == 5
    np.testing.assert_array_equal(oracle.emitted_tokens(d, a0, b0)[0], [5, -1, -1, -1, -1])


def test_rebuild_against_explicit_slot_lists():
    rng = np.random.default_rng(8)
    P = 16
    for trial in range(200):
        B, K = 4, int(rng.integers(1, 12))
        S = rng.integers(0, 100, size=B)
        Q = S + rng.integers(0, 30, size=B)
        max_pages = int(np.ceil((S.max() + 2 * K) / P)) + int(rng.integers(0, 2))
        num_pages = B * max_pages + 3
        pt = rng.permutation(num_pages)[: B * max_pages].reshape(B, max_pages)
        a = rng.integers(0, K + 1, size=B)
        out = oracle.rebuild_metadata(a, K, S, Q, pt, num_pages, P)
        for b in range(B):
            slots = np.concatenate([p * P + np.arange(P) for p in pt[b]])   # entry -> slot
            kept = min(a[b], K - 1) + 1
            assert out["status"][b] == oracle.REQ_OK
            assert S[b] + 1 <= out["seq_lens"][b] == S[b] + kept <= S[b] + K
            assert out["positions"][b] - Q[b] == a[b] + 1
            np.testing.assert_array_equal(out["slot_mapping"][b], slots[out["seq_lens"][b]: out["seq_lens"][b] + K])
            rb = out["rollback_slots"][b]
            n_rb = K - kept
            np.testing.assert_array_equal(rb[:n_rb], slots[S[b] + kept: S[b] + K])
            assert (rb[n_rb:] == -1).all()
            assert set(rb[:n_rb]) <= set(out["slot_mapping"][b])


def test_rebuild_capacity_and_bad_page_status():
    P, K = 16, 4
    pt = np.array([[0, 1], [2, 3], [4, -1]])
    S = np.array([27, 28, 10])
    Q = np.array([30, 30, 12])
    a = np.array([1, 1, 3])           # kept 2, 2, 4 -> S' = 29, 30, 14
    out = oracle.rebuild_metadata(a, K, S, Q, pt, num_pages=5, page_size=P)
    # request 0: S'+K = 33 > 32 -> capacity; request 1 likewise; request 2: entries 14..17
    # need page index 1 of its table, which is -1 -> bad page.
    np.testing.assert_array_equal(out["status"], [oracle.REQ_CAPACITY, oracle.REQ_CAPACITY, oracle.REQ_BAD_PAGE])
    np.testing.assert_array_equal(out["seq_lens"], S)
    np.testing.assert_array_equal(out["positions"], Q)
    assert (out["slot_mapping"] == -1).all() and (out["rollback_slots"] == -1).all()
    out2 = oracle.rebuild_metadata(np.array([0, 0, 0]), K, np.array([27, 0, 0]), Q, pt, 5, P)
    assert out2["status"][0] == oracle.REQ_OK            # 28 + 4 = 32 fits exactly
    np.testing.assert_array_equal(out2["slot_mapping"][0], [1 * P + 12, 1 * P + 13, 1 * P + 14, 1 * P + 15])


def test_rebuild_bad_input_status_on_out_of_range_lengths():
    # Negative lengths or positions, or values too close to 2^31 - 1 for the
    # next step's K entries, are rejected before any slot arithmetic.
    P, K = 16, 3
    lim = 2 ** 31 - 1 - 2 * K
    pt = np.array([[0, 1], [2, 3], [4, 5], [6, 7], [8, 9]])
    S = np.array([-1, 5, lim + 1, 5, 5])
    Q = np.array([7, -3, 7, lim + 1, 9])
    out = oracle.rebuild_metadata(np.array([1, 1, 1, 1, 1]), K, S, Q, pt, num_pages=10, page_size=P)
    np.testing.assert_array_equal(out["status"], [oracle.REQ_BAD_INPUT] * 4 + [oracle.REQ_OK])
    np.testing.assert_array_equal(out["seq_lens"][:4], S[:4])
    np.testing.assert_array_equal(out["positions"][:4], Q[:4])
    assert (out["slot_mapping"][:4] == -1).all() and (out["rollback_slots"][:4] == -1).all()
    assert out["seq_lens"][4] == 7 and out["positions"][4] == 11


# --------------------------------------------------------------- acceptance statistics

@pytest.mark.parametrize("alpha,K", [(0.7, 3), (0.55, 7), (0.3, 11), (0.8, 11), (0.6, 1)])
def test_planted_alpha_mean_tokens_matches_closed_form(alpha, K):
    n, V = 200_000, 1000
    rng = np.random.default_rng(9)
    d = rng.integers(0, V, size=(n, K))
    g = synth.plant_targets(d, np.full(n, alpha), V, seed=int(alpha * 100) + K)
    a, _ = oracle.verify(d, g)
    tokens = a + 1
    mean, sem = tokens.mean(), tokens.std(ddof=1) / np.sqrt(n)
    exact = oracle.expected_tokens_iid(alpha, K)
    assert abs(mean - exact) < 4 * sem
    # the lesson page's 1 + K*alpha bounds it from above, with equality at K = 1
    assert exact <= oracle.tokens_per_pass_linear(alpha, K) + 1e-12
    if K == 1:
        assert abs(exact - oracle.tokens_per_pass_linear(alpha, K)) < 1e-12


def test_expected_tokens_closed_form_by_enumeration():
    # E[a+1] = sum_a (a+1) P(a) with P(a) = alpha^a (1-alpha) for a<K, alpha^K for a=K.
    for alpha in (0.0, 0.3, 0.55, 0.8, 1.0):
        for K in range(1, 13):
            e = sum((a + 1) * alpha ** a * (1 - alpha) for a in range(K)) + (K + 1) * alpha ** K
            assert abs(oracle.expected_tokens_iid(alpha, K) - e) < 1e-12


def test_lesson_page_worked_example():
    with open(os.path.join(GOLDEN, "lesson_worked_example.json")) as f:
        gold = json.load(f)
    ex = gold["speedup_example"]
    assert abs(oracle.tokens_per_pass_linear(ex["alpha"], ex["K"]) - ex["tokens_per_pass"]) < 1e-12
    s = oracle.speedup_linear(ex["alpha"], ex["K"], ex["overhead"])
    assert abs(s - ex["speedup_fraction"][0] / ex["speedup_fraction"][1]) < 1e-12
    assert round(s, 1) == ex["speedup_printed"]
    be = gold["breakeven_example"]
    assert abs(oracle.breakeven_alpha(be["overhead"], be["K"]) - be["alpha_breakeven"]) < 1e-12
    assert abs(oracle.speedup_linear(be["alpha_breakeven"], be["K"], be["overhead"]) - 1.0) < 1e-12
