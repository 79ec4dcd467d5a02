"""Helpers for GPU-vs-oracle parity tests (test plumbing, no method arithmetic).

Tolerance rules (bf16 path vs float64 oracle; the logit and draft rules are the
stated parity bar of the method: 2e-2 relative on pre-argmax logits, drafts
compared where the top-2 gap exceeds 1e-2):
  * logits: per row, max_v |l_gpu - l_ref| <= 2e-2 * max_v |l_ref|;
  * drafts: equal wherever the oracle's top-2 logit gap exceeds 1e-2;
  * new KV rows: per row (all kv heads of one layer), the same 2e-2 rule;
  * acceptance, bonus, metadata: bit-exact.
"""

import numpy as np
import torch

import oracle
from speculative_drafting_pe_gb300 import synth

LOGIT_RTOL = 2e-2
GAP_MIN = 1e-2


def weights_to(W, dev):
    out = {k: v.to(dev) for k, v in W.items() if k != "layers"}
    out["layers"] = [{k: (v.to(dev) if v is not None else None) for k, v in L.items()} for L in W["layers"]]
    return out


def request_subproblem(inp, b, layers=None):
    """Inputs of request b alone, with a compact cache holding only its pages
    (host float64 arrays for the oracle) and the map page -> compact index."""
    pt = inp.page_table[b].cpu().numpy()
    used = pt[pt >= 0]
    remap = {int(p): i for i, p in enumerate(used)}
    idx = torch.as_tensor(used, dtype=torch.long, device=inp.k_cache.device)
    kc = inp.k_cache.index_select(1, idx).cpu().double().numpy()
    vc = inp.v_cache.index_select(1, idx).cpu().double().numpy()
    pt_c = np.array([[remap[int(p)] if p >= 0 else -1 for p in pt]])
    return dict(last_token=inp.last_token[b:b + 1].cpu().numpy(),
                target_hidden=inp.target_hidden[b:b + 1].cpu().double().numpy(),
                positions=inp.positions[b:b + 1].cpu().numpy(),
                seq_lens=inp.seq_lens[b:b + 1].cpu().numpy(),
                page_table=pt_c, k_cache=kc, v_cache=vc)


def oracle_request(shape, Wn, inp, b, K):
    sp = request_subproblem(inp, b)
    return oracle.draft_pass(shape, Wn, sp["last_token"], sp["target_hidden"], sp["positions"],
                             sp["seq_lens"], sp["page_table"], sp["k_cache"], sp["v_cache"], K)


def oracle_batch(shape, Wn, inp, K):
    return oracle.draft_pass(shape, Wn, inp.last_token.cpu().numpy(), inp.target_hidden.cpu().double().numpy(),
                             inp.positions.cpu().numpy(), inp.seq_lens.cpu().numpy(),
                             inp.page_table.cpu().numpy(), inp.k_cache.cpu().double().numpy(),
                             inp.v_cache.cpu().double().numpy(), K)


def assert_logits_close(lg, ref_lg, what="logits"):
    lg = np.asarray(lg, dtype=np.float64)
    err = np.abs(lg - ref_lg).max(axis=-1)
    scale = np.abs(ref_lg).max(axis=-1)
    bad = err > LOGIT_RTOL * scale
    assert not bad.any(), f"{what}: rows {np.argwhere(bad).tolist()} err {err[bad]} scale {scale[bad]}"
    return float((err / np.maximum(scale, 1e-30)).max())


def assert_drafts_match(d, ref):
    d = np.asarray(d)
    ok = ref["gap"] > GAP_MIN
    mism = (d != ref["drafts"]) & ok
    assert not mism.any(), f"drafts differ where gap > {GAP_MIN}: {np.argwhere(mism).tolist()}"
    return int(ok.sum())


def read_new_kv(inp, kc_dev, vc_dev, b, K, page_size=16):
    """The rows the pass wrote for request b: [L, K, nkv, hd] for k and v."""
    S = int(inp.seq_lens[b])
    pt = inp.page_table[b].cpu().numpy()
    ks, vs = [], []
    for j in range(K):
        e = S + j
        page, off = int(pt[e // page_size]), e % page_size
        ks.append(kc_dev[:, page, :, off, :].double().cpu().numpy())
        vs.append(vc_dev[:, page, :, off, :].double().cpu().numpy())
    return np.stack(ks, axis=1), np.stack(vs, axis=1)


def assert_kv_close(got, ref, what):
    # got/ref [L, K, nkv, hd]; rule applied per (layer, row)
    L, K = got.shape[:2]
    g = got.reshape(L, K, -1)
    r = ref.reshape(L, K, -1)
    err = np.abs(g - r).max(axis=-1)
    scale = np.abs(r).max(axis=-1)
    bad = err > LOGIT_RTOL * scale
    assert not bad.any(), f"{what}: (layer,row) {np.argwhere(bad).tolist()} err {err[bad]} scale {scale[bad]}"
