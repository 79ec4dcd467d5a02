"""GPU parity for sampled drafting (pe_sample_drafts) and speculative-sampling
acceptance (pe_verify_stochastic) against the oracle.

Floating point decides integers here (which index an inverse-CDF draw lands
on, whether u < p/q): the oracle (float64) reports each decision's margin,
and draws are compared exactly wherever that margin exceeds MARGIN; closer
calls are checked for validity only (a drawn index of positive weight)."""

import numpy as np
import pytest
import torch

import oracle
from speculative_drafting_pe_gb300 import binding, synth

from parity import weights_to

pytestmark = pytest.mark.gpu

MARGIN = 5e-6          # well above float32 rounding of the GPU's ordered sums (~1e-7 of the total)
TINY_V = synth.DrafterShape("stoch", 256, 4, 2, 64, 512, 5000)


def _drafter(shape, B, K):
    dev = torch.device("cuda")
    W = weights_to(synth.make_weights(shape, 81), dev)
    return binding.Drafter(shape, W, max_batch=B, k_max=K)


def _logits(B, K, V, seed, scale=2.0, extra=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(B, K + extra, V, generator=g, device="cuda") * scale


@pytest.mark.parametrize("V,T", [(5000, 1.0), (5000, 0.3), (151936, 0.3)])   # 0.3: the pages' temperature
def test_sample_drafts_match_oracle(V, T):
    B, K = 6, 5
    shape = synth.DrafterShape("stoch", 256, 4, 2, 64, 512, V)
    dr = _drafter(shape, B, K)
    lg = _logits(B, K, V, 3 + V)
    u = torch.rand(B, K, generator=torch.Generator(device="cuda").manual_seed(5), device="cuda")
    d = dr.sample_drafts(lg, T, u)
    torch.cuda.synchronize()
    ref, margin = oracle.sample_drafts(lg.double().cpu().numpy(), T, u.double().cpu().numpy())
    dn = d.cpu().numpy()
    sure = margin > MARGIN
    assert sure.mean() > 0.6
    np.testing.assert_array_equal(dn[sure], ref[sure])
    assert ((dn >= 0) & (dn < V)).all()


SMALL = synth.DrafterShape("stoch", 256, 4, 2, 64, 512, 128)   # 128 entries, all but the first few masked
MASKED = -1e30


def test_sample_drafts_follow_the_softmax():
    V, T, n = 8, 0.8, 8192
    dr = _drafter(SMALL, n // 8, 8)
    row = torch.full((SMALL.vocab,), MASKED, device="cuda")
    row[:V] = torch.randn(V, device="cuda", generator=torch.Generator(device="cuda").manual_seed(7)) * 1.5
    lg = row.expand(n // 8, 8, SMALL.vocab).contiguous()
    u = torch.rand(n // 8, 8, device="cuda", generator=torch.Generator(device="cuda").manual_seed(8))
    d = dr.sample_drafts(lg, T, u).cpu().numpy().ravel()
    assert (d < V).all()
    p = oracle.softmax_t(row[:V].double().cpu().numpy(), T)
    freq = np.bincount(d, minlength=V) / n
    assert (np.abs(freq - p) < 4 * np.sqrt(p * (1 - p) / n) + 1e-9).all(), (freq, p)


def _verify_inputs(B, K, V, seed, corr=0.8):
    g = torch.Generator(device="cuda").manual_seed(seed)
    dl = torch.randn(B, K, V, generator=g, device="cuda") * 2.0
    noise = torch.randn(B, K + 1, V, generator=g, device="cuda") * 2.0
    tl = noise.clone()
    tl[:, :K] = corr * dl + (1 - corr) * noise[:, :K]       # target close to the drafter: acceptances happen
    ua = torch.rand(B, K, generator=g, device="cuda")
    uf = torch.rand(B, generator=g, device="cuda")
    ud = torch.rand(B, K, generator=g, device="cuda")
    return dl, tl, ua, uf, ud


def _meta_inputs(B, K, seed):
    v = synth.make_verify_inputs(B, K, 1000, (0, 300), 0.5, seed=seed)
    t = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device="cuda")
    return v, t(v["page_table"]), v["num_pages"], t(v["positions"]), t(v["seq_lens"])


@pytest.mark.parametrize("V,T", [(5000, 1.0), (5000, 0.3), (151936, 0.3)])
def test_verify_stochastic_matches_oracle(V, T):
    B, K = 24, 5
    shape = synth.DrafterShape("stoch", 256, 4, 2, 64, 512, V)
    dr = _drafter(shape, B, K)
    dl, tl, ua, uf, ud = _verify_inputs(B, K, V, 11 + V)
    d = dr.sample_drafts(dl, T, ud)
    v, pt, npg, pos, sl = _meta_inputs(B, K, 12)
    out = dr.verify_stochastic(d, dl, tl, T, ua, uf, pt, npg, pos, sl)
    torch.cuda.synchronize()
    dn = d.cpu().numpy()
    ref = oracle.verify_stochastic(dn, dl.double().cpu().numpy(), tl.double().cpu().numpy(), T,
                                   ua.double().cpu().numpy(), uf.double().cpu().numpy())
    sure = ref["margin"] > MARGIN
    assert sure.mean() > 0.6
    a = out["accepted"].cpu().numpy()
    np.testing.assert_array_equal(a[sure], ref["accepted"][sure])
    np.testing.assert_array_equal(out["final"].cpu().numpy()[sure], ref["final"][sure])
    assert 0 < a.mean() < K                                  # the case exercises both outcomes
    # the rebuild follows the GPU's own acceptance exactly
    meta = oracle.rebuild_metadata(a, K, v["seq_lens"], v["positions"], v["page_table"], v["num_pages"])
    for k in ("seq_lens", "positions", "slot_mapping", "rollback_slots", "status"):
        np.testing.assert_array_equal(out[k].cpu().numpy(), meta[k], err_msg=k)
    np.testing.assert_array_equal(out["emitted"].cpu().numpy(),
                                  oracle.emitted_tokens(dn, a, out["final"].cpu().numpy()))


def test_stochastic_acceptance_emits_the_target_distribution_on_gpu():
    # the first emitted token is distributed as p_0 whatever the drafter's q_0
    V, T, K, B = 6, 0.9, 3, 8192
    dr = _drafter(SMALL, B, K)
    g = torch.Generator(device="cuda").manual_seed(21)
    dl = torch.full((1, K, SMALL.vocab), MASKED, device="cuda")
    tl = torch.full((1, K + 1, SMALL.vocab), MASKED, device="cuda")
    dl[..., :V] = torch.randn(1, K, V, generator=g, device="cuda") * 1.5
    tl[..., :V] = torch.randn(1, K + 1, V, generator=g, device="cuda") * 1.5
    dl = dl.expand(B, K, SMALL.vocab).contiguous()
    tl = tl.expand(B, K + 1, SMALL.vocab).contiguous()
    d = dr.sample_drafts(dl, T, torch.rand(B, K, generator=g, device="cuda"))
    v, pt, npg, pos, sl = _meta_inputs(B, K, 22)
    out = dr.verify_stochastic(d, dl, tl, T, torch.rand(B, K, generator=g, device="cuda"),
                               torch.rand(B, generator=g, device="cuda"), pt, npg, pos, sl)
    first = out["emitted"][:, 0].cpu().numpy()
    assert (first < V).all()
    p0 = oracle.softmax_t(tl[0, 0, :V].double().cpu().numpy(), T)
    q0 = oracle.softmax_t(dl[0, 0, :V].double().cpu().numpy(), T)
    freq = np.bincount(first, minlength=V) / B
    assert (np.abs(freq - p0) < 4 * np.sqrt(p0 * (1 - p0) / B) + 1e-9).all(), (freq, p0)
    acc = (out["accepted"].cpu().numpy() >= 1).mean()
    want = np.minimum(p0, q0).sum()
    assert abs(acc - want) < 4 * np.sqrt(want * (1 - want) / B)


def test_stochastic_at_low_temperature_is_the_greedy_verify():
    B, K, V, T = 64, 7, 3000, 1e-3
    shape = synth.DrafterShape("stoch", 256, 4, 2, 64, 512, V)
    dr = _drafter(shape, B, K)
    dl, tl, ua, uf, ud = _verify_inputs(B, K, V, 31, corr=0.0)
    for t_ in (dl, tl):           # every row's argmax leads its runner-up by >= 1
        flat = t_.view(-1, V)
        flat[torch.arange(flat.shape[0]), flat.argmax(-1)] += 1.0
    agree = torch.rand(B, K, device="cuda", generator=torch.Generator(device="cuda").manual_seed(32)) < 0.6
    am = dl.argmax(-1)
    for b in range(B):
        for j in range(K):
            if agree[b, j]:
                tl[b, j, am[b, j]] = tl[b, j].max() + 1.0
    d = dr.sample_drafts(dl, T, ud)
    assert torch.equal(d, am.to(torch.int32))
    v, pt, npg, pos, sl = _meta_inputs(B, K, 33)
    out = dr.verify_stochastic(d, dl, tl, T, ua, uf, pt, npg, pos, sl)
    gtok = tl.argmax(-1).to(torch.int32)
    ref = binding.verify_rebuild(d, gtok, pt, npg, pos, sl)
    torch.cuda.synchronize()
    assert torch.equal(out["accepted"], ref["accepted"])
    assert torch.equal(out["final"], ref["bonus"])
    for k in ("emitted", "slot_mapping", "rollback_slots", "status", "positions", "seq_lens"):
        assert torch.equal(out[k], ref[k]), k


def test_sampled_step_from_the_drafter():
    # pe_draft's logits feed the sampler; failed requests draft -1 throughout
    dev = torch.device("cuda")
    shape, B, K, T = TINY_V, 3, 4, 0.3
    wl = synth.Workload("stoch", shape, B, K, (20, 60), (0.7, 0.7), 34)
    W = weights_to(synth.make_weights(shape, 34), dev)
    inp = synth.make_step_inputs(wl, device=dev)
    inp.page_table[2, 0] = inp.num_pages + 3
    dr = binding.Drafter(shape, W, max_batch=B, k_max=K)
    lg = torch.empty(B, K, shape.vocab, device=dev)
    _, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table, inp.num_pages,
                     inp.k_cache.clone(), inp.v_cache.clone(), K, logits=lg)
    u = torch.rand(B, K, device=dev, generator=torch.Generator(device="cuda").manual_seed(35))
    d = dr.sample_drafts(lg, T, u, status=st)
    torch.cuda.synchronize()
    assert list(st.cpu().numpy()) == [0, 0, binding.PE_REQ_BAD_PAGE]
    dn = d.cpu().numpy()
    assert (dn[2] == -1).all()
    ref, margin = oracle.sample_drafts(lg[:2].double().cpu().numpy(), T, u[:2].double().cpu().numpy())
    sure = margin > MARGIN
    np.testing.assert_array_equal(dn[:2][sure], ref[sure])
    assert dr.device_errors() == 0
