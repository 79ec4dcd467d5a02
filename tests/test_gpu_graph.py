"""The step graph (draft + verify/rebuild captured once, replayed) and
programmatic dependent launch give the same results as plain launches."""

import os

import numpy as np
import pytest
import torch

import oracle
from speculative_drafting_pe_gb300 import binding, synth

from parity import weights_to

pytestmark = pytest.mark.gpu

SHAPE = synth.DrafterShape("mini-hd128", 384, 4, 1, 128, 960, 3001)


def _setup(B=3, K=5, seed=31):
    dev = torch.device("cuda")
    wl = synth.Workload("mini", SHAPE, B, K, (40, 300), (0.7, 0.7), seed)
    W = weights_to(synth.make_weights(SHAPE, seed), dev)
    inp = synth.make_step_inputs(wl, device=dev)
    return dev, wl, W, inp


def test_step_graph_matches_direct_calls():
    dev, wl, W, inp = _setup()
    K = wl.K
    dr = binding.Drafter(SHAPE, W, max_batch=wl.B, k_max=K)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                     inp.num_pages, kc, vc, K)
    torch.cuda.synchronize()
    g = torch.as_tensor(synth.plant_targets(d.cpu().numpy(), inp.alpha, SHAPE.vocab, 31), device=dev)
    ref = binding.verify_rebuild(d, g, inp.page_table, inp.num_pages, inp.positions, inp.seq_lens)
    torch.cuda.synchronize()

    kc2, vc2 = inp.k_cache.clone(), inp.v_cache.clone()
    sg = dr.step_graph(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                       inp.num_pages, kc2, vc2, K, g)
    for _ in range(3):
        sg.launch()
    torch.cuda.synchronize()
    o = sg.out
    assert torch.equal(o["drafts"], d)
    for k in ("accepted", "bonus", "emitted", "slot_mapping", "rollback_slots", "status", "positions", "seq_lens"):
        assert torch.equal(o[k], ref[k]), k
    assert torch.equal(kc2, kc) and torch.equal(vc2, vc)
    assert sg.launch_count() == dr.launch_count() + 1
    assert dr.device_errors() == 0


def test_step_graph_in_place_metadata_advances_like_direct_steps():
    dev, wl, W, inp = _setup(B=2, K=4, seed=32)
    K = wl.K
    dr = binding.Drafter(SHAPE, W, max_batch=wl.B, k_max=K)
    # two direct steps, metadata updated in place
    pos, sl = inp.positions.clone(), inp.seq_lens.clone()
    g = torch.full((wl.B, K + 1), 7, dtype=torch.int32, device=dev)   # fixed targets
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    for _ in range(2):
        d, _ = dr.draft(inp.last_token, inp.target_hidden, pos, sl, inp.page_table, inp.num_pages, kc, vc, K)
        binding.verify_rebuild(d, g, inp.page_table, inp.num_pages, pos, sl, positions_out=pos, seq_lens_out=sl)
    torch.cuda.synchronize()
    # the same two steps as graph replays over aliased metadata buffers
    pos2, sl2 = inp.positions.clone(), inp.seq_lens.clone()
    kc2, vc2 = inp.k_cache.clone(), inp.v_cache.clone()
    sg = dr.step_graph(inp.last_token, inp.target_hidden, pos2, sl2, inp.page_table, inp.num_pages, kc2, vc2, K, g,
                       positions_out=pos2, seq_lens_out=sl2)
    sg.launch()
    sg.launch()
    torch.cuda.synchronize()
    assert torch.equal(pos2, pos) and torch.equal(sl2, sl)
    assert torch.equal(kc2, kc) and torch.equal(vc2, vc)
    # the metadata advanced by accepted + 1 positions per step
    d_np = sg.out["drafts"].cpu().numpy()
    a, _ = oracle.verify(d_np, g.cpu().numpy())
    assert (pos2.cpu().numpy() - inp.positions.cpu().numpy() >= 2).all()
    assert (sl2.cpu().numpy() > inp.seq_lens.cpu().numpy()).all()


def test_pdl_on_and_off_give_identical_results(monkeypatch):
    dev, wl, W, inp = _setup(B=4, K=7, seed=33)
    outs = []
    for flag in ("1", "0"):
        monkeypatch.setenv("PE_PDL", flag)
        dr = binding.Drafter(SHAPE, W, max_batch=wl.B, k_max=wl.K)
        kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
        lg = torch.empty(wl.B, wl.K, SHAPE.vocab, device=dev)
        d, st = dr.draft(inp.last_token, inp.target_hidden, inp.positions, inp.seq_lens, inp.page_table,
                         inp.num_pages, kc, vc, wl.K, logits=lg)
        torch.cuda.synchronize()
        outs.append((d.clone(), lg.clone(), kc))
        dr.close()
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][2], outs[1][2])
