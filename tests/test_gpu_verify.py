"""GPU parity for the fused verify / metadata-rebuild / rollback kernel:
bit-exact against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from speculative_drafting_pe_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def _run(lib, v, K, dev):
    t = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device=dev)
    out = binding.verify_rebuild(t(v["drafts"]), t(v["targets"]), t(v["page_table"]), v["num_pages"],
                                 t(v["positions"]), t(v["seq_lens"]))
    torch.cuda.synchronize()
    return {k: (x.cpu().numpy() if x is not None else None) for k, x in out.items()}


def _expect(v, K):
    a, bonus = oracle.verify(v["drafts"], v["targets"])
    meta = oracle.rebuild_metadata(a, K, v["seq_lens"], v["positions"], v["page_table"], v["num_pages"])
    meta["accepted"], meta["bonus"] = a, bonus
    meta["emitted"] = oracle.emitted_tokens(v["drafts"], a, bonus)
    return meta


def _assert_equal(got, exp):
    for k in ("accepted", "bonus", "emitted", "slot_mapping", "rollback_slots", "status", "positions", "seq_lens"):
        np.testing.assert_array_equal(got[k], exp[k], err_msg=k)


@pytest.mark.parametrize("alpha", synth.VERIFY_STRESS["alphas"])
def test_verify_stress_bit_exact(lib, alpha):
    c = synth.VERIFY_STRESS
    v = synth.make_verify_inputs(c["B"], c["K"], c["vocab"], c["seq_lens"], alpha, c["seed"])
    got = _run(lib, v, c["K"], torch.device("cuda"))
    exp = _expect(v, c["K"])
    _assert_equal(got, exp)
    # acceptance follows the planted rate
    assert abs(got["accepted"].mean() + 1 - oracle.expected_tokens_iid(alpha, c["K"])) < 1.0


@pytest.mark.parametrize("K", [1, 2, 16, 31])
def test_verify_k_range(lib, K):
    v = synth.make_verify_inputs(37, K, 1000, (0, 300), 0.6, seed=11)
    _assert_equal(_run(lib, v, K, torch.device("cuda")), _expect(v, K))


def test_verify_all_accepted_and_none_accepted(lib):
    K = 5
    v = synth.make_verify_inputs(4, K, 50, (10, 40), 0.5, seed=12)
    v["targets"][0, :K] = v["drafts"][0]          # all accepted
    v["targets"][1, 0] = (v["drafts"][1, 0] + 1) % 50   # none accepted
    got = _run(lib, v, K, torch.device("cuda"))
    exp = _expect(v, K)
    _assert_equal(got, exp)
    assert got["accepted"][0] == K and got["bonus"][0] == v["targets"][0, K]
    assert got["accepted"][1] == 0


def test_verify_capacity_and_bad_page(lib):
    K = 4
    v = dict(drafts=np.array([[1, 2, 3, 4]] * 3), targets=np.array([[1, 2, 9, 9, 9]] * 3),
             page_table=np.array([[0, 1], [2, 3], [4, -1]]), num_pages=5,
             seq_lens=np.array([27, 26, 10]), positions=np.array([30, 30, 12]))
    v["targets"][1] = [1, 9, 9, 9, 9]
    got = _run(lib, v, K, torch.device("cuda"))
    exp = _expect(v, K)
    _assert_equal(got, exp)
    assert list(got["status"]) == [oracle.REQ_CAPACITY, oracle.REQ_OK, oracle.REQ_BAD_PAGE]


def test_verify_in_place_metadata(lib):
    K = 7
    v = synth.make_verify_inputs(64, K, 3000, (100, 900), 0.7, seed=13)
    dev = torch.device("cuda")
    t = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device=dev)
    pos, sl = t(v["positions"]), t(v["seq_lens"])
    out = binding.verify_rebuild(t(v["drafts"]), t(v["targets"]), t(v["page_table"]), v["num_pages"], pos, sl,
                                 positions_out=pos, seq_lens_out=sl)
    torch.cuda.synchronize()
    exp = _expect(v, K)
    np.testing.assert_array_equal(pos.cpu().numpy(), exp["positions"])
    np.testing.assert_array_equal(sl.cpu().numpy(), exp["seq_lens"])
    np.testing.assert_array_equal(out["slot_mapping"].cpu().numpy(), exp["slot_mapping"])


def test_verify_bad_input_lengths(lib):
    # negative lengths / positions and values too close to 2^31 - 1
    K = 3
    lim = 2 ** 31 - 1 - 2 * K
    v = dict(drafts=np.array([[1, 2, 3]] * 6), targets=np.array([[1, 2, 9, 9]] * 6),
             page_table=np.array([[0, 1], [2, 3], [4, 5], [6, 7], [8, 9], [10, 11]]), num_pages=12,
             seq_lens=np.array([-1, 5, lim + 1, 5, 5, lim]), positions=np.array([7, -3, 7, lim + 1, 9, 4]))
    got = _run(lib, v, K, torch.device("cuda"))
    exp = _expect(v, K)
    _assert_equal(got, exp)
    assert list(got["status"][:4]) == [oracle.REQ_BAD_INPUT] * 4
    assert got["status"][4] == oracle.REQ_OK and got["status"][5] == oracle.REQ_CAPACITY
