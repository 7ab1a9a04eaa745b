"""GPU parity of dcut_allocate_cost (the cost-unit D-cut policy of the
deep-dive page's scheduler listing) against the oracle: depths, offsets and
benefits bit-exact (both sides decide in fp64, operation by operation)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from draft_verification_02_b300 import specverify as sv
from draft_verification_02_b300.verifier import Verifier

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def run(v, conf, kmax, max_cost):
    B = kmax.size
    Kmax = conf.shape[1] if conf.ndim == 2 else 0
    c = torch.from_numpy(np.ascontiguousarray(conf, np.float32)).cuda()
    k = torch.from_numpy(np.ascontiguousarray(kmax, np.int32)).cuda()
    depth = torch.full((max(B, 1),), -7, dtype=torch.int32, device="cuda")
    cu = torch.full((B + 1,), -7, dtype=torch.int32, device="cuda")
    ben = torch.full((max(B, 1),), float("nan"), dtype=torch.float64, device="cuda")
    st = sv.dcut_allocate_cost(c, k, B, Kmax, max_cost, depth, cu, ben, v.workspace)
    assert st == sv.SPEC_OK
    torch.cuda.synchronize()
    return depth.cpu().numpy()[:B], cu.cpu().numpy(), ben.cpu().numpy()[:B]


def _padded(rows):
    K = max(len(r) for r in rows)
    c = np.zeros((len(rows), K), np.float32)
    for i, r in enumerate(rows):
        c[i, :len(r)] = r
    return c


def test_dcut_cost_golden_on_gpu():
    v = Verifier(8, 8, 1)
    for case in json.load(open(os.path.join(GOLDEN, "dcut_cost.json")))["cases"]:
        d, cu, _ = run(v, _padded(case["conf"]), np.array(case["kmax"], np.int32),
                       case["max_cost"])
        assert d.tolist() == case["expected_depth"], case["name"]
        assert cu.tolist() == [0] + np.cumsum(case["expected_depth"]).tolist(), case["name"]
    assert v.device_status() == sv.SPEC_OK


@pytest.mark.parametrize("B", [1, 7, 64, 300, 4096])
def test_dcut_cost_random_against_oracle(B):
    rng = np.random.default_rng(B)
    v = Verifier(8, 8, 1)
    for trial in range(6):
        Kmax = int(rng.integers(1, 33))
        kmax = rng.integers(0, Kmax + 1, size=B).astype(np.int32)
        conf = (rng.beta(8, 2, size=(B, Kmax)) * 0.95 ** np.arange(Kmax)).astype(np.float32)
        if trial % 3 == 2:  # many exact ties: a few distinct rows, powers of two
            conf = (0.5 ** rng.integers(0, 2, size=(B, Kmax))).astype(np.float32)
        max_cost = float(rng.choice([0.5, 3.0, B * 0.8, B * 1.7, 1e9]))
        d, cu, ben = run(v, conf, kmax, max_cost)
        o = O.dcut_schedule_cost(conf, kmax, max_cost)
        assert o.status == O.OK
        assert d.tolist() == o.depth.tolist(), trial
        assert cu.tolist() == o.cu.tolist(), trial
        assert ben.tobytes() == o.benefit.tobytes(), trial  # fp64, bit for bit
    assert v.device_status() == sv.SPEC_OK


def test_dcut_cost_invalid_confidence():
    v = Verifier(4, 4, 1)
    conf = torch.tensor([[0.5, 1.5], [0.2, 0.1]], device="cuda")
    depth = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    cu = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    st = sv.dcut_allocate_cost(conf, torch.tensor([2, 2], dtype=torch.int32, device="cuda"), 2, 2,
                               4.0, depth, cu, None, v.workspace)
    assert st == sv.SPEC_OK
    assert v.device_status() == sv.SPEC_ERR_INVALID_ARG
    assert depth.cpu().tolist() == [-1, -1] and cu.cpu().tolist() == [-1, -1, -1]


def test_dcut_cost_edge_values_against_oracle():
    """Values at the edges of the integer forms of the fp64 operations:
    zero confidences, confidences of 1 and 1 - 2^-24, subnormal confidences
    and products that underflow the normal range (the hardware path), and
    budgets equal to an exact running total of the costs and one ulp below
    it (the admission's <= decided on the rounded sum)."""
    v = Verifier(8, 8, 1)
    tiny = np.float32(1e-40)  # a subnormal float
    cases = []
    K = 16
    rows = [np.ones(K), np.zeros(K), np.full(K, np.float32(1 - 2.0 ** -24)),
            np.full(K, 1e-30), np.r_[np.ones(8), np.full(8, tiny)],
            np.linspace(1.0, 0.2, K), np.full(K, 0.5), np.r_[0.9, np.zeros(K - 1)]]
    conf = np.array(rows, np.float32)
    kmax = np.full(len(rows), K, np.int32)
    for max_cost in (0.0, 1.0, 3.0, 7.5, 1e9, -1.0, float("inf"), 5e-324):
        cases.append((conf, kmax, max_cost))
    # equal benefits everywhere: every request takes depth 2 at cost 1.2, and
    # the running total is the fp64 sum 1.2 + 1.2 + ...; a budget equal to
    # that sum admits n requests, one ulp below admits n - 1
    conf2 = np.ones((12, 2), np.float32)
    kmax2 = np.full(12, 2, np.int32)
    t = 0.0
    for n in range(1, 12):
        t = t + 1.2
        for mc in (t, float(np.nextafter(t, 0.0)), float(np.nextafter(t, 10.0))):
            cases.append((conf2, kmax2, mc))
    for conf_, kmax_, mc in cases:
        d, cu, ben = run(v, conf_, kmax_, mc)
        o = O.dcut_schedule_cost(conf_, kmax_, mc)
        assert o.status == O.OK
        assert d.tolist() == o.depth.tolist(), mc
        assert cu.tolist() == o.cu.tolist(), mc
        assert ben.tobytes() == o.benefit.tobytes(), mc
    assert v.device_status() == sv.SPEC_OK
