"""The bandwidth-adaptive level controller (cg_plan_levels,
cg_simulate_stream): host code, no GPU.  The oracle (oracle/plan.py) is
pinned by a hand-worked trace and by properties the rule fixes; the library
must then make the same choices and give the same timeline, bit for bit,
on seeded random traces."""
import os

import numpy as np
import pytest

from kv_cache_compression_02_gb300 import build, cachegen as cg
from oracle import plan

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    cg.lib()


def _golden():
    vals = {}
    for line in open(os.path.join(HERE, "golden", "hand_worked_plan.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=")
            vals[k.strip()] = [float(t) for t in v.split()]
    return vals


def test_oracle_hand_worked_trace():
    g = _golden()
    cb = np.array(g["chunk_bytes"], np.int64).reshape(-1, 2)
    trace = list(zip(g["trace"][0::2], g["trace"][1::2]))
    lv, tl, tot = plan.plan(cb.tolist(), trace, g["initial"][0], g["deadline"][0], g["decode"])
    assert lv == [int(v) for v in g["levels"]]
    assert np.allclose(np.array(tl).ravel(), g["timeline"], rtol=0, atol=1e-12)
    assert tot == pytest.approx(g["total"][0], abs=1e-12)
    _, _, t0 = plan.simulate(cb.tolist(), trace, [0, 0, 0], g["decode"])
    assert t0 == pytest.approx(g["fixed0_total"][0], abs=1e-12)
    _, tl1, _ = plan.simulate(cb.tolist(), trace, [1, 1, 1], g["decode"])
    assert np.allclose(np.array(tl1).ravel(), g["fixed1_timeline"], rtol=0, atol=1e-12)


def test_oracle_arrival_closed_forms():
    tr = [(2.0, 10.0), (1.0, 0.0), (5.0, 40.0)]  # a 1 s outage between two rates
    assert plan.arrival(tr, 0.0, 20.0) == 2.0
    assert plan.arrival(tr, 0.0, 30.0) == 3.0 + 10.0 / 40.0   # waits out the outage
    assert plan.arrival(tr, 2.5, 40.0) == 4.0                  # starts inside the outage
    assert plan.arrival(tr, 100.0, 80.0) == 102.0              # past the trace: last rate
    assert plan.arrival(tr, 1.0, 0.0) == 1.0


def test_oracle_limits():
    rng = np.random.default_rng(3)
    cb = np.sort(rng.integers(1000, 10 ** 6, (12, 4)), axis=1)[:, ::-1].tolist()  # coarser = smaller
    tr = [(0.5, 2e6), (1.0, 5e5), (2.0, 3e6)]
    dec = [0.01] * 12
    lv, _, _ = plan.plan(cb, [(1.0, 1e15)], 1e15, 10.0, dec)       # unlimited link: finest everywhere
    assert lv == [0] * 12
    lv, _, _ = plan.plan(cb, tr, 1e6, 0.0, dec)                     # no time at all: coarsest everywhere
    assert lv == [3] * 12
    # constant link, exact estimate: a slower link never picks a finer level
    prev = [0] * 12
    for rate in (4e6, 2e6, 1e6, 5e5, 2.5e5):
        lv, _, _ = plan.plan(cb, [(1.0, rate)], rate, 4.0, dec)
        assert all(a >= b for a, b in zip(lv, prev))
        prev = lv


def test_library_matches_oracle_hand_worked():
    g = _golden()
    cb = np.array(g["chunk_bytes"], np.int64).reshape(-1, 2)
    trace = list(zip(g["trace"][0::2], g["trace"][1::2]))
    rc, lv, tl, tot = cg.cg_plan_levels(cb, trace, g["initial"][0], g["deadline"][0], g["decode"])
    assert rc == cg.CG_OK
    assert lv.tolist() == [int(v) for v in g["levels"]]
    assert tl.ravel().tolist() == pytest.approx(g["timeline"], abs=1e-12)
    assert tot == pytest.approx(g["total"][0], abs=1e-12)


@pytest.mark.parametrize("seed", range(12))
def test_library_matches_oracle_random(seed):
    rng = np.random.default_rng(100 + seed)
    n, nl = int(rng.integers(1, 70)), int(rng.integers(1, 9))
    cb = np.sort(rng.integers(1, 1 << 40, (n, nl)), axis=1)[:, ::-1].copy()
    steps = int(rng.integers(1, 12))
    trace = [(float(rng.uniform(0, 50)), float(rng.choice([0.0, rng.uniform(1e8, 5e10)]))) for _ in range(steps)]
    trace[-1] = (trace[-1][0], float(rng.uniform(1e8, 5e10)))
    dec = rng.uniform(0, 0.5, n).tolist()
    init, dl = float(rng.uniform(1e8, 5e10)), float(rng.uniform(0, 400))
    rc, lv, tl, tot = cg.cg_plan_levels(cb, trace, init, dl, dec)
    assert rc == cg.CG_OK
    lv_o, tl_o, tot_o = plan.plan(cb.tolist(), trace, init, dl, dec)
    assert lv.tolist() == lv_o
    assert tl.tolist() == [list(t) for t in tl_o]   # same operations, same doubles
    assert tot == tot_o
    rc, tl2, tot2 = cg.cg_simulate_stream(cb, trace, lv, dec)
    assert rc == cg.CG_OK and tl2.tolist() == tl.tolist() and tot2 == tot


def test_library_rejects_bad_arguments():
    cb = [[10, 5]]
    ok = [(1.0, 10.0)]
    assert cg.cg_plan_levels(cb, ok, 10.0, 1.0, [0.0])[0] == cg.CG_OK
    for trace in ([(1.0, 0.0)], [(-1.0, 5.0), (1.0, 5.0)], [(float("nan"), 5.0), (1.0, 5.0)]):
        assert cg.cg_plan_levels(cb, trace, 10.0, 1.0, [0.0])[0] == cg.CG_ERR_INVALID_ARG
    assert cg.cg_plan_levels(cb, ok, 0.0, 1.0, [0.0])[0] == cg.CG_ERR_INVALID_ARG
    assert cg.cg_plan_levels(cb, ok, 10.0, 1.0, [-1.0])[0] == cg.CG_ERR_INVALID_ARG
    assert cg.cg_plan_levels(np.zeros((1, 9), np.int64), ok, 10.0, 1.0, [0.0])[0] == cg.CG_ERR_INVALID_ARG
    assert cg.cg_simulate_stream(cb, ok, [2], [0.0])[0] == cg.CG_ERR_INVALID_ARG
