"""Property tests of the oracle's planner in its three modes (CPU, hypothesis).

Invariants the pages fix for any input: the verified slots of a request are
a prefix of its draft ("동작" step 2 of the fosworld blog: survival only
falls along a draft); cu_seqlens counts the verified slots plus one row per
request; the budget never exceeds what the cost table covers; one draft
length for the batch (the DSD page) selects min(K, K_i) slots of every
request; a per-slot selection can only match or beat a per-batch one.
"""
import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings


@st.composite
def plan_case(draw):
    bs = draw(st.integers(1, 10))
    k_max = draw(st.integers(0, 6))
    dl = np.array(draw(st.lists(st.integers(0, k_max), min_size=bs, max_size=bs)), np.int32)
    N = int(dl.sum())
    conf = np.array(draw(st.lists(st.floats(-6, 6, width=32), min_size=N, max_size=N)),
                    np.float32)
    T = draw(st.integers(1, 12))
    L = T + draw(st.integers(0, N + 2))
    slope = draw(st.floats(0.0, 0.5))
    noise = np.array(draw(st.lists(st.floats(0.0, 0.3), min_size=L + 1, max_size=L + 1)))
    cost = (1.0 + slope * np.arange(L + 1) + noise).astype(np.float32)
    return dl, conf, k_max, cost, T


def _common(pl, dl, k_max, cost, T):
    n = pl["num_verified"]
    m = pl["slot_mask"]
    assert np.all(n <= dl)
    for i in range(len(dl)):
        assert list(m[i]) == [1] * int(n[i]) + [0] * (k_max - int(n[i]))
    assert pl["cu_seqlens"][0] == 0
    assert np.all(np.diff(pl["cu_seqlens"]) == n + 1)
    assert pl["B"] == int(n.sum())


@settings(max_examples=300, deadline=None)
@given(plan_case())
def test_adaptive_plan_invariants(case):
    dl, conf, k_max, cost, T = case
    pl = oracle.plan(conf, dl, k_max, cost, T)
    _common(pl, dl, k_max, cost, T)
    assert pl["B"] <= min(int(dl.sum()), len(cost) - 1 - T)


@settings(max_examples=300, deadline=None)
@given(plan_case())
def test_uniform_k_plan_invariants(case):
    dl, conf, k_max, cost, T = case
    un = oracle.plan(conf, dl, k_max, cost, T, mode=oracle.MODE_UNIFORM_K)
    _common(un, dl, k_max, cost, T)
    K = int(un["num_verified"].max())
    assert list(un["num_verified"]) == [min(K, int(k)) for k in dl]
    assert T + un["B"] <= len(cost) - 1
    ad = oracle.plan(conf, dl, k_max, cost, T)
    assert np.nanmax(un["obj"]) <= np.nanmax(ad["obj"]) * (1 + 1e-12)


@settings(max_examples=100, deadline=None)
@given(plan_case())
def test_all_slots_plan_invariants(case):
    dl, conf, k_max, cost, T = case
    pl = oracle.plan(None, dl, k_max, None, 0, mode=oracle.MODE_ALL_SLOTS)
    _common(pl, dl, k_max, cost, T)
    assert list(pl["num_verified"]) == list(dl)
