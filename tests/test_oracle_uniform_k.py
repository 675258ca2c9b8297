"""Pins of the oracle's uniform-K planning mode (CPU).

The mode follows the DSD page ("DSD feat. Cohere", section "동적 추측
디코딩(DSD)의 핵심 아이디어"): one draft length K for the whole batch,
chosen to maximise goodput = AL / ITL, where AL counts one token per request
plus the survival of its first min(K, K_i) draft slots and ITL is the
monotone step cost of the tokens verified.  The pins tie it to things fixed
outside its own code:

- one request: top-B over one draft is a prefix, so uniform K and the
  adaptive budget (pinned by brute force elsewhere) coincide;
- a flat cost verifies every slot (ALL_SLOTS), a per-token cost none;
- a per-slot selection can only do better: the adaptive optimum bounds the
  uniform one, size by size;
- the page's dense-model finding: with a cost that is flat up to a knee
  (bandwidth-bound) and linear beyond (compute-bound), the chosen K falls
  monotonically as the batch grows, down to no speculation.
"""
import math

import numpy as np
import pytest

import oracle

RNG_SEED = 20260712


def _logit(a):
    return math.log(a / (1.0 - a))


def _check_uniform_compaction(pl, dl, k_max):
    n = pl["num_verified"]
    K = int(n.max()) if len(n) else 0
    assert list(n) == [min(K, int(k)) for k in dl]
    assert pl["B"] == int(n.sum())
    assert np.all(np.diff(pl["cu_seqlens"]) == n + 1)
    for i in range(len(dl)):
        assert list(pl["slot_mask"][i]) == [1] * n[i] + [0] * (k_max - n[i])


@pytest.mark.parametrize("trial", range(30))
def test_one_request_uniform_equals_adaptive(trial):
    rng = np.random.default_rng(RNG_SEED + trial)
    k_max = int(rng.integers(1, 8))
    dl = np.array([int(rng.integers(0, k_max + 1))], np.int32)
    conf = rng.normal(1.0, 1.5, int(dl.sum())).astype(np.float32)
    T = int(rng.integers(1, 4))
    n = np.arange(T + k_max + 3)
    cost = (1.0 + rng.uniform(0.0, 0.4) * n + rng.uniform(0.0, 0.1, n.size)).astype(np.float32)
    ad = oracle.plan(conf, dl, k_max, cost, T)
    un = oracle.plan(conf, dl, k_max, cost, T, mode=oracle.MODE_UNIFORM_K)
    assert un["B"] == ad["B"]
    assert np.array_equal(un["slot_mask"], ad["slot_mask"])
    valid = ~np.isnan(un["obj"])
    m = min(int(valid.sum()), len(ad["obj"]))
    assert m >= 1
    np.testing.assert_allclose(un["obj"][:m], ad["obj"][:m], rtol=1e-15)


def test_flat_cost_verifies_every_slot():
    rng = np.random.default_rng(RNG_SEED)
    dl = np.array([3, 1, 0, 2, 3], np.int32)
    conf = rng.normal(0.0, 2.0, dl.sum()).astype(np.float32)
    un = oracle.plan(conf, dl, 3, np.ones(40, np.float32), T=5, mode=oracle.MODE_UNIFORM_K)
    al = oracle.plan(None, dl, 3, None, T=0, mode=oracle.MODE_ALL_SLOTS)
    assert np.array_equal(un["slot_mask"], al["slot_mask"])
    assert list(un["cu_seqlens"]) == list(al["cu_seqlens"])
    _check_uniform_compaction(un, dl, 3)


def test_per_token_cost_never_speculates():
    rng = np.random.default_rng(RNG_SEED + 1)
    dl = np.array([2, 3, 3], np.int32)
    conf = rng.normal(0.0, 2.0, dl.sum()).astype(np.float32)
    # cost(n) = n, T = R: AL / ITL = (R + sum s) / (R + tokens) < 1 = K = 0.
    un = oracle.plan(conf, dl, 3, np.arange(30, dtype=np.float32), T=3,
                     mode=oracle.MODE_UNIFORM_K)
    assert un["B"] == 0
    _check_uniform_compaction(un, dl, 3)


@pytest.mark.parametrize("trial", range(30))
def test_adaptive_selection_bounds_the_uniform_one(trial):
    rng = np.random.default_rng(RNG_SEED + 100 + trial)
    bs = int(rng.integers(1, 9))
    k_max = int(rng.integers(1, 8))
    dl = rng.integers(0, k_max + 1, bs).astype(np.int32)
    conf = rng.normal(1.0, 1.5, int(dl.sum())).astype(np.float32)
    T = bs
    n = np.arange(T + int(dl.sum()) + 2)
    cost = (1.0 + rng.uniform(0.0, 0.2) * n).astype(np.float32)
    ad = oracle.plan(conf, dl, k_max, cost, T)
    un = oracle.plan(conf, dl, k_max, cost, T, mode=oracle.MODE_UNIFORM_K)
    _check_uniform_compaction(un, dl, k_max)
    # every uniform choice is one prefix-closed subset of its size
    for K, o in enumerate(un["obj"]):
        if np.isnan(o):
            continue
        size = int(np.minimum(K, dl).sum())
        assert o <= ad["obj"][size] * (1 + 1e-12)
    assert np.nanmax(un["obj"]) <= np.nanmax(ad["obj"]) * (1 + 1e-12)


def test_short_cost_table_caps_k():
    dl = np.array([4, 4], np.int32)
    conf = np.full(8, _logit(0.95), np.float32)
    T = 2
    cost = np.ones(T + 5, np.float32)  # room for 4 draft tokens: K <= 2
    un = oracle.plan(conf, dl, 4, cost, T, mode=oracle.MODE_UNIFORM_K)
    assert list(un["num_verified"]) == [2, 2]
    assert np.isnan(un["obj"][3]) and np.isnan(un["obj"][4])
    assert not np.isnan(un["obj"][2])


def test_chosen_k_falls_with_batch_size():
    # Every request drafts 7 tokens with per-position acceptance 0.8; one
    # non-draft token a request (T = BS); a step costs 1 up to 64 tokens and
    # grows in proportion beyond (a bandwidth-bound then compute-bound model).
    k_max, knee = 7, 64
    a = _logit(0.8)
    ks = []
    for bs in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        dl = np.full(bs, k_max, np.int32)
        conf = np.full(bs * k_max, a, np.float32)
        n = np.arange(bs * (k_max + 1) + 1)
        cost = np.maximum(1.0, n / knee).astype(np.float32)
        pl = oracle.plan(conf, dl, k_max, cost, bs, mode=oracle.MODE_UNIFORM_K)
        _check_uniform_compaction(pl, dl, k_max)
        ks.append(int(pl["num_verified"].max()))
    assert all(x >= y for x, y in zip(ks, ks[1:])), ks
    assert ks[0] == k_max  # small batch: every draft slot is free
    assert ks[-1] == 0     # compute-bound: falls back to no speculation
    assert any(0 < k < k_max for k in ks)


def test_uniform_rejects_missing_inputs():
    with pytest.raises(oracle.OracleError):
        oracle.plan(None, [1, 1], 1, np.ones(10, np.float32), T=2, mode=oracle.MODE_UNIFORM_K)
    with pytest.raises(oracle.OracleError):
        oracle.plan(np.zeros(2, np.float32), [1, 1], 1, np.ones(3, np.float32), T=3,
                    mode=oracle.MODE_UNIFORM_K)
    with pytest.raises(oracle.OracleError):
        oracle.plan(np.array([np.nan, 0.0], np.float32), [1, 1], 1, np.ones(10, np.float32),
                    T=2, mode=oracle.MODE_UNIFORM_K)
