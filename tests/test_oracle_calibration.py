"""Pins of the oracle's online calibration step (CPU).

The fosworld blog's table under "동작" says that for model-based drafts the
per-position acceptance estimate comes from a small logistic model on the
draft's logits, corrected continuously with the verification results.  The
oracle reads that as a per-position logistic model a = sigmoid(w_j c + b_j)
of the confidence logit, moved by one gradient step on the mean logistic loss
of the slots a step observed (those up to and including the first
rejection).  The pins tie it to:

- the loss itself: the reported gradient equals central finite differences of
  the mean logistic loss, evaluated with scipy's log-sigmoid;
- constructed outcomes: which slots count, with which label, by hand;
- statistics: steps on outcomes drawn from a known model recover that model;
- descent: a small step lowers each observed position's loss by about lr·|grad|².
"""
import numpy as np
import pytest
from scipy import special

import oracle

RNG_SEED = 31415


def _observed(dl, nv, acc):
    """(request, position, label) of every observed slot, by hand."""
    out = []
    off = np.concatenate([[0], np.cumsum(dl)])
    for i in range(len(dl)):
        for j in range(min(nv[i], acc[i] + 1)):
            out.append((int(off[i] + j), j, 1.0 if j < acc[i] else 0.0))
    return out


def _mean_loss(conf, obs, j, w, b):
    z = np.array([w * conf[q] + b for q, jj, _ in obs if jj == j], np.float64)
    y = np.array([lab for _, jj, lab in obs if jj == j], np.float64)
    return float(np.mean(-(y * special.log_expit(z) + (1 - y) * special.log_expit(-z))))


def _random_step(rng, bs, k_max):
    dl = rng.integers(0, k_max + 1, bs).astype(np.int32)
    nv = np.array([rng.integers(0, k + 1) for k in dl], np.int32)
    acc = np.array([rng.integers(0, n + 1) for n in nv], np.int32)
    conf = rng.normal(0.5, 2.0, int(dl.sum())).astype(np.float32)
    return dl, nv, acc, conf


@pytest.mark.parametrize("trial", range(10))
def test_gradient_is_the_derivative_of_the_mean_logistic_loss(trial):
    rng = np.random.default_rng(RNG_SEED + trial)
    k_max = int(rng.integers(1, 8))
    dl, nv, acc, conf = _random_step(rng, int(rng.integers(8, 64)), k_max)
    w0 = rng.normal(1.0, 0.3, k_max)
    b0 = rng.normal(0.0, 0.5, k_max)
    r = oracle.calibrate(conf, dl, nv, acc, k_max, 0.0, w0, b0)
    obs = _observed(dl, nv, acc)
    c64 = conf.astype(np.float64)
    h = 1e-6
    for j in range(k_max):
        m = sum(1 for _, jj, _ in obs if jj == j)
        assert r["count"][j] == m
        if m == 0:
            assert r["grad_w"][j] == 0.0 and r["grad_b"][j] == 0.0
            continue
        fw = (_mean_loss(c64, obs, j, w0[j] + h, b0[j]) - _mean_loss(c64, obs, j, w0[j] - h, b0[j])) / (2 * h)
        fb = (_mean_loss(c64, obs, j, w0[j], b0[j] + h) - _mean_loss(c64, obs, j, w0[j], b0[j] - h)) / (2 * h)
        assert r["grad_w"][j] == pytest.approx(fw, rel=1e-6, abs=1e-8)
        assert r["grad_b"][j] == pytest.approx(fb, rel=1e-6, abs=1e-8)
    # lr = 0 leaves the parameters where they were
    assert np.array_equal(r["w"], w0) and np.array_equal(r["b"], b0)


def test_observation_rule_on_constructed_outcomes():
    # request 0: 4 drafted, 3 verified, 1 accepted -> j=0 accepted, j=1 rejected
    # request 1: 4 drafted, 4 verified, all accepted -> j=0..3 accepted
    # request 2: 2 drafted, none verified -> nothing observed
    # request 3: 3 drafted, 2 verified, 2 accepted -> j=0,1 accepted (j=2 untested)
    dl = np.array([4, 4, 2, 3], np.int32)
    nv = np.array([3, 4, 0, 2], np.int32)
    acc = np.array([1, 4, 0, 2], np.int32)
    conf = np.arange(1, 14, dtype=np.float32)  # slot values 1..13, packed
    k_max = 5
    r = oracle.calibrate(conf, dl, nv, acc, k_max, 0.5, np.zeros(k_max), np.zeros(k_max))
    assert list(r["count"]) == [3, 3, 1, 1, 0]
    # at w = b = 0 every estimate is 1/2, so e = 1/2 - y
    e = {(0, 0): -0.5, (0, 1): 0.5, (1, 0): -0.5, (1, 1): -0.5, (1, 2): -0.5, (1, 3): -0.5,
         (3, 0): -0.5, (3, 1): -0.5}
    c = {(0, 0): 1, (0, 1): 2, (1, 0): 5, (1, 1): 6, (1, 2): 7, (1, 3): 8, (3, 0): 11, (3, 1): 12}
    for j in range(4):
        keys = [k for k in e if k[1] == j]
        gb = sum(e[k] for k in keys) / len(keys)
        gw = sum(e[k] * c[k] for k in keys) / len(keys)
        assert r["grad_b"][j] == pytest.approx(gb, abs=1e-15)
        assert r["grad_w"][j] == pytest.approx(gw, abs=1e-15)
        assert r["b"][j] == pytest.approx(-0.5 * gb, abs=1e-15)
        assert r["w"][j] == pytest.approx(-0.5 * gw, abs=1e-15)
    assert r["w"][4] == 0.0 and r["b"][4] == 0.0 and r["grad_w"][4] == 0.0


def test_repeated_steps_recover_the_generating_model():
    """Outcomes drawn from a known per-position model: the calibrated
    parameters (averaged over the second half of the steps) approach it."""
    rng = np.random.default_rng(RNG_SEED + 99)
    k_max, bs, steps = 3, 256, 2000
    w_true = np.array([1.2, 0.8, 1.0])
    b_true = np.array([0.5, 0.0, -0.3])
    w, b = np.ones(k_max), np.zeros(k_max)
    tail_w, tail_b = [], []
    dl = np.full(bs, k_max, np.int32)
    for step in range(steps):
        conf = rng.normal(1.0, 1.5, (bs, k_max))
        a = special.expit(w_true * conf + b_true)
        ok = rng.uniform(size=(bs, k_max)) < a
        acc = np.where(ok.all(axis=1), k_max, np.argmin(ok, axis=1)).astype(np.int32)
        r = oracle.calibrate(conf.astype(np.float32).ravel(), dl, dl, acc, k_max, 1.0, w, b)
        w, b = r["w"], r["b"]
        if step >= steps // 2:
            tail_w.append(w)
            tail_b.append(b)
    np.testing.assert_allclose(np.mean(tail_w, axis=0), w_true, atol=0.08)
    np.testing.assert_allclose(np.mean(tail_b, axis=0), b_true, atol=0.08)


def test_calibrate_rejects_bad_inputs():
    dl = np.array([2, 2], np.int32)
    conf = np.zeros(4, np.float32)
    ok = dict(conf=conf, draft_lens=dl, num_verified=[2, 1], accepted_len=[1, 1], k_max=2,
              lr=0.1, w=np.ones(2), b=np.zeros(2))
    oracle.calibrate(**ok)
    for bad in (dict(accepted_len=[1, 2]),        # more accepted than verified
                dict(num_verified=[3, 1]),        # more verified than drafted
                dict(lr=-1.0),
                dict(draft_lens=np.array([3, 2], np.int32), conf=np.zeros(5, np.float32))):
        with pytest.raises(oracle.OracleError):
            oracle.calibrate(**dict(ok, **bad))
    nan = conf.copy()
    nan[0] = np.nan  # an observed slot
    with pytest.raises(oracle.OracleError):
        oracle.calibrate(**dict(ok, conf=nan))


@pytest.mark.parametrize("trial", range(20))
def test_a_small_step_lowers_each_positions_loss(trial):
    """The update is a descent step: with a small rate, the mean logistic loss
    of every observed position goes down (or stays, when its gradient is 0)."""
    rng = np.random.default_rng(RNG_SEED + 500 + trial)
    k_max = int(rng.integers(1, 8))
    dl, nv, acc, conf = _random_step(rng, int(rng.integers(8, 64)), k_max)
    w0 = rng.normal(1.0, 0.5, k_max)
    b0 = rng.normal(0.0, 1.0, k_max)
    r = oracle.calibrate(conf, dl, nv, acc, k_max, 1e-3, w0, b0)
    obs = _observed(dl, nv, acc)
    c64 = conf.astype(np.float64)
    for j in range(k_max):
        if r["count"][j] == 0:
            continue
        before = _mean_loss(c64, obs, j, w0[j], b0[j])
        after = _mean_loss(c64, obs, j, r["w"][j], r["b"][j])
        assert after <= before + 1e-15
        g2 = r["grad_w"][j] ** 2 + r["grad_b"][j] ** 2
        # first order: the decrease is about lr * |grad|^2
        assert before - after == pytest.approx(1e-3 * g2, rel=0.05, abs=1e-12)
