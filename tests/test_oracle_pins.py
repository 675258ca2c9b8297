"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test fixes the oracle against something it cannot have copied from itself:
the pages' worked examples (tests/golden/), brute-force enumeration on tiny
inputs, closed forms, invariants, textbook special cases and the statistical
guarantee of speculative rejection sampling (output tokens follow the target
distribution).  A plausible slip in the oracle -- a dropped term, a wrong sign,
a shifted index, a transposed operand -- fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
from scipy import special, stats

import oracle

RNG_SEED = 20261202


def _read_table(path):
    rows = []
    for line in path.read_text().splitlines():
        if line.strip() and not line.startswith("#"):
            rows.append(line.split())
    return rows


def _logit(a):
    a = np.asarray(a, np.float64)
    return np.log(a / (1.0 - a))


# ---------------------------------------------------------------------------
# a1 survival: worked examples W1 and W3


def test_w1_cumulative_acceptance(golden_dir):
    rows = _read_table(golden_dir / "position_acceptance_k7.txt")
    cond = np.array([float(r[2]) for r in rows]) / 100.0
    cum = np.array([float(r[1]) for r in rows])
    s = oracle.survival(_logit(cond).astype(np.float32), [len(cond)])
    np.testing.assert_array_equal(np.round(100.0 * s, 1), cum)
    # "평균 수락 길이": mean acceptance length = 1 + sum of the middle column.
    assert round(1.0 + s.sum(), 2) == 1.93


def test_w3_chain_of_seven():
    s = oracle.survival(np.full(7, _logit(0.55), np.float32), [7])
    assert round(100.0 * s[-1], 1) == 1.5
    # Survival only falls along a draft.
    assert np.all(np.diff(s) < 0)


def test_survival_packing_multiple_requests():
    conf = np.array([0.0, 0.0, 2.0, -1.0, 1.0, 1.0], np.float32)
    s = oracle.survival(conf, [2, 0, 1, 3])
    a = special.expit(conf.astype(np.float64))
    expect = [a[0], a[0] * a[1], a[2], a[3], a[3] * a[4], a[3] * a[4] * a[5]]
    np.testing.assert_allclose(s, expect, rtol=1e-15)


# ---------------------------------------------------------------------------
# a2-a4 planning: worked example W2, brute force, special cases


def test_w2_tokens_per_computed_position(golden_dir):
    w1 = _read_table(golden_dir / "position_acceptance_k7.txt")
    cond = np.array([float(r[2]) for r in w1]) / 100.0
    rows = _read_table(golden_dir / "tokens_per_position_k.txt")
    per_pos = np.array([float(r[3]) for r in rows])
    al = np.array([float(r[2]) for r in rows])
    # One request, R = 1, one non-draft token (T = 1) and cost(n) = n tokens.
    cost = np.arange(9, dtype=np.float32)
    pl = oracle.plan(_logit(cond).astype(np.float32), [7], 7, cost, T=1)
    np.testing.assert_array_equal(np.round(pl["obj"], 2), per_pos)
    np.testing.assert_array_equal(np.round(pl["obj"] * np.arange(1, 9), 2), al)
    # Computing positions is the whole cost: no speculation is best.
    assert pl["B"] == 0
    assert list(pl["cu_seqlens"]) == [0, 1]


def _prefix_closed(subset, dl):
    off = np.concatenate([[0], np.cumsum(dl)])
    for i, k in enumerate(dl):
        taken = [off[i] + j in subset for j in range(k)]
        if any(taken[j + 1] and not taken[j] for j in range(k - 1)):
            return False
    return True


def _brute_force(keys, dl, R, T, cost):
    """Best objective over every prefix-closed subset, by enumeration."""
    N = len(keys)
    L = len(cost) - 1
    cm = np.maximum.accumulate(np.where(np.arange(len(cost)) >= 1, cost.astype(np.float64), -np.inf))
    best_by_size = {}
    for size in range(0, min(N, L - T) + 1):
        for sub in itertools.combinations(range(N), size):
            if not _prefix_closed(set(sub), dl):
                continue
            v = sum(float(keys[q]) for q in sub)
            best_by_size[size] = max(best_by_size.get(size, -1.0), v)
    objs = {b: (R + v) / cm[T + b] for b, v in best_by_size.items()}
    return best_by_size, objs


@pytest.mark.parametrize("trial", range(40))
def test_plan_brute_force(trial):
    rng = np.random.default_rng(RNG_SEED + trial)
    bs = int(rng.integers(1, 5))
    k_max = int(rng.integers(1, 4))
    dl = rng.integers(0, k_max + 1, bs).astype(np.int32)
    N = int(dl.sum())
    conf = rng.normal(1.0, 1.5, N).astype(np.float32)
    T = int(rng.integers(1, 4))
    L = T + int(rng.integers(0, N + 2))
    kind = trial % 3
    n = np.arange(L + 1)
    if kind == 0:
        cost = 1.0 + rng.uniform(0.0, 0.3) * n
    elif kind == 1:
        cost = 1.0 + 0.1 * (4 * ((n + 3) // 4))
    else:  # not monotone: the planner must force it
        cost = 1.0 + 0.05 * n + rng.uniform(0, 0.2, n.size)
    cost = cost.astype(np.float32)
    pl = oracle.plan(conf, dl, k_max, cost, T)
    keys = oracle.survival(conf, dl).astype(np.float32)
    best_by_size, objs = _brute_force(keys, dl, bs, T, cost)
    best = max(objs.values())
    b_star = min(b for b, o in objs.items() if o >= best * (1 - 1e-12))
    if not pl["near"]:
        assert pl["B"] == b_star
    # The chosen mask is prefix-closed, has B slots and attains the best
    # survival sum among prefix-closed subsets of that size.
    off = np.concatenate([[0], np.cumsum(dl)])
    chosen = {int(off[i] + j) for i in range(bs) for j in range(k_max) if pl["slot_mask"][i, j]}
    assert len(chosen) == pl["B"]
    assert _prefix_closed(chosen, dl)
    assert math.isclose(sum(float(keys[q]) for q in chosen), best_by_size[pl["B"]], rel_tol=1e-12)
    # Objective values match the enumeration size by size.
    for b, o in objs.items():
        assert math.isclose(pl["obj"][b], o, rel_tol=1e-12)


def _check_compaction(pl, dl, k_max):
    m = pl["slot_mask"]
    n = pl["num_verified"]
    cu = pl["cu_seqlens"]
    assert cu[0] == 0
    assert np.all(np.diff(cu) == n + 1)
    assert cu[-1] == len(dl) + pl["B"]
    assert np.all(n <= dl)
    for i in range(len(dl)):
        assert list(m[i]) == [1] * n[i] + [0] * (k_max - n[i])


def test_constant_cost_verifies_everything():
    rng = np.random.default_rng(RNG_SEED)
    dl = np.array([3, 1, 2, 3], np.int32)
    conf = rng.normal(0.0, 2.0, dl.sum()).astype(np.float32)
    pl = oracle.plan(conf, dl, 3, np.ones(20, np.float32), T=4)
    assert pl["B"] == dl.sum()
    _check_compaction(pl, dl, 3)


def test_cost_per_token_never_speculates():
    rng = np.random.default_rng(RNG_SEED + 1)
    dl = np.array([2, 3, 3], np.int32)
    conf = rng.normal(0.0, 2.0, dl.sum()).astype(np.float32)
    # cost(n) = n and T = R: Obj(B) = (R + sum s)/(R + B) < 1 = Obj(0).
    pl = oracle.plan(conf, dl, 3, np.arange(30, dtype=np.float32), T=3)
    assert pl["B"] == 0
    _check_compaction(pl, dl, 3)


def test_all_slots_mode():
    dl = np.array([3, 0, 2], np.int32)
    pl = oracle.plan(None, dl, 3, None, T=0, mode=oracle.MODE_ALL_SLOTS)
    assert pl["B"] == 5
    assert list(pl["cu_seqlens"]) == [0, 4, 5, 8]
    _check_compaction(pl, dl, 3)


def test_tie_break_by_slot_index():
    # Two requests with identical confidence have equal keys; when the budget
    # is one slot it goes to the lower packed index (request 0).
    conf = np.array([3.0, 3.0], np.float32)
    # T = 1: Obj(0) = 2/1, Obj(1) = (2+s)/1, Obj(2) = (2+2s)/10 -> B = 1.
    pl = oracle.plan(conf, [1, 1], 1, np.array([1.0, 1.0, 1.0, 10.0], np.float32), T=1)
    assert pl["B"] == 1
    assert list(pl["slot_mask"][:, 0]) == [1, 0]
    assert pl["near"] & oracle.NEAR_TOPB


def test_budget_from_previous_step():
    rng = np.random.default_rng(RNG_SEED + 2)
    dl_prev = np.array([3, 3, 3, 3], np.int32)
    conf_prev = rng.normal(1.0, 1.0, dl_prev.sum()).astype(np.float32)
    dl = np.array([3, 1, 2, 3], np.int32)
    conf = rng.normal(1.0, 1.0, dl.sum()).astype(np.float32)
    cost = (1.0 + 0.08 * np.arange(40)).astype(np.float32)
    T = 4
    prev_alone = oracle.plan(conf_prev, dl_prev, 3, cost, T)
    pl = oracle.plan(conf, dl, 3, cost, T, budget_conf=conf_prev, budget_draft_lens=dl_prev)
    assert pl["B"] == min(prev_alone["B"], dl.sum(), len(cost) - 1 - T)
    # Assignment follows the current keys: the chosen slots are the top-B.
    keys = oracle.survival(conf, dl).astype(np.float32)
    order = sorted(range(len(keys)), key=lambda q: (-keys[q], q))[: pl["B"]]
    off = np.concatenate([[0], np.cumsum(dl)])
    chosen = sorted(int(off[i] + j) for i in range(4) for j in range(3) if pl["slot_mask"][i, j])
    assert chosen == sorted(order)
    _check_compaction(pl, dl, 3)


def test_plan_rejects_bad_inputs():
    with pytest.raises(oracle.OracleError):
        oracle.plan(np.zeros(2, np.float32), [1, 4], 3, np.ones(10, np.float32), T=2)
    with pytest.raises(oracle.OracleError):
        oracle.plan(np.zeros(2, np.float32), [1, 1], 3, np.ones(3, np.float32), T=3)
    with pytest.raises(oracle.OracleError):
        oracle.plan(np.array([np.nan, 0.0], np.float32), [1, 1], 3, np.ones(10, np.float32), T=2)


# ---------------------------------------------------------------------------
# a5 row statistics


def test_softmax_two_tokens_is_sigmoid():
    row = np.array([0.3, 1.7], np.float32)
    for tau in (0.5, 1.0, 2.0):
        p = oracle.softmax(row, oracle.F32, tau)
        d = float(row[1]) - float(row[0])  # exact difference of the stored values
        assert math.isclose(p[1], special.expit(d / tau), rel_tol=1e-12)
        assert math.isclose(p.sum(), 1.0, rel_tol=1e-15)


def test_softmax_matches_library_and_is_shift_invariant():
    rng = np.random.default_rng(RNG_SEED + 3)
    row = rng.normal(0, 3, 4096).astype(np.float32)
    for tau in (0.7, 1.0):
        p = oracle.softmax(row, oracle.F32, tau)
        np.testing.assert_allclose(p, special.softmax(row.astype(np.float64) / tau), rtol=1e-12)
        assert abs(p.sum() - 1.0) < 1e-12
    # bf16 decoding: the bit pattern of 1.0 is 0x3F80.
    pb = oracle.softmax(np.array([0x3F80, 0x0000], np.uint16), oracle.BF16, 1.0)
    assert math.isclose(pb[0], special.expit(1.0), rel_tol=1e-15)
    shifted = oracle.softmax((row + np.float32(8.0)).astype(np.float32), oracle.F32, 1.0)
    np.testing.assert_allclose(shifted, oracle.softmax(row, oracle.F32, 1.0), rtol=1e-5)


# ---------------------------------------------------------------------------
# a6-a8 sampling: constructed cases whose outcome is known, closed forms, chi^2


def _one_hot_rows(tokens, V, big=60.0, second=None):
    rows = np.zeros((len(tokens), V), np.float32)
    for r, t in enumerate(tokens):
        rows[r, t] = big
        if second is not None and second[r] is not None:
            rows[r, second[r]] = big
    return rows


def test_constructed_paths_follow_target_tokens():
    """Peaked rows make every decision certain, so the whole output is known:
    the emitted tokens are the target's own tokens along the path."""
    V, k_max = 16, 3
    cu = np.array([0, 4, 5, 8, 12], np.int32)  # n = 3, 0, 2, 3
    n = np.diff(cu) - 1
    ttok = [[1, 2, 3, 4], [5], [6, 7, 8], [9, 10, 11, 12]]
    dtok = [[1, 2, 0], [], [6, 3], [9, 10, 11]]
    target = _one_hot_rows([t for r in ttok for t in r], V)
    draft = _one_hot_rows([t for r in dtok for t in r], V)
    ids = np.array([t for r in dtok for t in r], np.int32)
    u = np.full((4, k_max + 1), 0.5, np.float32)
    for temps in (np.zeros(4, np.float32), np.ones(4, np.float32), np.array([0, 1, 0.5, 2], np.float32)):
        r = oracle.verify(target, draft, oracle.F32, V, ids, u, temps, cu, k_max)
        assert list(r["accepted_len"]) == [2, 0, 1, 3]
        assert list(r["out_tokens"][0]) == [1, 2, 3, -1]
        assert list(r["out_tokens"][1]) == [5, -1, -1, -1]
        assert list(r["out_tokens"][2]) == [6, 7, -1, -1]
        assert list(r["out_tokens"][3]) == [9, 10, 11, 12]
    assert list(n) == [3, 0, 2, 3]


def test_uniform_indexing_is_per_slot():
    """p(x) = 1/2 and q(x) = 1 at every slot: slot j is accepted iff
    uniforms[i][j] <= 1/2, which reveals which uniform each test reads."""
    V, k_max = 8, 3
    cu = np.array([0, 4, 8], np.int32)
    target = _one_hot_rows([2, 2, 2, 2, 2, 2, 2, 2], V, second=[5] * 8)
    draft = _one_hot_rows([5] * 6, V)
    ids = np.full(6, 5, np.int32)
    u = np.array([[0.25, 0.75, 0.25, 0.25], [0.25, 0.25, 0.75, 0.25]], np.float32)
    r = oracle.verify(target, draft, oracle.F32, V, ids, u, np.ones(2, np.float32), cu, k_max)
    assert list(r["accepted_len"]) == [1, 2]
    # After a rejection at x = 5 the residual max(p - q, 0) is all on token 2.
    assert list(r["out_tokens"][0]) == [5, 2, -1, -1]
    assert list(r["out_tokens"][1]) == [5, 5, 2, -1]
    # p(x), q(x) are reported for the slots tested (up to the first rejection).
    tested = np.array([1, 1, 0, 1, 1, 1], bool)
    np.testing.assert_allclose(r["px"][tested], 0.5, rtol=1e-12)
    np.testing.assert_allclose(r["qx"][tested], 1.0, rtol=1e-12)
    assert np.all(np.isnan(r["px"][~tested]))


def test_final_draw_uses_last_uniform_and_strict_cdf():
    """Bonus row with p = (1/2 on token 1, 1/2 on token 6), every other token
    masked (-inf, p = 0): the final draw reads the last uniform; u < 1/2 gives
    token 1, u >= 1/2 token 6, and u = 0 must not give the zero-mass token 0
    (strict '>' in the inverse CDF)."""
    V, k_max = 8, 2
    target = np.full((1, V), -np.inf, np.float32)
    target[0, 1] = target[0, 6] = 3.0
    cu = np.array([0, 1], np.int32)
    for u_last, expect in ((0.0, 1), (0.25, 1), (0.5, 6), (0.75, 6)):
        u = np.array([[0.9, 0.9, u_last]], np.float32)
        r = oracle.verify(target, np.zeros((0, V), np.float32), oracle.F32, V,
                          np.zeros(0, np.int32), u, np.ones(1, np.float32), cu, k_max)
        assert r["out_tokens"][0, 0] == expect


def test_residual_skips_tokens_where_draft_dominates():
    """After a rejection the residual max(p - q, 0) is zero wherever q >= p:
    with u = 0 the draw is the first token where p > q, not token 0."""
    V, k_max = 4, 1
    target = np.array([[0.0, 0.0, 2.0, 0.0], [0.0, 0.0, 0.0, 0.0]], np.float32)
    draft = np.array([[3.0, 0.0, -1.0, 0.0]], np.float32)  # q_0 > p_0, q_2 < p_2
    cu = np.array([0, 2], np.int32)
    u = np.array([[0.999, 0.0]], np.float32)  # slot 0 (x = 0) is rejected
    r = oracle.verify(target, draft, oracle.F32, V, np.array([0], np.int32), u,
                      np.ones(1, np.float32), cu, k_max)
    assert r["accepted_len"][0] == 0
    p = special.softmax(target[0].astype(np.float64))
    q = special.softmax(draft[0].astype(np.float64))
    first_positive = int(np.argmax(p - q > 0))
    assert r["out_tokens"][0, 0] == first_positive


def test_greedy_equals_target_argmax():
    rng = np.random.default_rng(RNG_SEED + 4)
    V, k_max, bs = 300, 4, 6
    n = np.array([4, 0, 2, 4, 1, 3])
    cu = np.concatenate([[0], np.cumsum(n + 1)]).astype(np.int32)
    target = rng.normal(0, 2, (cu[-1], V)).astype(np.float32)
    amax = target.argmax(axis=1)
    ids, nd = [], []
    for i in range(bs):
        m = rng.integers(0, n[i] + 1)  # first m drafts agree with the target
        for j in range(n[i]):
            t = amax[cu[i] + j]
            ids.append(t if j < m else (t + 1) % V)
        nd.append(m)
    draft = rng.normal(0, 2, (cu[-1] - bs, V)).astype(np.float32)
    u = rng.uniform(0, 1, (bs, k_max + 1)).astype(np.float32)
    r = oracle.verify(target, draft, oracle.F32, V, np.array(ids, np.int32), u,
                      np.zeros(bs, np.float32), cu, k_max)
    for i in range(bs):
        a = r["accepted_len"][i]
        assert a == nd[i]
        assert list(r["out_tokens"][i, : a + 1]) == [int(amax[cu[i] + j]) for j in range(a + 1)]


def _trial_batch(p_logits, q_logits, tau, trials, n_draft, seed):
    """trials independent requests sharing the same rows; draft ids ~ q."""
    rng = np.random.default_rng(seed)
    V = p_logits.shape[-1]
    q = special.softmax(q_logits.astype(np.float64) / tau)
    k_max = n_draft
    cu = np.arange(trials + 1, dtype=np.int32) * (n_draft + 1)
    target = np.tile(p_logits.astype(np.float32), (trials * (n_draft + 1), 1))
    draft = np.tile(q_logits.astype(np.float32), (trials * n_draft, 1))
    ids = rng.choice(V, size=trials * n_draft, p=q).astype(np.int32)
    u = (rng.integers(0, 1 << 24, (trials, k_max + 1)) / float(1 << 24)).astype(np.float32)
    temps = np.full(trials, tau, np.float32)
    r = oracle.verify(target, draft, oracle.F32, V, ids, u, temps, cu, k_max)
    return r


@pytest.mark.parametrize("tau", [0.7, 1.0, 1.6])
def test_acceptance_probability_closed_form(tau):
    rng = np.random.default_rng(RNG_SEED + 5)
    pl = rng.normal(0, 1.5, 8).astype(np.float32)
    ql = (pl + rng.normal(0, 1.0, 8)).astype(np.float32)
    trials = 400_000
    r = _trial_batch(pl, ql, tau, trials, 1, RNG_SEED + 6)
    p = special.softmax(pl.astype(np.float64) / tau)
    q = special.softmax(ql.astype(np.float64) / tau)
    alpha = np.minimum(p, q).sum()
    freq = (r["accepted_len"] == 1).mean()
    sigma = math.sqrt(alpha * (1 - alpha) / trials)
    assert abs(freq - alpha) < 4 * sigma


@pytest.mark.parametrize("tau", [0.7, 1.0, 1.6])
def test_emitted_tokens_follow_target_distribution(tau):
    """Leviathan et al. / Chen et al.: whatever the draft, the first emitted
    token is distributed as p; a bonus token drawn after full acceptance is
    distributed as the next row's p."""
    rng = np.random.default_rng(RNG_SEED + 7)
    pl = rng.normal(0, 1.5, 8).astype(np.float32)
    ql = (pl[::-1] * 0.7 + rng.normal(0, 1.0, 8)).astype(np.float32)  # p and q quite different
    trials = 1_000_000
    r = _trial_batch(pl, ql, tau, trials, 1, RNG_SEED + 8)
    p = special.softmax(pl.astype(np.float64) / tau)
    first = r["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=8)
    assert stats.chisquare(counts, p * trials).pvalue > 1e-3
    bonus = r["out_tokens"][r["accepted_len"] == 1, 1]
    cb = np.bincount(bonus, minlength=8)
    assert stats.chisquare(cb, p * len(bonus)).pvalue > 1e-3


def test_bonus_only_request_samples_p():
    rng = np.random.default_rng(RNG_SEED + 9)
    pl = rng.normal(0, 1.0, 8).astype(np.float32)
    trials = 400_000
    r = _trial_batch(pl, pl, 1.0, trials, 0, RNG_SEED + 10)
    p = special.softmax(pl.astype(np.float64))
    counts = np.bincount(r["out_tokens"][:, 0], minlength=8)
    assert stats.chisquare(counts, p * trials).pvalue > 1e-3
    assert np.all(r["accepted_len"] == 0)


def test_request_subset_matches_full_run():
    rng = np.random.default_rng(RNG_SEED + 11)
    V, k_max, bs = 64, 3, 5
    n = np.array([3, 1, 0, 2, 3])
    cu = np.concatenate([[0], np.cumsum(n + 1)]).astype(np.int32)
    target = rng.normal(0, 2, (cu[-1], V)).astype(np.float32)
    draft = (target[: cu[-1] - bs] + rng.normal(0, 1, (cu[-1] - bs, V))).astype(np.float32)
    ids = rng.integers(0, V, cu[-1] - bs).astype(np.int32)
    u = rng.uniform(0, 1, (bs, k_max + 1)).astype(np.float32)
    temps = np.array([1.0, 0.0, 0.7, 1.0, 0.0], np.float32)
    full = oracle.verify(target, draft, oracle.F32, V, ids, u, temps, cu, k_max)
    part = oracle.verify(target, draft, oracle.F32, V, ids, u, temps, cu, k_max, requests=[3, 0])
    for i in (0, 3):
        assert full["accepted_len"][i] == part["accepted_len"][i]
        assert list(full["out_tokens"][i]) == list(part["out_tokens"][i])


def test_verify_rejects_bad_inputs():
    V = 8
    t = np.zeros((2, V), np.float32)
    d = np.zeros((1, V), np.float32)
    ok = dict(target=t, draft=d, dtype=oracle.F32, V=V, draft_ids=np.array([1], np.int32),
              uniforms=np.zeros((1, 2), np.float32), temps=np.ones(1, np.float32),
              cu_seqlens=np.array([0, 2], np.int32), k_max=1)
    oracle.verify(**ok)
    for key, bad in (("draft_ids", np.array([V], np.int32)),
                     ("uniforms", np.array([[0.2, 1.0]], np.float32)),
                     ("temps", np.array([-1.0], np.float32)),
                     ("cu_seqlens", np.array([0, 3], np.int32))):
        with pytest.raises(oracle.OracleError):
            oracle.verify(**{**ok, key: bad})
    for bad in (np.inf, np.nan):
        tn = t.copy()
        tn[0, 3] = bad
        with pytest.raises(oracle.OracleError):
            oracle.verify(**{**ok, "target": tn})
    tm = t.copy()
    tm[0, 3] = -np.inf  # a masked token is allowed
    oracle.verify(**{**ok, "target": tm})
    with pytest.raises(oracle.OracleError):  # but not a fully masked row
        oracle.verify(**{**ok, "target": np.full((2, V), -np.inf, np.float32)})
