"""Pins of the oracle's confidence-scheduled verify-length pre-pass (no GPU).

The DSpark review (vllmbangkok.com, Sec. 4.2.1-4.2.2) fixes: survival is the
prefix product of per-token confidences and never increases; draft tokens of all
requests are ranked by survival and added one at a time; the step time comes from
a table profiled at startup; the production scheduler searches the whole table.
Pinned here by a hand-computed case, a step-shaped table where the first drop is
not the optimum, exhaustive search over every allocation, and a Monte-Carlo check
that the sum of prefix products is the expected accepted length.
"""
import itertools

import numpy as np
import pytest


def test_hand_computed_two_requests(oracle_mod):
    # S_0 = [0.9, 0.72, 0.36], S_1 = [0.6, 0.3, 0.27]; min_len 1 -> n0 = 2, E0 = 1.5
    # ranked candidates: 0.72, 0.36, 0.30, 0.27
    # F(2) = 3.5/12, F(3) = 4.22/13, F(4) = 4.58/14 (best), F(5) = 4.88/15, F(6) = 5.15/16
    conf = np.array([[0.9, 0.8, 0.5], [0.6, 0.5, 0.9]], np.float32)
    tau = (10.0 + np.arange(7)).astype(np.float32)
    out = oracle_mod.schedule_verify_len(conf, None, tau, budget=6, min_len=1)
    assert list(out["len"]) == [3, 1]
    assert out["n"] == 4
    assert abs(out["expected_tokens"] - 4.58) < 1e-6
    assert abs(out["tokens_per_us"] - 4.58 / 14) < 1e-7
    # a budget of 3 caps the search at n = 3
    out = oracle_mod.schedule_verify_len(conf, None, tau, budget=3, min_len=1)
    assert list(out["len"]) == [2, 1] and out["n"] == 3


def test_full_search_beats_first_drop(oracle_mod):
    """Step-shaped table: F = 1/10, 2/11, 3/30, 4/30, 5/20.  The first drop is at
    n = 2 (stopping there keeps n = 1); the whole-table search keeps n = 4."""
    conf = np.ones((1, 4), np.float32)
    tau = np.array([10, 11, 30, 30, 20], np.float32)
    out = oracle_mod.schedule_verify_len(conf, None, tau, budget=4, min_len=0)
    assert out["n"] == 4 and list(out["len"]) == [4]


def _bruteforce(conf, max_len, tau, budget, min_len):
    B, K = conf.shape
    c = np.clip(np.nan_to_num(conf.astype(np.float64), nan=0.0), 0.0, 1.0)
    S = np.cumprod(c, axis=1)
    ml = [K if max_len is None else int(np.clip(max_len[b], 0, K)) for b in range(B)]
    lo = [min(min_len, ml[b]) for b in range(B)]
    best = -np.inf
    for L in itertools.product(*[range(lo[b], ml[b] + 1) for b in range(B)]):
        n = sum(L)
        if n > budget or n > len(tau) - 1 or tau[n] <= 0:
            continue
        E = sum(S[b, :L[b]].sum() for b in range(B))
        best = max(best, (B + E) / float(tau[n]))
    return best


@pytest.mark.parametrize("seed", range(12))
def test_exhaustive_search_agrees(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    B, K = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    conf = rng.beta(4, 1.5, size=(B, K)).astype(np.float32)
    if seed % 3 == 0:
        conf[0, -1] = 1.0  # survival plateau: tie broken by position
    max_len = rng.integers(0, K + 1, size=B).astype(np.int32) if seed % 2 else None
    n_tab = B * K + 1
    base = rng.uniform(5, 15)
    tau = (base + rng.uniform(0.0, 3.0) * np.arange(n_tab) + 4.0 * (np.arange(n_tab) > n_tab // 2)
           ).astype(np.float32)
    min_len = int(rng.integers(0, 2))
    budget = int(rng.integers(B * min_len, B * K + 1))
    out = oracle_mod.schedule_verify_len(conf, max_len, tau, budget, min_len)
    bf = _bruteforce(conf, max_len, tau, budget, min_len)
    assert abs(out["tokens_per_us"] - bf) <= 1e-9 * bf
    # the allocation achieves it and respects the limits
    c = np.clip(conf.astype(np.float64), 0, 1)
    S = np.cumprod(c, axis=1)
    L = out["len"]
    assert L.sum() == out["n"] <= budget
    E = sum(S[b, :L[b]].sum() for b in range(B))
    assert abs((B + E) / float(tau[L.sum()]) - bf) <= 1e-9 * bf
    for b in range(B):
        mlb = K if max_len is None else int(max_len[b])
        assert min(min_len, mlb) <= L[b] <= mlb


def test_expected_accepted_length_monte_carlo():
    """Sum of prefix products = E[number accepted] when position i is accepted with
    probability c_i given that every earlier one was (sequential acceptance)."""
    rng = np.random.default_rng(0)
    c = np.array([0.9, 0.7, 0.95, 0.5, 0.8])
    N = 400000
    acc = rng.random((N, c.size)) < c
    first_fail = np.where(acc.all(axis=1), c.size, np.argmin(acc, axis=1))
    mc = first_fail.mean()
    closed = np.cumprod(c).sum()
    assert abs(mc - closed) < 5 * first_fail.std() / np.sqrt(N)


def test_expected_tokens_report(oracle_mod):
    conf = np.array([[0.9, 0.7, 0.95, 0.5, 0.8]], np.float32)
    tau = np.full(6, 10.0, np.float32)  # flat table: verify everything
    out = oracle_mod.schedule_verify_len(conf, None, tau, budget=5, min_len=0)
    assert out["n"] == 5
    assert abs(out["expected_tokens"] - (1 + np.cumprod(conf[0].astype(np.float64)).sum())) < 1e-12


def test_clamping_and_bad_arguments(oracle_mod):
    conf = np.array([[1.5, np.nan, 0.5], [-0.2, 0.9, 0.9]], np.float32)
    tau = np.full(7, 10.0, np.float32)
    out = oracle_mod.schedule_verify_len(conf, None, tau, budget=6, min_len=0)
    # clamped: S_0 = [1, 0, 0], S_1 = [0, 0, 0]; flat table -> take all (ties go to the smallest n
    # only when F is equal; adding zero-survival slots keeps F equal, so n stays at the first max)
    assert out["n"] == 1 and list(out["len"]) == [1, 0]
    assert oracle_mod.schedule_verify_len(conf, None, tau, budget=1, min_len=1) is None
    assert oracle_mod.schedule_verify_len(conf, None, tau[:2], budget=6, min_len=1) is None


def test_prefix_property_and_budget(oracle_mod):
    rng = np.random.default_rng(4)
    B, K = 64, 16
    conf = (rng.beta(4, 1.5, size=(B, K)) * 0.95 ** np.arange(K)).astype(np.float32)
    tau = (12 + 0.02 * np.arange(1025)).astype(np.float32)
    for budget in (64, 300, 1024):
        out = oracle_mod.schedule_verify_len(conf, None, tau, budget=budget, min_len=1)
        L = out["len"]
        assert L.sum() == out["n"] <= budget and (L >= 1).all() and (L <= K).all()
        # every kept slot has survival >= every dropped slot (ranking by survival)
        S = np.cumprod(conf.astype(np.float64), axis=1)
        kept = [S[b, i] for b in range(B) for i in range(1, L[b])]
        dropped = [S[b, i] for b in range(B) for i in range(L[b], K)]
        if kept and dropped:
            assert min(kept) >= max(dropped)


# ---------------------------------------------------------------------------
# Scheduler variants: static threshold truncation ("Accelerating Large-Model
# Inference ... DSpark", prefix scheduler: scan left to right, truncate at the
# first score below the threshold; "DSpark paper review" Sec. 3: a fixed cutoff)
# and two-step-stale batch sizing ("DSpark paper review" Sec. 4.2.2: the batch
# size from the scores of two steps earlier, the tokens from the latest ones).

def test_threshold_hand_computed(oracle_mod):
    conf = np.array([[0.9, 0.8, 0.3, 0.9], [0.2, 0.9, 0.9, 0.9], [0.5, 0.5, 0.5, 0.5]], np.float32)
    assert list(oracle_mod.schedule_threshold(conf, None, 0.5)) == [2, 0, 4]  # 0.5 >= 0.5 is kept
    assert list(oracle_mod.schedule_threshold(conf, np.array([1, 3, 2], np.int32), 0.5)) == [1, 0, 2]
    assert list(oracle_mod.schedule_threshold(conf, None, 0.0)) == [4, 4, 4]
    assert list(oracle_mod.schedule_threshold(conf, None, 1.01)) == [0, 0, 0]


def test_threshold_nan_truncates(oracle_mod):
    conf = np.array([[0.9, np.nan, 0.9]], np.float32)
    assert list(oracle_mod.schedule_threshold(conf, None, 0.1)) == [1]
    assert oracle_mod.schedule_threshold(conf, None, float("nan")) is None


@pytest.mark.parametrize("seed", range(5))
def test_threshold_invariants(oracle_mod, seed):
    """Every kept position is at or above the threshold, the first cut one is
    below it, and raising the threshold never lengthens a draft."""
    rng = np.random.default_rng(seed)
    B, K = 200, 16
    conf = (rng.beta(4, 1.5, size=(B, K)) * 0.95 ** np.arange(K)).astype(np.float32)
    ml = rng.integers(0, K + 1, size=B).astype(np.int32)
    prev = None
    for thr in (0.2, 0.4, 0.6, 0.8):
        L = oracle_mod.schedule_threshold(conf, ml, thr)
        for b in range(B):
            assert 0 <= L[b] <= ml[b]
            assert (conf[b, :L[b]] >= np.float32(thr)).all()
            if L[b] < ml[b]:
                assert conf[b, L[b]] < np.float32(thr)
        if prev is not None:
            assert (L <= prev).all()
        prev = L


def test_stale_equals_plain_when_scores_agree(oracle_mod):
    rng = np.random.default_rng(3)
    conf = rng.beta(4, 1.5, size=(20, 6)).astype(np.float32)
    tau = (12 + 0.3 * np.arange(121)).astype(np.float32)
    a = oracle_mod.schedule_verify_len(conf, None, tau, 90, 1)
    s = oracle_mod.schedule_verify_len_stale(conf, conf, None, tau, 90, 1)
    assert (a["len"] == s["len"]).all() and a["n"] == s["n"]
    assert abs(a["expected_tokens"] - s["expected_tokens"]) < 1e-12


def test_stale_hand_computed(oracle_mod):
    """Stale scores size the batch, the latest ones pick the slots.  Stale:
    request 0 confident, request 1 not; latest: the reverse.  min_len 0 and
    tau = 10 + n: F(n) = E(n) / (10 + n)."""
    stale = np.array([[0.9, 0.9], [0.1, 0.1]], np.float32)
    now = np.array([[0.1, 0.1], [0.9, 0.9]], np.float32)
    tau = (10.0 + np.arange(5)).astype(np.float32)
    # stale ranking 0.9, 0.81, 0.1, 0.01: F = 0, 0.9/11, 1.71/12, 1.81/13, 1.82/14 -> n* = 2
    s = oracle_mod.schedule_verify_len_stale(stale, now, None, tau, 4, 0)
    assert s["n"] == 2
    assert list(s["len"]) == [0, 2]  # the two slots go to request 1 under the latest scores
    assert abs(s["expected_tokens"] - (2 + 0.9 + 0.81)) < 1e-6
    assert abs(s["tokens_per_us"] - (2 + 0.9 + 0.81) / 12) < 1e-7


@pytest.mark.parametrize("seed", range(6))
def test_stale_allocation_is_best_for_the_latest_scores(oracle_mod, seed):
    """Exhaustive: among every allocation of n* slots (each request a prefix of at
    least m_b and at most maxlen_b), none has a larger expected accepted length
    under the latest scores."""
    rng = np.random.default_rng(seed)
    B, K = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    stale = rng.uniform(0.05, 1.0, size=(B, K)).astype(np.float32)
    now = rng.uniform(0.05, 1.0, size=(B, K)).astype(np.float32)
    ml = rng.integers(0, K + 1, size=B).astype(np.int32)
    min_len = int(rng.integers(0, 2))
    tau = (8 + rng.uniform(0.5, 3.0) * np.arange(B * K + 1)).astype(np.float32)
    s = oracle_mod.schedule_verify_len_stale(stale, now, ml, tau, B * K, min_len)
    assert s is not None
    surv = np.cumprod(now.astype(np.float64), axis=1)
    mand = np.minimum(min_len, ml)
    best = -1.0
    for L in itertools.product(*[range(int(mand[b]), int(ml[b]) + 1) for b in range(B)]):
        if sum(L) != s["n"]:
            continue
        best = max(best, sum(surv[b, :L[b]].sum() for b in range(B)))
    got = sum(surv[b, :s["len"][b]].sum() for b in range(B))
    assert sum(s["len"]) == s["n"]
    assert got >= best - 1e-12
