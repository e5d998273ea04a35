"""Pins of the oracle's verify/commit step against what the pages and the
mathematics fix (no GPU).

* the worked examples printed on the pages (tests/golden/worked_examples.json);
* closed forms: P(accept | x ~ q) = sum_v min(p_v, q_v), sum_v max(0, p_v - q_v)
  = total-variation distance;
* losslessness by brute-force enumeration of every draft sequence and every
  accept / correct / bonus branch on a prefix-dependent toy model;
* chi-square tests of the oracle's full sampling path (Philox + Gumbel-max)
  against the target's autoregressive distribution and against the exact
  per-branch law;
* greedy ties (lowest index), status codes, bf16 decoding, softmax invariants.
"""
import itertools
import json
import math
import os
from collections import defaultdict

import numpy as np
import pytest
from scipy import special, stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


# ----------------------------------------------------------------- helpers
def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (uint16)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(f)
    out[nan] = 0x7FC0
    return out


def _table_row(spec: dict, vocab: list) -> np.ndarray:
    p = np.zeros(len(vocab))
    for w, pr in spec.items():
        p[vocab.index(w)] = pr
    return p


def _log(p):
    with np.errstate(divide="ignore"):
        return np.log(p)


def _example_arrays(ex, vocab, T):
    K = len(ex["drafts"])
    V = len(vocab)
    target = np.full((1, K + 1, V), np.nan, np.float32)
    draft = np.full((1, K, V), np.nan, np.float32)
    for i, row in enumerate(ex["target"]):
        target[0, i] = T * _log(_table_row(row, vocab))
    for i, row in enumerate(ex["draft"]):
        draft[0, i] = T * _log(_table_row(row, vocab))
    kb = ex["num_draft"]
    if ex.get("unused_rows_nan"):
        target[0, kb + 1:] = np.nan
        draft[0, kb:] = np.nan
    x = np.array([[vocab.index(w) for w in ex["drafts"]]], np.int32)
    return target, draft, x, np.array([kb], np.int32)


# ---------------------------------------------------------- worked examples
@pytest.mark.parametrize("T", [1.0, 0.7])
@pytest.mark.parametrize("as_bf16", [False, True])
def test_worked_examples_every_seed(oracle_mod, T, as_bf16):
    gold = json.load(open(GOLDEN))
    vocab = gold["vocab"]
    for ex in gold["examples"]:
        target, draft, x, kb = _example_arrays(ex, vocab, T)
        if as_bf16:
            target, draft = _bf16_bits(target), _bf16_bits(draft)
        exp_tokens = [vocab.index(w) for w in ex["expected"]["tokens"]]
        for seed in range(25):
            for step in (0, 1, 2**40 + 3):
                out = oracle_mod.verify_sample(target, draft, x, kb, np.array([T], np.float32),
                                               seed, step)
                assert out["status"][0] == 0, ex["name"]
                A = int(out["accepted"][0])
                assert A == ex["expected"]["accepted"], (ex["name"], seed, step)
                assert A + 1 == ex["expected"]["committed"]
                assert list(out["tokens"][0, :A + 1]) == exp_tokens, (ex["name"], seed, step)
                assert (out["tokens"][0, A + 1:] == -1).all()


# ------------------------------------------------------------ closed forms
def _rand_dist(rng, V, zero_frac=0.25):
    p = rng.dirichlet(np.full(V, 0.7))
    p[rng.random(V) < zero_frac] = 0.0
    if p.sum() == 0:
        p[rng.integers(V)] = 1.0
    return p / p.sum()


def test_acceptance_closed_form_exact(oracle_mod):
    """E_{x~q}[min(1, p(x)/q(x))] = sum_v min(p_v, q_v)."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        V = int(rng.integers(2, 9))
        p, q = _rand_dist(rng, V), _rand_dist(rng, V)
        lhs = sum(q[v] * oracle_mod.accept_prob(p[v], q[v]) for v in range(V) if q[v] > 0)
        assert abs(lhs - np.minimum(p, q).sum()) < 1e-14


def test_accept_prob_special_cases(oracle_mod):
    assert oracle_mod.accept_prob(0.3, 0.3) == 1.0
    assert oracle_mod.accept_prob(0.9, 0.3) == 1.0
    assert oracle_mod.accept_prob(0.0, 0.3) == 0.0
    assert oracle_mod.accept_prob(0.2, 0.0) == 1.0
    assert oracle_mod.accept_prob(0.0, 0.0) == 0.0
    assert abs(oracle_mod.accept_prob(0.1, 0.4) - 0.25) < 1e-16


def test_residual_mass_is_total_variation(oracle_mod):
    rng = np.random.default_rng(4)
    for _ in range(200):
        V = int(rng.integers(2, 12))
        p, q = _rand_dist(rng, V), _rand_dist(rng, V)
        r = oracle_mod.residual_weights(p, q)
        assert (r >= 0).all()
        assert abs(r.sum() - 0.5 * np.abs(p - q).sum()) < 1e-14
        # support: exactly where p exceeds q
        assert ((r > 0) == (p > q)).all()


def test_acceptance_rate_empirical_matches_closed_form(oracle_mod):
    """Many requests with the same rows, drafts x ~ q: acceptance at position 0
    lies within a 5-sigma binomial band of sum_v min(p_v, q_v)."""
    rng = np.random.default_rng(5)
    V, N = 8, 40000
    p, q = _rand_dist(rng, V, 0.1), _rand_dist(rng, V, 0.1)
    x = rng.choice(V, size=N, p=q).astype(np.int32)
    target = np.broadcast_to(_log(p).astype(np.float32), (N, 2, V)).copy()
    draft = np.broadcast_to(_log(q).astype(np.float32), (N, 1, V)).copy()
    out = oracle_mod.verify_sample(target, draft, x[:, None], None, np.ones(N, np.float32), 11, 0)
    rate = (out["accepted"] >= 1).mean()
    a = np.minimum(p, q).sum()
    assert abs(rate - a) < 5 * math.sqrt(a * (1 - a) / N), (rate, a)


# ------------------------------------------------- brute-force losslessness
class ToyModel:
    """Prefix-dependent next-token tables p(.|s), q(.|s) over a V-word vocabulary."""

    def __init__(self, V, seed, zero_frac=0.2):
        self.V, self.seed, self.zero_frac = V, seed, zero_frac
        self._p, self._q = {}, {}

    def _draw(self, s, which):
        h = hash((self.seed, which) + tuple(s)) & 0xFFFFFFFF
        return _rand_dist(np.random.default_rng(h), self.V, self.zero_frac)

    def p(self, s):
        s = tuple(s)
        if s not in self._p:
            self._p[s] = self._draw(s, 1)
        return self._p[s]

    def q(self, s):
        s = tuple(s)
        if s not in self._q:
            self._q[s] = self._draw(s, 2)
        return self._q[s]


def _emitted_law(oracle_mod, m: ToyModel, K: int):
    """Exact law of the emitted sequence (accepted drafts + one extra token),
    enumerating every draft sequence and every accept/reject branch with the
    oracle's acceptance rule and residual weights."""
    law = defaultdict(float)
    V = m.V
    for xs in itertools.product(range(V), repeat=K):
        w = 1.0
        for i in range(K):
            w *= m.q(xs[:i])[xs[i]]
        if w == 0.0:
            continue
        reach = w
        for a in range(K + 1):
            if a == K:
                pk = m.p(xs)
                for y in range(V):
                    law[xs + (y,)] += reach * pk[y]
                break
            s = xs[:a]
            alpha = oracle_mod.accept_prob(m.p(s)[xs[a]], m.q(s)[xs[a]])
            if alpha < 1.0:
                r = oracle_mod.residual_weights(m.p(s), m.q(s))
                R = r.sum()
                assert R > 0
                for y in range(V):
                    if r[y] > 0:
                        law[s + (y,)] += reach * (1.0 - alpha) * r[y] / R
            reach *= alpha
            if reach == 0.0:
                break
    return law


@pytest.mark.parametrize("V,K,seed", [(3, 1, 0), (4, 2, 1), (5, 3, 2), (8, 3, 3), (6, 3, 4)])
def test_lossless_bruteforce(oracle_mod, V, K, seed):
    """For every L and emitted prefix s: P(y_L = y | y_<L = s, at least L+1 emitted) = p(y|s)."""
    m = ToyModel(V, seed)
    law = _emitted_law(oracle_mod, m, K)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    for L in range(K + 1):
        joint = defaultdict(lambda: np.zeros(V))
        for e, pr in law.items():
            if len(e) > L:
                joint[e[:L]][e[L]] += pr
        for s, row in joint.items():
            tot = row.sum()
            if tot < 1e-300:
                continue
            np.testing.assert_allclose(row / tot, m.p(s), atol=1e-12, err_msg=f"L={L} s={s}")


def test_lossless_bruteforce_detects_wrong_residual(oracle_mod):
    """Guard on the enumeration itself: the law built with the residual flipped
    (max(0, q - p)) is not the target's."""
    m = ToyModel(5, 9)

    class Flipped:
        accept_prob = staticmethod(oracle_mod.accept_prob)

        @staticmethod
        def residual_weights(p, q):
            return oracle_mod.residual_weights(q, p)

    law = _emitted_law(Flipped, m, 2)
    row = np.zeros(5)
    for e, pr in law.items():
        row[e[0]] += pr
    assert np.abs(row - m.p(())).max() > 1e-3


# --------------------------------------------- chi-square of the full sampler
def _simulate(oracle_mod, m: ToyModel, K, N, seed, T=1.0):
    """N independent requests: drafts proposed autoregressively from q (numpy),
    verified by the oracle's full sampling path (Philox + Gumbel-max)."""
    V = m.V
    rng = np.random.default_rng(seed)
    x = np.zeros((N, K), np.int32)
    target = np.zeros((N, K + 1, V), np.float32)
    draft = np.zeros((N, K, V), np.float32)
    for n in range(N):
        for i in range(K):
            s = tuple(x[n, :i])
            qd = m.q(s)
            x[n, i] = rng.choice(V, p=qd)
            draft[n, i] = T * _log(qd)
            target[n, i] = T * _log(m.p(s))
        target[n, K] = T * _log(m.p(tuple(x[n])))
    out = oracle_mod.verify_sample(target, draft, x, None, np.full(N, T, np.float32), seed, 7)
    assert (out["status"] == 0).all()
    return x, out


def _chi2_ok(counts, probs, alpha=1e-3):
    keep = probs > 0
    assert counts[~keep].sum() == 0, "mass on a zero-probability outcome"
    n = counts.sum()
    exp = probs[keep] * n
    if keep.sum() < 2:
        return True
    chi2, pval = stats.chisquare(counts[keep], exp)
    return pval > alpha


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_chi_square_first_two_emitted_tokens(oracle_mod, T):
    m = ToyModel(6, 21, zero_frac=0.15)
    K, N = 3, 30000
    x, out = _simulate(oracle_mod, m, K, N, seed=123, T=T)
    A = out["accepted"]
    y0 = out["tokens"][np.arange(N), 0]
    assert _chi2_ok(np.bincount(y0, minlength=6), m.p(()))
    sel = A >= 1
    for a in range(6):
        grp = sel & (y0 == a)
        if grp.sum() < 500:
            continue
        y1 = out["tokens"][grp, 1]
        assert _chi2_ok(np.bincount(y1, minlength=6), m.p((a,))), a


def test_chi_square_joint_accept_and_token_fixed_drafts(oracle_mod):
    """Fixed rows and drafts: the joint law of (A, emitted token) is
    prod_{i<A} a_i * (1 - a_A) * r_A / sum r_A, or prod a_i * p_K at A = K."""
    rng = np.random.default_rng(8)
    V, K, N = 5, 3, 60000
    P = [_rand_dist(rng, V, 0.2) for _ in range(K + 1)]
    Q = [_rand_dist(rng, V, 0.2) for _ in range(K)]
    xs = [int(np.argmax(Q[i])) for i in range(K)]
    target = np.broadcast_to(np.stack([_log(p) for p in P]).astype(np.float32), (N, K + 1, V)).copy()
    draft = np.broadcast_to(np.stack([_log(q) for q in Q]).astype(np.float32), (N, K, V)).copy()
    x = np.broadcast_to(np.array(xs, np.int32), (N, K)).copy()
    out = oracle_mod.verify_sample(target, draft, x, None, np.ones(N, np.float32), 77, 1)
    A = out["accepted"]
    tok = out["tokens"][np.arange(N), A]
    probs = np.zeros((K + 1, V))
    reach = 1.0
    for a in range(K + 1):
        if a == K:
            probs[a] = reach * P[K]
            break
        alpha = min(1.0, P[a][xs[a]] / Q[a][xs[a]])
        r = np.maximum(P[a] - Q[a], 0.0)
        if r.sum() > 0:
            probs[a] = reach * (1 - alpha) * r / r.sum()
        reach *= alpha
    counts = np.zeros((K + 1, V))
    np.add.at(counts, (A, tok), 1)
    assert _chi2_ok(counts.ravel(), probs.ravel())


def test_gumbel_sample_frequencies(oracle_mod):
    w = np.array([0.05, 0.0, 0.3, 0.15, 0.0, 0.5])
    N = 30000
    counts = np.zeros(6)
    for n in range(N):
        counts[oracle_mod.gumbel_sample(w, seed=5, step=n, b=n % 7, row=1, purpose=1)] += 1
    assert _chi2_ok(counts, w / w.sum())


def test_gumbel_sample_single_support(oracle_mod):
    w = np.zeros(40)
    w[17] = 1e-30
    for n in range(200):
        assert oracle_mod.gumbel_sample(w, seed=n, step=3) == 17
    assert oracle_mod.gumbel_sample(np.zeros(5), seed=1, step=1) == -1


# ------------------------------------------------------------ softmax rows
def test_row_logprobs_vs_scipy_and_invariants(oracle_mod):
    rng = np.random.default_rng(6)
    for V in (1, 2, 7, 1000):
        x = rng.normal(0, 4, V)
        for T in (1.0, 0.6, 2.5):
            lp = oracle_mod.row_logprobs(x, T)
            np.testing.assert_allclose(lp, special.log_softmax(x / T), atol=1e-12)
            assert abs(math.fsum(np.exp(lp)) - 1.0) < 1e-13
            np.testing.assert_allclose(oracle_mod.row_logprobs(x + 123.25, T), lp, atol=1e-11)
    lp = oracle_mod.row_logprobs(np.array([0.0, -np.inf, 1.0]), 1.0)
    assert lp[1] == -np.inf and abs(np.exp(lp[0]) + np.exp(lp[2]) - 1) < 1e-15


# ------------------------------------------------------------------- greedy
def test_greedy_ties_lowest_index_and_paths(oracle_mod):
    V, K = 9, 3
    t = np.zeros((3, K + 1, V), np.float32)
    # request 0: ties at the max in every row, draft = lowest tied index -> all accepted
    for i in range(K + 1):
        t[0, i, [2, 5]] = 4.0
    # request 1: first position mismatch (draft picks the higher tied index)
    t[1, :, [3, 7]] = 2.5
    # request 2: argmax 1, 2, 3, then bonus row argmax 8
    for i in range(K):
        t[2, i, i + 1] = 1.0
    t[2, K, 8] = 0.5
    x = np.array([[2, 2, 2], [7, 3, 3], [1, 2, 3]], np.int32)
    out = oracle_mod.verify_greedy(t, x, None)
    assert list(out["accepted"]) == [3, 0, 3]
    assert list(out["tokens"][0]) == [2, 2, 2, 2]
    assert list(out["tokens"][1]) == [3, -1, -1, -1]
    assert list(out["tokens"][2]) == [1, 2, 3, 8]
    # sampling entry point with T = 0 is the same greedy rule; draft logits unread (NaN)
    d = np.full((3, K, V), np.nan, np.float32)
    out2 = oracle_mod.verify_sample(t, d, x, None, np.zeros(3, np.float32), 1, 1)
    assert (out2["tokens"] == out["tokens"]).all() and (out2["status"] == 0).all()


def test_greedy_ragged_k(oracle_mod):
    V, K = 6, 4
    rng = np.random.default_rng(2)
    t = rng.normal(size=(2, K + 1, V)).astype(np.float32)
    x = np.argmax(t[:, :K], axis=-1).astype(np.int32)
    t[0, 2:] = np.nan  # k_0 = 1: rows 0..1 needed only
    out = oracle_mod.verify_greedy(t, x, np.array([1, 0], np.int32))
    assert list(out["accepted"]) == [1, 0]
    assert out["tokens"][0, 0] == x[0, 0] and out["tokens"][0, 1] == np.argmax(t[0, 1])
    assert out["tokens"][1, 0] == np.argmax(t[1, 0]) and (out["tokens"][1, 1:] == -1).all()


# --------------------------------------------------------------- statuses
def test_status_codes(oracle_mod):
    V, K, B = 7, 2, 7
    rng = np.random.default_rng(9)
    t = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    d = rng.normal(size=(B, K, V)).astype(np.float32)
    x = rng.integers(0, V, size=(B, K)).astype(np.int32)
    nd = np.full(B, K, np.int32)
    T = np.ones(B, np.float32)
    nd[1] = K + 1          # k_b out of range -> 2
    T[2] = -0.5            # bad temperature -> 3
    x[3, 1] = V            # token out of range -> 1
    t[4, 1, 3] = np.nan    # NaN in a needed row -> 4
    d[5, 0, :] = -np.inf   # all -inf draft row -> 4
    t[6, 0, 2] = np.inf    # +inf -> 4
    out = oracle_mod.verify_sample(t, d, x, nd, T, 3, 3)
    assert list(out["status"]) == [0, 2, 3, 1, 4, 4, 4]
    for b in range(1, B):
        assert out["accepted"][b] == 0 and (out["tokens"][b] == -1).all()
    T2 = np.ones(B, np.float32)
    T2[0] = np.nan
    T2[1] = np.inf
    out = oracle_mod.verify_sample(t, d, x, None, T2, 3, 3)
    assert out["status"][0] == 3 and out["status"][1] == 3


def test_unneeded_rows_are_not_read(oracle_mod):
    V, K = 11, 5
    rng = np.random.default_rng(10)
    t = rng.normal(size=(1, K + 1, V)).astype(np.float32)
    d = rng.normal(size=(1, K, V)).astype(np.float32)
    x = rng.integers(0, V, size=(1, K)).astype(np.int32)
    ref = oracle_mod.verify_sample(t, d, x, np.array([2], np.int32), np.ones(1, np.float32), 4, 4)
    t[0, 3:] = np.nan
    d[0, 2:] = np.nan
    out = oracle_mod.verify_sample(t, d, x, np.array([2], np.int32), np.ones(1, np.float32), 4, 4)
    assert out["status"][0] == 0
    assert (out["tokens"] == ref["tokens"]).all()


def test_bf16_decoding_matches_fp32_of_same_values(oracle_mod):
    rng = np.random.default_rng(12)
    B, K, V = 5, 3, 300
    t32 = rng.normal(0, 3, size=(B, K + 1, V)).astype(np.float32)
    d32 = (t32[:, :K] + rng.normal(0, 1, size=(B, K, V))).astype(np.float32)
    tb, db = _bf16_bits(t32), _bf16_bits(d32)
    # bf16 values widened exactly to fp32
    tw = (tb.astype(np.uint32) << 16).view(np.float32)
    dw = (db.astype(np.uint32) << 16).view(np.float32)
    x = rng.integers(0, V, size=(B, K)).astype(np.int32)
    T = np.full(B, 0.8, np.float32)
    a = oracle_mod.verify_sample(tb, db, x, None, T, 9, 9)
    b = oracle_mod.verify_sample(tw, dw, x, None, T, 9, 9)
    for k in ("tokens", "accepted", "status"):
        assert (a[k] == b[k]).all()
    np.testing.assert_array_equal(a["p"], b["p"])


def test_zero_drafts_is_a_bonus_draw(oracle_mod):
    """k_b = 0: nothing to verify; the one emitted token is drawn from target row 0."""
    V, N = 4, 20000
    p = np.array([0.1, 0.2, 0.3, 0.4])
    t = np.broadcast_to(_log(p).astype(np.float32), (N, 1, V)).copy()
    d = np.zeros((N, 0, V), np.float32)
    out = oracle_mod.verify_sample(t, d, np.zeros((N, 0), np.int32), None, np.ones(N, np.float32), 2, 2)
    assert (out["accepted"] == 0).all()
    assert _chi2_ok(np.bincount(out["tokens"][:, 0], minlength=V), p)


def _bonus_row_case(kind):
    """Request with K = 2 whose target row 2 (after the last draft) is NaN."""
    V, K = 16, 2
    rng = np.random.default_rng(21)
    p = [_rand_dist(rng, V, 0.0) for _ in range(K)]
    t = np.zeros((1, K + 1, V), np.float32)
    d = np.zeros((1, K, V), np.float32)
    for i in range(K):
        t[0, i] = np.log(p[i])
        d[0, i] = np.log(p[i])  # q == p: every draft accepted
    t[0, K] = np.nan
    x = np.array([[int(np.argmax(p[0])), int(np.argmax(p[1]))]], np.int32)
    if kind == "reject":
        t[0, 0, x[0, 0]] = -np.inf  # p(x_0) = 0: rejected at position 0, row 2 never read
    return t, d, x


def test_bonus_row_checked_only_when_read(oracle_mod):
    t, d, x = _bonus_row_case("accept")
    out = oracle_mod.verify_sample(t, d, x, None, np.ones(1, np.float32), 1, 1)
    assert out["status"][0] == 4 and out["accepted"][0] == 0
    assert (out["tokens"] == -1).all() and (out["p"] == -1).all()
    g = oracle_mod.verify_greedy(t, x, None)
    assert g["status"][0] == 4 and (g["tokens"] == -1).all()
    t, d, x = _bonus_row_case("reject")
    out = oracle_mod.verify_sample(t, d, x, None, np.ones(1, np.float32), 1, 1)
    assert out["status"][0] == 0 and out["accepted"][0] == 0 and out["tokens"][0, 0] >= 0
    g = oracle_mod.verify_greedy(t, x, None)
    assert g["status"][0] == 0 and g["accepted"][0] == 0
