"""Pins of the oracle's Markov-head drafting ("Accelerating Large-Model Inference ...
DSpark", drafting-engine table, layer 2: a low-rank bias applied left to right, set
at position k+1 by the token chosen at position k; "DSpark paper review" Sec. 4.1;
"Bringing DSpark to vLLM Metal", "Making the draft cheaper": top-K Markov drafting).

Each pin fixes the oracle by something other than its own formula: hand-computed
rank-1 chains, the page's "of course / no problem" example, the reduction to plain
Gumbel-max sampling when the factors vanish, the exact joint law of a two-token
block against the empirical law of many draws, and the top-K special cases.
"""
import itertools

import numpy as np
import pytest
from scipy import stats


def _bf16_bits(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)  # exact for values with 8 significant bits


def test_rank1_hand_chains(oracle_mod):
    """V=3, r=1: emb = (1, 0, -1), proj = (2, 0, -2), zero base logits.  The bias row
    after token p is emb[p] * proj: p=0 -> (2, 0, -2), p=2 -> (-2, 0, 2), p=1 -> 0."""
    U = np.zeros((3, 4, 3), np.float32)
    emb = np.array([[1], [0], [-1]], np.float32)
    proj = np.array([[2], [0], [-2]], np.float32)
    out = oracle_mod.markov_draft(U, np.array([0, 2, 1], np.int32), emb, proj, None, 1, 1)
    assert out["tokens"].tolist() == [[0, 0, 0, 0], [2, 2, 2, 2], [0, 0, 0, 0]]
    assert out["logits"][0, 0].tolist() == [2.0, 0.0, -2.0]
    assert out["logits"][1, 0].tolist() == [-2.0, 0.0, 2.0]
    assert out["logits"][2, 0].tolist() == [0.0, 0.0, 0.0]
    assert out["logits"][2, 1].tolist() == [2.0, 0.0, -2.0]  # after the tie went to token 0
    assert out["status"].tolist() == [0, 0, 0]
    assert out["tie"].tolist() == [4, 4, 0]  # the exact tie at request 2, position 0
    # the same chains from bf16 bit patterns
    outb = oracle_mod.markov_draft(_bf16_bits(U), np.array([0, 2, 1], np.int32), _bf16_bits(emb),
                                   _bf16_bits(proj), None, 1, 1)
    assert (outb["tokens"] == out["tokens"]).all() and (outb["logits"] == out["logits"]).all()


def test_page_example_pairs_stay_coherent(oracle_mod):
    """"DSpark paper review" Sec. 4.1: both "of course" and "no problem" fit; the
    backbone alone guesses of/no then course/problem; once position 1 drew "of",
    the head boosts "course" and suppresses "problem" at position 2."""
    OF, NO, COURSE, PROBLEM = range(4)
    B = 4000
    U = np.full((B, 2, 4), -20.0, np.float32)
    U[:, 0, [OF, NO]] = 5.0
    U[:, 1, [COURSE, PROBLEM]] = 5.0
    emb = np.zeros((4, 2), np.float32)
    emb[OF] = [1, 0]
    emb[NO] = [0, 1]
    proj = np.zeros((4, 2), np.float32)
    proj[COURSE] = [10, -10]
    proj[PROBLEM] = [-10, 10]
    anchor = np.full(B, COURSE, np.int32)  # emb[course] = 0: no bias at the first position
    out = oracle_mod.markov_draft(U, anchor, emb, proj, np.ones(B, np.float32), 17, 3, nthreads=4,
                                  want_logits=False)
    pairs = [tuple(t) for t in out["tokens"].tolist()]
    assert set(pairs) == {(OF, COURSE), (NO, PROBLEM)}
    n_of = sum(p[0] == OF for p in pairs)
    assert abs(n_of - B / 2) < 5 * np.sqrt(B / 4)
    # without the head the pairs mix
    out0 = oracle_mod.markov_draft(U, anchor, np.zeros_like(emb), proj, np.ones(B, np.float32), 17, 3,
                                   nthreads=4, want_logits=False)
    assert set(tuple(t) for t in out0["tokens"].tolist()) == {(OF, COURSE), (OF, PROBLEM), (NO, COURSE),
                                                              (NO, PROBLEM)}


def test_zero_factors_reduce_to_gumbel_sampling(oracle_mod):
    """With emb = 0 the corrected logits are the base logits and every position is
    an independent draw from softmax(U / T) with purpose-3 noise at row k."""
    rng = np.random.default_rng(3)
    B, K, V, r = 5, 3, 40, 4
    U = rng.normal(scale=2.0, size=(B, K, V)).astype(np.float32)
    emb = np.zeros((V, r), np.float32)
    proj = rng.normal(size=(V, r)).astype(np.float32)
    T = np.array([0.5, 0.8, 1.0, 1.3, 2.0], np.float32)
    out = oracle_mod.markov_draft(U, np.arange(B, dtype=np.int32), emb, proj, T, 99, 7)
    assert (out["logits"] == U.astype(np.float64)).all()
    for b in range(B):
        for k in range(K):
            w = np.exp(U[b, k].astype(np.float64) / T[b] - (U[b, k] / T[b]).max())
            assert out["tokens"][b, k] == oracle_mod.gumbel_sample(w, 99, 7, b=b, row=k, purpose=3)
    g = oracle_mod.markov_draft(U, np.arange(B, dtype=np.int32), emb, proj, None, 99, 7)
    assert (g["tokens"] == U.argmax(-1)).all()


def test_two_token_law_chi2(oracle_mod):
    """V=5, r=2, K=2, T=0.9: the empirical law of (x_0, x_1) over 20000 draws against
    the exact law P(x_0) P(x_1 | x_0), each factor a softmax of the corrected row
    built by hand from the factors."""
    rng = np.random.default_rng(11)
    V, r, T = 5, 2, 0.9
    U1 = rng.normal(size=(2, V))
    emb = rng.normal(size=(V, r))
    proj = rng.normal(size=(V, r))
    a = 3

    def softmax(x):
        e = np.exp(x - x.max())
        return e / e.sum()

    B = 20000
    U = np.broadcast_to(U1.astype(np.float32), (B, 2, V)).copy()
    cnt = np.zeros((V, V))
    for step in range(2):
        # float32 factors: the law below is built from the same rounded values
        out = oracle_mod.markov_draft(U, np.full(B, a, np.int32), emb.astype(np.float32), proj.astype(np.float32),
                                      np.full(B, T, np.float32), 5, step, nthreads=4, want_logits=False)
        for x0, x1 in out["tokens"].tolist():
            cnt[x0, x1] += 1
    emb32, proj32, U32 = (x.astype(np.float32).astype(np.float64) for x in (emb, proj, U1))
    T32 = np.float64(np.float32(T))
    law = np.zeros((V, V))
    for x0, x1 in itertools.product(range(V), range(V)):
        z0 = U32[0] + np.array([emb32[a] @ proj32[v] for v in range(V)])
        z1 = U32[1] + np.array([emb32[x0] @ proj32[v] for v in range(V)])
        law[x0, x1] = softmax(z0 / T32)[x0] * softmax(z1 / T32)[x1]
    exp = law.ravel() * cnt.sum()
    keep = exp >= 5
    chi2 = (((cnt.ravel() - exp) ** 2) / exp)[keep].sum()
    assert stats.chi2.sf(chi2, keep.sum() - 1) > 1e-4


def test_topk_special_cases(oracle_mod):
    rng = np.random.default_rng(2)
    B, K, V, r = 4, 3, 30, 3
    U = rng.normal(scale=2.0, size=(B, K, V)).astype(np.float32)
    emb = rng.normal(size=(V, r)).astype(np.float32)
    proj = (3 * rng.normal(size=(V, r))).astype(np.float32)
    T = np.array([0.0, 0.7, 1.0, 1.5], np.float32)
    anchor = np.array([1, 5, 7, 29], np.int32)
    full = oracle_mod.markov_draft(U, anchor, emb, proj, T, 4, 4)
    # every candidate: the full vocabulary
    allk = oracle_mod.markov_draft(U, anchor, emb, proj, T, 4, 4, topk=V)
    assert (allk["tokens"] == full["tokens"]).all() and (allk["logits"] == full["logits"]).all()
    # one candidate: the base argmax, whatever the bias
    one = oracle_mod.markov_draft(U, anchor, emb, proj, T, 4, 4, topk=1)
    assert (one["tokens"] == U.argmax(-1)).all()
    # outside the candidates the corrected logits are -inf
    k3 = oracle_mod.markov_draft(U, anchor, emb, proj, T, 4, 4, topk=3)
    assert (np.isfinite(k3["logits"]).sum(-1) == 3).all()
    for b in range(B):
        for k in range(K):
            top3 = set(np.argsort(-U[b, k], kind="stable")[:3].tolist())
            assert set(np.nonzero(np.isfinite(k3["logits"][b, k]))[0].tolist()) == top3
            assert k3["tokens"][b, k] in top3


def test_topk_excludes_a_token_the_bias_would_pick(oracle_mod):
    """U = (3, 2, 1, 0) with a bias of +10 on token 3 after the anchor: the full draft
    picks 3, the top-2 draft can only pick among (0, 1); ties at the cut keep the
    lower index."""
    U = np.array([[[3.0, 2.0, 1.0, 0.0]]], np.float32)
    emb = np.array([[1.0], [0.0], [0.0], [0.0]], np.float32)
    proj = np.array([[0.0], [0.0], [0.0], [10.0]], np.float32)
    a = np.array([0], np.int32)
    assert oracle_mod.markov_draft(U, a, emb, proj, None, 1, 1)["tokens"].tolist() == [[3]]
    t2 = oracle_mod.markov_draft(U, a, emb, proj, None, 1, 1, topk=2)
    assert t2["tokens"].tolist() == [[0]] and t2["logits"][0, 0].tolist()[2:] == [-np.inf, -np.inf]
    Ut = np.array([[[1.0, 1.0, 1.0, 0.0]]], np.float32)
    t2t = oracle_mod.markov_draft(Ut, a, emb, proj, None, 1, 1, topk=2)
    assert np.isfinite(t2t["logits"][0, 0]).tolist() == [True, True, False, False]


@pytest.mark.parametrize("topk", [0, 4])
def test_status_codes(oracle_mod, topk):
    rng = np.random.default_rng(8)
    B, K, V, r = 5, 3, 16, 2
    U = rng.normal(size=(B, K, V)).astype(np.float32)
    emb = rng.normal(size=(V, r)).astype(np.float32)
    proj = rng.normal(size=(V, r)).astype(np.float32)
    anchor = np.array([-1, V, 3, 3, 3], np.int32)
    T = np.array([1.0, 1.0, np.nan, 1.0, 0.0], np.float32)
    U[3, 1, 9] = np.nan  # a NaN is always a candidate
    U[4, 2, :] = -np.inf
    out = oracle_mod.markov_draft(U, anchor, emb, proj, T, 1, 1, topk=topk)
    assert out["status"].tolist() == [1, 1, 3, 4, 4]
    assert (out["tokens"] == -1).all()
    ok = oracle_mod.markov_draft(U[:1], np.array([2], np.int32), emb, proj, T[:1], 1, 1, topk=topk)
    assert ok["status"].tolist() == [0] and (ok["tokens"] >= 0).all()
