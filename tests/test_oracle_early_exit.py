"""Pins of the oracle's early-exit mode (rows read in position order, reading stops
at the first rejection): the worked examples give the same commits; on random
batches the accepted counts, tokens and statuses equal the full scan's and p / q
equal it up to the first rejected position; a non-finite row after the first
rejection is never seen, one at or before it gives status 4."""
import json
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _table(ex, vocab, T):
    from test_oracle_verify import _example_arrays

    return _example_arrays(ex, vocab, T)


def test_worked_examples_same_commit(oracle_mod):
    gold = json.load(open(GOLDEN))
    vocab = gold["vocab"]
    for ex in gold["examples"]:
        target, draft, x, kb = _table(ex, vocab, 1.0)
        exp_tokens = [vocab.index(w) for w in ex["expected"]["tokens"]]
        for seed in range(10):
            out = oracle_mod.verify_sample(target, draft, x, kb, np.array([1.0], np.float32), seed, 3,
                                           early_exit=True)
            A = int(out["accepted"][0])
            assert out["status"][0] == 0
            assert A == ex["expected"]["accepted"]
            assert list(out["tokens"][0, :A + 1]) == exp_tokens


def _check_same_as_full(oracle_mod, batch, seed, step):
    nd = batch.get("num_draft")
    args = (synth.as_oracle_array(batch["target"]), synth.as_oracle_array(batch["draft"]),
            batch["draft_tokens"].numpy(), None if nd is None else np.asarray(nd, np.int32),
            batch["temperature"].numpy(), seed, step)
    full = oracle_mod.verify_sample(*args, nthreads=4)
    ee = oracle_mod.verify_sample(*args, nthreads=4, early_exit=True)
    assert (ee["status"] == full["status"]).all()
    assert (ee["accepted"] == full["accepted"]).all()
    assert (ee["tokens"] == full["tokens"]).all()
    assert (ee["flags"] == full["flags"]).all()
    T = batch["temperature"].numpy()
    K = full["p"].shape[1]
    for b in range(full["p"].shape[0]):
        if full["status"][b] != 0 or T[b] == 0:
            continue
        A = int(full["accepted"][b])
        n = min(A + 1, K)  # positions read: up to and including the first rejection
        assert (ee["p"][b, :n] == full["p"][b, :n]).all()
        assert (ee["q"][b, :n] == full["q"][b, :n]).all()
        assert (ee["p"][b, n:] == -1).all() and (ee["q"][b, n:] == -1).all()
    return full


@pytest.mark.parametrize("step", [0, 1])
def test_same_as_full_scan_small(oracle_mod, step):
    b = synth.small(step)
    _check_same_as_full(oracle_mod, b, b["seed"], step)


def test_same_as_full_scan_tiny_many_steps(oracle_mod):
    for step in range(200):
        b = synth.tiny(step)
        _check_same_as_full(oracle_mod, b, b["seed"], step)


def _planted(rng, B=6, K=5, V=40):
    t = rng.normal(scale=2.0, size=(B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(size=(B, K, V))).astype(np.float32)
    x = rng.integers(0, V, size=(B, K)).astype(np.int32)
    return t, d, x


def test_nonfinite_after_first_rejection_is_not_read(oracle_mod):
    rng = np.random.default_rng(5)
    t, d, x = _planted(rng)
    B, K1, V = t.shape
    K = K1 - 1
    T = np.full(B, 0.9, np.float32)
    clean = oracle_mod.verify_sample(t, d, x, None, T, 11, 7)
    t2, d2 = t.copy(), d.copy()
    seen = 0
    for b in range(B):
        A = int(clean["accepted"][b])
        if A + 1 < K:  # plant NaN / +inf strictly after the first rejected position
            t2[b, A + 1, 0] = np.nan
            d2[b, K - 1, 1] = np.inf
            seen += 1
    assert seen > 0
    full = oracle_mod.verify_sample(t2, d2, x, None, T, 11, 7)
    ee = oracle_mod.verify_sample(t2, d2, x, None, T, 11, 7, early_exit=True)
    for b in range(B):
        A = int(clean["accepted"][b])
        if A + 1 < K:
            assert full["status"][b] == 4
            assert ee["status"][b] == 0
            assert ee["accepted"][b] == A
            assert (ee["tokens"][b] == clean["tokens"][b]).all()


def test_nonfinite_at_or_before_first_rejection_is_status_4(oracle_mod):
    rng = np.random.default_rng(6)
    t, d, x = _planted(rng)
    B, K1, V = t.shape
    T = np.full(B, 0.9, np.float32)
    clean = oracle_mod.verify_sample(t, d, x, None, T, 12, 1)
    for b in range(B):
        A = int(clean["accepted"][b])
        j = min(A, K1 - 2)
        for which in ("t", "d"):
            t2, d2 = t.copy(), d.copy()
            (t2 if which == "t" else d2)[b, j, 3] = np.nan
            ee = oracle_mod.verify_sample(t2, d2, x, None, T, 12, 1, early_exit=True)
            assert ee["status"][b] == 4 and ee["accepted"][b] == 0
            assert (ee["tokens"][b] == -1).all() and (ee["p"][b] == -1).all()


def test_greedy_early_exit(oracle_mod):
    rng = np.random.default_rng(7)
    B, K, V = 8, 4, 30
    t = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    y = np.argmax(t[:, :K], axis=-1).astype(np.int32)
    x = y.copy()
    for b in range(B):  # request b mismatches at position b % (K + 1) (none when b % (K + 1) == K)
        j = b % (K + 1)
        if j < K:
            x[b, j] = (y[b, j] + 1) % V
    full = oracle_mod.verify_greedy(t, x, None)
    ee = oracle_mod.verify_greedy(t, x, None, early_exit=True)
    assert (ee["accepted"] == full["accepted"]).all() and (ee["tokens"] == full["tokens"]).all()
    assert list(full["accepted"]) == [b % (K + 1) for b in range(B)]
    # NaN after the mismatch: unseen by the early exit, status 4 for the full scan
    t2 = t.copy()
    for b in range(B):
        j = b % (K + 1)
        if j + 1 < K:
            t2[b, j + 1:K, 0] = np.nan
    full2 = oracle_mod.verify_greedy(t2, x, None)
    ee2 = oracle_mod.verify_greedy(t2, x, None, early_exit=True)
    for b in range(B):
        j = b % (K + 1)
        if j + 1 < K:
            assert full2["status"][b] == 4 and ee2["status"][b] == 0
            assert (ee2["tokens"][b] == full["tokens"][b]).all()
