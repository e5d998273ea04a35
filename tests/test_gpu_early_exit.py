"""Early-exit verify through the C ABI ("Accelerating Large-Model Inference ...
DSpark", Sec. 1: only the accepted prefix and one more token are committed, so the
rows after a request's first rejection are never needed).

The early-exit calls are checked against the oracle's early-exit mode, which reads
rows in position order and stops at the first rejection: statuses everywhere,
tokens and accepted counts away from near-ties, p / q within 1e-5 up to the first
rejected position and -1 after it.  Non-finite rows after the first rejection are
never read (status 0); at or before it they give status 4.  They are also checked
against the two-kernel path on the same inputs, and greedy early exit is bit-exact.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import compare_sample, run_gpu_sample, to_dev

pytestmark = pytest.mark.gpu

CORES = len(os.sched_getaffinity(0))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def _np(out):
    return {k: v.cpu().numpy() for k, v in out.items()}


def gpu_ee_sample(batch, seed, step):
    import speculative_decoding_verification_15_gb300 as pkg

    d = to_dev(batch)
    out = pkg.verify_sample_early_exit(d["target"], d["draft"], d["draft_tokens"], d["temperature"], seed, step,
                                       num_draft=d["num_draft"])
    torch.cuda.synchronize()
    return _np(out)


def gpu_ee_greedy(batch):
    import speculative_decoding_verification_15_gb300 as pkg

    d = to_dev(batch)
    out = pkg.verify_greedy_early_exit(d["target"], d["draft_tokens"], num_draft=d["num_draft"])
    torch.cuda.synchronize()
    return _np(out)


def oracle_ee_sample(batch, seed, step):
    nd = batch.get("num_draft")
    return oracle.verify_sample(synth.as_oracle_array(batch["target"]), synth.as_oracle_array(batch["draft"]),
                                batch["draft_tokens"].numpy(), None if nd is None else np.asarray(nd),
                                batch["temperature"].numpy(), seed, step, nthreads=CORES, early_exit=True)


def oracle_ee_greedy(batch):
    nd = batch.get("num_draft")
    return oracle.verify_greedy(synth.as_oracle_array(batch["target"]), batch["draft_tokens"].numpy(),
                                None if nd is None else np.asarray(nd), nthreads=CORES, early_exit=True)


def test_tiny_many_steps_both_modes():
    """B=1, K=4, V=1024 fp32: 300 steps of independent inputs and seeds."""
    n = flagged = 0
    for step in range(300):
        batch = synth.tiny(step)
        g = gpu_ee_greedy(batch)
        r = oracle_ee_greedy(batch)
        assert (g["tokens"] == r["tokens"]).all() and (g["accepted"] == r["accepted"]).all()
        assert (g["status"] == r["status"]).all()
        res = compare_sample(gpu_ee_sample(batch, batch["seed"], step), oracle_ee_sample(batch, batch["seed"], step),
                             batch["temperature"].numpy())
        n += res["n"]
        flagged += res["flagged"]
    assert flagged <= max(1, n // 200), (flagged, n)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_ragged_mixed_batch(dt):
    """Ragged num_draft (0 and Kmax included), mixed greedy / sampling requests,
    a vocabulary that is not a multiple of the cluster's shares."""
    B, K, V = 24, 7, 50021
    nd = [0, 1, 2, 3, 4, 5, 6, 7] * 3
    batch = synth.make_batch(B, K, V, dt, 123, zipf=True, noise_sigmas=(0.25, 0.5, 1.0, 2.0),
                             temperature=(0.6, 1.3), greedy_mask=[b % 4 == 1 for b in range(B)], num_draft=nd)
    for step in range(2):
        res = compare_sample(gpu_ee_sample(batch, 5, step), oracle_ee_sample(batch, 5, step),
                             batch["temperature"].numpy())
        assert res["flagged"] <= 1


def test_main_batch_full_size():
    """B=64, K=7, V=151936 bf16 (sampling and greedy), and the same tokens as the
    two-kernel path on every request the oracle does not flag."""
    for step in range(2):
        batch = synth.main(step)
        ee = gpu_ee_sample(batch, batch["seed"], step)
        ref = oracle_ee_sample(batch, batch["seed"], step)
        res = compare_sample(ee, ref, batch["temperature"].numpy())
        assert res["flagged"] <= 1
        full = run_gpu_sample(batch, batch["seed"], step)
        ok = ref["flags"] == 0
        assert (ee["tokens"][ok] == full["tokens"][ok]).all()
        assert (ee["accepted"][ok] == full["accepted"][ok]).all()
        K = ee["p"].shape[1]
        for b in np.nonzero(ok)[0]:  # the rows both read: same p / q to rounding
            n = min(int(ee["accepted"][b]) + 1, K)
            assert np.abs(ee["p"][b, :n] - full["p"][b, :n]).max(initial=0) <= 1e-6
            assert (ee["p"][b, n:] == -1).all()
    batch = synth.main(0)
    g = gpu_ee_greedy(batch)
    r = oracle_ee_greedy(batch)
    assert (g["tokens"] == r["tokens"]).all() and (g["accepted"] == r["accepted"]).all()
    assert (g["status"] == 0).all()


def _planted(seed, dt=torch.bfloat16, B=10, K=5, V=70001):
    return synth.make_batch(B, K, V, dt, seed, zipf=True, noise_sigmas=(0.5, 1.0), temperature=(0.8, 1.0))


def test_nonfinite_after_first_rejection_is_not_read():
    batch = _planted(41)
    clean = oracle_ee_sample(batch, 3, 2)
    K = batch["draft_tokens"].shape[1]
    planted = 0
    for b in range(batch["target"].shape[0]):
        A = int(clean["accepted"][b])
        if A + 1 < K:
            batch["target"][b, A + 1, 17] = float("nan")
            batch["draft"][b, K - 1, 5] = float("inf")
            planted += 1
    assert planted > 0
    ee = gpu_ee_sample(batch, 3, 2)
    ref = oracle_ee_sample(batch, 3, 2)
    compare_sample(ee, ref, batch["temperature"].numpy())
    for b in range(batch["target"].shape[0]):
        if clean["flags"][b] == 0:
            assert ee["status"][b] == 0
            assert (ee["tokens"][b] == clean["tokens"][b]).all()


@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_nonfinite_at_or_before_first_rejection_is_status_4(where):
    """NaN in a read row (target or draft) at its first, a middle or its last
    element: status 4 from the early-exit path and from the two-kernel path (a NaN
    early in a long row must survive the running max being replaced by later
    chunks' maxima)."""
    batch = _planted(42)
    V = batch["target"].shape[2]
    col = {"first": 0, "middle": V // 2 + 3, "last": V - 1}[where]
    clean = oracle_ee_sample(batch, 4, 9)
    B = batch["target"].shape[0]
    for b in range(B):
        j = min(int(clean["accepted"][b]), batch["draft_tokens"].shape[1] - 1)
        (batch["target"] if b % 2 == 0 else batch["draft"])[b, j, col] = float("nan")
    ee = gpu_ee_sample(batch, 4, 9)
    full = run_gpu_sample(batch, 4, 9)
    assert (ee["status"] == 4).all(), ee["status"]
    assert (full["status"] == 4).all(), full["status"]
    assert (ee["tokens"] == -1).all() and (ee["accepted"] == 0).all() and (ee["p"] == -1).all()


def test_nonfinite_first_element_full_size():
    """B=64, K=7, V=151936 bf16 with a NaN at the first element of row 0 (always
    read): target row 0 for even requests, draft row 0 for odd ones.  Every lane
    streams several chunks of a row here, so the NaN's chunk is followed by others."""
    batch = synth.main(0)
    B = batch["target"].shape[0]
    for b in range(B):
        (batch["target"] if b % 2 == 0 else batch["draft"])[b, 0, 0] = float("nan")
    ee = gpu_ee_sample(batch, batch["seed"], 0)
    full = run_gpu_sample(batch, batch["seed"], 0)
    assert (ee["status"] == 4).all(), ee["status"]
    assert (full["status"] == 4).all(), full["status"]


def test_greedy_mismatch_and_nan_after_it():
    """Request b mismatches at position b % (K + 1); NaN rows after the mismatch are
    not read (status 0), the full greedy path reports them (status 4)."""
    import speculative_decoding_verification_15_gb300 as pkg

    B, K, V = 12, 5, 40000
    batch = synth.make_batch(B, K, V, torch.bfloat16, 7, zipf=True, noise_sigmas=(0.1,))
    y = batch["target"][:, :K].float().argmax(-1).to(torch.int32)
    x = y.clone()
    for b in range(B):
        j = b % (K + 1)
        if j < K:
            x[b, j] = (y[b, j] + 1) % V
        if j + 1 < K:
            batch["target"][b, j + 1:K, 11] = float("nan")
    batch["draft_tokens"] = x
    g = gpu_ee_greedy(batch)
    r = oracle_ee_greedy(batch)
    assert (g["tokens"] == r["tokens"]).all() and (g["accepted"] == r["accepted"]).all()
    assert (g["status"] == r["status"]).all()
    assert list(g["accepted"]) == [min(b % (K + 1), K) for b in range(B)]
    assert (g["status"] == 0).all()
    d = to_dev(batch)
    full = _np(pkg.verify_greedy(d["target"], d["draft_tokens"]))
    for b in range(B):
        assert full["status"][b] == (4 if b % (K + 1) + 1 < K else 0)


def test_empty_batch_and_zero_drafts():
    import speculative_decoding_verification_15_gb300 as pkg

    V = 3001
    t = torch.randn(0, 4, V, device="cuda")
    out = pkg.verify_sample_early_exit(t, torch.randn(0, 3, V, device="cuda"),
                                       torch.zeros(0, 3, dtype=torch.int32, device="cuda"),
                                       torch.ones(0, device="cuda"), 1, 1)
    assert out["tokens"].shape == (0, 4)
    # Kmax = 0: the bonus token alone
    batch = synth.make_batch(3, 0, V, torch.float32, 9, temperature=(0.7, 0.7), greedy_mask=[True, False, False])
    ee = gpu_ee_sample(batch, 2, 2)
    ref = oracle_ee_sample(batch, 2, 2)
    assert (ee["tokens"] == ref["tokens"]).all() and (ee["accepted"] == 0).all()


def test_status_codes():
    """Bad k_b (status 2), bad draft token (3), bad temperature (1) as the
    two-kernel path reports them."""
    B, K, V = 4, 3, 5000
    batch = synth.make_batch(B, K, V, torch.float32, 3, temperature=(0.9, 0.9))
    batch["num_draft"] = torch.tensor([3, 4, 2, -1], dtype=torch.int32)
    batch["draft_tokens"][2, 1] = V
    batch["temperature"][0] = float("nan")
    ee = gpu_ee_sample(batch, 1, 1)
    full = run_gpu_sample(batch, 1, 1)
    assert (ee["status"] == full["status"]).all(), (ee["status"], full["status"])
    assert list(ee["status"]) == [3, 2, 1, 2]
    assert (ee["tokens"][ee["status"] != 0] == -1).all()
