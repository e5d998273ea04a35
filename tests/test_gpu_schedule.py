"""GPU parity of the confidence-scheduled verify-length kernel against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _gpu(conf, max_len, tau, budget, min_len):
    import speculative_decoding_verification_15_gb300 as pkg

    c = torch.as_tensor(conf, dtype=torch.float32, device="cuda")
    ml = None if max_len is None else torch.as_tensor(max_len, dtype=torch.int32, device="cuda")
    t = torch.as_tensor(tau, dtype=torch.float32, device="cuda")
    L, info = pkg.schedule_verify_len(c, t, budget, min_len, max_len=ml)
    torch.cuda.synchronize()
    return L.cpu().numpy(), info.cpu().numpy()


def _check(conf, max_len, tau, budget, min_len):
    ref = oracle.schedule_verify_len(conf, max_len, tau, budget, min_len)
    L, info = _gpu(conf, max_len, tau, budget, min_len)
    if ref["flags"] == 0:
        assert (L == ref["len"]).all(), (L, ref["len"])
        assert int(info[0]) == ref["n"]
    assert abs(info[1] - ref["expected_tokens"]) <= 1e-9 * max(1.0, ref["expected_tokens"]) or ref["flags"]
    assert abs(info[2] - ref["tokens_per_us"]) <= 1e-9 * max(1.0, ref["tokens_per_us"]) or ref["flags"]
    return ref["flags"]


def test_hand_computed():
    conf = np.array([[0.9, 0.8, 0.5], [0.6, 0.5, 0.9]], np.float32)
    tau = (10.0 + np.arange(7)).astype(np.float32)
    L, info = _gpu(conf, None, tau, 6, 1)
    assert list(L) == [3, 1] and int(info[0]) == 4 and abs(info[1] - 4.58) < 1e-6


def test_full_search_step_table():
    L, info = _gpu(np.ones((1, 4), np.float32), None, np.array([10, 11, 30, 30, 20], np.float32), 4, 0)
    assert int(info[0]) == 4 and list(L) == [4]


@pytest.mark.parametrize("seed", range(10))
def test_random_parity(seed):
    rng = np.random.default_rng(seed)
    B, K = int(rng.integers(1, 300)), int(rng.integers(1, 17))
    conf = (rng.beta(4, 1.5, size=(B, K)) * 0.95 ** np.arange(K)).astype(np.float32)
    if seed % 4 == 1:
        conf[rng.random((B, K)) < 0.1] = 1.0
    max_len = rng.integers(0, K + 1, size=B).astype(np.int32) if seed % 2 else None
    n_tab = B * K + 1
    tau = (12 + rng.uniform(0.005, 0.05) * np.arange(n_tab) + 3.0 * (np.arange(n_tab) % 128 == 0).cumsum()
           ).astype(np.float32)
    min_len = int(rng.integers(0, 2))
    budget = int(rng.integers(B * min_len, B * K + 1))
    _check(conf, max_len, tau, budget, min_len)


def test_ragged_workload_scheduler():
    s = synth.ragged_schedule_inputs(0)
    flags = _check(s["conf"].numpy(), None, s["step_time_us"].numpy(), s["budget"], s["min_len"])
    assert flags == 0


def test_largest_supported_batch():
    rng = np.random.default_rng(1)
    B, K = 512, 16  # 8192 slots, the maximum
    conf = rng.beta(4, 1.5, size=(B, K)).astype(np.float32)
    tau = (12 + 0.02 * np.arange(B * K + 1)).astype(np.float32)
    _check(conf, None, tau, 6000, 1)


# ---- scheduler variants: two-step-stale sizing and static threshold truncation

def _gpu_stale(stale, conf, max_len, tau, budget, min_len):
    import speculative_decoding_verification_15_gb300 as pkg

    dev = "cuda"
    ml = None if max_len is None else torch.as_tensor(max_len, dtype=torch.int32, device=dev)
    L, info = pkg.schedule_verify_len_stale(torch.as_tensor(stale, device=dev), torch.as_tensor(conf, device=dev),
                                            torch.as_tensor(tau, device=dev), budget, min_len, max_len=ml)
    torch.cuda.synchronize()
    return L.cpu().numpy(), info.cpu().numpy()


@pytest.mark.parametrize("seed", range(8))
def test_stale_parity(seed):
    rng = np.random.default_rng(100 + seed)
    B, K = int(rng.integers(1, 300)), int(rng.integers(1, 17))
    decay = 0.95 ** np.arange(K)
    stale = (rng.beta(4, 1.5, size=(B, K)) * decay).astype(np.float32)
    conf = (rng.beta(4, 1.5, size=(B, K)) * decay).astype(np.float32)
    max_len = rng.integers(0, K + 1, size=B).astype(np.int32) if seed % 2 else None
    n_tab = B * K + 1
    tau = (12 + 0.02 * np.arange(n_tab)).astype(np.float32)
    min_len = int(rng.integers(0, 2))
    budget = int(rng.integers(B * min_len, B * K + 1))
    ref = oracle.schedule_verify_len_stale(stale, conf, max_len, tau, budget, min_len)
    L, info = _gpu_stale(stale, conf, max_len, tau, budget, min_len)
    assert int(info[0]) == ref["n"] or ref["flags"] & 1
    if ref["flags"] == 0:
        assert (L == ref["len"]).all()
        assert abs(info[1] - ref["expected_tokens"]) <= 1e-9 * max(1.0, ref["expected_tokens"])


def test_stale_ragged_workload():
    """The ragged workload's scheduler inputs, with the stale scores drawn from the
    same law as the latest ones (independently)."""
    s = synth.ragged_schedule_inputs(0)
    conf = s["conf"].numpy()
    rng = np.random.default_rng(7)
    stale = (rng.beta(4, 1.5, size=conf.shape) * 0.95 ** np.arange(conf.shape[1])).astype(np.float32)
    tau = s["step_time_us"].numpy()
    ref = oracle.schedule_verify_len_stale(stale, conf, None, tau, s["budget"], s["min_len"])
    L, info = _gpu_stale(stale, conf, None, tau, s["budget"], s["min_len"])
    assert ref["flags"] == 0
    assert (L == ref["len"]).all() and int(info[0]) == ref["n"]


@pytest.mark.parametrize("seed", range(4))
def test_threshold_parity(seed):
    import speculative_decoding_verification_15_gb300 as pkg

    rng = np.random.default_rng(200 + seed)
    B, K = int(rng.integers(1, 4000)), int(rng.integers(0, 33))
    conf = (rng.beta(4, 1.5, size=(B, K)) * 0.95 ** np.arange(K)).astype(np.float32)
    conf[rng.random((B, K)) < 0.01] = np.nan
    max_len = rng.integers(-1, K + 2, size=B).astype(np.int32) if seed % 2 else None
    for thr in (0.0, 0.3, 0.55, 0.9, 1.5):
        ref = oracle.schedule_threshold(conf, max_len, thr)
        ml = None if max_len is None else torch.as_tensor(max_len, device="cuda")
        L = pkg.schedule_threshold(torch.as_tensor(conf, device="cuda"), thr, max_len=ml)
        torch.cuda.synchronize()
        assert (L.cpu().numpy() == ref).all()
