"""The header's limits and the temperature extremes on the GPU, against the oracle,
through the C ABI: Kmax = SPEC_MAX_DRAFTS (255) with ragged k_b up to it, B =
SPEC_MAX_BATCH (8192) with a small vocabulary, and temperatures 0.05 (logits / T
in the hundreds) and 3.0 (a flat distribution: most groups survive the Gumbel-max
pruning)."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import compare_sample, run_gpu_sample, run_oracle_sample, to_dev

pytestmark = pytest.mark.gpu

CORES = len(os.sched_getaffinity(0))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def _greedy_check(batch):
    import speculative_decoding_verification_15_gb300 as pkg

    d = to_dev(batch)
    out = pkg.verify_greedy(d["target"], d["draft_tokens"], num_draft=d["num_draft"])
    torch.cuda.synchronize()
    nd = batch.get("num_draft")
    ref = oracle.verify_greedy(synth.as_oracle_array(batch["target"]), batch["draft_tokens"].numpy(),
                               None if nd is None else nd.numpy(), nthreads=CORES)
    assert np.array_equal(out["status"].cpu().numpy(), ref["status"])
    assert np.array_equal(out["accepted"].cpu().numpy(), ref["accepted"])
    assert np.array_equal(out["tokens"].cpu().numpy(), ref["tokens"])
    return ref


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_max_drafts(dt):
    """Kmax = 255: k_b in {255, 0, 100, 255, 17, 254}; low draft noise, so that
    scans run deep (the positions past 32 use the scan's later rounds)."""
    K = 255
    nd = [255, 0, 100, 255, 17, 254]
    batch = synth.make_batch(len(nd), K, 1000, dt, 2551, noise_sigmas=(0.02, 0.05), temperature=(0.9, 1.1),
                             num_draft=nd)
    for step in range(2):
        gpu = run_gpu_sample(batch, 9, step)
        ref = run_oracle_sample(batch, 9, step, nthreads=CORES)
        r = compare_sample(gpu, ref, batch["temperature"].numpy())
        assert r["flagged"] <= 1
    assert ref["accepted"].max() > 32
    # greedy: drafts are the draft rows' argmaxes, close to the target's
    g = _greedy_check(synth.make_batch(len(nd), K, 1000, dt, 2552, noise_sigmas=(0.01,), num_draft=nd,
                                       greedy_mask=[True] * len(nd)))
    assert g["accepted"].max() > 32


def test_max_drafts_early_exit():
    import speculative_decoding_verification_15_gb300 as pkg

    nd = [255, 3, 255, 40]
    batch = synth.make_batch(len(nd), 255, 777, torch.float32, 2553, noise_sigmas=(0.02,), num_draft=nd)
    d = to_dev(batch)
    out = pkg.verify_sample_early_exit(d["target"], d["draft"], d["draft_tokens"], d["temperature"], 4, 1,
                                       num_draft=d["num_draft"])
    torch.cuda.synchronize()
    ref = oracle.verify_sample(synth.as_oracle_array(batch["target"]), synth.as_oracle_array(batch["draft"]),
                               batch["draft_tokens"].numpy(), np.asarray(nd, np.int32),
                               batch["temperature"].numpy(), 4, 1, nthreads=CORES, early_exit=True)
    compare_sample({k: v.cpu().numpy() for k, v in out.items()}, ref, batch["temperature"].numpy())


def test_max_batch_small_vocab():
    """B = 8192, K = 3, V = 97 (a ragged 16-byte tail in every bf16 row)."""
    batch = synth.make_batch(8192, 3, 97, torch.bfloat16, 8191, noise_sigmas=(0.5, 2.0), temperature=(0.5, 1.5),
                             greedy_mask=[b % 5 == 0 for b in range(8192)])
    gpu = run_gpu_sample(batch, 0xFEDCBA9876543210, 5)
    ref = run_oracle_sample(batch, 0xFEDCBA9876543210, 5, nthreads=CORES)
    r = compare_sample(gpu, ref, batch["temperature"].numpy())
    assert r["flagged"] <= 3
    _greedy_check(batch)


@pytest.mark.parametrize("T", [0.05, 3.0])
def test_temperature_extremes(T):
    """T = 0.05: x / T reaches the hundreds; T = 3.0: a flat p and q."""
    batch = synth.make_batch(16, 6, 40000, torch.bfloat16, int(T * 1000), t_sigma=3.0, zipf=True,
                             noise_sigmas=(0.25, 1.0), temperature=(T, T))
    for step in range(2):
        gpu = run_gpu_sample(batch, 21, step)
        ref = run_oracle_sample(batch, 21, step, nthreads=CORES)
        r = compare_sample(gpu, ref, batch["temperature"].numpy())
        assert r["flagged"] <= 1
