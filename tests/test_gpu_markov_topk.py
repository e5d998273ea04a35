"""Top-K Markov-head drafting through the C ABI ("Bringing DSpark to vLLM Metal" --
"Making the draft cheaper": only the top-K candidates of each position are
corrected), against the fp64 oracle's markov_draft(topk=...) on the same seeded
inputs.  The comparison follows the full-vocabulary test: tokens equal up to the
oracle's first near-tie position, corrected logits within 1e-4 * max(1, |z|) up to
and including it (-inf outside the candidates on both sides), statuses equal."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

CORES = len(os.sched_getaffinity(0))
Z_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def run_gpu(m, topk, greedy=False):
    import speculative_decoding_verification_15_gb300 as pkg

    out = pkg.markov_draft_topk(m["base"].cuda(), m["anchor"].cuda(), m["emb"].cuda(), m["proj"].cuda(), topk,
                                None if greedy else m["temperature"].cuda(), m["seed"], m["step"])
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out.items()}


def run_oracle(m, topk, greedy=False):
    return oracle.markov_draft(synth.as_oracle_array(m["base"]), m["anchor"].numpy(),
                               synth.as_oracle_array(m["emb"]), synth.as_oracle_array(m["proj"]),
                               None if greedy else m["temperature"].numpy(), m["seed"], m["step"], topk=topk,
                               nthreads=CORES)


def compare(gpu, ref):
    assert (gpu["status"] == ref["status"]).all(), (gpu["status"], ref["status"])
    B, K = ref["tokens"].shape
    ties = 0
    for b in range(B):
        if ref["status"][b] != 0:
            assert (gpu["tokens"][b] == -1).all()
            continue
        t = int(ref["tie"][b])
        ties += t < K
        assert (gpu["tokens"][b, :t] == ref["tokens"][b, :t]).all(), (b, gpu["tokens"][b], ref["tokens"][b], t)
        n = min(t + 1, K)
        z, zr = gpu["logits"][b, :n], ref["logits"][b, :n]
        fin = np.isfinite(zr)
        assert np.array_equal(np.isfinite(z), fin), b  # the same candidate sets
        assert np.all(np.abs(z[fin] - zr[fin]) <= Z_TOL * np.maximum(1.0, np.abs(zr[fin]))), b
        assert (gpu["tokens"][b] >= 0).all()
    return ties


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("topk", [1, 64, 300])
def test_small_mixed(dt, topk):
    """B=6, K=4, V=5003, r=64, every third request greedy; topk 1 (the largest base
    logit always wins), 64, and 300 (spans several 512-entry blocks of the scan)."""
    ties = 0
    for step in range(2):
        m = synth.markov(step, B=6, K=4, V=5003, r=64, dtype=dt, greedy_every=3)
        gpu, ref = run_gpu(m, topk), run_oracle(m, topk)
        ties += compare(gpu, ref)
        if topk == 1:
            U = m["base"].float().numpy()
            assert np.array_equal(gpu["tokens"], U.argmax(axis=2))
    assert ties <= 1


def test_ties_and_nan_in_the_base_logits():
    """Exact ties at the selection threshold (lower v first), -0 against +0, and a
    NaN among the base logits (a candidate: status 4)."""
    m = synth.markov(3, B=4, K=2, V=3000, r=16, dtype=torch.float32)
    m["base"] = torch.round(m["base"])  # many equal values around the 40th largest
    m["base"][1, 0, :] = 0.0
    m["base"][1, 0, ::2] = -0.0
    m["base"][2, 1, 1234] = float("nan")
    for topk in (7, 40):
        gpu, ref = run_gpu(m, topk), run_oracle(m, topk)
        assert ref["status"].tolist() == [0, 0, 4, 0]
        compare(gpu, ref)


def test_gather_overflow_falls_back_exactly():
    """A constant row of V = 9000 (every entry ties: more than the fast path gathers)
    and a row whose largest values sit in one thread's stride (v = 512 j): both take
    the exact whole-row selection."""
    m = synth.markov(11, B=3, K=2, V=9000, r=8, dtype=torch.bfloat16)
    m["base"][0, 1, :] = 1.5
    m["base"][2, 0, ::512] = 60.0
    for topk in (5, 64):
        compare(run_gpu(m, topk), run_oracle(m, topk))


def test_topk_at_least_vocab_equals_full_vocab():
    import speculative_decoding_verification_15_gb300 as pkg

    m = synth.markov(4, B=3, K=3, V=700, r=8, dtype=torch.float32)
    gpu = run_gpu(m, 1000)
    full = pkg.markov_draft(m["base"].cuda(), m["anchor"].cuda(), m["emb"].cuda(), m["proj"].cuda(),
                            m["temperature"].cuda(), m["seed"], m["step"])
    ref = run_oracle(m, 0)
    compare(gpu, ref)
    assert np.array_equal(gpu["tokens"][ref["tie"] == 3], full["tokens"].cpu().numpy()[ref["tie"] == 3])


def test_main_size():
    """B=64, K=7, V=151936, r=256, bf16, top-64: the benchmarked drafting block."""
    m = synth.markov(0)
    ties = compare(run_gpu(m, 64), run_oracle(m, 64))
    assert ties <= max(2, m["B"] * m["K"] // 50)


def test_status_codes_and_no_logits():
    import speculative_decoding_verification_15_gb300 as pkg

    m = synth.markov(7, B=5, K=3, V=1024, r=8, dtype=torch.float32)
    m["anchor"][0] = -1
    m["temperature"][1] = float("nan")
    m["base"][3, 2, :] = float("-inf")
    gpu, ref = run_gpu(m, 16), run_oracle(m, 16)
    assert ref["status"].tolist() == [1, 3, 0, 4, 0]
    compare(gpu, ref)
    out = pkg.markov_draft_topk(m["base"].cuda(), m["anchor"].cuda(), m["emb"].cuda(), m["proj"].cuda(), 16,
                                m["temperature"].cuda(), m["seed"], m["step"], want_logits=False)
    torch.cuda.synchronize()
    assert out["logits"] is None and np.array_equal(out["tokens"].cpu().numpy(), gpu["tokens"])
