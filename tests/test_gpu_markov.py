"""Markov-head drafting through the C ABI ("Accelerating Large-Model Inference ...
DSpark", drafting-engine table, layer 2; "DSpark paper review" Sec. 4.1), against
the fp64 oracle on the same seeded inputs.

Each position's draw depends on the token drawn before it, so the comparison runs
position by position up to the oracle's first near-tie (two best scores within
1e-3 relative, where fp32 and fp64 may pick differently): tokens equal before it,
corrected logits within 1e-4 * max(1, |z|) up to and including it, statuses equal
everywhere.  Near-ties must stay rare.
"""
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


def run_gpu(m, greedy=False):
    import speculative_decoding_verification_15_gb300 as pkg

    out = pkg.markov_draft(m["base"].cuda(), m["anchor"].cuda(), m["emb"].cuda(), m["proj"].cuda(),
                           None if greedy else m["temperature"].cuda(), m["seed"], m["step"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_oracle(m, greedy=False):
    return oracle.markov_draft(synth.as_oracle_array(m["base"]), m["anchor"].numpy(),
                               synth.as_oracle_array(m["emb"]), synth.as_oracle_array(m["proj"]),
                               None if greedy else m["temperature"].numpy(), m["seed"], m["step"],
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
        n = min(t + 1, K)  # row t still follows an agreed token
        z, zr = gpu["logits"][b, :n], ref["logits"][b, :n]
        assert np.all(np.abs(z - zr) <= Z_TOL * np.maximum(1.0, np.abs(zr))), (b, np.abs(z - zr).max())
        assert (gpu["tokens"][b] >= 0).all()
    return ties


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_small_mixed(dt):
    """B=6, K=4, V=5003 (not a multiple of 4 or 32), r=64, every third request greedy."""
    ties = 0
    for step in range(3):
        m = synth.markov(step, B=6, K=4, V=5003, r=64, dtype=dt, greedy_every=3)
        ties += compare(run_gpu(m), run_oracle(m))
    assert ties <= 1


def test_bf16_tiles_two_request_chunks():
    """bf16 factors on the tensor-core path: B = 70 (a full chunk of 64 requests and a
    partial one), V = 5000 (the last 64-entry tile holds 8), r = 32 (the staged product
    tile is larger than the tile's projection rows), every fifth request greedy."""
    m = synth.markov(11, B=70, K=2, V=5000, r=32, dtype=torch.bfloat16, greedy_every=5)
    assert compare(run_gpu(m), run_oracle(m)) <= 1


def test_bf16_rank_512():
    """bf16 at the header's largest rank (r = 512): the two-CTA bias kernel (the
    role-split one serves r <= 256), B = 66 (two request chunks), V = 3001."""
    m = synth.markov(13, B=66, K=2, V=3001, r=512, dtype=torch.bfloat16, greedy_every=4)
    assert compare(run_gpu(m), run_oracle(m)) <= 1


def test_bf16_padded_rows():
    """bf16, base rows padded to an odd stride (4101 entries for V = 4099): the
    epilogue's scalar path; r = 48."""
    import speculative_decoding_verification_15_gb300 as pkg

    m = synth.markov(12, B=5, K=3, V=4099, r=48, dtype=torch.bfloat16)
    padded = torch.full((5, 3, 4101), float("nan"), dtype=torch.bfloat16)
    padded[:, :, :4099] = m["base"]
    out = pkg.markov_draft(padded.cuda()[:, :, :4099], m["anchor"].cuda(), m["emb"].cuda(), m["proj"].cuda(),
                           m["temperature"].cuda(), m["seed"], m["step"])
    torch.cuda.synchronize()
    assert compare({k: v.cpu().numpy() for k, v in out.items()}, run_oracle(m)) <= 1


def test_greedy_and_rank_4():
    m = synth.markov(5, B=9, K=5, V=2053, r=4, dtype=torch.float32)
    assert compare(run_gpu(m, greedy=True), run_oracle(m, greedy=True)) <= 1


def test_main_size():
    """B=64, K=7, V=151936, r=256, bf16: the drafting block of the benchmarked batch."""
    m = synth.markov(0)
    ties = compare(run_gpu(m), run_oracle(m))
    assert ties <= max(2, m["B"] * m["K"] // 50)  # the band flags under 2 % of the 448 draws


def test_status_codes():
    m = synth.markov(7, B=6, K=3, V=1024, r=8, dtype=torch.float32)
    m["anchor"][0] = -1
    m["anchor"][1] = 1024
    m["temperature"][2] = float("nan")
    m["base"][3, 1, 100] = float("nan")
    m["base"][4, 2, :] = float("-inf")
    m["base"][5, 0, 7] = float("inf")
    gpu, ref = run_gpu(m), run_oracle(m)
    assert ref["status"].tolist() == [1, 1, 3, 4, 4, 4]
    compare(gpu, ref)


def test_zero_positions_and_empty_batch():
    import speculative_decoding_verification_15_gb300 as pkg

    m = synth.markov(8, B=4, K=1, V=512, r=8, dtype=torch.float32)
    m["anchor"][2] = 600
    base0 = m["base"][:, :0].contiguous().cuda()
    out = pkg.markov_draft(base0, m["anchor"].cuda(), m["emb"].cuda(), m["proj"].cuda(), m["temperature"].cuda(),
                           1, 1)
    torch.cuda.synchronize()
    assert out["status"].cpu().tolist() == [0, 0, 1, 0]
    e = torch.empty((0, 3, 512), device="cuda")
    out = pkg.markov_draft(e, torch.empty(0, dtype=torch.int32, device="cuda"), m["emb"].cuda(), m["proj"].cuda())
    assert out["tokens"].shape == (0, 3)


def test_zero_factors_match_plain_draws():
    """emb = 0: every position is an independent draw from softmax(U / T) (the
    oracle's pinned Gumbel-max with purpose 3), so the GPU's tokens equal those."""
    m = synth.markov(9, B=4, K=3, V=3001, r=16, dtype=torch.float32)
    m["emb"].zero_()
    gpu, ref = run_gpu(m), run_oracle(m)
    compare(gpu, ref)
    assert np.array_equal(gpu["logits"], m["base"].numpy())
