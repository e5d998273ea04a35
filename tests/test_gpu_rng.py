"""Direct checks of the library's device Philox4x32-10 stream against the oracle's.

The two implementations were written separately (the oracle's is pinned to
cuRAND's host generator and Triton's interpreter).  Here each draw is arranged so
that the token it returns is decided by the Philox words alone, and the GPU's
tokens are compared with the oracle's for every request:

- Markov drafting with a zero head and constant base logits: x_k = argmax_v g_v,
  the largest word of purpose 3 at row k (every row of a 20-position block);
- verify with target = draft (p = q, every draft accepted): the bonus token is the
  largest word of purpose 2 at row k_b (k_b from 0 to 20);
- verify with a uniform target and a one-hot draft at x_i: the draft is accepted
  iff u_i < 1/V (purpose 0), and the correction is the largest purpose-1 word at
  row j among v != x_j; rows before j have target = draft and are always accepted,
  so j reaches 17.

Every case runs B = 8192 requests (counter word 1 up to 8191), with a seed whose
high word is not zero (the key's second word), and with a step at or above 2^32,
whose low word alone enters the counter (both sides truncate it the same way).
"""
import os

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CORES = len(os.sched_getaffinity(0))
SEEDS = [0xFEDCBA9876543210, 0x00000001_00000000, 3]
STEPS = [(1 << 32) + 7, 0xFFFFFFFF, 11]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("seed,step", list(zip(SEEDS, STEPS)))
def test_markov_zero_head_draws_follow_the_words(seed, step):
    import speculative_decoding_verification_15_gb300 as pkg

    B, K, V, r = 8192, 20, 64, 4
    base = torch.zeros((B, K, V), dtype=torch.bfloat16)
    emb = torch.zeros((V, r), dtype=torch.bfloat16)
    proj = torch.ones((V, r), dtype=torch.bfloat16)
    anchor = torch.arange(B, dtype=torch.int32) % V
    T = torch.ones(B, dtype=torch.float32)
    out = pkg.markov_draft(base.cuda(), anchor.cuda(), emb.cuda(), proj.cuda(), T.cuda(), seed, step)
    torch.cuda.synchronize()
    ref = oracle.markov_draft(base.view(torch.int16).numpy().view(np.uint16), anchor.numpy(),
                              emb.view(torch.int16).numpy().view(np.uint16),
                              proj.view(torch.int16).numpy().view(np.uint16), T.numpy(), seed, step,
                              nthreads=CORES, want_logits=False)
    assert (ref["status"] == 0).all() and (out["status"].cpu().numpy() == 0).all()
    tok = out["tokens"].cpu().numpy()
    tie = ref["tie"]
    assert (tie < K).sum() <= 3  # two noise values within fp32 rounding of each other: rare
    for b in np.nonzero(tie < K)[0]:
        assert np.array_equal(tok[b, : tie[b]], ref["tokens"][b, : tie[b]])
    clean = tie == K
    assert np.array_equal(tok[clean], ref["tokens"][clean])
    # the counter holds the step's low word only
    if step >= (1 << 32):
        low = pkg.markov_draft(base.cuda(), anchor.cuda(), emb.cuda(), proj.cuda(), T.cuda(), seed,
                               step & 0xFFFFFFFF)
        assert torch.equal(low["tokens"], out["tokens"])


@pytest.mark.parametrize("seed,step", list(zip(SEEDS, STEPS)))
def test_bonus_draws_follow_the_words(seed, step):
    import speculative_decoding_verification_15_gb300 as pkg

    B, K, V = 8192, 20, 64
    t = torch.zeros((B, K + 1, V), dtype=torch.float32)
    d = torch.zeros((B, K, V), dtype=torch.float32)
    x = (torch.arange(B * K, dtype=torch.int32) % V).reshape(B, K)
    nd = torch.arange(B, dtype=torch.int32) % (K + 1)
    T = torch.ones(B, dtype=torch.float32)
    out = pkg.verify_sample(t.cuda(), d.cuda(), x.cuda(), T.cuda(), seed, step, num_draft=nd.cuda())
    torch.cuda.synchronize()
    ref = oracle.verify_sample(t.numpy(), d.numpy(), x.numpy(), nd.numpy(), T.numpy(), seed, step, nthreads=CORES)
    assert (ref["status"] == 0).all() and (ref["accepted"] == nd.numpy()).all()
    ok = ref["flags"] == 0  # a top-2 noise gap within 1e-5 may go either way in fp32
    assert ok.sum() >= B - 3
    assert np.array_equal(out["status"].cpu().numpy(), ref["status"])
    assert np.array_equal(out["accepted"].cpu().numpy(), ref["accepted"])
    assert np.array_equal(out["tokens"].cpu().numpy()[ok], ref["tokens"][ok])


@pytest.mark.parametrize("seed,step", list(zip(SEEDS, STEPS)))
def test_acceptance_and_correction_follow_the_words(seed, step):
    import speculative_decoding_verification_15_gb300 as pkg

    B, K, V, J = 8192, 20, 64, 17
    t = torch.zeros((B, K + 1, V), dtype=torch.float32)
    d = torch.zeros((B, K, V), dtype=torch.float32)
    x = (torch.arange(B * K, dtype=torch.int32) * 7 % V).reshape(B, K)
    # rows J.. : uniform target, one-hot draft at x_i (q(x_i) = 1, p(x_i) = 1/V)
    d[:, J:, :] = float("-inf")
    for i in range(J, K):
        d[torch.arange(B), i, x[:, i].long()] = 0.0
    T = torch.ones(B, dtype=torch.float32)
    out = pkg.verify_sample(t.cuda(), d.cuda(), x.cuda(), T.cuda(), seed, step)
    torch.cuda.synchronize()
    ref = oracle.verify_sample(t.numpy(), d.numpy(), x.numpy(), None, T.numpy(), seed, step, nthreads=CORES)
    assert (ref["status"] == 0).all()
    A = ref["accepted"]
    assert (A >= J).all() and (A < K).sum() > B // 2 and (A > J).sum() > 0
    ok = ref["flags"] == 0
    assert ok.sum() >= B - 3
    assert np.array_equal(out["status"].cpu().numpy(), ref["status"])
    assert np.array_equal(out["accepted"].cpu().numpy()[ok], A[ok])
    assert np.array_equal(out["tokens"].cpu().numpy()[ok], ref["tokens"][ok])
    assert np.abs(out["p"].cpu().numpy() - ref["p"]).max() <= 1e-5
