"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that still span many
warp ranges and end in ragged tails.  Greedy results must be bit-exact; sampling
results must be identical outside the oracle's reported near-ties, with p(x_i) and
q(x_i) within 1e-5."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import compare_sample, run_gpu_sample, run_oracle_sample, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


CASES = [
    # B, K, V, dtype, temperature range, noise sigmas
    (3, 4, 5000, torch.bfloat16, (0.7, 1.0), (0.5, 1.0)),
    (4, 7, 33000, torch.bfloat16, (0.6, 1.0), (0.25, 1.0, 2.0)),
    (5, 3, 20011, torch.float32, (1.0, 1.0), (1.0,)),          # odd V: scalar path
    (6, 5, 40000, torch.float32, (0.8, 0.8), (0.5, 2.0)),
    (2, 2, 7, torch.float32, (1.0, 1.0), (1.0,)),              # V below one vector per lane
    (2, 0, 1000, torch.bfloat16, (1.0, 1.0), (1.0,)),          # no drafts: bonus only
    (16, 3, 4099, torch.bfloat16, (0.5, 1.5), (0.25, 0.5)),    # odd V, bf16 scalar path
    (9, 6, 65536, torch.bfloat16, (0.9, 0.9), (0.1, 0.3)),     # high acceptance
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}K{c[1]}V{c[2]}{str(c[3])[6:]}" for c in CASES])
def test_sample_parity(case):
    B, K, V, dt, trange, sig = case
    tot = dict(n=0, flagged=0)
    for step in range(3):
        batch = synth.make_batch(B, K, V, dt, 100 + step, t_sigma=3.0, zipf=True, noise_sigmas=sig,
                                 temperature=trange)
        gpu = run_gpu_sample(batch, seed=5, step=step)
        ref = run_oracle_sample(batch, seed=5, step=step)
        r = compare_sample(gpu, ref, batch["temperature"].numpy())
        tot["n"] += r["n"]
        tot["flagged"] += r["flagged"]
    assert tot["flagged"] <= max(1, tot["n"] // 200)


def test_sample_ragged_num_draft_and_unread_rows():
    B, K, V = 12, 6, 12000
    nd = [0, 1, 2, 3, 4, 5, 6, 6, 3, 0, 1, 2]
    batch = synth.make_batch(B, K, V, torch.bfloat16, 42, zipf=True, noise_sigmas=(0.5, 1.0),
                             temperature=(0.7, 1.0), num_draft=nd)
    # rows beyond k_b are NaN: reading them would set status 4
    gpu = run_gpu_sample(batch, seed=9, step=1)
    ref = run_oracle_sample(batch, seed=9, step=1)
    assert (ref["status"] == 0).all()
    compare_sample(gpu, ref, batch["temperature"].numpy())


def test_sample_mixed_greedy_requests():
    B, K, V = 10, 4, 9000
    mask = np.arange(B) % 3 == 0
    batch = synth.make_batch(B, K, V, torch.float32, 7, zipf=True, noise_sigmas=(0.3,),
                             temperature=(1.0, 1.0), greedy_mask=mask)
    batch["draft"][torch.as_tensor(mask)] = float("nan")  # greedy requests never read draft logits
    gpu = run_gpu_sample(batch, seed=3, step=3)
    ref = run_oracle_sample(batch, seed=3, step=3)
    assert (ref["status"] == 0).all()
    compare_sample(gpu, ref, batch["temperature"].numpy())
    assert (gpu["p"][mask] == -1).all()


def test_padded_row_stride():
    B, K, V, LD = 3, 3, 1000, 1024
    full = synth.make_batch(B, K, LD, torch.bfloat16, 8, zipf=True, temperature=(0.8, 0.8))
    batch = dict(full)
    batch["target"] = full["target"][..., :V]
    batch["draft"] = full["draft"][..., :V]
    batch["draft_tokens"] = full["draft_tokens"].clamp(max=V - 1)
    gpu = run_gpu_sample(batch, seed=1, step=1)  # strided views: ld_row = 1024
    ref_batch = dict(batch, target=batch["target"].contiguous(), draft=batch["draft"].contiguous())
    ref = run_oracle_sample(ref_batch, seed=1, step=1)
    compare_sample(gpu, ref, batch["temperature"].numpy())


def test_worked_examples_on_gpu():
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
    vocab = gold["vocab"]
    import speculative_decoding_verification_15_gb300 as pkg

    for ex in gold["examples"]:
        K, V = len(ex["drafts"]), len(vocab)
        t = np.full((1, K + 1, V), np.nan, np.float32)
        d = np.full((1, K, V), np.nan, np.float32)
        with np.errstate(divide="ignore"):
            for i, row in enumerate(ex["target"]):
                p = np.zeros(V)
                for w, pr in row.items():
                    p[vocab.index(w)] = pr
                t[0, i] = np.log(p)
            for i, row in enumerate(ex["draft"]):
                q = np.zeros(V)
                for w, pr in row.items():
                    q[vocab.index(w)] = pr
                d[0, i] = np.log(q)
        kb = ex["num_draft"]
        if ex.get("unused_rows_nan"):
            t[0, kb + 1:] = np.nan
            d[0, kb:] = np.nan
        x = torch.tensor([[vocab.index(w) for w in ex["drafts"]]], dtype=torch.int32, device="cuda")
        exp = [vocab.index(w) for w in ex["expected"]["tokens"]]
        for dt in (torch.float32, torch.bfloat16):
            tt = torch.from_numpy(t).to(dt).cuda()
            dd = torch.from_numpy(d).to(dt).cuda()
            for seed in range(20):
                out = pkg.verify_sample(tt, dd, x, torch.ones(1, device="cuda"), seed, seed * 7 + 1,
                                        num_draft=torch.tensor([kb], dtype=torch.int32, device="cuda"))
                A = int(out["accepted"][0])
                assert int(out["status"][0]) == 0
                assert A == ex["expected"]["accepted"], (ex["name"], seed)
                assert out["tokens"][0, :A + 1].tolist() == exp, (ex["name"], seed)


def test_status_codes_on_gpu():
    V, K, B = 64, 2, 7
    rng = np.random.default_rng(9)
    t = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    d = rng.normal(size=(B, K, V)).astype(np.float32)
    x = rng.integers(0, V, size=(B, K)).astype(np.int32)
    nd = np.full(B, K, np.int32)
    T = np.ones(B, np.float32)
    nd[1] = K + 1
    T[2] = -0.5
    x[3, 1] = V
    t[4, 1, 3] = np.nan
    d[5, 0, :] = -np.inf
    t[6, 0, 2] = np.inf
    batch = dict(target=torch.from_numpy(t), draft=torch.from_numpy(d), draft_tokens=torch.from_numpy(x),
                 num_draft=torch.from_numpy(nd), temperature=torch.from_numpy(T))
    gpu = run_gpu_sample(batch, 3, 3)
    ref = run_oracle_sample(batch, 3, 3)
    assert list(ref["status"]) == [0, 2, 3, 1, 4, 4, 4]
    compare_sample(gpu, ref, T)


def _greedy(batch):
    import speculative_decoding_verification_15_gb300 as pkg

    d = to_dev(batch)
    out = pkg.verify_greedy(d["target"], d["draft_tokens"], num_draft=d["num_draft"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("V,dt", [(151936, torch.bfloat16), (32000, torch.float32), (1001, torch.bfloat16),
                                  (3, torch.float32)])
def test_greedy_parity_bit_exact(V, dt):
    B, K = 8, 5
    batch = synth.make_batch(B, K, V, dt, 3, zipf=True, noise_sigmas=(0.05, 0.2), temperature=(0.0, 0.0),
                             num_draft=[5, 4, 3, 2, 1, 0, 5, 5])
    gpu = _greedy(batch)
    ref = oracle.verify_greedy(synth.as_oracle_array(batch["target"]), batch["draft_tokens"].numpy(),
                               batch["num_draft"].numpy())
    assert (gpu["status"] == ref["status"]).all()
    assert (gpu["accepted"] == ref["accepted"]).all()
    assert (gpu["tokens"] == ref["tokens"]).all()


def test_greedy_ties_lowest_index():
    B, K, V = 4, 3, 50000
    rng = np.random.default_rng(0)
    t = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    # exact ties at the max far apart (different warp ranges), draft = the higher index
    for b in range(B):
        for i in range(K + 1):
            lo, hi = int(rng.integers(0, V // 2)), int(rng.integers(V // 2, V))
            t[b, i, lo] = t[b, i, hi] = 10.0
    x = np.zeros((B, K), np.int32)
    for b in range(B):
        for i in range(K):
            x[b, i] = int(np.nonzero(t[b, i] == 10.0)[0][0 if b % 2 == 0 else -1])
    for dt in (torch.float32, torch.bfloat16):
        batch = dict(target=torch.from_numpy(t).to(dt), draft_tokens=torch.from_numpy(x), num_draft=None)
        gpu = _greedy(batch)
        ref = oracle.verify_greedy(synth.as_oracle_array(batch["target"]), x, None)
        assert (gpu["tokens"] == ref["tokens"]).all() and (gpu["accepted"] == ref["accepted"]).all()
        assert list(ref["accepted"]) == [K, 0, K, 0]


def test_empty_batch_and_repeat_calls():
    import speculative_decoding_verification_15_gb300 as pkg

    t = torch.zeros((0, 3, 100), dtype=torch.bfloat16, device="cuda")
    out = pkg.verify_greedy(t, torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    assert out["tokens"].shape == (0, 3)
    # repeated calls on the same workspace give identical results
    batch = synth.make_batch(4, 3, 3000, torch.bfloat16, 1, zipf=True)
    a = run_gpu_sample(batch, 1, 1)
    b = run_gpu_sample(batch, 1, 1)
    for k in ("tokens", "accepted", "status", "p", "q"):
        assert (a[k] == b[k]).all()


def test_bonus_row_status_on_gpu():
    from test_oracle_verify import _bonus_row_case
    import speculative_decoding_verification_15_gb300 as pkg

    for kind in ("accept", "reject"):
        t, d, x = _bonus_row_case(kind)
        batch = dict(target=torch.from_numpy(t), draft=torch.from_numpy(d), draft_tokens=torch.from_numpy(x),
                     num_draft=None, temperature=torch.ones(1))
        gpu = run_gpu_sample(batch, 1, 1)
        ref = run_oracle_sample(batch, 1, 1)
        compare_sample(gpu, ref, np.ones(1, np.float32))
        g = pkg.verify_greedy(torch.from_numpy(t).cuda(), torch.from_numpy(x).cuda())
        gref = oracle.verify_greedy(t, x, None)
        assert int(g["status"][0]) == int(gref["status"][0])
        assert g["tokens"].cpu().numpy().tolist() == gref["tokens"].tolist()
