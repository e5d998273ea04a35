"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, and compare them."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

P_ATOL = 1e-5  # |p_gpu - p_oracle| and |q_gpu - q_oracle| bound for p(x_i), q(x_i)


def to_dev(batch: dict, dev="cuda"):
    out = {}
    for k in ("target", "draft", "draft_tokens", "num_draft", "temperature"):
        v = batch.get(k)
        out[k] = None if v is None else v.to(dev)
    return out


def run_gpu_sample(batch: dict, seed: int, step: int, dev="cuda") -> dict:
    import speculative_decoding_verification_15_gb300 as pkg

    d = to_dev(batch, dev)
    out = pkg.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["temperature"], seed, step,
                            num_draft=d["num_draft"])
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out.items()}


def run_oracle_sample(batch: dict, seed: int, step: int, nthreads: int = 8) -> dict:
    nd = batch.get("num_draft")
    return oracle.verify_sample(synth.as_oracle_array(batch["target"]), synth.as_oracle_array(batch["draft"]),
                                batch["draft_tokens"].numpy(), None if nd is None else nd.numpy(),
                                batch["temperature"].numpy(), seed, step, nthreads=nthreads)


def compare_sample(gpu: dict, ref: dict, temperature: np.ndarray, num_draft=None, K=None) -> dict:
    """Statuses everywhere, accepted lengths and tokens on every request the oracle
    does not flag as a near-tie (greedy requests: always), p/q within P_ATOL."""
    B = ref["status"].shape[0]
    assert (gpu["status"] == ref["status"]).all(), (gpu["status"], ref["status"])
    flagged = ref["flags"] != 0
    greedy = temperature == 0
    check = (ref["status"] == 0) & (~flagged | greedy)
    bad = np.nonzero(check & (gpu["accepted"] != ref["accepted"]))[0]
    assert bad.size == 0, f"accepted differ at {bad[:10]}: gpu {gpu['accepted'][bad[:10]]} oracle {ref['accepted'][bad[:10]]}"
    tok_bad = np.nonzero(check & (gpu["tokens"] != ref["tokens"]).any(axis=1))[0]
    assert tok_bad.size == 0, f"tokens differ at {tok_bad[:10]}:\n{gpu['tokens'][tok_bad[:4]]}\n{ref['tokens'][tok_bad[:4]]}"
    bad_status = ref["status"] != 0
    assert (gpu["accepted"][bad_status] == 0).all() and (gpu["tokens"][bad_status] == -1).all()
    if gpu.get("p") is not None:
        valid = ref["p"] >= 0
        assert ((gpu["p"] >= 0) == valid).all()
        assert np.abs(gpu["p"][valid] - ref["p"][valid]).max(initial=0) <= P_ATOL
        assert np.abs(gpu["q"][valid] - ref["q"][valid]).max(initial=0) <= P_ATOL
        assert (gpu["p"][~valid] == -1).all() and (gpu["q"][~valid] == -1).all()
    return dict(n=B, flagged=int((flagged & ~greedy & (ref["status"] == 0)).sum()),
                mismatched_flagged=int((flagged & ~greedy & (gpu["accepted"] != ref["accepted"])).sum()))
