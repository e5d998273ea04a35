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
    """Compare one batch of the CUDA path with the oracle, request by request.

    The parity rule: greedy requests bit-exact; sampling requests
    identical in accepted length and tokens except at a near-tie, where the
    threshold gap (bit 1) or the top-2 Gumbel gap (bit 2) is below 1e-5 relative,
    or where the residual has no support (bit 4, reachable only by rounding).
    What a near-tie leaves open is only what follows it:
      - bit 1 at position f: drafts 0 .. f-1 are still accepted by both and their
        tokens equal (the decision at f and everything after may differ);
      - bit 2 or 4 only: the accepted length and the accepted drafts are equal;
        the drawn token may differ.
    Bit 8 (the residual's conditioning band) is counted, never excluded: a request
    carrying only bit 8 must match exactly.  Statuses match everywhere; p/q match
    within P_ATOL wherever both sides computed them.  Returns the counts.
    """
    B = ref["status"].shape[0]
    assert (gpu["status"] == ref["status"]).all(), (gpu["status"], ref["status"])
    flags = ref["flags"]
    fpos = ref.get("flag_pos")
    greedy = temperature == 0
    ok = ref["status"] == 0
    counts = dict(n=B, thresh=0, gumbel=0, degenerate=0, illcond=0, mismatched_flagged=0)
    for b in range(B):
        if not ok[b]:
            continue
        fl = 0 if greedy[b] else int(flags[b])
        ga, ra = int(gpu["accepted"][b]), int(ref["accepted"][b])
        gt, rt = gpu["tokens"][b], ref["tokens"][b]
        counts["thresh"] += bool(fl & oracle.FL_THRESH)
        counts["gumbel"] += bool(fl & oracle.FL_GUMBEL)
        counts["degenerate"] += bool(fl & oracle.FL_DEGENERATE)
        counts["illcond"] += bool(fl & oracle.FL_ILLCOND)
        exact = ga == ra and np.array_equal(gt, rt)
        if fl & oracle.FL_THRESH:
            f = int(fpos[b]) if fpos is not None else 0
            assert 0 <= f <= ra, (b, f, ra)
            assert ga >= f and np.array_equal(gt[:f], rt[:f]), (b, f, gt, rt)
        elif fl & (oracle.FL_GUMBEL | oracle.FL_DEGENERATE):
            assert ga == ra and np.array_equal(gt[:ra], rt[:ra]), (b, gt, rt)
            assert (gt[ra + 1:] == -1).all()
        else:
            assert exact, f"request {b} (flags {fl}) differs: accepted gpu {ga} oracle {ra}\n{gt}\n{rt}"
        if not exact:
            counts["mismatched_flagged"] += 1
    bad_status = ~ok
    assert (gpu["accepted"][bad_status] == 0).all() and (gpu["tokens"][bad_status] == -1).all()
    if gpu.get("p") is not None:
        gv, rv = gpu["p"] >= 0, ref["p"] >= 0
        both = gv & rv
        # the positions each side computed agree except after a decision that a
        # near-tie left open (early exit stops at its own first rejection)
        same_decisions = gpu["accepted"] == ref["accepted"]
        assert (gv[same_decisions] == rv[same_decisions]).all()
        assert np.abs(gpu["p"][both] - ref["p"][both]).max(initial=0) <= P_ATOL
        assert np.abs(gpu["q"][both] - ref["q"][both]).max(initial=0) <= P_ATOL
        assert (gpu["p"][~gv] == -1).all() and (gpu["q"][~gv] == -1).all()
    counts["flagged"] = counts["thresh"] + counts["gumbel"] + counts["degenerate"]
    return counts
