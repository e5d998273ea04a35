"""The fixed-scratch entry point spec_verify_sample_noalloc against the workspace
entry point spec_verify_sample, through the C ABI.

Named to be collected last, so that it runs both after every other GPU test (the
library already set up on the device) and, run alone, in a fresh process (the first
call does the per-device set-up)."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import P_ATOL, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def _outputs(B, K):
    dev = "cuda"
    return dict(tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
                accepted=torch.full((B,), -7, dtype=torch.int32, device=dev),
                p=torch.full((B, K), -7.0, device=dev), q=torch.full((B, K), -7.0, device=dev),
                status=torch.full((B,), -7, dtype=torch.int32, device=dev))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_noalloc_matches_workspace_entry_point(dt):
    from speculative_decoding_verification_15_gb300 import binding

    B, K, V = 12, 5, 30011
    nd = [5, 4, 3, 2, 1, 0, 5, 5, 5, 2, 3, 4]
    mask = np.zeros(B, bool)
    mask[7] = True  # one greedy request (temperature 0)
    batch = synth.make_batch(B, K, V, dt, 77, zipf=True, noise_sigmas=(0.3, 1.0), temperature=(0.7, 1.0),
                             num_draft=nd, greedy_mask=mask)
    d = to_dev(batch)
    args = (d["target"], d["draft"], d["draft_tokens"], d["num_draft"], d["temperature"], 11, 4)
    ref = _outputs(B, K)
    ws = torch.zeros(binding.spec_verify_workspace_size(B, K, V, binding._dtype_code(d["target"])),
                     dtype=torch.uint8, device="cuda")
    binding.spec_verify_sample(*args, ref["tokens"], ref["accepted"], ref["p"], ref["q"], ref["status"], ws)
    torch.cuda.synchronize()
    assert (ref["status"] == 0).all()
    for _ in range(2):  # two consecutive calls on the same fixed scratch
        out = _outputs(B, K)
        binding.spec_verify_sample_noalloc(*args, out["tokens"], out["accepted"], out["p"], out["q"],
                                           out["status"])
        torch.cuda.synchronize()
        assert torch.equal(out["status"], ref["status"])
        assert torch.equal(out["accepted"], ref["accepted"])
        assert torch.equal(out["tokens"], ref["tokens"])
        valid = ref["p"] >= 0
        assert torch.equal(out["p"] >= 0, valid)
        assert (out["p"][valid] - ref["p"][valid]).abs().max().item() <= P_ATOL
        assert (out["q"][valid] - ref["q"][valid]).abs().max().item() <= P_ATOL


def test_noalloc_rejects_sizes_beyond_the_scratch():
    from speculative_decoding_verification_15_gb300 import binding

    lib = binding.load()
    B, K, V = 8192, 8, 1 << 20
    assert binding.spec_verify_workspace_size(B, K, V, binding.SPEC_F32) > 4 << 20
    P = ctypes.c_void_p(256)  # never dereferenced: the size check returns before any launch
    rc = lib.spec_verify_sample_noalloc(P, P, binding.SPEC_F32, B, K, V, V, P, None, P, 0, 0, P, P, None,
                                        None, P, None)
    assert rc == binding.SPEC_ESCRATCH
    assert b"fixed scratch" in lib.spec_error_string(rc)
    # an empty batch is still a no-op
    assert lib.spec_verify_sample_noalloc(P, P, 0, 0, K, V, V, P, None, P, 0, 0, P, P, None, None, P, None) == 0
