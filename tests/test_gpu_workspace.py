"""The verify calls' contract with their caller, on the GPU and through the C ABI:
pointers must be on the current device, and a workspace must start with its ticket
counter at zero.  Batches of fewer requests than SMs run main_kernel + commit_kernel:
there a counter that is not zero (a workspace that was not zero-filled) makes the
main pass skip chunks; the commit pass then finds partials carrying another call's
tag and reports status 5 for those requests (nothing hangs: no wait depends on the
skipped work), and leaves the counter zero, so the next call on the same workspace
is correct.  Larger batches run the single persistent kernel, whose counters and
per-request lines are zeroed in stream order before every launch: any workspace
contents serve, and one workspace may alternate between the two paths."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import compare_sample, run_oracle_sample, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    assert torch.cuda.is_available()


def _call(lib, t, d, x, T, outs, ws, B, K, V):
    P = ctypes.c_void_p
    return lib.spec_verify_sample(P(t.data_ptr()), P(d.data_ptr()), 0, B, K, V, V, P(x.data_ptr()), None,
                                  P(T.data_ptr()), 3, 1, P(outs["tok"].data_ptr()), P(outs["acc"].data_ptr()),
                                  P(outs["p"].data_ptr()), P(outs["q"].data_ptr()), P(outs["st"].data_ptr()),
                                  P(ws.data_ptr()), ws.numel(), None)


def _outs(B, K):
    return dict(tok=torch.empty((B, K + 1), dtype=torch.int32, device="cuda"),
                acc=torch.empty(B, dtype=torch.int32, device="cuda"),
                p=torch.empty((B, K), device="cuda"), q=torch.empty((B, K), device="cuda"),
                st=torch.empty(B, dtype=torch.int32, device="cuda"))


def test_logits_not_on_the_device_are_rejected():
    from speculative_decoding_verification_15_gb300 import binding

    lib = binding.load()
    B, K, V = 2, 2, 64
    batch = synth.make_batch(B, K, V, torch.bfloat16, 4, temperature=(1.0, 1.0))
    d = to_dev(batch)
    ws = torch.zeros(binding.spec_verify_workspace_size(B, K, V, 0), dtype=torch.uint8, device="cuda")
    host_t = batch["target"].pin_memory()  # host memory, mapped but not device memory
    outs = _outs(B, K)
    assert _call(lib, host_t, d["draft"], d["draft_tokens"], d["temperature"], outs, ws, B, K, V) == 1  # EINVAL
    assert _call(lib, d["target"], d["draft"], d["draft_tokens"], d["temperature"], outs, ws, B, K, V) == 0


def test_workspace_with_a_nonzero_ticket_counter_reports_status_5_then_recovers():
    from speculative_decoding_verification_15_gb300 import binding

    lib = binding.load()
    B, K, V = 64, 7, 151936
    batch = synth.main(0)
    d = to_dev(batch)
    ws = torch.zeros(binding.spec_verify_workspace_size(B, K, V, 0), dtype=torch.uint8, device="cuda")
    ws[:4] = torch.tensor([0x00, 0x00, 0x00, 0x40], dtype=torch.uint8)  # ticket counter 2^30: chunks skipped
    outs = _outs(B, K)
    assert _call(lib, d["target"], d["draft"], d["draft_tokens"], d["temperature"], outs, ws, B, K, V) == 0
    torch.cuda.synchronize()
    st = outs["st"].cpu().numpy()
    assert (st == 5).sum() > B // 2 and np.isin(st, (0, 5)).all()
    tok = outs["tok"].cpu().numpy()
    assert (tok[st == 5] == -1).all() and (outs["acc"].cpu().numpy()[st == 5] == 0).all()
    assert int(ws[:4].view(torch.int32).item()) == 0  # the counter is zero again
    # the same workspace, next call: every request verified, equal to the oracle
    assert _call(lib, d["target"], d["draft"], d["draft_tokens"], d["temperature"], outs, ws, B, K, V) == 0
    torch.cuda.synchronize()
    gpu = {"tokens": outs["tok"].cpu().numpy(), "accepted": outs["acc"].cpu().numpy(),
           "status": outs["st"].cpu().numpy(), "p": outs["p"].cpu().numpy(), "q": outs["q"].cpu().numpy()}
    ref = run_oracle_sample(batch, 3, 1)
    compare_sample(gpu, ref, batch["temperature"].numpy())


def _outs_np(outs):
    return {"tokens": outs["tok"].cpu().numpy(), "accepted": outs["acc"].cpu().numpy(),
            "status": outs["st"].cpu().numpy(), "p": outs["p"].cpu().numpy(), "q": outs["q"].cpu().numpy()}


def _sized(B, K, V, seed):
    batch = synth.make_batch(B, K, V, torch.bfloat16, seed, noise_sigmas=(0.3, 1.0), temperature=(0.6, 1.4),
                             greedy_mask=[b % 7 == 3 for b in range(B)])
    return batch, to_dev(batch)


def test_single_kernel_path_ignores_what_the_workspace_held():
    """B = 320 (at least one request per SM): a workspace of 0xA5 bytes, then one
    of 0xFF bytes; both calls equal the oracle."""
    from speculative_decoding_verification_15_gb300 import binding

    lib = binding.load()
    B, K, V = 320, 3, 5000
    assert B >= torch.cuda.get_device_properties(0).multi_processor_count
    batch, d = _sized(B, K, V, 3201)
    ref = run_oracle_sample(batch, 3, 1)
    ws = torch.full((binding.spec_verify_workspace_size(B, K, V, 0),), 0xA5, dtype=torch.uint8, device="cuda")
    for fill in (0xA5, 0xFF):
        ws.fill_(fill)
        outs = _outs(B, K)
        assert _call(lib, d["target"], d["draft"], d["draft_tokens"], d["temperature"], outs, ws, B, K, V) == 0
        torch.cuda.synchronize()
        compare_sample(_outs_np(outs), ref, batch["temperature"].numpy())
        assert (outs["st"].cpu().numpy() == 0).all()
        assert int(ws[:4].view(torch.int32).item()) == 0  # the shared chunk counter


def test_one_workspace_alternates_between_the_two_paths():
    """B = 320 (single kernel, V = 5000), B = 16 (two kernels, K = 8, V = 151936: 1280
    chunks, more than the two static chunks of each of main_kernel's CTAs, so the
    ticket counter the single kernel shares must be zero again), then both once more,
    on one zero-filled workspace: every call equals the oracle."""
    from speculative_decoding_verification_15_gb300 import binding

    lib = binding.load()
    shapes = [(320, 3, 5000, 3202), (16, 8, 151936, 3203), (320, 3, 5000, 3204), (16, 8, 151936, 3205)]
    size = max(binding.spec_verify_workspace_size(B, K, V, 0) for B, K, V, _ in shapes)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for B, K, V, seed in shapes:
        batch, d = _sized(B, K, V, seed)
        outs = _outs(B, K)
        assert _call(lib, d["target"], d["draft"], d["draft_tokens"], d["temperature"], outs, ws, B, K, V) == 0
        torch.cuda.synchronize()
        compare_sample(_outs_np(outs), run_oracle_sample(batch, 3, 1), batch["temperature"].numpy())
        assert (outs["st"].cpu().numpy() == 0).all()
        assert int(ws[:4].view(torch.int32).item()) == 0  # the shared chunk counter


@pytest.mark.parametrize("offset", [0, -1])
def test_batch_at_the_sm_count(offset):
    """B = the SM count runs the single kernel with two commit items a request
    (Q = 2 CTAs per SM / 1 request per SM); B = SM count - 1 runs the two kernels.
    K = 3, V = 151936 bf16 (5 chunks a row), every seventh request greedy."""
    import speculative_decoding_verification_15_gb300 as pkg

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, K, V = sms + offset, 3, 151936
    batch, d = _sized(B, K, V, 3300 + B)
    out = pkg.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["temperature"], 3, 1)
    torch.cuda.synchronize()
    gpu = {k: v.cpu().numpy() for k, v in out.items()}
    compare_sample(gpu, run_oracle_sample(batch, 3, 1), batch["temperature"].numpy())
    assert (gpu["status"] == 0).all()
