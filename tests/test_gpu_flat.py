"""The flattened ragged layout ("DSpark paper review", Sec. 4: the engine flattens
every token of the batch and tracks each one's request) through the C ABI.

The flat entry points compute what the padded ones compute; only the addressing
differs.  So they are checked against the padded path on the same requests
(flattening is pure data movement, done here with torch indexing), against the
fp64 oracle, and under CUDA-graph capture with new inputs replayed.
"""
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


def flatten(batch: dict, base: int = 0):
    """Padded [B, K+1, V] / [B, K, V] / [B, K] -> flat rows; cu_draft starts at `base`
    (with `base` unused leading draft positions and target rows)."""
    nd = batch["num_draft"]
    B, K1, V = batch["target"].shape
    kb = nd.tolist() if nd is not None else [K1 - 1] * B
    t_rows = [batch["target"][b, : kb[b] + 1] for b in range(B)]
    d_rows = [batch["draft"][b, : kb[b]] for b in range(B)]
    x = [batch["draft_tokens"][b, : kb[b]] for b in range(B)]
    pad_t = torch.full((base, V), float("nan"), dtype=batch["target"].dtype)
    target = torch.cat([pad_t] + t_rows)
    draft = torch.cat([pad_t] + d_rows)
    tokens = torch.cat([torch.zeros(base, dtype=torch.int32)] + x)
    cu = torch.tensor([base] + list(np.cumsum(kb) + base), dtype=torch.int32)
    return dict(target=target, draft=draft, tokens=tokens, cu=cu, kb=kb)


def unflatten_tokens(flat_tokens, cu, kb, K):
    B = len(kb)
    out = np.full((B, K + 1), -1, np.int32)
    for b in range(B):
        t0 = int(cu[b]) + b
        out[b, : kb[b] + 1] = flat_tokens[t0 : t0 + kb[b] + 1]
    return out


def unflatten_pq(flat, cu, kb, K):
    out = np.full((len(kb), K), -1.0, np.float32)
    for b in range(len(kb)):
        out[b, : kb[b]] = flat[int(cu[b]) : int(cu[b]) + kb[b]]
    return out


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("base", [0, 3])
def test_sample_flat_matches_padded_and_oracle(dt, base):
    import speculative_decoding_verification_15_gb300 as pkg

    B, K, V = 14, 6, 23011
    nd = [0, 1, 2, 3, 4, 5, 6, 6, 3, 0, 1, 2, 6, 5]
    batch = synth.make_batch(B, K, V, dt, 31, zipf=True, noise_sigmas=(0.5, 1.0), temperature=(0.6, 1.0),
                             num_draft=nd)
    f = flatten(batch, base)
    dev = "cuda"
    out = pkg.verify_sample_flat(f["target"].to(dev), f["draft"].to(dev), f["cu"].to(dev), f["tokens"].to(dev),
                                 batch["temperature"].to(dev), 9, 4, K)
    d = to_dev(batch, dev)
    pad = pkg.verify_sample(d["target"], d["draft"], d["draft_tokens"], d["temperature"], 9, 4,
                            num_draft=d["num_draft"])
    torch.cuda.synchronize()
    cu = f["cu"].numpy()
    tok = unflatten_tokens(out["tokens"].cpu().numpy(), cu, f["kb"], K)
    p = unflatten_pq(out["p"].cpu().numpy(), cu, f["kb"], K)
    q = unflatten_pq(out["q"].cpu().numpy(), cu, f["kb"], K)
    # The same arithmetic on the same rows.  Rows whose byte length is not a
    # multiple of 16 start at other alignments in the two layouts, which changes
    # the lanes' summation order, so p and q agree to rounding, not bit for bit;
    # outputs agree exactly away from the oracle's near-ties.
    ref = run_oracle_sample(batch, 9, 4)
    ok = ref["flags"] == 0
    assert (tok[ok] == pad["tokens"].cpu().numpy()[ok]).all()
    assert (out["accepted"].cpu().numpy()[ok] == pad["accepted"].cpu().numpy()[ok]).all()
    assert (out["status"].cpu().numpy() == pad["status"].cpu().numpy()).all()
    assert np.abs(p - pad["p"].cpu().numpy()).max() <= 1e-6 and np.abs(q - pad["q"].cpu().numpy()).max() <= 1e-6
    gpu = dict(tokens=tok, accepted=out["accepted"].cpu().numpy(), status=out["status"].cpu().numpy(), p=p, q=q)
    compare_sample(gpu, ref, batch["temperature"].numpy())


def test_sample_flat_single_kernel():
    """The flattened layout at B = 256 (the single-kernel path), ragged k_b from 0 to
    6, against the oracle."""
    import speculative_decoding_verification_15_gb300 as pkg

    B, K, V = 256, 6, 23011
    nd = [(5 * b + 3) % (K + 1) for b in range(B)]
    batch = synth.make_batch(B, K, V, torch.bfloat16, 41, zipf=True, noise_sigmas=(0.5, 1.0),
                             temperature=(0.6, 1.0), num_draft=nd, greedy_mask=[b % 9 == 4 for b in range(B)])
    f = flatten(batch)
    out = pkg.verify_sample_flat(f["target"].cuda(), f["draft"].cuda(), f["cu"].cuda(), f["tokens"].cuda(),
                                 batch["temperature"].cuda(), 5, 6, K)
    torch.cuda.synchronize()
    cu = f["cu"].numpy()
    gpu = dict(tokens=unflatten_tokens(out["tokens"].cpu().numpy(), cu, f["kb"], K),
               accepted=out["accepted"].cpu().numpy(), status=out["status"].cpu().numpy(),
               p=unflatten_pq(out["p"].cpu().numpy(), cu, f["kb"], K), q=unflatten_pq(out["q"].cpu().numpy(), cu,
                                                                                      f["kb"], K))
    compare_sample(gpu, run_oracle_sample(batch, 5, 6), batch["temperature"].numpy())
    assert (gpu["status"] == 0).all()


def test_greedy_flat_matches_padded():
    import speculative_decoding_verification_15_gb300 as pkg

    B, K, V = 9, 5, 40000
    nd = [5, 0, 1, 2, 3, 4, 5, 5, 2]
    batch = synth.make_batch(B, K, V, torch.bfloat16, 77, zipf=True, noise_sigmas=(0.1,), num_draft=nd)
    f = flatten(batch, 2)
    out = pkg.verify_greedy_flat(f["target"].cuda(), f["cu"].cuda(), f["tokens"].cuda(), K)
    d = to_dev(batch)
    pad = pkg.verify_greedy(d["target"], d["draft_tokens"], num_draft=d["num_draft"])
    torch.cuda.synchronize()
    tok = unflatten_tokens(out["tokens"].cpu().numpy(), f["cu"].numpy(), f["kb"], K)
    # greedy compares raw values: exact whatever the summation order
    assert (tok == pad["tokens"].cpu().numpy()).all()
    assert (out["accepted"].cpu().numpy() == pad["accepted"].cpu().numpy()).all()
    assert (out["status"].cpu().numpy() == 0).all()


def test_flat_bad_offsets_report_status_2():
    import speculative_decoding_verification_15_gb300 as pkg

    V = 4096
    t = torch.randn(12, V, device="cuda")
    dft = torch.randn(12, V, device="cuda")
    # request 1 runs backwards (k = -1), request 2 exceeds Kmax = 3 (k = 4)
    cu = torch.tensor([0, 2, 1, 5, 6], dtype=torch.int32, device="cuda")
    x = torch.zeros(12, dtype=torch.int32, device="cuda")
    out = pkg.verify_sample_flat(t, dft, cu, x, torch.ones(4, device="cuda"), 1, 1, 3)
    torch.cuda.synchronize()
    assert out["status"].cpu().tolist() == [0, 2, 2, 0]
    assert out["accepted"].cpu().tolist()[1:3] == [0, 0]


def test_scheduler_lengths_feed_flat_verify():
    """The scheduler's lengths become the offsets of a flat batch with no padding."""
    import speculative_decoding_verification_15_gb300 as pkg

    s = synth.ragged_schedule_inputs(0, B=64, Kmax=16)
    L, _ = pkg.schedule_verify_len(s["conf"].cuda(), s["step_time_us"].cuda(), s["budget"] // 4, s["min_len"])
    nd = L.cpu().tolist()
    batch = synth.ragged(0, num_draft=nd, V=32000, B=64, Kmax=16)
    f = flatten(batch)
    out = pkg.verify_sample_flat(f["target"].cuda(), f["draft"].cuda(), f["cu"].cuda(), f["tokens"].cuda(),
                                 batch["temperature"].cuda(), 2, 8, 16)
    torch.cuda.synchronize()
    gpu = dict(tokens=unflatten_tokens(out["tokens"].cpu().numpy(), f["cu"].numpy(), f["kb"], 16),
               accepted=out["accepted"].cpu().numpy(), status=out["status"].cpu().numpy(),
               p=unflatten_pq(out["p"].cpu().numpy(), f["cu"].numpy(), f["kb"], 16),
               q=unflatten_pq(out["q"].cpu().numpy(), f["cu"].numpy(), f["kb"], 16))
    compare_sample(gpu, run_oracle_sample(batch, 2, 8), batch["temperature"].numpy())


@pytest.mark.parametrize("B", [8, 200])
def test_flat_verify_under_cuda_graph_capture(B):
    """Capture one flat sampling verify in a CUDA graph, then replay it on new
    inputs copied into the captured buffers: same results as eager calls.  B = 200
    (at least one request per SM) captures the single kernel with the memset of
    its counters before it."""
    from speculative_decoding_verification_15_gb300 import api, binding

    K, V = 4, 30000
    nd = ([4, 1, 0, 3, 4, 2, 4, 1] * 32)[:B]
    batches = [synth.make_batch(B, K, V, torch.bfloat16, 500 + i, zipf=True, noise_sigmas=(0.5, 1.0),
                                temperature=(0.7, 1.0), num_draft=nd) for i in range(3)]
    flats = [flatten(b) for b in batches]
    dev = torch.device("cuda")
    t = flats[0]["target"].to(dev)
    d = flats[0]["draft"].to(dev)
    cu = flats[0]["cu"].to(dev)
    x = flats[0]["tokens"].to(dev)
    T = batches[0]["temperature"].to(dev)
    out = dict(tokens=torch.empty(t.shape[0], dtype=torch.int32, device=dev),
               accepted=torch.empty(B, dtype=torch.int32, device=dev),
               p=torch.empty(d.shape[0], device=dev), q=torch.empty(d.shape[0], device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    ws = api.workspace(dev, binding.spec_verify_workspace_size(B, K, V, binding.SPEC_BF16))

    def call():
        binding.spec_verify_sample_flat(t, d, cu, x, T, 17, 3, out["tokens"], out["accepted"], out["p"], out["q"],
                                        out["status"], ws, K)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # first call on the device does the set-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for i in (1, 2, 0):
        t.copy_(flats[i]["target"])
        d.copy_(flats[i]["draft"])
        x.copy_(flats[i]["tokens"])
        T.copy_(batches[i]["temperature"])
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.clone() for k, v in out.items()}
        call()
        torch.cuda.synchronize()
        for k in out:
            assert torch.equal(got[k], out[k]), k
        ref = run_oracle_sample(batches[i], 17, 3)
        gpu = dict(tokens=unflatten_tokens(got["tokens"].cpu().numpy(), flats[i]["cu"].numpy(), nd, K),
                   accepted=got["accepted"].cpu().numpy(), status=got["status"].cpu().numpy(),
                   p=unflatten_pq(got["p"].cpu().numpy(), flats[i]["cu"].numpy(), nd, K),
                   q=unflatten_pq(got["q"].cpu().numpy(), flats[i]["cu"].numpy(), nd, K))
        compare_sample(gpu, ref, batches[i]["temperature"].numpy())
