#!/usr/bin/env python
"""Benchmark of the batched speculative-decoding verify/commit step on GB300.

One step = one spec_verify_sample call over the "main" workload: B=64 requests,
K=7 drafts each, V=151,936, bf16 target [64, 8, V] and draft [64, 7, V] logits,
temperatures U[0.6, 1.0] (synthetic, seeded; see synth.py).  The metric is
verified draft tokens per second (sum_b k_b = 448 per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: inputs resident in HBM; an L2 flush (256 MiB write) before every step,
outside the per-step CUDA events; the value is the sum of those events over the
K timed steps, max over ranks.  For N > 1 (launched by torchrun) every rank
verifies its own batch on its own GPU (replicas, no data-path collective).
`--impl reference` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/sec and HBM GB/s (% of GB300 peak), B=64 K=7 V=151936 bf16"
UNIT = "tokens/s"
WORKLOAD = "main: B=64 K=7 V=151936, bf16 target+draft logits, sampling, T~U[0.6,1.0]"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = ["speculative_decoding_verification_15_gb300/csrc/verify.cu",
                  "speculative_decoding_verification_15_gb300/csrc/spec_common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "main_kernel_main.md")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic() -> float | None:
    """dram read+write bytes per main_kernel launch from the committed ncu summary,
    if it was taken on the current kernel source."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    sha, traffic = None, None
    for line in text.splitlines():
        if line.startswith("source_sha:"):
            sha = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if sha == kernel_source_sha() else None


def hbm_peak() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self) -> dict | None:
        if self.proc is None:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def replica_batch(rank: int) -> dict:
    """The requests rank `rank` verifies: replicas share no request (the data seed
    differs per rank), so ranks never exchange data."""
    import synth

    return synth.main(step=rank)


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over the ranks of the default process group (x with one rank)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_step: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: units every rank processed over the slowest rank's time."""
    return world * units_per_step * steps / (total_ms * 1e-3)


def oracle_cpu_rate(batch: dict, seed: int, min_seconds: float, max_reps: int) -> dict:
    """Time the fp64 oracle on the host cores over whole copies of the batch."""
    import oracle
    import synth

    cores = len(os.sched_getaffinity(0))
    t = synth.as_oracle_array(batch["target"])
    d = synth.as_oracle_array(batch["draft"])
    x = batch["draft_tokens"].numpy()
    T = batch["temperature"].numpy()
    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.verify_sample(t, d, x, None, T, seed, reps, nthreads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    tokens = int(batch["draft_tokens"].shape[0] * batch["draft_tokens"].shape[1]) * reps
    return {"value": tokens / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} x the full {batch['B']}-request batch, OpenMP over requests, {el:.2f} s wall"}


def run_reference(args) -> None:
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import synth

    full = synth.main(0)
    n_req = 16  # bounded sample: the first 16 of the 64 requests per step
    batch = dict(full, B=n_req, target=full["target"][:n_req], draft=full["draft"][:n_req],
                 draft_tokens=full["draft_tokens"][:n_req], temperature=full["temperature"][:n_req])
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        r = oracle_cpu_rate(batch, 3, 0.0, 1)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
        cores = r["cores"]
    tok = n_req * 7
    total = sum(times)
    value = tok * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "B": 64, "K": 7, "V": 151936},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "16 of the 64 requests per step, OpenMP over requests"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args) -> None:
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import __graft_entry__
    import synth

    __graft_entry__.build()
    import speculative_decoding_verification_15_gb300 as pkg
    from speculative_decoding_verification_15_gb300 import binding

    batch = replica_batch(rank)
    B, K, V = batch["B"], batch["K"], batch["V"]
    t = batch["target"].to(dev)
    d = batch["draft"].to(dev)
    x = batch["draft_tokens"].to(dev)
    T = batch["temperature"].to(dev)
    tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    st = torch.empty(B, dtype=torch.int32, device=dev)
    pp = torch.empty((B, K), dtype=torch.float32, device=dev)
    qq = torch.empty((B, K), dtype=torch.float32, device=dev)
    ws = pkg.workspace(dev, binding.spec_verify_workspace_size(B, K, V, binding.SPEC_BF16))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write 256 MiB, then read another 256 MiB: L2 ends up holding clean lines of an
        # unrelated buffer, so no write-back of the flush lands inside the timed step
        flush.zero_()
        flush_rd.sum()
    stream = torch.cuda.current_stream(dev)
    verified = B * K  # every request verifies all K drafts
    esz = t.element_size()
    algo_bytes = B * (2 * K + 1) * V * esz  # step: one read of every needed logit row
    main_bytes = B * 2 * K * V * esz        # main_kernel: the target and draft rows of the drafts

    def step(i):
        binding.spec_verify_sample(t, d, x, None, T, 3, i, tokens, acc, pp, qq, st, ws, stream)

    for i in range(args.warmup):
        flush_l2()
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index if world == 1 else local) as clk:
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush_l2()
            starts[i].record(stream)
            step(args.warmup + i)
            ends[i].record(stream)
        torch.cuda.synchronize()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # Per-kernel times: a second timed pass with the library recording CUDA events
    # around each of its launches (events between the launches serialise them, so
    # the step time above is taken without them).
    binding.profile_enable(True)
    kern_ms = []
    for i in range(args.steps):
        flush_l2()
        step(args.warmup + args.steps + i)
        kern_ms.append(binding.profile_read(2))  # waits for this step's kernel events
    binding.profile_enable(False)
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, dev)
    assert int((st != 0).sum()) == 0, "a request reported a non-zero status"
    emitted = int(acc.sum().item()) + B
    rows_ms = statistics.mean(k[0] for k in kern_ms)
    per_kernel = [statistics.mean(k[j] for k in kern_ms) for j in range(len(kern_ms[0]))]

    # Early exit on the same workload, timed the same way and reported beside the
    # headline: one kernel, each request's rows read in position order up to its
    # first rejection.
    ee_ms = []
    for i in range(args.warmup + args.steps):
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        binding.spec_verify_sample_early_exit(t, d, x, None, T, 3, i, tokens, acc, pp, qq, st, stream)
        e1.record(stream)
        ee_ms.append((e0, e1))
    torch.cuda.synchronize()
    ee_ms = [a.elapsed_time(b) for a, b in ee_ms[args.warmup:]]
    assert int((st != 0).sum()) == 0, "a request reported a non-zero status (early exit)"
    ee_rows = int((2 * torch.clamp(acc + 1, max=K) + (acc == K).to(torch.int32)).sum().item())

    # Markov-head drafting of the same block shape (B, K, V), rank 256, random
    # factors: the draft-side step before verify, timed beside the headline.
    mk = synth.markov(0, B=B, K=K, V=V, r=256, dtype=t.dtype)
    mk_dev = {n: mk[n].to(dev) for n in ("base", "anchor", "emb", "proj", "temperature")}
    mk_tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    mk_z = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    mk_st = torch.empty(B, dtype=torch.int32, device=dev)
    mk_ev = []
    for i in range(args.warmup + min(args.steps, 10)):
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        binding.spec_markov_draft(mk_dev["base"], mk_dev["anchor"], mk_dev["emb"], mk_dev["proj"],
                                  mk_dev["temperature"], 6, i, mk_tok, mk_z, mk_st, stream)
        e1.record(stream)
        mk_ev.append((e0, e1))
    torch.cuda.synchronize()
    mk_ms = statistics.mean(a.elapsed_time(b) for a, b in mk_ev[args.warmup:])
    assert int((mk_st != 0).sum()) == 0, "a Markov draft request reported a non-zero status"
    del mk_dev, mk_z

    # end to end: pinned host inputs -> device, verify, outputs -> host, every step
    th, dh = t.cpu().pin_memory(), d.cpu().pin_memory()
    xh, Th = x.cpu().pin_memory(), T.cpu().pin_memory()
    out_h = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in
             dict(tokens=tokens, acc=acc, st=st).items()}
    h2d = th.numel() * th.element_size() + dh.numel() * dh.element_size() + xh.numel() * 4 + Th.numel() * 4
    d2h = sum(v.numel() * v.element_size() for v in out_h.values())
    e2e_steps = max(3, min(args.steps, 20))
    for i in range(2):  # warm the copy path
        t.copy_(th, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        t.copy_(th, non_blocking=True)
        d.copy_(dh, non_blocking=True)
        x.copy_(xh, non_blocking=True)
        T.copy_(Th, non_blocking=True)
        step(10_000 + i)
        out_h["tokens"].copy_(tokens, non_blocking=True)
        out_h["acc"].copy_(acc, non_blocking=True)
        out_h["st"].copy_(st, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    if rank == 0:
        peak, peak_kind = hbm_peak()
        achieved = main_bytes / (rows_ms * 1e-3) / 1e9
        cpu = oracle_cpu_rate(batch, 3, min_seconds=12.0, max_reps=1000) if world == 1 else None
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": job_rate(world, verified, args.steps, total_ms), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": B, "K": K, "V": V, "logits": "bf16",
                       "l2": "flushed before every step (256 MiB write + 256 MiB read of other buffers), outside the "
                             "per-step events; "
                             "inputs 292 MB > L2",
                       "parallelism": f"replicas x{world}"},
            "emitted_tokens_per_s": world * emitted * args.steps / (total_ms * 1e-3),
            "step_hbm_gbs": algo_bytes / (total_ms / args.steps * 1e-3) / 1e9,
            "kernel_ms": {"main": per_kernel[0], "commit": per_kernel[1] if len(per_kernel) > 1 else None},
            "roofline": {"bound": "hbm", "kernel": "main_kernel", "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "algorithmic_bytes": main_bytes, "traffic": measured_traffic()},
            "step_algorithmic_bytes": algo_bytes,
            "e2e": {"value": world * verified / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "early_exit": {"ms_per_step": statistics.mean(ee_ms),
                           "value": world * verified / (statistics.mean(ee_ms) * 1e-3), "unit": UNIT,
                           "rows_read_per_step": ee_rows, "rows_full_scan": B * (2 * K + 1)},
            "markov_draft": {"ms_per_call": mk_ms, "positions": K, "rank": 256,
                             "draft_tokens_per_s": world * B * K / (mk_ms * 1e-3)},
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
