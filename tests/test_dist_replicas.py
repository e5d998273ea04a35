"""The multi-rank path of bench.py on CPU (gloo, world size 2): replicas verify
disjoint requests, timing is the slowest rank's, and the whole-job rate counts the
units of every rank.  Each rank also runs the oracle on a small slice of its own
batch, so the replica inputs are exercised end to end without a GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import synth

    batch = bench.replica_batch(rank)
    x = batch["draft_tokens"][:2].numpy()
    res = oracle.verify_sample(synth.as_oracle_array(batch["target"][:2, :, :4096]),
                               synth.as_oracle_array(batch["draft"][:2, :, :4096]),
                               np.minimum(x, 4095), None, batch["temperature"][:2].numpy(), 3, rank)
    # every rank's own time; the job time is the largest
    local_ms = 10.0 + 5.0 * rank
    job_ms = bench.max_over_ranks(local_ms)
    rate = bench.job_rate(world, 448, 3, job_ms)
    sig = torch.tensor([float(batch["draft_tokens"].sum())], dtype=torch.float64)
    sigs = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(sigs, sig)
    np.save(os.path.join(out_dir, f"rank{rank}.npy"),
            np.array([job_ms, rate, sigs[0].item(), sigs[1].item(), float(res["status"].sum())]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas(tmp_path):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    r0, r1 = (np.load(tmp_path / f"rank{r}.npy") for r in range(world))
    assert r0[0] == r1[0] == 15.0                       # slowest rank's time on every rank
    assert r0[1] == pytest.approx(2 * 448 * 3 / 15e-3)  # units of both ranks
    assert r0[2] != r0[3]                               # the replicas verify different requests
    assert r0[4] == 0 and r1[4] == 0                    # and their own slices verify cleanly


def test_single_process_helpers():
    import bench

    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_rate(1, 448, 10, 1.0) == pytest.approx(448 * 10 / 1e-3)
