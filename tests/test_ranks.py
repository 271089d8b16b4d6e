"""Host logic of the multi-process bench (one process per GPU), on CPU ranks
with the gloo backend: every rank decodes its own batch (no data-path
collective), the job's time is the slowest rank's, and its frame count is
every rank's frames."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench
    from ctc_prefix_beam_gb300 import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synth.workload("tiny", B=3, T=20)
    wr = bench.rank_workload(w, rank)
    lp, lens = synth.gen_batch(wr)
    mine = 1.0 + rank  # this rank's "time"
    slowest = bench.max_over_ranks(mine, dist, torch.device("cpu"))
    sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(sums, torch.tensor([float(np.nansum(lp))], dtype=torch.float64))
    out[rank] = (slowest, [float(x) for x in sums], bench.job_frames(world, lp.shape[0], lp.shape[1]), wr.seed)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_shard_rows_and_take_the_slowest_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        slowest, sums, frames, seed = res[r]
        assert slowest == float(world)           # max over ranks, seen by every rank
        assert frames == world * 3 * 20          # whole-job frames
        assert seed == r                         # tiny's seed 0 offset by the rank
    s0, s1 = res[0][1]
    assert s0 != s1                              # the two ranks decode different batches


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(2.5, None, None) == 2.5
    assert bench.job_frames(1, 32, 500) == 16000
