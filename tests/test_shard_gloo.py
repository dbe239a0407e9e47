"""The multi-process path on the CPU: two ranks over gloo (world size 2).

Each rank takes its contiguous shard of the branches (verify_spec_draft_gb300.shard),
computes its share of the mean survival with the oracle standing in for
spec_e2etv_shard (the GPU is not needed for the host logic), and the shares are
combined by the one scalar all-reduce.  The result must be the whole batch's loss, and
every shard's gradient rows the whole batch's rows (normalised by the global count).
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from verify_spec_draft_gb300 import shard, synth
from oracle import e2etv as oe

WORLD = 2


def test_shard_range_partitions():
    for n in (1, 2, 5, 7, 1024):
        for world in (1, 2, 3, 8):
            got = []
            for r in range(world):
                s, c = shard.shard_range(n, r, world)
                got.extend(range(s, s + c))
                assert c in (n // world, n // world + 1)
            assert got == list(range(n))
    with pytest.raises(ValueError):
        shard.shard_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, N, Wb, V):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        t, d = synth.e2etv_rows(N, Wb, V, 1.0, seed=77)
        t = t.double().numpy()
        d = d.double().numpy()
        full = oe.e2etv(t, d, N, Wb)
        b0, n = shard.shard_range(N, rank, WORLD)
        share = 0.0
        for b in range(b0, b0 + n):
            rows = slice(b * Wb, (b + 1) * Wb)
            br = oe.branch(t[rows], d[rows], N * Wb)
            share += br["sum_surv"] / (N * Wb)
            # the shard's gradient, normalised by the whole batch, is the batch's own
            assert np.abs(br["grad"] - full["grad"][rows]).max() <= 1e-15
        loss = shard.e2etv_loss_from_shares(torch.tensor([share], dtype=torch.float64))
        assert abs(float(loss.item()) - full["loss"]) <= 1e-12, (float(loss.item()), full["loss"])
        # timings are combined by the slowest rank
        assert shard.max_over_ranks(0.25 + rank, "cpu") == 0.25 + (WORLD - 1)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("N", [5, 8])
def test_two_ranks_combine_the_loss(N):
    mp.start_processes(_rank_main, args=(_free_port(), N, 3, 64), nprocs=WORLD, start_method="spawn", join=True)
