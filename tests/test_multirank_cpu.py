"""The multi-rank logic of the benchmark on CPU with two gloo ranks: each
rank draws its own independent batch, the timed region's time is the maximum
over ranks, the whole-job value counts every rank's FLOPs (weak scaling), and
the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from exact_io_aware_27_gb300 import inputs as wl
    w = wl.SINGLE_HEAD_128
    seed = bench.rank_seed(w, rank)
    q = wl.attention_inputs(1, 1, 8, 8, 64, seed)[0]
    ms = 1.0 + rank  # rank 1 is slower
    worst = bench.max_over_ranks(ms)
    gathered = [torch.zeros_like(q) for _ in range(world)]
    dist.all_gather(gathered, q)
    distinct = not torch.equal(gathered[0], gathered[1])
    value = bench.weak_value(1e12, world, worst)

    class Args:
        steps, warmup = 1, 1
    ref_rc = bench.run_reference(Args) if rank == 1 else 0
    out[rank] = (seed, worst, distinct, value, ref_rc)
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    (s0, w0, d0, v0, r0), (s1, w1, d1, v1, r1) = out[0], out[1]
    assert s0 != s1 and d0 and d1                 # independent batches per rank
    assert w0 == w1 == 2.0                        # slowest rank's time everywhere
    assert v0 == pytest.approx(1e12 * 2 / 2e-3 / 1e12)  # both ranks' FLOPs / max time
    assert r1 == 0                                # non-zero ranks leave the reference arm
