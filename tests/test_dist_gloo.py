"""The multi-process (torchrun) path of bench.py, on CPU with gloo ranks.

The layer is row-independent, so data-parallel replicas need no collective on
the data path: each rank runs its own batch of tokens against the same
weights; only the timing uses a barrier and a max over ranks.  These tests run
that host logic with two gloo ranks."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle.lynx_oracle as O
    import synth

    w, r, _ = bench.dist_env()
    t = synth.layer_tensors("tiny", "linear", batch=r)
    rows = np.arange(8)
    y = O.linear(t["X"], t["W"], t["LA"], t["LB"], rows=rows)
    bench.barrier(w)
    elapsed = 1.0 + r  # a rank-local "timed region"
    mx = bench.max_over_ranks(elapsed, w, device="cpu")
    q.put((r, w, mx, t["X"][:2].copy(), t["W"][:2].copy(), y))
    dist.destroy_process_group()


def test_two_gloo_replicas_share_weights_not_batches():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, mx0, x0, wt0, y0), (r1, w1, mx1, x1, wt1, y1) = out
    assert (r0, r1) == (0, 1) and w0 == w1 == 2
    assert mx0 == mx1 == 2.0                       # max over ranks of 1.0 and 2.0
    assert np.array_equal(wt0, wt1)                # same weights on every replica
    assert not np.array_equal(x0, x1)              # independent batches of tokens
    assert not np.allclose(y0, y1)


def test_single_process_path_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
