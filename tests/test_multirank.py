"""The N > 1 benchmark path on CPU: two gloo ranks, weak scaling, max-over-ranks time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from invariant_paged_kv_gb300 import workload as wl
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank builds its own independent step (seed offset by rank)
        class A:
            workload, small, layers, kv = "decode_batch", True, None, "bf16"
        step, layers, name = bench.make_step(A, rank)
        ms_local = 1.0 + rank  # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local, world)
        val = bench.weak_scaling_value(1000, world, ms)
        out[rank] = (ms, val, int(step.ctx_lens.sum()), name)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    (ms0, v0, c0, n0), (ms1, v1, c1, n1) = out[0], out[1]
    assert ms0 == ms1 == 2.0          # both ranks see the slowest rank's time
    assert v0 == v1 == pytest.approx(1000 * 2 / 2e-3 / 1e9)
    assert c0 != c1                   # independent work per rank
    assert n0 == n1 == "decode_batch"


def test_single_rank_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.weak_scaling_value(2e9, 1, 1.0) == pytest.approx(2000.0)
