"""The N > 1 paths on CPU: two gloo ranks -- the benchmark's weak scaling and
max-over-ranks time, and the KV-parallel exchange (each owner's partials of its
own splits, an all-gather, the ordered fold in global split order)."""
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


def _canonical(step):
    """(row, split) -> entry in the canonical partial layout: rows in flat
    order, each row's splits in order."""
    import split_rule
    idx, e = {}, 0
    pos = step.row_positions()
    for r in range(step.T):
        for i, _ in enumerate(split_rule.split_starts(int(pos[r]) + 1)):
            idx[(r, i)] = e
            e += 1
    return idx, e


def _kvp_rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle.paged_attention as opa
    import split_rule
    from helpers import to_store
    from invariant_paged_kv_gb300 import kv_parallel, workload as wl
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        geom = wl.Geometry(4, 2, 16, 16, "f32")
        ctx = [1100, 9, 1537, 600, 2100]
        q_lens = [1, 3, 1, 40, 1]
        step = wl.build_step(geom, q_lens, ctx, sum(-(-c // 16) for c in ctx) + 3,
                             np.random.default_rng(3))
        t = wl.make_tensors(step, 77, "cpu")
        q = opa.widen(to_store(t["q"][0]), "f32")
        kc, vc = to_store(t["k_cache"][0]), to_store(t["v_cache"][0])
        bounds = kv_parallel.owner_bounds(step.ctx_lens, world)
        idx, E = _canonical(step)
        lane_of, pos = step.row_lane(), step.row_positions()
        H, D = geom.H, geom.D
        scale = opa.default_scale(D)

        def seq(b):
            K = opa.widen(opa.gather(kc, step.block_tables[b], int(step.ctx_lens[b]), 16), "f32")
            V = opa.widen(opa.gather(vc, step.block_tables[b], int(step.ctx_lens[b]), 16), "f32")
            return K, V

        def partials_fn(buf):
            view = buf.view(torch.float64).view(E, H, D + 2)
            for r in range(step.T):
                b, p = int(lane_of[r]), int(pos[r])
                K, V = seq(b)
                starts = split_rule.split_starts(p + 1)
                sl = split_rule.split_length(p + 1)
                for i, k0 in enumerate(starts):
                    if not (bounds[rank, b] <= k0 < bounds[rank + 1, b]):
                        continue  # another owner's split
                    for h in range(H):
                        m, l, a = opa.row_partial(q[r], K, V, k0, min(k0 + sl, p + 1), scale, h)
                        view[idx[(r, i)], h, 0], view[idx[(r, i)], h, 1] = m, l
                        view[idx[(r, i)], h, 2:] = torch.from_numpy(a)

        def merge_fn(gathered, W):
            views = gathered.view(torch.float64).view(W, E, H, D + 2)
            res = np.zeros((step.T, H, D))
            for r in range(step.T):
                b, p = int(lane_of[r]), int(pos[r])
                for h in range(H):
                    parts = []
                    for i, k0 in enumerate(split_rule.split_starts(p + 1)):
                        w = max(x for x in range(W) if bounds[x, b] <= k0)
                        e = views[w, idx[(r, i)], h]
                        parts.append((float(e[0]), float(e[1]), e[2:].numpy()))
                    res[r, h] = opa.fold_partials(parts)
            return res

        local = torch.full((E * H * (D + 2) * 8,), 0xFF, dtype=torch.uint8)
        got = kv_parallel.kv_parallel_attention(partials_fn, merge_fn, local)
        want, _, _ = opa.attention(to_store(t["q"][0]), kc, vc, step.block_tables,
                                   step.cu_seqlens_q, step.ctx_lens, scale, "f32", 16)
        out[rank] = (got.tobytes(), float(np.max(np.abs(got - want))),
                     int(sum(1 for b in range(step.B) if 0 < bounds[1, b] < step.ctx_lens[b])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_kv_parallel_exchange_two_gloo_ranks():
    """Two page owners: each computes only its own splits, the buffers are
    all-gathered, both fold every row in global split order -- both ranks get
    the same bits, and they agree with the single-owner oracle."""
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_kvp_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    (b0, e0, split0), (b1, e1, _) = out[0], out[1]
    assert b0 == b1              # every rank merges to the same bits
    assert e0 <= 1e-12 and e1 <= 1e-12
    assert split0 >= 2           # lanes really were shared between the owners


def test_split_rule_named_values():
    """The tests' copy of the library's split rule: named values of the rule
    pa_attention documents, its defining property, and agreement with the
    host copy the KV-parallel owner bounds use."""
    import sys
    sys.path.insert(0, ROOT)
    import split_rule
    from invariant_paged_kv_gb300 import kv_parallel
    cases = {1: 512, 512: 512, 65536: 512, 65537: 1024, 131072: 1024, 131073: 2048,
             10 ** 6: 8192}
    for keys, want in cases.items():
        assert split_rule.split_length(keys) == want
    for keys in (1, 7, 513, 40000, 70000, 300000, 2 ** 21 + 3):
        s = split_rule.split_length(keys)
        assert -(-keys // s) <= 128 and (s == 512 or -(-keys // (s // 2)) > 128)
        st = split_rule.split_starts(keys)
        assert st[0] == 0 and st[-1] < keys and all(b - a == s for a, b in zip(st, st[1:]))
        assert kv_parallel.split_len(keys) == s
