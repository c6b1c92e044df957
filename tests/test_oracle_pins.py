"""The oracle agrees with every fact it is pinned to (CPU only)."""
import numpy as np
import pytest
import torch

import oracle.paged_attention as pa
import oracle_pins
from invariant_paged_kv_gb300 import workload
from helpers import to_store


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    msg = check()
    assert msg is None, msg


def test_f32_evaluation_within_tolerance_bar():
    """The tiny fp32 case evaluated entirely in float32 stays within 1e-6 of
    the fp64 oracle, so the 1e-5 fp32 parity bar leaves room for the GPU's
    different (but still fp32) rounding order."""
    step = workload.tiny_f32(0)
    t = workload.make_tensors(step, 1001)
    g = step.geom
    scale = pa.default_scale(g.D)
    args = dict(q=to_store(t["q"][0]), k_cache=to_store(t["k_cache"][0]),
                v_cache=to_store(t["v_cache"][0]), block_tables=step.block_tables,
                cu_seqlens_q=step.cu_seqlens_q, ctx_lens=step.ctx_lens,
                scale=scale, dtype="f32", block_size=g.block_size,
                slot_mapping=step.slot_mapping, k_new=to_store(t["k_new"][0]),
                v_new=to_store(t["v_new"][0]))
    ref, kc, vc = pa.attention(**args)
    # float32 evaluation of the same rows, written with torch ops
    q = t["q"][0]
    out32 = torch.empty_like(q)
    kcf = torch.from_numpy(kc)
    vcf = torch.from_numpy(vc)
    for b in range(step.B):
        c = int(step.ctx_lens[b])
        pos = torch.arange(c)
        blk = torch.from_numpy(step.block_tables[b].astype(np.int64))[pos // g.block_size]
        K = kcf[blk, pos % g.block_size]
        V = vcf[blk, pos % g.block_size]
        r = int(step.cu_seqlens_q[b])
        for h in range(g.H):
            s = (K[:, h // g.group] @ q[r, h]) * np.float32(scale)
            out32[r, h] = torch.softmax(s, 0) @ V[:, h // g.group]
    err = np.max(np.abs(out32.numpy().astype(np.float64) - ref))
    assert err < 1e-6, err


def test_rows_subset_matches_full():
    rng = np.random.default_rng(5)
    geom = workload.Geometry(4, 2, 16, 4, "bf16")
    step = workload.build_step(geom, [1, 5, 1], [9, 12, 1], 16, rng)
    t = workload.make_tensors(step, 7)
    common = dict(q=to_store(t["q"][0]), k_cache=to_store(t["k_cache"][0]),
                  v_cache=to_store(t["v_cache"][0]), block_tables=step.block_tables,
                  cu_seqlens_q=step.cu_seqlens_q, ctx_lens=step.ctx_lens,
                  scale=0.25, dtype="bf16", block_size=4)
    full, _, _ = pa.attention(**common)
    part, _, _ = pa.attention(rows=[2, 6], **common)
    assert np.array_equal(full[[2, 6]], part[[2, 6]])
    assert np.isnan(part[0]).all()
