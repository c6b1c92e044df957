"""Helpers shared by the GPU tests: move a step to the device, call the C ABI,
and call the oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle.paged_attention as opa
import parity_bound as pb
from helpers import to_store
from invariant_paged_kv_gb300 import pa, workload as wl


def device_step(step: wl.Step, device="cuda"):
    return dict(
        block_tables=torch.from_numpy(np.ascontiguousarray(step.block_tables)).to(device),
        cu_seqlens_q=torch.from_numpy(step.cu_seqlens_q).to(device),
        ctx_lens=torch.from_numpy(step.ctx_lens.astype(np.int32)).to(device),
        slot_mapping=torch.from_numpy(step.slot_mapping).to(device),
    )


def cache_torch_dtype(g: wl.Geometry):
    return {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}[g.dtype]


def workspace_for(step: wl.Step, mode="batch"):
    g = step.geom
    dt = cache_torch_dtype(g)
    n = pa.workspace_bytes(step.B, step.T, step.max_q_len, step.max_ctx_len,
                           int(step.ctx_lens.sum()), g.H, g.Hkv, g.D, g.block_size, dt,
                           mode=mode)
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def run_attention(step: wl.Step, t: dict, layer=0, write=True, scale=None, status=None,
                  out=None, dev=None, workspace=None, mode="batch", reuse_plan=False):
    """One pa_attention call; returns out (device) and the status flags."""
    g = step.geom
    dev = dev or device_step(step)
    q = t["q"][layer]
    if out is None:
        out = torch.full_like(q, float("nan"))
    st = status if status is not None else pa.new_status()
    ws = workspace if workspace is not None else workspace_for(step, mode)
    kw = {}
    if write:
        kw = dict(slot_mapping=dev["slot_mapping"], k_new=t["k_new"][layer],
                  v_new=t["v_new"][layer])
    pa.attention(q, t["k_cache"][layer], t["v_cache"][layer], dev["block_tables"],
                 dev["cu_seqlens_q"], dev["ctx_lens"], out,
                 max_q_len=step.max_q_len, max_ctx_len=step.max_ctx_len,
                 scale=opa.default_scale(g.D) if scale is None else scale,
                 workspace=ws, status=st, mode=mode, reuse_plan=reuse_plan, **SCALES, **kw)
    flags = pa.read_status(st)
    return out, flags


SCALES = dict(k_scale=wl.FP8_K_SCALE, v_scale=wl.FP8_V_SCALE)


def oracle_attention(step: wl.Step, t_cpu: dict, layer=0, write=True, rows=None, scale=None,
                     caches=None, terms=False):
    """Oracle output (float64) plus the caches after the write, from CPU copies
    (and, with ``terms``, the rows' bound terms as a fourth item)."""
    g = step.geom
    kc = caches[0] if caches is not None else to_store(t_cpu["k_cache"][layer])
    vc = caches[1] if caches is not None else to_store(t_cpu["v_cache"][layer])
    kw = {}
    if write:
        kw = dict(slot_mapping=step.slot_mapping, k_new=to_store(t_cpu["k_new"][layer]),
                  v_new=to_store(t_cpu["v_new"][layer]))
    return opa.attention(to_store(t_cpu["q"][layer]), kc, vc, step.block_tables,
                         step.cu_seqlens_q, step.ctx_lens,
                         opa.default_scale(g.D) if scale is None else scale, g.dtype,
                         g.block_size, rows=rows, terms=terms, **SCALES, **kw)


def to_cpu(t: dict) -> dict:
    return {k: [x.cpu() for x in v] for k, v in t.items()}


def max_abs(gpu_out: torch.Tensor, ref: np.ndarray, rows=None) -> float:
    got = gpu_out.detach().cpu().to(torch.float64).numpy()
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert not np.isnan(got).any(), "GPU output has NaN"
    assert not np.isnan(ref).any(), "oracle output has NaN on compared rows"
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


TOL = {"f32": 1e-5, "bf16": 2e-2, "fp8": 2e-2}

# (test, stats) of every parity comparison in this session, printed at the end
PARITY_LOG = []


def check_parity(gpu_out, ref: np.ndarray, terms: dict, positions, geom: wl.Geometry,
                 label: str, scale=None) -> dict:
    """Compare GPU rows with the oracle's: the acceptance bar (max-abs TOL) and
    the derived per-element rounding bound of parity_bound (every element
    within its bound, no per-row slope). ref / terms / positions are the
    same rows as gpu_out, in order."""
    got = gpu_out.detach().cpu().to(torch.float64).numpy() if torch.is_tensor(gpu_out) \
        else np.asarray(gpu_out, dtype=np.float64)
    assert not np.isnan(got).any(), "GPU output has NaN"
    assert not np.isnan(ref).any(), "oracle output has NaN on compared rows"
    sc = opa.default_scale(geom.D) if scale is None else scale
    st = pb.compare(got, ref, terms, positions, geom.D, sc, geom.dtype)
    st["rows"] = int(ref.shape[0])
    PARITY_LOG.append((label, geom.dtype, st))
    assert st["max_abs"] <= TOL[geom.dtype], (label, st)
    assert st["ratio"] <= 1.0, f"{label}: an element exceeds its rounding bound: {st}"
    assert st["slope_ratio"] <= 1.0, f"{label}: a row's errors have a slope: {st}"
    return st


def rows_of(terms: dict, idx) -> dict:
    return {k: v[idx] for k, v in terms.items()}


def compact_lanes(step: wl.Step, t: dict, lanes, layer=0):
    """Sub-step holding only `lanes` (blocks renumbered into a compact pool
    copied to the host), its host tensors, the original rows of its rows, and
    the device index of its blocks."""
    sub, blocks, rows = wl.sub_step(step, lanes)
    idx = torch.from_numpy(blocks if len(blocks) else np.zeros(1, np.int64)).to(
        t["k_cache"][layer].device)
    ridx = torch.from_numpy(rows).to(t["q"][layer].device)
    sub_t = {
        "q": [t["q"][layer].index_select(0, ridx).cpu()],
        "k_cache": [t["k_cache"][layer].index_select(0, idx).cpu()],
        "v_cache": [t["v_cache"][layer].index_select(0, idx).cpu()],
        "k_new": [t["k_new"][layer].index_select(0, ridx).cpu()],
        "v_new": [t["v_new"][layer].index_select(0, ridx).cpu()],
    }
    return sub, sub_t, rows, idx
