"""KV-parallel page owners emulated on one GPU (GPU).

"Numerics envelopes", Layout invariance of query context parallelism: the
partials of the KV-parallel page owners are merged with the ordered fold; The
hierarchy: a reduction is data movement plus a fixed-order fp32 fold. W
virtual owners each hold a split-aligned share of every lane's keys -- their
block tables keep only their own pages, the rest are -1 -- and compute the
partials of their splits into their own buffer; the buffers side by side are
what an all-gather leaves, and the merge must give bitwise the single-owner
(row-invariant) output.
"""
import numpy as np
import pytest
import torch

from gpu_harness import SCALES, cache_torch_dtype, device_step, run_attention
from invariant_paged_kv_gb300 import build, kv_parallel, pa, workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    pa.load()


def _owner_table(step, lo, hi):
    """The block table an owner of keys [lo[b], hi[b]) holds: -1 elsewhere."""
    bt = step.block_tables.copy()
    bs = step.geom.block_size
    for b in range(step.B):
        keep = np.zeros(bt.shape[1], bool)
        if hi[b] > lo[b]:
            keep[lo[b] // bs: -(-int(hi[b]) // bs)] = True
        bt[b, ~keep] = -1
    return bt


def _kv_parallel(step, t, bounds, status_check=True):
    g = step.geom
    W = bounds.shape[0] - 1
    dev = device_step(step)
    q = t["q"][0]
    pb = pa.partials_bytes(step.T, step.max_ctx_len, g.H, g.D)
    gathered = torch.full((W * pb,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN filler
    ws = torch.empty(pa.partials_workspace_bytes(step.B, step.T, step.max_ctx_len),
                     dtype=torch.uint8, device="cuda")
    st = pa.new_status()
    for w in range(W):
        lo, hi = bounds[w], bounds[w + 1]
        bt = torch.from_numpy(_owner_table(step, lo, hi)).cuda()
        pa.attention_partials(q, t["k_cache"][0], t["v_cache"][0], bt, dev["cu_seqlens_q"],
                              dev["ctx_lens"], torch.from_numpy(lo).cuda(),
                              torch.from_numpy(hi).cuda(), gathered[w * pb:(w + 1) * pb],
                              max_q_len=step.max_q_len, max_ctx_len=step.max_ctx_len,
                              scale=1.0 / np.sqrt(g.D), workspace=ws, status=st, **SCALES)
        flags = pa.read_status(st)
        if status_check:
            assert flags == 0, (w, flags)
    out = torch.full_like(q, float("nan"))
    pa.merge_partials(gathered, W, torch.from_numpy(bounds).cuda(), dev["cu_seqlens_q"],
                      dev["ctx_lens"], out, max_q_len=step.max_q_len,
                      max_ctx_len=step.max_ctx_len, workspace=ws,
                      kv_dtype=cache_torch_dtype(g), v_scale=SCALES["v_scale"], status=st)
    return out, pa.read_status(st)


def _random_bounds(step, W, seed):
    """Random split-aligned partitions (owners may hold nothing of a lane)."""
    rng = np.random.default_rng(seed)
    out = np.zeros((W + 1, step.B), np.int64)
    for b in range(step.B):
        c = int(step.ctx_lens[b])
        sl = kv_parallel.split_len(max(c, 1))
        n = -(-c // sl)
        cuts = np.sort(rng.integers(0, n + 1, size=W - 1))
        out[1:W, b] = np.minimum(cuts * sl, c)
        out[W, b] = c
    return out.astype(np.int32)


def _bits(x):
    return x.contiguous().view(torch.int32 if x.dtype == torch.float32 else torch.int16)


STEPS = {
    "decode_bf16": lambda: wl.decode_batch(0, lanes=24),
    "decode_e4m3": lambda: wl.decode_batch(1, lanes=24, dtype="fp8"),
    "tiny_f32": lambda: wl.tiny_f32(2),
    "chunks_bf16": lambda: wl.build_step(wl.Geometry(40, 8, 128, 16, "bf16"),
                                         [1, 130, 1, 64, 1], [3000, 1700, 70000, 600, 513],
                                         (3000 + 1700 + 70000 + 600 + 513) // 16 + 40,
                                         np.random.default_rng(5)),
}


@pytest.mark.parametrize("name", sorted(STEPS))
@pytest.mark.parametrize("W", [1, 2, 3, 5])
def test_owners_merge_bitwise(name, W):
    step = STEPS[name]()
    t = wl.make_tensors(step, 7000 + W, "cuda", poison=True)
    ref, flags = run_attention(step, t, write=False, mode="row")
    assert flags == 0
    for bounds in (kv_parallel.owner_bounds(step.ctx_lens, W),
                   _random_bounds(step, W, 17 + W)):
        out, flags = _kv_parallel(step, t, bounds)
        assert flags == 0
        assert torch.equal(_bits(out), _bits(ref)), (name, W)


def test_misaligned_bounds_are_flagged():
    step = wl.decode_batch(0, lanes=8)
    t = wl.make_tensors(step, 7100, "cuda")
    bounds = kv_parallel.owner_bounds(step.ctx_lens, 2)
    lane = int(np.argmax(step.ctx_lens))
    assert 0 < bounds[1, lane] < step.ctx_lens[lane]
    bounds[1, lane] += 16  # no longer a multiple of the split length
    _, flags = _kv_parallel(step, t, bounds, status_check=False)
    assert flags & pa.FLAGS["OWNER_RANGE"]
