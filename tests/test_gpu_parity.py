"""CUDA path vs the CPU oracle, element by element, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import oracle.paged_attention as opa
from gpu_harness import (TOL, check_parity, compact_lanes, device_step, max_abs,
                         oracle_attention, rows_of, run_attention, to_cpu, workspace_for)
from helpers import to_store
from invariant_paged_kv_gb300 import build, pa, workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    pa.load()


def _bytes(t):
    return to_store(t).view(np.uint8)


# ---------------------------------------------------------------------------
# KV append
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("make,seed", [(wl.tiny_f32, 1001), (wl.decode_batch, 2001),
                                       (wl.mixed_step, 3001)])
def test_write_kv_bit_exact(make, seed):
    step = make(0)
    t = wl.make_tensors(step, seed, "cuda", poison=True)
    slots = step.slot_mapping.copy()
    slots[::7] = -1  # padding rows are skipped
    tc = to_cpu(t)
    pa.write_kv(t["k_new"][0], t["v_new"][0], t["k_cache"][0], t["v_cache"][0],
                torch.from_numpy(slots).cuda())
    kc, vc = opa.write_kv(to_store(tc["k_cache"][0]), to_store(tc["v_cache"][0]),
                          to_store(tc["k_new"][0]), to_store(tc["v_new"][0]), slots,
                          step.geom.block_size)
    assert np.array_equal(_bytes(t["k_cache"][0]), kc.view(np.uint8))
    assert np.array_equal(_bytes(t["v_cache"][0]), vc.view(np.uint8))


@pytest.mark.parametrize("make,seed", [(lambda s: wl.decode_batch(s, dtype="fp8"), 2002),
                                       (lambda s: wl.long_tail(s, lanes=24, pool_bytes_per_layer=2e8,
                                                               dtype="fp8"), 5002)])
def test_write_kv_e4m3_bit_exact(make, seed):
    """New bf16 rows land in e4m3 caches as exactly the oracle's codes."""
    step = make(0)
    t = wl.make_tensors(step, seed, "cuda", poison=True)
    # rows spanning the whole code range: tiny (subnormal codes), ordinary,
    # ties, beyond 448 * scale (saturation) and exact zeros of both signs
    g = torch.Generator(device="cuda").manual_seed(seed)
    for name in ("k_new", "v_new"):
        x = t[name][0]
        mag = torch.exp2(torch.randint(-24, 6, x.shape, generator=g, device="cuda").float())
        x.copy_((torch.randn(x.shape, generator=g, device="cuda") * mag).to(torch.bfloat16))
        x.view(-1)[:64] = 0.0
        x.view(-1)[64:128] = -0.0
    slots = step.slot_mapping.copy()
    slots[::5] = -1
    tc = to_cpu(t)
    pa.write_kv(t["k_new"][0], t["v_new"][0], t["k_cache"][0], t["v_cache"][0],
                torch.from_numpy(slots).cuda(), k_scale=wl.FP8_K_SCALE, v_scale=wl.FP8_V_SCALE)
    import oracle.e4m3 as e4m3
    kn = e4m3.quantize_bf16(to_store(tc["k_new"][0]), wl.FP8_K_SCALE)
    vn = e4m3.quantize_bf16(to_store(tc["v_new"][0]), wl.FP8_V_SCALE)
    kc, vc = opa.write_kv(to_store(tc["k_cache"][0]), to_store(tc["v_cache"][0]), kn, vn, slots,
                          step.geom.block_size)
    assert np.array_equal(to_store(t["k_cache"][0]), kc)
    assert np.array_equal(to_store(t["v_cache"][0]), vc)
    # the inputs really reached saturation and subnormal codes
    assert np.any((kn & 0x7F) == 0x7E) and np.any(((kn & 0x7F) > 0) & ((kn & 0x7F) < 8))


def test_write_kv_flags_out_of_range_slot():
    step = wl.tiny_f32(0)
    t = wl.make_tensors(step, 5, "cuda")
    before = _bytes(t["k_cache"][0]).copy()
    slots = np.array([step.num_blocks * 16 + 3, -1, 5, -1], dtype=np.int64)
    st = pa.new_status()
    pa.write_kv(t["k_new"][0], t["v_new"][0], t["k_cache"][0], t["v_cache"][0],
                torch.from_numpy(slots).cuda(), status=st)
    assert pa.read_status(st) == pa.FLAGS["SLOT_RANGE"]
    after = _bytes(t["k_cache"][0]).reshape(step.num_blocks * 16, -1)
    want = before.reshape(step.num_blocks * 16, -1).copy()
    want[5] = _bytes(t["k_new"][0]).reshape(4, -1)[2]
    assert np.array_equal(after, want)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _check_step(step, seed, rows=None, poison=True, layers=1, mode="batch", label=None):
    """Run the step through the C ABI (invariance ``mode``) and compare with the oracle.

    The oracle sees a compact copy of the lanes that own the checked rows
    (all rows when ``rows`` is None): their blocks, before the step's write.
    Every checked element must meet the fixed bar and its derived rounding
    bound (gpu_harness.check_parity).
    """
    t = wl.make_tensors(step, seed, "cuda", layers=layers, poison=poison)
    lane_of = step.row_lane()
    lanes = range(step.B) if rows is None else sorted(set(int(lane_of[r]) for r in rows))
    label = label or f"{step.geom} {mode} seed {seed}"
    worst = 0.0
    for layer in range(layers):
        sub, sub_t, sub_rows, blk = compact_lanes(step, t, lanes, layer)
        out, flags = run_attention(step, t, layer=layer, mode=mode)
        assert flags == 0, flags
        want = rows if rows is not None else list(range(step.T))
        pos = {int(r): i for i, r in enumerate(sub_rows)}
        idx = [pos[int(r)] for r in want]
        ref, kc, vc, terms = oracle_attention(sub, sub_t, rows=idx, terms=True)
        # the write inside the call is bit-exact on every block the lanes use
        assert np.array_equal(_bytes(t["k_cache"][layer].index_select(0, blk)), kc.view(np.uint8))
        assert np.array_equal(_bytes(t["v_cache"][layer].index_select(0, blk)), vc.view(np.uint8))
        got = out[torch.tensor(want, dtype=torch.long, device=out.device)]
        st = check_parity(got, ref[idx], rows_of(terms, idx), sub.row_positions()[idx],
                          step.geom, f"{label} layer {layer}")
        worst = max(worst, st["max_abs"])
    return worst


@pytest.mark.parametrize("sample", range(5))
def test_tiny_f32(sample):
    _check_step(wl.tiny_f32(sample), 1000 * 1 + sample)


@pytest.mark.parametrize("sample", range(2))
def test_decode_batch_bf16(sample):
    """Decode-only bf16 step, all 64 lanes (lognormal ctx, median 2048)."""
    _check_step(wl.decode_batch(sample), 2000 + sample)


def _ragged(geom, q_lens, ctx, seed, pool_extra=1.3):
    rng = np.random.default_rng(seed)
    used = sum(-(-c // geom.block_size) for c in ctx)
    return wl.build_step(geom, q_lens, ctx, int(used * pool_extra) + 2, rng)


@pytest.mark.parametrize("mode", ["batch", "row"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "fp8"])
@pytest.mark.parametrize("D,bs", [(64, 16), (128, 32)])
def test_ragged_edges(dtype, D, bs, mode):
    """ctx = 1, ctx on and off split / chunk / block edges, empty lanes, prefill chunks."""
    geom = wl.Geometry(8, 2, D, bs, dtype)
    # 65536 / 65537 keys: 512- and 1024-key splits
    ctx = [1, 15, 16, 17, 511, 512, 513, 1024, 1500, 2049, 7, 40, 600, 12000, 65536, 65537]
    q = [1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 0, 9, 23, 1, 1, 1]
    step = _ragged(geom, q, ctx, 7)
    _check_step(step, 77, mode=mode)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("H,Hkv", [(16, 1), (40, 8), (64, 4), (4, 4)])
def test_gqa_groups_bf16(H, Hkv, dtype):
    """Group sizes 16, 5, 16 and 1 (two n tiles, padded tile, MHA)."""
    geom = wl.Geometry(H, Hkv, 128, 16, dtype)
    step = _ragged(geom, [1, 1, 1, 3], [700, 33, 1025, 80], 11)
    _check_step(step, 91)


@pytest.mark.parametrize("mode", ["batch", "row"])
@pytest.mark.parametrize("D,bs", [(128, 16), (64, 32), (128, 32)])
def test_prefill_chunk_edges_bf16(D, bs, mode):
    """Prefill chunks on and off 128-row / 128-key tile edges, chunks starting
    at key 0, a 2-row chunk, next to decode rows (tensor-core prefill in
    batch mode, the split path in row mode)."""
    geom = wl.Geometry(16, 2, D, bs, "bf16")
    q = [128, 129, 300, 2, 257, 1, 64, 1]
    ctx = [128, 300, 1000, 2, 384, 700, 64 + 191, 5]
    step = _ragged(geom, q, ctx, 21)
    _check_step(step, 211, mode=mode)


@pytest.mark.parametrize("sample", range(2))
def test_decode_batch_e4m3(sample):
    """Decode-only step over e4m3 caches, all 64 lanes."""
    _check_step(wl.decode_batch(sample, dtype="fp8"), 2100 + sample)


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 32)])
def test_prefill_chunks_e4m3(D, bs):
    """Prefill chunks over e4m3 caches take the split path, row by row."""
    geom = wl.Geometry(16, 2, D, bs, "fp8")
    q = [128, 129, 300, 2, 257, 1, 64, 1]
    ctx = [128, 300, 1000, 2, 384, 700, 64 + 191, 5]
    _check_step(_ragged(geom, q, ctx, 23), 213)


def _long_tail_rows(step, n_short=10):
    """Every long row (16k-40k keys) of the long-tail step and a seeded
    sample of the short ones."""
    longs = [int(x) for x in np.nonzero(step.ctx_lens >= 16384)[0]]
    shorts = np.nonzero(step.ctx_lens < 16384)[0]
    rng = np.random.default_rng(55)
    return sorted(longs + [int(x) for x in rng.choice(shorts, n_short, replace=False)])


def test_long_tail_e4m3_sampled():
    """Long-context heavy tail over e4m3 caches (one layer): every long row
    and a sample of short ones, unreferenced cache bytes poisoned."""
    free, _ = torch.cuda.mem_get_info()
    step = wl.long_tail(0, pool_bytes_per_layer=min(15e9, 0.3 * free), dtype="fp8")
    rows = _long_tail_rows(step)
    assert sum(step.ctx_lens[r] >= 16384 for r in rows) == 26
    _check_step(step, 5100, rows=rows, poison=True, label="long_tail e4m3 (26 long + 10 short)")


def test_mixed_small_full():
    """Mixed bf16 step, small enough for the oracle on every row."""
    geom = wl.Geometry(40, 8, 128, 16, "bf16")
    rng = np.random.default_rng(3)
    ctx = [int(x) for x in rng.integers(16, 3000, size=10)] + [600, 130]
    q = [1] * 10 + [64, 40]
    step = wl.build_step(geom, q, ctx, sum(-(-c // 16) for c in ctx) + 40, rng)
    _check_step(step, 3100)


@pytest.mark.parametrize("mode", ["batch", "row"])
def test_mixed_step_sampled(mode):
    """Mixed bf16 step at full size (8 x 512 chunks + 120 decodes); sampled rows."""
    step = wl.mixed_step(0)
    cu = step.cu_seqlens_q
    rows = list(range(0, 120, 7))
    for b in range(120, step.B):
        rows += [int(cu[b]), int(cu[b]) + 255, int(cu[b + 1]) - 1]
    _check_step(step, 3000, rows=rows, mode=mode)


def test_long_tail_sampled():
    """Long-context heavy tail at full size (one layer of the 4): every long
    row and a sample of short ones, unreferenced cache bytes poisoned."""
    free, _ = torch.cuda.mem_get_info()
    pool = min(15e9, 0.3 * free)
    step = wl.long_tail(0, pool_bytes_per_layer=pool)
    rows = _long_tail_rows(step)
    assert sum(step.ctx_lens[r] >= 16384 for r in rows) == 26
    _check_step(step, 5000, rows=rows, poison=True, label="long_tail bf16 (26 long + 10 short)")


def test_empty_step_is_noop():
    geom = wl.Geometry(4, 2, 64, 16, "bf16")
    step = _ragged(geom, [0, 0], [5, 9], 1)
    t = wl.make_tensors(step, 1, "cuda")
    dev = device_step(step)
    out = torch.empty(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    pa.attention(t["q"][0], t["k_cache"][0], t["v_cache"][0], dev["block_tables"],
                 dev["cu_seqlens_q"], dev["ctx_lens"], out, max_q_len=0, max_ctx_len=9,
                 scale=0.125, workspace=workspace_for(step))
    torch.cuda.synchronize()


def test_device_flags_bad_lane_and_block():
    """Out-of-range ctx and block ids are reported in the status word, no fault."""
    geom = wl.Geometry(4, 2, 64, 16, "bf16")
    step = _ragged(geom, [1, 1, 1], [20, 40, 9], 2)
    t = wl.make_tensors(step, 2, "cuda")
    dev = device_step(step)
    dev["ctx_lens"][0] = 16 * step.max_blocks_per_seq + 1  # beyond its table row
    dev["block_tables"][1, 1] = step.num_blocks + 5       # block id out of range
    st = pa.new_status()
    out, flags = run_attention(step, t, dev=dev, status=st, write=False)
    assert flags & pa.FLAGS["CTX_RANGE"]
    assert flags & pa.FLAGS["BLOCK_RANGE"]
    # the untouched lane is still right
    ref, _, _, terms = oracle_attention(step, to_cpu(t), write=False, rows=[2], terms=True)
    check_parity(out[2:3], ref[2:3], rows_of(terms, [2]), step.row_positions()[[2]], geom,
                 "flagged step, untouched lane")


def test_workspace_too_small_is_flagged():
    step = wl.decode_batch(0, lanes=8)
    t = wl.make_tensors(step, 4, "cuda")
    small = torch.empty(40000, dtype=torch.uint8, device="cuda")  # room for 2 splits
    out, flags = run_attention(step, t, workspace=small)
    assert flags & pa.FLAGS["WORKSPACE"]


def test_repeat_runs_bitwise_equal():
    step = wl.decode_batch(1, lanes=16)
    t = wl.make_tensors(step, 9, "cuda")
    a, _ = run_attention(step, t)
    b, _ = run_attention(step, t)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
