"""Row invariance on the GPU: in the row-invariant mode a query row has the
same bits however its own lane's rows are cut into chunks (GPU).

"Numerics envelopes", Prefix hits resume at any token: a query row depends
only on the K/V rows it attends, so a prefix hit at any token, chunked
prefill and a cold run give the same bits; "P3: native paged-KV
continuous-batching sampler", Evidence, item 2: batch invariance holds under
chunk sizes 1, 2 and 64. One cached sequence of P tokens is cut into lanes
in several ways (one chunk, 64-row chunks, one decode row per token, random
cut points, the same cuts with unrelated lanes around them); every row's
output must be bitwise equal across the cuts, and equal to the default
mode's decode path (a row fed as a q_len = 1 lane).
"""
import numpy as np
import pytest
import torch

import oracle.paged_attention as opa
from gpu_harness import SCALES, check_parity, run_attention
from helpers import to_store
from invariant_paged_kv_gb300 import build, pa, workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    pa.load()


def _sequence(geom, P, seed, extra_blocks=7):
    """Cache of one P-token sequence (NaN everywhere else), its block list and
    one q row per position."""
    bs = geom.block_size
    nblk = -(-P // bs)
    NB = nblk + extra_blocks
    rng = np.random.default_rng(seed)
    blocks = rng.permutation(NB)[:nblk].astype(np.int32)
    dt = torch.float32 if geom.dtype == "f32" else torch.bfloat16
    g = torch.Generator(device="cuda").manual_seed(seed)
    shape = (NB, bs, geom.Hkv, geom.D)
    pos = np.arange(P)
    flat = torch.from_numpy(blocks[pos // bs].astype(np.int64) * bs + pos % bs).cuda()

    def cache(scale):
        x = torch.randn(P, geom.Hkv, geom.D, generator=g, device="cuda", dtype=dt)
        if geom.dtype == "fp8":  # e4m3 codes (NaN code elsewhere)
            c = torch.full(shape, 0x7F, device="cuda", dtype=torch.uint8)
            x = (x.float() / scale).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            c = torch.full(shape, float("nan"), device="cuda", dtype=dt)
        c.view(-1, geom.Hkv, geom.D)[flat] = x
        return c

    kc, vc = cache(wl.FP8_K_SCALE), cache(wl.FP8_V_SCALE)
    q = torch.randn(P, geom.H, geom.D, generator=g, device="cuda", dtype=dt)
    return NB, blocks, dict(k_cache=kc, v_cache=vc, q=q)


def _run_cuts(geom, NB, blocks, seq, cuts, mode, others=()):
    """Lanes (start, end) of the sequence -- lane attends keys 0..end-1 with
    rows start..end-1 -- plus unrelated `others` lanes (q_len, ctx) reading
    the same blocks; returns the output rows of the sequence's positions, in
    the order of `cuts`."""
    lanes = [(e - s, e, True) for s, e in cuts] + [(q, c, False) for q, c in others]
    order = np.random.default_rng(len(cuts) + 31 * len(others)).permutation(len(lanes)) \
        if others else np.arange(len(lanes))
    lanes = [lanes[i] for i in order]
    width = len(blocks)
    bt = np.tile(blocks, (len(lanes), 1)).astype(np.int32)
    q_lens = np.array([x[0] for x in lanes], np.int32)
    ctx = np.array([x[1] for x in lanes], np.int32)
    step = wl.Step(geom, NB, q_lens, ctx, bt.reshape(len(lanes), width),
                   np.zeros(int(q_lens.sum()), np.int64))
    rows_q = []
    seq_rows = {}
    r = 0
    for (q, c, mine) in lanes:
        for j in range(q):
            p = c - q + j
            rows_q.append(p)
            if mine:
                seq_rows[p] = r
            r += 1
    idx = torch.tensor(rows_q, dtype=torch.long, device="cuda")
    t = {"q": [seq["q"].index_select(0, idx).contiguous()], "k_cache": [seq["k_cache"]],
         "v_cache": [seq["v_cache"]]}
    out, flags = run_attention(step, t, write=False, mode=mode)
    assert flags == 0, flags
    want = [p for s, e in cuts for p in range(s, e)]
    return out[torch.tensor([seq_rows[p] for p in want], device="cuda")], want


def _bits(x):
    return x.contiguous().view(torch.int32 if x.dtype == torch.float32 else torch.int16).cpu()


def _random_cuts(lo, hi, n, seed):
    rng = np.random.default_rng(seed)
    pts = sorted(set(int(x) for x in rng.integers(lo + 1, hi, size=n)))
    edges = [lo] + pts + [hi]
    return [(a, b) for a, b in zip(edges[:-1], edges[1:])]


GEOMS = [wl.Geometry(32, 8, 128, 16, "bf16"), wl.Geometry(40, 8, 128, 16, "bf16"),
         wl.Geometry(8, 8, 64, 32, "bf16"), wl.Geometry(32, 2, 128, 16, "bf16"),
         wl.Geometry(16, 1, 64, 32, "bf16"), wl.Geometry(4, 2, 64, 16, "f32"),
         wl.Geometry(40, 8, 128, 16, "fp8"), wl.Geometry(16, 1, 64, 32, "fp8")]


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"H{g.H}kv{g.Hkv}D{g.D}bs{g.block_size}{g.dtype}")
def test_row_bits_independent_of_chunking(geom):
    P = 1300  # rows with 1, 2 and 3 splits
    NB, blocks, seq = _sequence(geom, P, 9001)
    ref, want = _run_cuts(geom, NB, blocks, seq, [(0, P)], "row")
    ref_bits = _bits(ref)
    decomps = {
        "chunks of 64": [(s, min(P, s + 64)) for s in range(0, P, 64)],
        "one row per lane": [(j, j + 1) for j in range(P)],
        "random cuts": _random_cuts(0, P, 9, 5),
        "random cuts among other lanes": _random_cuts(0, P, 4, 6),
    }
    for name, cuts in decomps.items():
        others = [(1, 900), (37, 800), (1, 5), (128, 1300)] if "other" in name else ()
        got, w = _run_cuts(geom, NB, blocks, seq, cuts, "row", others)
        assert w == want
        assert torch.equal(_bits(got), ref_bits), name
    # the default mode's decode path gives the same bits for q_len = 1 lanes
    dec, _ = _run_cuts(geom, NB, blocks, seq, [(j, j + 1) for j in range(P)], "batch")
    assert torch.equal(_bits(dec), ref_bits)
    # and the rows are right
    kc, vc = to_store(seq["k_cache"].cpu()), to_store(seq["v_cache"].cpu())
    rows = [0, 1, 511, 512, 513, 1023, 1024, 1299]
    bt = blocks[None, :].astype(np.int32)
    for p in rows:
        q1 = to_store(seq["q"][p:p + 1].cpu())
        o, _, _, terms = opa.attention(q1, kc, vc, bt, np.array([0, 1], np.int32),
                                       np.array([p + 1], np.int32), opa.default_scale(geom.D),
                                       geom.dtype, geom.block_size, terms=True, **SCALES)
        check_parity(ref[p:p + 1], o, terms, [p], geom, f"row mode {geom} position {p}")


def test_row_bits_across_split_length_change():
    """A chunk whose rows straddle 65536 keys: rows up to 65536 keys use
    512-key splits, later rows 1024-key splits, in the same lane."""
    geom = wl.Geometry(16, 4, 128, 32, "bf16")
    P = 65700
    NB, blocks, seq = _sequence(geom, P, 9100)
    lo = 65400
    ref, _ = _run_cuts(geom, NB, blocks, seq, [(lo, P)], "row")
    for cuts in ([(j, j + 1) for j in range(lo, P)], _random_cuts(lo, P, 5, 8)):
        got, _ = _run_cuts(geom, NB, blocks, seq, cuts, "row")
        assert torch.equal(_bits(got), _bits(ref))
    dec, _ = _run_cuts(geom, NB, blocks, seq, [(j, j + 1) for j in range(lo, P)], "batch")
    assert torch.equal(_bits(dec), _bits(ref))


def test_batch_mode_chunk_differs_only_within_tolerance():
    """The default mode's tensor-core prefill is not row invariant across
    paths, but it stays within the bf16 bar of the row-invariant result."""
    geom = wl.Geometry(32, 8, 128, 16, "bf16")
    P = 700
    NB, blocks, seq = _sequence(geom, P, 9200)
    row, _ = _run_cuts(geom, NB, blocks, seq, [(0, P)], "row")
    bat, _ = _run_cuts(geom, NB, blocks, seq, [(0, P)], "batch")
    diff = (row.float() - bat.float()).abs().max().item()
    assert diff <= 2e-2
