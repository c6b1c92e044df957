"""CPU oracle for batch-invariant paged-KV attention over one flat ragged step.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import or call this module. It shares
no code with the CUDA library and imports nothing from it.

It is the plain definition, written for a reader to check by eye:

* write  -- byte copy of every new K/V row into ``cache[slot // bs, slot % bs]``
  ("P3: native paged-KV continuous-batching sampler", section Design, paged.py:
  PagedKVCache copy-free append that scatters into (block, offset));
* gather -- contiguous ``[L, Hkv, D]`` keys of one sequence, read block by
  block through its block-table row (same section: ``gather()`` returns the
  sequence's keys in one contiguous layout whatever else is in the batch);
* attend -- for every query row, softmax attention over exactly its own keys
  (same section: TorchPagedAttention 'row' mode, one attention per query row;
  the step first writes the new K/V, then returns ``[T, H, D]``), causal by
  absolute position inside a prefill chunk, query head h reading kv head
  ``h // (H / Hkv)`` (blocked GQA map, "Tensor parallelism" Design, GQA).

Everything is widened exactly to float64 before any arithmetic. bf16 data is
carried as raw uint16 bit patterns (bfloat16 is the upper half of an IEEE
binary32, so widening is a 16-bit shift); fp32 data as float32. With the
'fp8' dtype the queries and new rows are bf16 and the caches hold e4m3 codes
under one scale per tensor: the write quantises the new rows and the gather
reads codes back as decode(code) * scale (oracle/e4m3.py).

``attend_row_terms`` adds, for the tests' rounding-error bound, plain sums over
a row's softmax weights (weighted magnitudes of V and of the scores' terms);
they are pinned like the rest and do not enter the output.

Readings where the pages leave a step open (listed with their reasons in the
design notes of this repository):
  * ``ctx_lens`` counts the keys after this step's write, so a lane with
    ``q_len`` rows has its row j at position ``ctx - q_len + j``;
  * a negative slot means "no write" (padding);
  * ``scale`` is the caller's float32 value, widened.
"""
from __future__ import annotations

import math

import numpy as np

from . import e4m3


# ---------------------------------------------------------------------------
# element widening
# ---------------------------------------------------------------------------

def widen(x, dtype: str) -> np.ndarray:
    """Exact float64 values of stored elements ('f32': float32, 'bf16': uint16 bits)."""
    x = np.asarray(x)
    if dtype == "f32":
        if x.dtype != np.float32:
            raise TypeError("f32 data must be float32")
        return x.astype(np.float64)
    if dtype == "bf16":
        if x.dtype != np.uint16:
            raise TypeError("bf16 data must be carried as uint16 bit patterns")
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# ---------------------------------------------------------------------------
# memory accounting
# ---------------------------------------------------------------------------

def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int,
                       tp_degree: int = 1) -> int:
    """K and V bytes one token occupies across all layers on one rank.

    "P3: native paged-KV continuous-batching sampler", section Memory
    accounting: layers x 2 (K and V) x kv heads x head dim x element bytes;
    kv heads are split evenly over tensor-parallel ranks ("Tensor
    parallelism", Design: the cache is sharded by kv head).
    """
    if kv_heads % tp_degree:
        raise ValueError("tp degree must divide the kv heads")
    return layers * 2 * (kv_heads // tp_degree) * head_dim * elem_bytes


# ---------------------------------------------------------------------------
# write
# ---------------------------------------------------------------------------

def slot_location(slot: int, block_size: int):
    """(block, offset) that a flat slot number names."""
    return slot // block_size, slot % block_size


def write_kv(k_cache, v_cache, k_new, v_new, slot_mapping, block_size: int):
    """Return copies of the caches with every new row stored at its slot.

    Bytes move unchanged; rows whose slot is negative are skipped.
    Caches are ``[NB, bs, Hkv, D]``, new rows ``[T, Hkv, D]``.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        blk, off = slot_location(int(slot), block_size)
        k_out[blk, off] = k_new[t]
        v_out[blk, off] = v_new[t]
    return k_out, v_out


# ---------------------------------------------------------------------------
# gather
# ---------------------------------------------------------------------------

def gather(cache, table_row, ctx_len: int, block_size: int) -> np.ndarray:
    """Contiguous ``[ctx_len, Hkv, D]`` keys (or values) of one sequence."""
    rows = []
    for p in range(ctx_len):
        blk = int(table_row[p // block_size])
        rows.append(cache[blk, p % block_size])
    if not rows:
        return np.zeros((0,) + tuple(cache.shape[2:]), dtype=cache.dtype)
    return np.stack(rows)


# ---------------------------------------------------------------------------
# attend
# ---------------------------------------------------------------------------

def kv_head_of(h: int, H: int, Hkv: int) -> int:
    """Blocked GQA map: query heads [g*k, g*k + g) read kv head k, g = H / Hkv."""
    return h // (H // Hkv)


def visible_keys(position: int) -> int:
    """A row at absolute position p attends keys 0..p (causal)."""
    return position + 1


def softmax_weights(scores: np.ndarray) -> np.ndarray:
    """exp(s - max s) / sum exp(s - max s), in float64."""
    m = np.max(scores)
    e = np.exp(scores - m)
    return e / np.sum(e)


def attend_row(q_row, K, V, position: int, scale: float):
    """Output ``[H, D]`` (float64) of one query row.

    q_row ``[H, D]``, K and V ``[L, Hkv, D]``, all float64.
    """
    H, D = q_row.shape
    Hkv = K.shape[1]
    n = visible_keys(position)
    out = np.empty((H, D), dtype=np.float64)
    for h in range(H):
        kv = kv_head_of(h, H, Hkv)
        s = scale * (K[:n, kv, :] @ q_row[h])
        w = softmax_weights(s)
        out[h] = w @ V[:n, kv, :]
    return out


def row_weights(q_row, K, position: int, scale: float, h: int) -> np.ndarray:
    """Softmax weights of head h of one row (for invariant checks)."""
    H = q_row.shape[0]
    kv = kv_head_of(h, H, K.shape[1])
    n = visible_keys(position)
    return softmax_weights(scale * (K[:n, kv, :] @ q_row[h]))


def attend_row_terms(q_row, K, V, position: int, scale: float) -> dict:
    """Sums over one row's softmax weights that size a rounding-error bound
    for a computed version of ``attend_row`` (the weights are ``row_weights``;
    nothing here changes what attention computes).

    For head h, its kv head k, the row's weights w_i over its visible keys
    and c_i = sum_d |q[h, d]| |K[i, k, d]| (the size of key i's score before
    scaling), all float64:
        wv[h, d]   = sum_i w_i |V[i, k, d]|
        w2v2[h, d] = sum_i w_i^2 V[i, k, d]^2
        w2v[h, d]  = sum_i w_i^2 |V[i, k, d]|
        wcv[h, d]  = sum_i w_i c_i |V[i, k, d]|
        w2[h]      = sum_i w_i^2
        wc[h]      = sum_i w_i c_i
        cmax[h]    = max_i c_i
    """
    H, D = q_row.shape
    Hkv = K.shape[1]
    n = visible_keys(position)
    t = {name: np.empty((H, D)) for name in ("wv", "w2v2", "w2v", "wcv")}
    t.update({name: np.empty(H) for name in ("w2", "wc", "cmax")})
    for h in range(H):
        kv = kv_head_of(h, H, Hkv)
        w = row_weights(q_row, K, position, scale, h)
        v = V[:n, kv, :]
        c = np.abs(K[:n, kv, :]) @ np.abs(q_row[h])
        t["wv"][h] = w @ np.abs(v)
        t["w2v2"][h] = (w * w) @ (v * v)
        t["w2v"][h] = (w * w) @ np.abs(v)
        t["wcv"][h] = (w * c) @ np.abs(v)
        t["w2"][h] = np.sum(w * w)
        t["wc"][h] = np.sum(w * c)
        t["cmax"][h] = np.max(c)
    return t


def widen_kv(x, dtype: str, kv_scale: float) -> np.ndarray:
    """Exact float64 values of cache elements: e4m3 codes times their
    tensor's scale for 'fp8', ``widen`` otherwise."""
    if dtype == "fp8":
        return e4m3.dequantize(x, kv_scale)
    return widen(x, dtype)


def attention(q, k_cache, v_cache, block_tables, cu_seqlens_q, ctx_lens,
              scale: float, dtype: str, block_size: int,
              slot_mapping=None, k_new=None, v_new=None, rows=None,
              k_scale: float = 1.0, v_scale: float = 1.0, terms: bool = False):
    """Reference output of one flat ragged step, float64 ``[T, H, D]``.

    When new rows are given they are written first (the step writes, then
    attends); with dtype 'fp8' they are quantised under ``k_scale`` /
    ``v_scale`` on the way in. ``rows`` optionally restricts the work to a
    subset of flat rows (others are left NaN), for sampled checks of large
    steps. Returns (out, k_cache_after, v_cache_after), and with ``terms``
    a fourth item: ``attend_row_terms`` of every computed row, stacked into
    ``[T, H, D]`` / ``[T, H]`` arrays (NaN elsewhere).
    """
    if k_new is not None:
        if dtype == "fp8":
            k_new = e4m3.quantize_bf16(k_new, k_scale)
            v_new = e4m3.quantize_bf16(v_new, v_scale)
        k_cache, v_cache = write_kv(k_cache, v_cache, k_new, v_new,
                                    slot_mapping, block_size)
    q_dtype = "bf16" if dtype == "fp8" else dtype
    scale = float(np.float32(scale))
    T, H, D = q.shape
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    B = ctx.shape[0]
    want = None if rows is None else set(int(r) for r in rows)
    out = np.full((T, H, D), np.nan, dtype=np.float64)
    tt = None
    if terms:
        tt = {name: np.full((T, H, D), np.nan) for name in ("wv", "w2v2", "w2v", "wcv")}
        tt.update({name: np.full((T, H), np.nan) for name in ("w2", "wc", "cmax")})
    for b in range(B):
        q_len = int(cu[b + 1] - cu[b])
        if q_len == 0:
            continue
        lane_rows = [int(cu[b]) + j for j in range(q_len)]
        if want is not None and not want.intersection(lane_rows):
            continue
        K = widen_kv(gather(k_cache, block_tables[b], int(ctx[b]), block_size), dtype, k_scale)
        V = widen_kv(gather(v_cache, block_tables[b], int(ctx[b]), block_size), dtype, v_scale)
        for j, r in enumerate(lane_rows):
            if want is not None and r not in want:
                continue
            position = int(ctx[b]) - q_len + j
            out[r] = attend_row(widen(q[r], q_dtype), K, V, position, scale)
            if terms:
                for name, val in attend_row_terms(widen(q[r], q_dtype), K, V, position,
                                                  scale).items():
                    tt[name][r] = val
    if terms:
        return out, k_cache, v_cache, tt
    return out, k_cache, v_cache


# ---------------------------------------------------------------------------
# partials and their ordered fold (KV-parallel page owners)
# ---------------------------------------------------------------------------

def row_partial(q_row, K, V, lo: int, hi: int, scale: float, h: int):
    """Unnormalised softmax partial of head h over keys [lo, hi), float64:
    m = max s_i, l = sum exp(s_i - m), acc = sum exp(s_i - m) V_i."""
    H = q_row.shape[0]
    kv = kv_head_of(h, H, K.shape[1])
    s = scale * (K[lo:hi, kv, :] @ q_row[h])
    m = float(np.max(s))
    e = np.exp(s - m)
    return m, float(np.sum(e)), e @ V[lo:hi, kv, :]


def fold_partials(parts):
    """Ordered fold of partials (m_i, l_i, acc_i), i = 0, 1, ... in list
    order ("Numerics envelopes", The hierarchy: a reduction is data movement
    plus a fixed-order fold of ranks 0..W-1; Layout invariance of query
    context parallelism: combine_attention_partials merges the partials of
    KV-parallel page owners with that fold): M, L, A from the first; for each
    next M' = max(M, m), L = L e^(M - M') + l e^(m - M'), A likewise; the
    result is A / L."""
    M, L, A = parts[0][0], parts[0][1], np.array(parts[0][2], dtype=np.float64)
    for m, l, a in parts[1:]:
        Mn = max(M, m)
        ea, eb = math.exp(M - Mn), math.exp(m - Mn)
        L = L * ea + l * eb
        A = A * ea + np.asarray(a, dtype=np.float64) * eb
        M = Mn
    return A / L


def default_scale(D: int) -> float:
    """1/sqrt(D) rounded to float32, the scale the workloads use."""
    return float(np.float32(1.0 / math.sqrt(D)))
