"""Pins of the CPU oracle to facts outside itself.

Each ``check_*`` returns None when the oracle agrees with the pinned fact and a
string describing the disagreement otherwise; ``test_oracle_pins.py`` asserts
every check passes and ``test_oracle_mutants.py`` plants plausible mistakes in
the oracle and asserts that some check catches each one.

What pins what:
  * single key            -> out = V_0 exactly (closed form; GQA map)
  * zero query            -> out = mean of the visible V rows (closed form, via numpy.mean)
  * position code         -> V_i = i and q = 0 give out = p / 2 (causal extent, gather)
  * constant V per head   -> out_h = c_{h // g} (GQA map)
  * one-hot keys          -> out picks the V row whose key matches q (operand roles)
  * brute force           -> paged oracle == scipy softmax on the unpaged sequence
  * block permutation     -> relabelling physical blocks changes no bit
  * weights sum           -> softmax weights sum to 1 within 1e-15
  * write bytes           -> write == a flat-index scatter, other bytes untouched
  * kv bytes golden       -> the memory-accounting values the P3 page prints
"""
import json
import math
import os

import numpy as np
import scipy.special
import torch

import oracle.paged_attention as pa
from helpers import as_f64, to_store

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _paged_from_sequences(seqs_k, seqs_v, block_size, num_blocks, rng):
    """Scatter contiguous per-sequence [L, Hkv, D] arrays into a random pool.

    Written independently of the oracle: a flat [NB*bs] view and explicit
    position arithmetic. Unreferenced pool entries hold NaN.
    """
    Hkv, D = seqs_k[0].shape[1:]
    dt = seqs_k[0].dtype
    fill = np.nan if dt == np.float32 else 0x7FC0  # a bf16 NaN bit pattern
    kc = np.full((num_blocks * block_size, Hkv, D), fill, dtype=dt)
    vc = np.full_like(kc, fill)
    perm = list(rng.permutation(num_blocks))
    tables = []
    for K, V in zip(seqs_k, seqs_v):
        nblk = -(-K.shape[0] // block_size)
        blocks = [int(perm.pop()) for _ in range(nblk)]
        tables.append(blocks)
        for p in range(K.shape[0]):
            flat = blocks[p // block_size] * block_size + (p % block_size)
            kc[flat] = K[p]
            vc[flat] = V[p]
    width = max(len(t) for t in tables)
    bt = np.full((len(tables), width), -1, dtype=np.int64)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    shape = (num_blocks, block_size, Hkv, D)
    return kc.reshape(shape), vc.reshape(shape), bt


def _run(q, kc, vc, bt, q_lens, ctx, scale, bs, dtype="f32"):
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int64)
    out, _, _ = pa.attention(q, kc, vc, bt, cu, ctx, scale, dtype, bs)
    return out


def _f32(a):
    return np.asarray(a, dtype=np.float32)


def check_single_key():
    rng = np.random.default_rng(11)
    H, Hkv, D, bs = 4, 2, 8, 4
    K = [_f32(rng.standard_normal((1, Hkv, D)))]
    V = [_f32(rng.standard_normal((1, Hkv, D)))]
    kc, vc, bt = _paged_from_sequences(K, V, bs, 6, rng)
    q = _f32(rng.standard_normal((1, H, D)))
    out = _run(q, kc, vc, bt, [1], [1], 0.3, bs)
    for h in range(H):
        want = V[0][0, h // (H // Hkv)].astype(np.float64)
        if not np.array_equal(out[0, h], want):
            return f"single key: head {h} != V0 of its kv head"
    return None


def check_zero_query_mean():
    rng = np.random.default_rng(12)
    H, Hkv, D, bs = 6, 3, 8, 4
    lens = [13, 7]
    q_lens = [5, 1]
    K = [_f32(rng.standard_normal((L, Hkv, D))) for L in lens]
    V = [_f32(rng.standard_normal((L, Hkv, D))) for L in lens]
    kc, vc, bt = _paged_from_sequences(K, V, bs, 12, rng)
    q = np.zeros((sum(q_lens), H, D), dtype=np.float32)
    out = _run(q, kc, vc, bt, q_lens, lens, 0.5, bs)
    r = 0
    for b, (L, ql) in enumerate(zip(lens, q_lens)):
        for j in range(ql):
            p = L - ql + j
            for h in range(H):
                want = np.mean(V[b][:p + 1, h // 2].astype(np.float64), axis=0)
                if np.max(np.abs(out[r, h] - want)) > 1e-12:
                    return f"zero query: lane {b} row {j} head {h} is not the mean of V[0..{p}]"
            r += 1
    return None


def check_position_code():
    rng = np.random.default_rng(13)
    H, Hkv, D, bs = 2, 1, 4, 4
    lens = [11, 6, 1]
    q_lens = [4, 1, 1]
    K = [_f32(rng.standard_normal((L, Hkv, D))) for L in lens]
    V = [np.broadcast_to(np.arange(L, dtype=np.float32)[:, None, None], (L, Hkv, D)).copy()
         for L in lens]
    kc, vc, bt = _paged_from_sequences(K, V, bs, 9, rng)
    q = np.zeros((sum(q_lens), H, D), dtype=np.float32)
    out = _run(q, kc, vc, bt, q_lens, lens, 1.0, bs)
    r = 0
    for L, ql in zip(lens, q_lens):
        for j in range(ql):
            p = L - ql + j
            if np.max(np.abs(out[r] - p / 2.0)) > 1e-12:
                return f"position code: row at position {p} gave {out[r, 0, 0]}, want {p / 2}"
            r += 1
    return None


def check_constant_v_per_head():
    rng = np.random.default_rng(14)
    H, Hkv, D, bs = 8, 4, 8, 4
    L = 10
    K = [_f32(rng.standard_normal((L, Hkv, D)))]
    c = np.array([1.5, -2.0, 3.25, 0.5], dtype=np.float32)
    V = [np.broadcast_to(c[None, :, None], (L, Hkv, D)).copy()]
    kc, vc, bt = _paged_from_sequences(K, V, bs, 5, rng)
    q = _f32(rng.standard_normal((1, H, D)))
    out = _run(q, kc, vc, bt, [1], [L], 0.7, bs)
    for h in range(H):
        if np.max(np.abs(out[0, h] - c[h // 2])) > 1e-12:
            return f"constant V: head {h} gave {out[0, h, 0]}, want {c[h // 2]}"
    return None


def check_one_hot():
    """Key i = 30 * e_i; the query aims at key j, so out ~ V_j (weight error < e^-29)."""
    rng = np.random.default_rng(15)
    H, Hkv, D, bs = 2, 2, 8, 4
    L = 7
    K = np.zeros((L, Hkv, D), dtype=np.float32)
    for i in range(L):
        K[i, :, i] = 30.0
    V = _f32(rng.standard_normal((L, Hkv, D)))
    kc, vc, bt = _paged_from_sequences([K], [V], bs, 4, rng)
    for j in range(L):
        q = np.zeros((1, H, D), dtype=np.float32)
        q[0, :, j] = 1.0
        out = _run(q, kc, vc, bt, [1], [L], 1.0, bs)
        for h in range(H):
            if np.max(np.abs(out[0, h] - V[j, h])) > 1e-9:
                return f"one-hot: query aimed at key {j} (head {h}) did not return V_{j}"
    return None


def _brute_force_case(dtype, seed):
    rng = np.random.default_rng(seed)
    H, Hkv, D, bs = 6, 2, 16, 4
    lens = [1, 5, 9, 14, 4]
    q_lens = [1, 1, 6, 3, 0]
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(seed)
    Kt = [torch.randn(L, Hkv, D, generator=g).to(tdt) for L in lens]
    Vt = [torch.randn(L, Hkv, D, generator=g).to(tdt) for L in lens]
    qt = torch.randn(sum(q_lens), H, D, generator=g).to(tdt)
    kc, vc, bt = _paged_from_sequences([to_store(x) for x in Kt],
                                       [to_store(x) for x in Vt], bs, 16, rng)
    scale = 0.37
    out = _run(to_store(qt), kc, vc, bt, q_lens, lens, scale, bs, dtype)
    # reference: contiguous sequences, torch's own widening, scipy softmax
    qf = as_f64(qt)
    s32 = float(np.float32(scale))
    r = 0
    worst = 0.0
    for b, (L, ql) in enumerate(zip(lens, q_lens)):
        Kf, Vf = as_f64(Kt[b]), as_f64(Vt[b])
        for j in range(ql):
            p = L - ql + j
            for h in range(H):
                kv = h * Hkv // H
                logits = s32 * np.einsum("ld,d->l", Kf[:p + 1, kv], qf[r, h])
                w = scipy.special.softmax(logits)
                want = np.einsum("l,ld->d", w, Vf[:p + 1, kv])
                worst = max(worst, float(np.max(np.abs(out[r, h] - want))))
            r += 1
    return worst


def check_brute_force():
    for dtype in ("f32", "bf16"):
        for seed in (21, 22):
            worst = _brute_force_case(dtype, seed)
            if not worst <= 1e-12:
                return f"brute force ({dtype}, seed {seed}): max |diff| {worst}"
    return None


def check_block_permutation():
    rng = np.random.default_rng(31)
    H, Hkv, D, bs, NB = 4, 2, 8, 4, 20
    lens = [9, 14, 3]
    q_lens = [1, 4, 1]
    K = [_f32(rng.standard_normal((L, Hkv, D))) for L in lens]
    V = [_f32(rng.standard_normal((L, Hkv, D))) for L in lens]
    kc, vc, bt = _paged_from_sequences(K, V, bs, NB, rng)
    q = _f32(rng.standard_normal((sum(q_lens), H, D)))
    base = _run(q, kc, vc, bt, q_lens, lens, 0.4, bs)
    perm = rng.permutation(NB)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    moved = _run(q, kc2, vc2, bt2, q_lens, lens, 0.4, bs)
    if not np.array_equal(base, moved):
        return "relabelling physical blocks changed the output"
    return None


def check_weights_sum():
    rng = np.random.default_rng(41)
    for L in (1, 2, 17, 300):
        K = rng.standard_normal((L, 2, 16))
        q = rng.standard_normal((4, 16))
        for h in range(4):
            w = pa.row_weights(q, K, L - 1, 0.25 * 3, h)
            if w.shape != (L,) or abs(np.sum(w) - 1.0) > 1e-15 or np.any(w < 0):
                return f"weights of a {L}-key row do not form a distribution"
    return None


def check_write_bytes():
    rng = np.random.default_rng(51)
    NB, bs, Hkv, D = 6, 4, 2, 8
    for dt in (np.float32, np.uint16):
        kc = rng.integers(0, 60000, size=(NB, bs, Hkv, D)).astype(dt)
        vc = rng.integers(0, 60000, size=(NB, bs, Hkv, D)).astype(dt)
        T = 7
        kn = rng.integers(0, 60000, size=(T, Hkv, D)).astype(dt)
        vn = rng.integers(0, 60000, size=(T, Hkv, D)).astype(dt)
        slots = rng.choice(NB * bs, size=T, replace=False).astype(np.int64)
        slots[2] = -1
        k2, v2 = pa.write_kv(kc, vc, kn, vn, slots, bs)
        want_k = kc.reshape(NB * bs, Hkv, D).copy()
        want_v = vc.reshape(NB * bs, Hkv, D).copy()
        for t, s in enumerate(slots):
            if s >= 0:
                want_k[s] = kn[t]
                want_v[s] = vn[t]
        if not (np.array_equal(k2.reshape(NB * bs, Hkv, D).view(np.uint8),
                               want_k.view(np.uint8)) and
                np.array_equal(v2.reshape(NB * bs, Hkv, D).view(np.uint8),
                               want_v.view(np.uint8))):
            return "write: cache bytes differ from a flat-index scatter"
        if not np.array_equal(kc, kc):  # inputs untouched
            return "write modified its input"
    return None


def check_kv_bytes_golden():
    with open(os.path.join(GOLDEN, "kv_bytes_per_token.json")) as f:
        data = json.load(f)
    for c in data["cases"]:
        got = pa.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"],
                                    c["elem_bytes"], c["tp_degree"])
        if got != c["bytes"]:
            return f"kv_bytes_per_token({c['what']}) = {got}, page prints {c['bytes']}"
    return None


ALL_CHECKS = [check_single_key, check_zero_query_mean, check_position_code,
              check_constant_v_per_head, check_one_hot, check_brute_force,
              check_block_permutation, check_weights_sum, check_write_bytes,
              check_kv_bytes_golden]


def failures():
    out = []
    for c in ALL_CHECKS:
        try:
            msg = c()
        except Exception as e:  # a crash is a failed pin too
            msg = f"{c.__name__} raised {type(e).__name__}: {e}"
        if msg is not None:
            out.append(msg)
    return out
