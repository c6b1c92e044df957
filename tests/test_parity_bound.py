"""The parity bound on the CPU: it admits what the kernel's rounding can do and
rejects plausible kernel mistakes on a long row.

On one 40,960-key decode row of the long-tail geometry (H 64, Hkv 8, D 128,
block 32, bf16, N(0, 1) data):
  * the oracle's output rounded to bf16 passes, and so does a float32 model of
    the split path's rounding points (p rounded to bf16, fp32 sums in 512-key
    splits, the ordered fp32 fold, one bf16 rounding);
  * the oracle's output with one 512-key split dropped, with one block id
    pointing at another block, or with V scaled by 1.01, each fails.
"""
import math

import numpy as np
import torch

import oracle.paged_attention as opa
import parity_bound as pb
import split_rule
from helpers import to_store
from invariant_paged_kv_gb300 import workload as wl

GEOM = wl.Geometry(64, 8, 128, 32, "bf16")


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _row(n, seed):
    rng = np.random.default_rng(seed)
    used = -(-n // GEOM.block_size)
    step = wl.build_step(GEOM, [1], [n], used + 8, rng)
    t = wl.make_tensors(step, seed, "cpu")
    q, kc, vc = to_store(t["q"][0]), to_store(t["k_cache"][0]), to_store(t["v_cache"][0])
    scale = opa.default_scale(GEOM.D)
    return step, q, kc, vc, scale


def _oracle(step, q, kc, vc, scale, block_tables=None):
    bt = step.block_tables if block_tables is None else block_tables
    out, _, _, terms = opa.attention(q, kc, vc, bt, step.cu_seqlens_q, step.ctx_lens, scale,
                                     "bf16", GEOM.block_size, terms=True)
    return out, terms


def _split_path_model(step, q, kc, vc, scale):
    """float32 model of the split path: scores, p = 2^(t - m) rounded to bf16,
    l from the rounded p, acc = p V per split; splits folded in order."""
    n = int(step.ctx_lens[0])
    K = opa.widen(opa.gather(kc, step.block_tables[0], n, GEOM.block_size), "bf16")
    V = opa.widen(opa.gather(vc, step.block_tables[0], n, GEOM.block_size), "bf16")
    qf = opa.widen(q[0], "bf16").astype(np.float32)
    c2 = np.float32(scale * math.log2(math.e))
    S = split_rule.split_length(n)
    g = GEOM.H // GEOM.Hkv
    out = np.empty((GEOM.H, GEOM.D))
    for h in range(GEOM.H):
        kv = h // g
        M = L = A = None
        for s0 in range(0, n, S):
            k = K[s0:s0 + S, kv].astype(np.float32)
            v = V[s0:s0 + S, kv].astype(np.float32)
            t = (k @ qf[h]) * c2
            m = np.float32(t.max())
            p = _bf16(np.exp2(t - m)).astype(np.float32)
            l = np.float32(p.sum(dtype=np.float32))
            acc = (p @ v).astype(np.float32)
            if M is None:
                M, L, A = m, l, acc
            else:
                Mn = np.float32(max(M, m))
                ea, eb = np.float32(np.exp2(M - Mn)), np.float32(np.exp2(m - Mn))
                L = np.float32(L * ea + l * eb)
                A = (A * ea + acc * eb).astype(np.float32)
                M = Mn
        out[h] = _bf16(A / L)
    return out


def _stats(got, ref, terms, step, scale):
    return pb.compare(got[None], ref[None], {k: v[:1] for k, v in terms.items()},
                      step.row_positions()[:1], GEOM.D, scale, "bf16")


def test_bound_admits_rounding_and_rejects_mistakes_on_a_long_row():
    n = 40960
    step, q, kc, vc, scale = _row(n, 71)
    ref, terms = _oracle(step, q, kc, vc, scale)
    ref, terms = ref[0], {k: v[:1] for k, v in terms.items()}
    terms = {k: np.concatenate([v]) for k, v in terms.items()}
    ok = {"oracle rounded to bf16": _bf16(ref), "fp32 split-path model": _split_path_model(
        step, q, kc, vc, scale)}
    for name, got in ok.items():
        s = _stats(got, ref, terms, step, scale)
        print(f"{name}: {s}")
        assert pb.passes(s), (name, s)
        assert s["max_abs"] <= 2e-2

    # one 512-key split dropped (split 40 of 80): fold of the others
    K = opa.widen(opa.gather(kc, step.block_tables[0], n, GEOM.block_size), "bf16")
    V = opa.widen(opa.gather(vc, step.block_tables[0], n, GEOM.block_size), "bf16")
    qf = opa.widen(q[0], "bf16")
    dropped = np.empty_like(ref)
    for h in range(GEOM.H):
        parts = [opa.row_partial(qf, K, V, s0, min(s0 + 512, n), scale, h)
                 for s0 in range(0, n, 512) if s0 != 40 * 512]
        dropped[h] = opa.fold_partials(parts)
    # one block id pointing at a spare block
    bt = step.block_tables.copy()
    bt[0, 500] = step.num_blocks - 1
    swapped = _oracle(step, q, kc, vc, scale, block_tables=bt)[0][0]
    bad = {"split dropped": _bf16(dropped), "block swapped": _bf16(swapped),
           "V scaled by 1.01": _bf16(ref * 1.01)}
    for name, got in bad.items():
        s = _stats(got, ref, terms, step, scale)
        print(f"{name}: {s}")
        assert s["max_abs"] <= 2e-2, "the fixed tolerance alone would pass it"
        assert not pb.passes(s), (name, s)


def test_bound_admits_short_rows():
    for n, seed in ((1, 72), (3, 73), (700, 74), (4096, 75)):
        step, q, kc, vc, scale = _row(n, seed)
        ref, terms = _oracle(step, q, kc, vc, scale)
        got = _split_path_model(step, q, kc, vc, scale)
        s = _stats(got, ref[0], terms, step, scale)
        print(f"n={n}: {s}")
        assert pb.passes(s), (n, s)
