"""Seeded synthetic flat ragged steps and the host-side block allocator.

This module only builds inputs: lane lengths, block tables, slot maps and
N(0, 1) tensors. It holds none of the attention arithmetic, so both the CUDA
path and the CPU oracle can be fed from it.

Layout follows the paged KV cache of "P3: native paged-KV continuous-batching
sampler", section Design (paged.py): per layer K and V are each
``[num_blocks, block_size, Hkv, D]``; a lane's block table row lists the
physical blocks holding its positions 0, bs, 2*bs, ...; the flat step stacks
the query rows of every lane in ``cu_seqlens_q`` order (engine.py: decodes
first, prefill chunks after, all in one ragged step).

Conventions used throughout the library:
  * ``ctx_lens[b]`` counts every key lane ``b`` attends after this step's
    write, its own new rows included; row ``j`` of a lane with ``q_len`` rows
    sits at absolute position ``ctx - q_len + j``.
  * block table rows are padded with -1 past ``ceil(ctx / bs)``.
  * ``slot_mapping[t] = block * bs + offset`` for the position of new row t.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

DTYPES = ("f32", "bf16", "fp8")

# Per-tensor scales of the synthetic e4m3 caches ("fp8" geometry): N(0, 1)
# data over millions of elements reaches |x| ~ 5.6, and 5.6 / 448 = 0.0125;
# V gets a slightly different scale so a K/V mix-up cannot go unseen.
FP8_K_SCALE = 0.0125
FP8_V_SCALE = 0.011


class AllocatorError(RuntimeError):
    pass


class BlockAllocator:
    """LIFO free list with reference counts.

    Mirrors the allocator described in "P3: native paged-KV continuous-batching
    sampler", section Design (paged.py: BlockAllocator): freeing a block whose
    count is already zero raises (a double free would hand one block to two
    sequences), and ``check_consistent`` proves that free + referenced equals
    the pool with no duplicates.  ``order`` seeds the initial free list so that
    block tables come out as a seeded permutation of the pool.
    """

    def __init__(self, num_blocks: int, order: Optional[Sequence[int]] = None):
        if num_blocks <= 0:
            raise AllocatorError("pool must hold at least one block")
        self.num_blocks = int(num_blocks)
        if order is None:
            order = range(num_blocks)
        order = [int(b) for b in order]
        if sorted(order) != list(range(num_blocks)):
            raise AllocatorError("initial order must be a permutation of the pool")
        # pop() takes from the end: reverse so the first entry of `order` goes out first
        self._free: List[int] = list(reversed(order))
        self._ref = np.zeros(num_blocks, dtype=np.int64)

    @property
    def num_free(self) -> int:
        return len(self._free)

    def refcount(self, block: int) -> int:
        return int(self._ref[block])

    def alloc(self, n: int) -> List[int]:
        """All-or-nothing: either n blocks come out or none do."""
        if n < 0:
            raise AllocatorError("negative allocation")
        if n > len(self._free):
            raise AllocatorError(f"out of blocks: want {n}, have {len(self._free)}")
        out = [self._free.pop() for _ in range(n)]
        for b in out:
            assert self._ref[b] == 0
            self._ref[b] = 1
        return out

    def incref(self, blocks: Sequence[int]) -> None:
        for b in blocks:
            if self._ref[b] <= 0:
                raise AllocatorError(f"incref of free block {b}")
            self._ref[b] += 1

    def free(self, blocks: Sequence[int]) -> None:
        for b in blocks:
            if self._ref[b] <= 0:
                raise AllocatorError(f"free of block {b} with refcount 0")
            self._ref[b] -= 1
            if self._ref[b] == 0:
                self._free.append(int(b))

    def check_consistent(self) -> None:
        free = self._free
        if len(set(free)) != len(free):
            raise AllocatorError("duplicate block on the free list")
        for b in free:
            if self._ref[b] != 0:
                raise AllocatorError(f"free block {b} has refcount {self._ref[b]}")
        referenced = int(np.count_nonzero(self._ref > 0))
        if referenced + len(free) != self.num_blocks:
            raise AllocatorError(
                f"books do not balance: free {len(free)} + referenced {referenced}"
                f" != total {self.num_blocks}")
        if np.any(self._ref < 0):
            raise AllocatorError("negative refcount")


@dataclasses.dataclass
class Geometry:
    H: int
    Hkv: int
    D: int
    block_size: int
    dtype: str  # "f32" | "bf16" | "fp8" (bf16 q / new rows, e4m3 code caches)

    def __post_init__(self):
        if self.dtype not in DTYPES:
            raise ValueError(f"dtype must be one of {DTYPES}")
        if self.H % self.Hkv:
            raise ValueError("H must be a multiple of Hkv")

    @property
    def elem_bytes(self) -> int:
        """Bytes of one cache element."""
        return {"f32": 4, "bf16": 2, "fp8": 1}[self.dtype]

    @property
    def q_bytes(self) -> int:
        """Bytes of one q / out / new-row element."""
        return 4 if self.dtype == "f32" else 2

    @property
    def group(self) -> int:
        return self.H // self.Hkv

    @property
    def kv_row_bytes(self) -> int:
        """Bytes of one token's K (or V) row across all kv heads."""
        return self.Hkv * self.D * self.elem_bytes


@dataclasses.dataclass
class Step:
    """Descriptor of one flat ragged step (host arrays, untimed)."""
    geom: Geometry
    num_blocks: int
    q_lens: np.ndarray        # int32 [B]
    ctx_lens: np.ndarray      # int32 [B]
    block_tables: np.ndarray  # int32 [B, max_blocks], -1 padded
    slot_mapping: np.ndarray  # int64 [T]
    shared_blocks: np.ndarray = dataclasses.field(
        default_factory=lambda: np.zeros(0, np.int64))  # blocks with refcount > 1

    @property
    def B(self) -> int:
        return int(self.q_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.q_lens.sum())

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        cu = np.zeros(self.B + 1, dtype=np.int32)
        np.cumsum(self.q_lens, out=cu[1:])
        return cu

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.B else 0

    @property
    def max_ctx_len(self) -> int:
        return int(self.ctx_lens.max()) if self.B else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def row_positions(self) -> np.ndarray:
        """Absolute position of every flat query row (int64 [T])."""
        pos = np.empty(self.T, dtype=np.int64)
        cu = self.cu_seqlens_q
        for b in range(self.B):
            q, c = int(self.q_lens[b]), int(self.ctx_lens[b])
            pos[cu[b]:cu[b + 1]] = np.arange(c - q, c)
        return pos

    def row_lane(self) -> np.ndarray:
        return np.repeat(np.arange(self.B, dtype=np.int64), self.q_lens)


def _table_and_slots(lane_blocks, q_lens, ctx_lens, bs):
    B = len(lane_blocks)
    max_blocks = max([len(x) for x in lane_blocks] + [1])
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    slots = []
    for b, blocks in enumerate(lane_blocks):
        bt[b, :len(blocks)] = blocks
        c, q = int(ctx_lens[b]), int(q_lens[b])
        for p in range(c - q, c):
            slots.append(blocks[p // bs] * bs + p % bs)
    return bt, np.asarray(slots, dtype=np.int64)


def build_step(geom: Geometry, q_lens, ctx_lens, num_blocks: int, rng,
               share=None) -> Step:
    """Allocate every lane's blocks from a seeded permutation of the pool.

    ``share`` optionally maps a lane to (leader lane, n_full_blocks): the lane
    adopts the leader's first n FULL blocks (refcount > 1) and allocates the
    rest privately, as prefix sharing does in the P3 engine design.
    """
    q_lens = np.asarray(q_lens, dtype=np.int32)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
    if np.any(q_lens < 0) or np.any(q_lens > ctx_lens):
        raise ValueError("need 0 <= q_len <= ctx_len")
    bs = geom.block_size
    alloc = BlockAllocator(num_blocks, order=rng.permutation(num_blocks))
    share = share or {}
    lane_blocks: List[List[int]] = [None] * len(q_lens)  # type: ignore
    order = sorted(range(len(q_lens)), key=lambda b: (b in share, b))
    for b in order:
        need = -(-int(ctx_lens[b]) // bs)
        if b in share:
            leader, nfull = share[b]
            prefix = lane_blocks[leader][:nfull]
            alloc.incref(prefix)
            lane_blocks[b] = list(prefix) + alloc.alloc(need - nfull)
        else:
            lane_blocks[b] = alloc.alloc(need)
    alloc.check_consistent()
    bt, slots = _table_and_slots(lane_blocks, q_lens, ctx_lens, bs)
    shared = np.nonzero(alloc._ref > 1)[0].astype(np.int64)
    return Step(geom, num_blocks, q_lens, ctx_lens, bt, slots, shared)


def _pool_for(ctx_lens, bs, factor=1.1):
    used = int(sum(-(-int(c) // bs) for c in ctx_lens))
    return max(1, int(math.ceil(used * factor)))


# ---------------------------------------------------------------------------
# The five workloads. Seeds: seed = 1000 * config + sample.
# ---------------------------------------------------------------------------

def tiny_f32(sample: int = 0) -> Step:
    """Tiny fp32 case: H4/Hkv2/D64/bs16, 64-block pool, ctx {3, 9, 17, 40}."""
    rng = np.random.default_rng(1000 * 1 + sample)
    geom = Geometry(4, 2, 64, 16, "f32")
    ctx = [3, 9, 17, 40]
    return build_step(geom, [1] * 4, ctx, 64, rng)


def decode_batch(sample: int = 0, lanes: int = 64, dtype: str = "bf16") -> Step:
    """Decode-only bf16: H32/Hkv8/D128/bs16, lognormal ctx (median 2048, sigma 1)."""
    rng = np.random.default_rng(1000 * 2 + sample)
    geom = Geometry(32, 8, 128, 16, dtype)
    ctx = np.clip(np.rint(2048.0 * np.exp(rng.standard_normal(lanes))), 16, 16384)
    ctx = ctx.astype(np.int32)
    return build_step(geom, [1] * lanes, ctx, _pool_for(ctx, 16), rng)


def mixed_step(sample: int = 0, chunks: int = 8, chunk_len: int = 512,
               decodes: int = 120) -> Step:
    """Mixed bf16 step: H40/Hkv8/D128/bs16; decode lanes first, then chunks.

    Chunks of ``chunk_len`` new rows start at prior offsets U{0..4096};
    decode ctx lognormal (median 3000, sigma 1) clipped to [16, 16384].
    """
    rng = np.random.default_rng(1000 * 3 + sample)
    geom = Geometry(40, 8, 128, 16, "bf16")
    dctx = np.clip(np.rint(3000.0 * np.exp(rng.standard_normal(decodes))), 16, 16384)
    offs = rng.integers(0, 4096, size=chunks, endpoint=True)
    q = [1] * decodes + [chunk_len] * chunks
    ctx = list(dctx.astype(np.int64)) + list(offs + chunk_len)
    return build_step(geom, q, ctx, _pool_for(ctx, 16), rng)


def prefill_chunks(sample: int = 0) -> Step:
    """The prefill chunks of ``mixed_step`` alone (the same seeded offsets,
    8 chunks of 512 rows, H40/Hkv8/D128/bs16 bf16): a step whose every row
    takes the tensor-core prefill path, for measuring that path on its own."""
    rng = np.random.default_rng(1000 * 3 + sample)
    geom = Geometry(40, 8, 128, 16, "bf16")
    rng.standard_normal(120)  # the mixed step's decode lengths, drawn first
    offs = rng.integers(0, 4096, size=8, endpoint=True)
    ctx = list(offs + 512)
    return build_step(geom, [512] * 8, ctx, _pool_for(ctx, 16), rng)


INVARIANCE_TARGET_CTX = 4096
INVARIANCE_SIBLINGS = 7


def invariance_step(t: int, sample: int = 0) -> (Step, int):
    """One composition of the batch-invariance sweep (H32/Hkv8/D128/bs16).

    The target is a decode row at ctx 4096. ``t`` counts lanes in the step
    (target + t-1 neighbours). Up to 7 neighbours are siblings of the target
    (GRPO samples of one prompt): they share its first 255 FULL blocks
    (refcount > 1, read-only) and own their last block. The other neighbours
    are decode rows (p = 0.75, ctx U{1..16384}) or 256-row prefill chunks
    (p = 0.25, ctx U{256..16384}). The target lane's index is random. Returns
    (step, index of the target's flat row).
    """
    if t < 1:
        raise ValueError("t >= 1")
    rng = np.random.default_rng(1000 * 4 + 97 * t + sample)
    geom = Geometry(32, 8, 128, 16, "bf16")
    bs = 16
    n_sib = min(INVARIANCE_SIBLINGS, t - 1)
    lanes = []  # (q_len, ctx, kind)
    for _ in range(n_sib):
        lanes.append((1, INVARIANCE_TARGET_CTX, "sib"))
    for _ in range(t - 1 - n_sib):
        if rng.random() < 0.75:
            lanes.append((1, int(rng.integers(1, 16384, endpoint=True)), "dec"))
        else:
            lanes.append((256, int(rng.integers(256, 16384, endpoint=True)), "pre"))
    pos = int(rng.integers(0, t))
    lanes.insert(pos, (1, INVARIANCE_TARGET_CTX, "target"))
    q = [x[0] for x in lanes]
    ctx = [x[1] for x in lanes]
    nfull = (INVARIANCE_TARGET_CTX - 1) // bs
    share = {b: (pos, nfull) for b, x in enumerate(lanes) if x[2] == "sib"}
    # the target's physical block ids differ between compositions; the caller
    # writes the same bytes into them, so only the addresses change
    step = build_step(geom, q, ctx, _pool_for(ctx, bs, 1.1) + 8, rng, share=share)
    cu = step.cu_seqlens_q
    return step, int(cu[pos])


def long_tail(sample: int = 0, lanes: int = 256, long_frac: float = 0.1,
              pool_bytes_per_layer: float = 15e9, dtype: str = "bf16") -> Step:
    """Long-context heavy tail bf16: H64/Hkv8/D128/bs32, 256 decode lanes.

    90% of lanes U{1024..4096}, 10% U{16384..40960} (230 + 26 at 256 lanes),
    order shuffled by the seed. The pool fills ``pool_bytes_per_layer`` of K+V.
    """
    rng = np.random.default_rng(1000 * 5 + sample)
    geom = Geometry(64, 8, 128, 32, dtype)
    n_long = int(round(lanes * long_frac))
    short = rng.integers(1024, 4096, size=lanes - n_long, endpoint=True)
    longs = rng.integers(16384, 40960, size=n_long, endpoint=True)
    ctx = np.concatenate([short, longs])
    rng.shuffle(ctx)
    per_block = geom.block_size * geom.kv_row_bytes * 2
    pool = max(_pool_for(ctx, 32, 1.0), int(pool_bytes_per_layer // per_block))
    return build_step(geom, [1] * lanes, ctx, pool, rng)


# ---------------------------------------------------------------------------
# Tensors
# ---------------------------------------------------------------------------

def make_tensors(step: Step, seed: int, device="cpu", layers: int = 1,
                 poison: bool = False):
    """N(0, 1) q / caches / new rows in the step's dtype from one torch.Generator.

    Returns a dict with q [layers][T,H,D], k_cache / v_cache
    [layers][NB,bs,Hkv,D], k_new / v_new [layers][T,Hkv,D]; for the "fp8"
    geometry q and new rows are bf16 and the caches uint8 e4m3 codes (scales
    FP8_K_SCALE / FP8_V_SCALE). With ``poison`` every cache position that is
    not one of the step's keys (tails of last blocks and unreferenced blocks)
    holds NaN (the NaN code for e4m3), so any stray read shows.
    """
    import torch

    g = step.geom
    dt = torch.float32 if g.dtype == "f32" else torch.bfloat16
    gen = torch.Generator(device=device).manual_seed(int(seed))
    out = {"q": [], "k_cache": [], "v_cache": [], "k_new": [], "v_new": []}
    T, NB = step.T, step.num_blocks

    def cache(scale):
        x = torch.randn(NB, g.block_size, g.Hkv, g.D, generator=gen, device=device, dtype=dt)
        if g.dtype != "fp8":
            return x
        # e4m3 codes drawn with torch's own cast (a random-code generator
        # here, not the library's quantiser): N(0, 1) / scale, clamped to
        # the finite range
        return (x.float() / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)

    for _ in range(layers):
        out["q"].append(torch.randn(T, g.H, g.D, generator=gen, device=device, dtype=dt))
        out["k_cache"].append(cache(FP8_K_SCALE))
        out["v_cache"].append(cache(FP8_V_SCALE))
        for name in ("k_new", "v_new"):
            out[name].append(torch.randn(T, g.Hkv, g.D, generator=gen,
                                         device=device, dtype=dt))
    if poison:
        mask = key_mask(step)
        m = torch.from_numpy(~mask).to(device)
        for name in ("k_cache", "v_cache"):
            for c in out[name]:
                c.view(NB * g.block_size, g.Hkv, g.D)[m] = 0x7F if g.dtype == "fp8" else float("nan")
    return out


def key_mask(step: Step) -> np.ndarray:
    """bool [NB*bs]: True where a cache position holds one of the step's keys."""
    bs = step.geom.block_size
    mask = np.zeros(step.num_blocks * bs, dtype=bool)
    for b in range(step.B):
        c = int(step.ctx_lens[b])
        nblk = -(-c // bs)
        for i in range(nblk):
            blk = int(step.block_tables[b, i])
            n = min(bs, c - i * bs)
            mask[blk * bs: blk * bs + n] = True
    return mask


def sub_step(step: Step, lanes):
    """Descriptor of the step restricted to `lanes`, blocks renumbered 0.. in
    order of first use. Returns (sub step, original ids of its blocks,
    original flat rows of its rows).

    Renumbering physical blocks changes no attention result; it lets a host
    check or a CPU baseline work on a compact copy of a few lanes of a large
    pool.
    """
    bs = step.geom.block_size
    lanes = sorted(set(int(b) for b in lanes))
    seen = {}
    blocks = []
    for b in lanes:
        n = -(-int(step.ctx_lens[b]) // bs)
        for x in step.block_tables[b, :n]:
            x = int(x)
            if x not in seen:
                seen[x] = len(blocks)
                blocks.append(x)
    width = max([1] + [-(-int(step.ctx_lens[b]) // bs) for b in lanes])
    bt = np.full((len(lanes), width), -1, dtype=np.int32)
    cu = step.cu_seqlens_q
    rows, slots = [], []
    for i, b in enumerate(lanes):
        n = -(-int(step.ctx_lens[b]) // bs)
        bt[i, :n] = [seen[int(x)] for x in step.block_tables[b, :n]]
        rows += list(range(int(cu[b]), int(cu[b + 1])))
        c, q = int(step.ctx_lens[b]), int(step.q_lens[b])
        slots += [int(bt[i, p // bs]) * bs + p % bs for p in range(c - q, c)]
    sub = Step(step.geom, max(1, len(blocks)), step.q_lens[lanes].copy(),
               step.ctx_lens[lanes].copy(), bt, np.asarray(slots, dtype=np.int64))
    return sub, np.asarray(blocks, dtype=np.int64), np.asarray(rows, dtype=np.int64)


def kv_bytes(step: Step) -> int:
    """K+V bytes of every key every row of the step attends, counted once per lane."""
    return int(step.ctx_lens.astype(np.int64).sum()) * 2 * step.geom.kv_row_bytes


def algorithmic_bytes(step: Step, write: bool = True) -> dict:
    """Bytes the step must move at minimum, per part.

    decode (split path): every key's K and V once per lane, q in, out, and the
    4-byte block-table entries read; partial results of the split path are
    overhead and are not counted. write: each new K and V row read once and
    written once, plus its 8-byte slot.
    """
    g = step.geom
    e = g.q_bytes
    bs = g.block_size
    qo = 2 * step.T * g.H * g.D * e
    bt = 4 * int(sum(-(-int(c) // bs) for c in step.ctx_lens))
    out = {"kv": kv_bytes(step), "q_out": qo, "block_table": bt}
    new_rows = 2 * step.T * g.Hkv * g.D * (g.q_bytes + g.elem_bytes)  # K and V: read + write
    out["write"] = (new_rows + 8 * step.T) if write else 0
    out["decode_kernel"] = out["kv"] + step.T * g.H * g.D * e + bt
    out["total"] = out["kv"] + qo + bt + out["write"]
    return out


def prefill_flops(step: Step) -> int:
    """Dense-contraction flops of the prefill lanes (q_len >= 2): per row and
    head, 2 D flops for q.k and 2 D for p.v over each attended key; a lane of q
    rows after `off` earlier keys attends q * off + q (q + 1) / 2 keys per head."""
    g = step.geom
    tot = 0
    for q, c in zip(step.q_lens.tolist(), step.ctx_lens.tolist()):
        if q >= 2:
            off = c - q
            tot += g.H * 4 * g.D * (q * off + q * (q + 1) // 2)
    return int(tot)


def decode_rows_kv_bytes(step: Step) -> int:
    """K+V bytes the decode lanes (q_len == 1) attend."""
    m = step.q_lens == 1
    return int(step.ctx_lens[m].astype(np.int64).sum()) * 2 * step.geom.kv_row_bytes
