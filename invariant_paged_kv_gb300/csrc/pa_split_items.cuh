// Work items of the split kernels: (row, split, kv head) triples drawn from
// the split plan, the order warps take them in, and the window of block ids
// an item reads. Shared by the bf16 and the e4m3 split kernels so both walk
// the plan the same way.
#pragma once

#include "pa_common.cuh"

namespace pa {

struct Item {
  int pair, kvh, row, lane, keys, t0, len, nchunks, single;
};

// k-th item of warp gw among nw warps: passes over the item list alternate
// direction (snake order), so with items sorted by size every warp gets a
// near-equal share of the work. Which warp runs an item never changes its
// arithmetic.
__device__ __forceinline__ long long item_at(long long k, long long gw, long long nw) {
  return k * nw + ((k & 1) ? (nw - 1 - gw) : gw);
}

__device__ __forceinline__ Item load_item(const StepParams& p, long long item, int nfull) {
  Item it;
  const int k = (int)(item / p.Hkv);
  it.kvh = (int)(item - (long long)k * p.Hkv);
  it.pair = pair_slot(p.plan, k, nfull);
  const int4 pr = p.plan.pairs[it.pair];
  it.row = pr.x;
  it.lane = pr.z;
  it.keys = pr.w;
  const int sl = split_len(it.keys);
  it.t0 = pr.y * sl;
  it.len = min(sl, it.keys - it.t0);
  it.nchunks = (it.len + kChunk - 1) / kChunk;
  it.single = it.keys <= sl;
  return it;
}

// Block ids w0 .. w0 + 31 of the item's range (relative to its first block):
// lane i holds entry w0 + i.
__device__ __forceinline__ int load_blocks(const StepParams& p, const Item& it, int w0, int lane) {
  const int nblk = (it.len + p.bs - 1) / p.bs;
  if (w0 + lane >= nblk) return 0;
  return p.block_tables[(size_t)it.lane * p.max_blocks + it.t0 / p.bs + w0 + lane];
}

}  // namespace pa
