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

// The next item for the calling warp: a warp that finishes early takes more
// items, so all warps end within about one item of each other (items go out
// in list order, largest first). The counter only hands out indices: an
// item's arithmetic and where its result goes depend on the item alone,
// never on which warp runs it or when.
__device__ __forceinline__ long long take_item(const StepParams& p, int lane) {
  unsigned long long v = 0;
  if (lane == 0) v = atomicAdd(item_counter(p.plan, kCounterSplit), 1ull);
  return (long long)__shfl_sync(0xffffffffu, v, 0);
}

// Items a warp's producer has taken and its consumer has not finished: the
// producer runs at most kStages chunks ahead, so at most kStages items beyond
// the consumer's current one; slot k & (kItemSlots - 1) holds the warp's k-th.
constexpr int kItemSlots = 4;

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
