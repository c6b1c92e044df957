// Split-KV decode partials, bf16 caches (the decode path of the paged-attention
// kernel contract in "P3: native paged-KV continuous-batching sampler", Design,
// paged.py: fixed KV split per context length, no atomics).
//
// Work item = (row, split, kv head); splits follow split_len (512 keys for
// rows up to 65,536 keys, longer for longer rows). Warps take items from a
// counter in list order (largest first), so a warp that finishes early takes
// more; the counter only decides who computes an item -- no partial result
// is ever accumulated atomically. One warp owns an item: it streams the
// split's keys in 16-key chunks through a private 3-stage ring of swizzled
// shared-memory tiles filled by TMA (one 64-element box per half row), and
// computes, for the g = H / Hkv query heads that read this kv head,
//   t_j = log2(e) * scale * <q_h, k_j>    (tensor cores, fp32 accumulate)
//   m   = max_j t_j,  p_j = 2^(t_j - m) rounded to bf16,  l = sum_j p_j
//   acc = sum_j p_j v_j                   (tensor cores, fp32 accumulate)
// with the usual running rescale when m grows, keys in ascending order.
// The products are arranged so the kv head's keys are the M side of the mma:
// S^T = K Q^T (M = 16 keys, N = 8 heads, K = 16 dims) and O^T = V^T P^T
// (M = 16 dims, N = 8 heads, K = 16 keys), so a GQA group of up to 8 heads
// fills one N tile. P^T moves from the accumulator layout of the first
// product to the operand layout of the second with movmatrix.
//
// A row whose keys fit one split writes its normalised output directly; the
// others leave (m, l, acc) for the fixed-order combine. Every item's
// arithmetic depends only on its own row's q and keys: which warp runs it and
// what else is in the step do not enter.
//
// The work is written as the code of one CTA of kW warps (decode_bf16_warps)
// so that it runs both as its own kernel (4 warps per CTA, 2 CTAs per SM) and
// as the decode role of the mixed-step kernel (8 warps per CTA).
#pragma once

#include "pa_split_bf16_row.cuh"
#include "pa_split_items.cuh"

namespace pa {

constexpr int kDecStages = 3;  // ring depth per warp

template <int D>
struct DecTile {
  static constexpr int kHalves = D / 64;              // 128-byte swizzled boxes per row
  static constexpr int kHalfBytes = kChunk * 128;     // one box: 16 keys x 64 elements
  static constexpr int kBytes = kChunk * D * 2;       // one K (or V) chunk
  static constexpr int kStageBytes = 2 * kBytes;      // K + V
  static constexpr int kWarpBytes = kDecStages * kStageBytes;
  // dynamic shared memory of a CTA of w such warps (+ alignment slack)
  static constexpr int smem_bytes(int w) { return w * kWarpBytes + 1024; }
};

// The decode split work of one CTA of kW independent warps: warp w of the
// CTA streams its items through ring w of dsmem (kW * DecTile<D>::kWarpBytes
// bytes after 1024-byte alignment).
template <int D, int NT, bool kOwner, int kW>
__device__ __forceinline__ void decode_bf16_warps(const StepParams& p, const CUtensorMap* tmK,
                                                  const CUtensorMap* tmV, uint8_t* dsmem) {
  using TL = DecTile<D>;
  constexpr int kStages = kDecStages;
  constexpr int KS = D / 16;  // 16-wide steps along D
  __shared__ __align__(8) uint64_t bars[kW][kStages];
  __shared__ long long s_items[kW][kItemSlots];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t wbase = base + warp * TL::kWarpBytes;
  uint32_t bar[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) bar[s] = smem_u32(&bars[warp][s]);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(bar[s], 1);
    fence_mbar_init();
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
  }
  __syncwarp();

  const long long n_items = (long long)p.plan.header[0] * p.Hkv;
  const int nfull = p.plan.header[1];
  static_assert(kStages < kItemSlots, "item slots");
  long long* const wq = s_items[warp];

  // ---- producer cursor: runs up to kStages chunks ahead of the consumer ----
  long long p_k = 0;
  long long p_item = take_item(p, lane);
  if (lane == 0) wq[0] = p_item;
  int p_chunk = 0, p_w0 = 0;
  Item pi;
  int p_blk = 0;
  if (p_item < n_items) {
    pi = load_item(p, p_item, nfull);
    p_blk = load_blocks(p, pi, 0, lane);
  }
  uint32_t issued = 0;
  auto produce = [&]() {
    if (p_item >= n_items) return;
    const int stage = issued % kStages;
    const int off = p_chunk * kChunk;  // key offset inside the split
    if (off / p.bs - p_w0 >= 32) {     // next window of block ids
      p_w0 += 32;
      p_blk = load_blocks(p, pi, p_w0, lane);
    }
    int blk = __shfl_sync(0xffffffffu, p_blk, off / p.bs - p_w0);
    // (test hook: no copy for the first chunk of item skip_item, so its
    // consumer's bounded wait runs out; -1 on every ordinary step)
    if (lane == 0 && !(p_chunk == 0 && p_item == p.skip_item)) {
      if (blk < 0 || blk >= p.NB) {
        raise_flag(p.status, PA_FLAG_BLOCK_RANGE);
        blk = 0;
      }
      const int tok = blk * p.bs + (pi.t0 + off) % p.bs;
      const uint32_t ks = wbase + stage * TL::kStageBytes;
      const uint32_t vs = ks + TL::kBytes;
      mbar_expect_tx(bar[stage], TL::kStageBytes);
      // keys are read once: their L2 lines go first, so the split partials
      // (stored evict-last) are still in L2 when the combine reads them
      const uint64_t pol = l2_evict_first();
#pragma unroll
      for (int h = 0; h < TL::kHalves; ++h) {
        tma_load_3d_hint(ks + h * TL::kHalfBytes, tmK, h * 64, pi.kvh, tok, bar[stage], pol);
        tma_load_3d_hint(vs + h * TL::kHalfBytes, tmV, h * 64, pi.kvh, tok, bar[stage], pol);
      }
    }
    ++issued;
    if (++p_chunk == pi.nchunks) {
      p_chunk = 0;
      p_w0 = 0;
      p_item = take_item(p, lane);
      if (lane == 0) wq[++p_k & (kItemSlots - 1)] = p_item;
      if (p_item < n_items) {
        pi = load_item(p, p_item, nfull);
        p_blk = load_blocks(p, pi, 0, lane);
      }
    }
  };
#pragma unroll 1
  for (int s = 0; s < kStages; ++s) produce();

  uint32_t consumed = 0;

#pragma unroll 1
  for (long long c_k = 0;; ++c_k) {
    __syncwarp();
    const long long c_item = wq[c_k & (kItemSlots - 1)];
    if (c_item >= n_items) break;
    const Item it = load_item(p, c_item, nfull);

    RowAcc<D, NT> ra;
    ra.init(p, it.row, it.kvh, gid, tig);

#pragma unroll 1
    for (int ch = 0; ch < it.nchunks; ++ch) {
      const int stage = consumed % kStages;
      const uint32_t parity = (consumed / kStages) & 1u;
      // every lane waits (so every lane sees the landed bytes); the outcome is
      // made warp-uniform before anyone acts on it
      const bool landed = __all_sync(0xffffffffu, mbar_wait_bounded(bar[stage], parity, p.wait_cycles));
      if (!landed) {
        if (lane == 0) raise_flag(p.status, PA_FLAG_TIMEOUT);
        // let copies already in flight land before the warp leaves
        for (uint32_t c = consumed + 1; c < issued; ++c)
          mbar_wait_bounded(bar[c % kStages], (c / kStages) & 1u, p.wait_cycles);
        return;
      }
      const uint32_t ks = wbase + stage * TL::kStageBytes;
      const uint32_t vs = ks + TL::kBytes;
      const int nvalid = min(kChunk, it.len - ch * kChunk);
      if (nvalid < kChunk) {
        // keys past the end: zero their V rows so 0 * (stale bytes) cannot
        // turn into NaN inside the second product
        const int nz = (kChunk - nvalid) * TL::kHalves * 8;
        for (int i = lane; i < nz; i += 32) {
          const int c16 = i & 7, rest = i >> 3;
          const int half = rest % TL::kHalves, tok = nvalid + rest / TL::kHalves;
          const uint32_t a = vs + half * TL::kHalfBytes + tok * 128 + c16 * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

      // S^T = K Q^T : 16 keys x 8 heads per n tile
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      {
        const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(bf16_tile_addr(ks, tok, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_bf16_16816(s[nt], a0, a1, a2, a3, ra.qf[nt][kk][0], ra.qf[nt][kk][1]);
        }
      }

      // online softmax over this chunk; this thread holds keys gid and gid + 8
      // for heads 2 * tig and 2 * tig + 1 of each n tile
      uint32_t pbt[NT][2];
      ra.softmax(s, nvalid, gid, p.scale_log2, pbt);

      // O^T += V^T P^T : 16 dims x 8 heads per (m tile, n tile)
      {
        const int tok = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(bf16_tile_addr(vs, tok, mt * 2 + ((lane >> 3) & 1)), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_bf16_16816(ra.o[mt][nt], a0, a1, a2, a3, pbt[nt][0], pbt[nt][1]);
        }
      }
      __syncwarp();  // every lane is done reading this stage
      ++consumed;
      produce();
    }

    // ---- finish the item ----
    ra.finish(p, it.row, it.kvh, it.single && !kOwner,
              kOwner ? (long long)p.plan.row_info[it.row].x + it.t0 / split_len(it.keys)
                     : (long long)it.pair,
              gid, tig);
  }
}

}  // namespace pa
