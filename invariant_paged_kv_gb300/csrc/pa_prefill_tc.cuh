// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05), bf16.
//
// A lane with q_len >= 2 is a causal prefill chunk ("P3: native paged-KV
// continuous-batching sampler", Design, engine.py: prefill chunks and decode
// tokens share one flat step; Evidence, mutant "prefill causal mask off by
// one"): its row j sits at position ctx - q_len + j and attends keys
// 0..position. Work item = (128-row q tile of one lane, a pair of query heads
// that read the same kv head). Per item, key tiles of 128 keys go in
// ascending order; for each head of the pair and each key tile:
//   S = Q K^T           tcgen05.mma, M = 128 rows, N = 128 keys, K = D, fp32 in TMEM
//   m, p, l             one thread per row: running max, p = 2^(t - m) rounded
//                       to bf16 and written back over S in TMEM, l += sum of
//                       the p (fp32, before rounding) -- all within the thread
//   O = O * alpha + P V tcgen05.mma with A = P read from TMEM, B = V (MN-major
//                       smem), O in TMEM
// and finally out = O * (1 / l). The running max moves only when a tile's max
// exceeds it by more than 8 (log2 units), so O is rescaled rarely. A row's
// arithmetic depends on its q row, its keys and the fixed 128-key tiling from
// key 0 -- never on other lanes. (N = 128 keys: a 128 x 128 x 16 product runs
// at the tensor core's full rate, where a 128 x 64 x 16 one reaches ~70%.)
//
// Warp roles (320 threads): warps 0-3 and 4-7 are two softmax groups (one per
// head of the pair; thread r of a group owns row r = TMEM lane r), warp 8
// issues the MMAs (one elected thread), warp 9 streams Q / K / V in by TMA (K /
// V through the block table, 16 keys per box) into 2-deep K and V rings shared
// by both heads. TMEM per head slot (256 of the 512 columns): S / P (128), O
// (128). Each head has one S / P buffer; the MMA warp serves the two heads in
// turn -- P V of tile t for a head, then (once that P is consumed) its S of
// tile t + 1 -- so one head's softmax runs while the tensor core works for the
// other. Every wait is bounded (timeout -> PA_FLAG_TIMEOUT). No parity wait
// ever meets a barrier more than one phase away from the awaited one, ahead
// or behind (the P V barriers alternate by tile parity for that reason).
//
// The work is written as the code of one CTA (prefill_tc_cta): it runs as the
// prefill role of the mixed-step kernel (pa_mixed.cu), which gives every CTA
// this role when a step has no decode rows.
#pragma once

#include "pa_tcgen05.cuh"

namespace pa {
namespace pftc {


constexpr int kRows = 128;  // query rows per item (M)
constexpr int kKeys = 128;  // keys per tile (N of S, K of PV)
constexpr int kStages = 2;  // depth of the K and V rings
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct PfLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kRows * 128;         // Q: 128 rows x 128 bytes
  static constexpr int kKHalfBytes = kKeys * 128;        // K / V: 128 keys x 128 bytes
  static constexpr int kQBytes = kHalves * kHalfBytes;   // one Q tile
  static constexpr int kKBytes = kHalves * kKHalfBytes;  // one K tile
  static constexpr int kVBytes = kHalves * kKHalfBytes;  // one V tile
  static constexpr int kQ = 0;                           // Q of head A, then head B
  static constexpr int kK0 = kQ + 2 * kQBytes;
  static constexpr int kV0 = kK0 + kStages * kKBytes;
  static constexpr int kEnd = kV0 + kStages * kVBytes;
  // + alignment slack; at least 116 KB so one CTA (and one 512-column TMEM
  // allocation) per SM
  static constexpr int kSmemBytes = (kEnd + 1024) > 118784 ? (kEnd + 1024) : 118784;
};

struct Bars {
  uint64_t kfull[kStages], kempty[kStages], vfull[kStages], vempty[kStages];
  uint64_t q, s[2], p[2], o[2][2];  // [head slot] ([tile parity] for o)
};

struct ItemInfo {
  int lane, tile, head0, has_b, cu0, q_len, ctx, nrows, p_first, nkt, kvh;
};

__device__ __forceinline__ ItemInfo item_info(const StepParams& p, int item, int g) {
  ItemInfo it;
  const int npair = (g + 1) / 2;
  const int per_tile = p.Hkv * npair;
  const int t = item / per_tile;
  const int rem = item - t * per_tile;
  it.kvh = rem / npair;
  const int j = rem - it.kvh * npair;
  it.head0 = it.kvh * g + 2 * j;
  it.has_b = (2 * j + 1) < g;
  const int4 e = p.plan.ptiles[t];
  it.lane = e.x;
  it.tile = e.y;
  it.cu0 = p.cu_seqlens[it.lane];
  it.q_len = p.cu_seqlens[it.lane + 1] - it.cu0;
  it.ctx = p.ctx_lens[it.lane];
  const int row0 = it.tile * kRows;
  it.nrows = min(kRows, it.q_len - row0);
  it.p_first = it.ctx - it.q_len + row0;
  const int p_last = it.p_first + it.nrows - 1;
  it.nkt = p_last / kKeys + 1;
  return it;
}

// Wait with the CTA-wide abort flag: returns false (and sets the flag) on timeout.
__device__ __forceinline__ bool wait_or_abort_1(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, int* status,
                                                long long limit) {
  if (*abort_flag) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      raise_flag(status, PA_FLAG_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Every lane of the warp waits; the verdict is made warp-uniform.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int* status,
                                              long long limit) {
  return __all_sync(0xffffffffu, wait_or_abort_1(bar, parity, abort_flag, status, limit));
}

// The work of one CTA of kThreads threads (see the roles above); dsmem
// holds PfLayout<D>::kSmemBytes bytes.
template <int D>
__device__ __forceinline__ void prefill_tc_cta(const StepParams& p, const CUtensorMap* tmQ,
                                               const CUtensorMap* tmK, const CUtensorMap* tmV,
                                               uint8_t* dsmem) {
  using L = PfLayout<D>;
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  // items are taken from the prefill item counter in list order (heaviest
  // tiles first): thread 0 takes item n + 1 during item n into slot
  // (n + 1) & 1, and the end-of-item barrier publishes it
  __shared__ long long s_item[2];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sQ = base + L::kQ, sK0 = base + L::kK0, sV0 = base + L::kV0;
  const uint32_t bq = smem_u32(&bars.q);
  uint32_t bkf[kStages], bke[kStages], bvf[kStages], bve[kStages];
#pragma unroll
  for (int i = 0; i < kStages; ++i) {
    bkf[i] = smem_u32(&bars.kfull[i]);
    bke[i] = smem_u32(&bars.kempty[i]);
    bvf[i] = smem_u32(&bars.vfull[i]);
    bve[i] = smem_u32(&bars.vempty[i]);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bkf[i], 1);
      mbar_init(bke[i], 1);
      mbar_init(bvf[i], 1);
      mbar_init(bve[i], 1);
    }
    mbar_init(bq, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&bars.s[h]), 1);
      mbar_init(smem_u32(&bars.p[h]), kRows);
      mbar_init(smem_u32(&bars.o[h][0]), 1);
      mbar_init(smem_u32(&bars.o[h][1]), 1);
    }
    s_abort = 0;
    s_item[0] = (long long)atomicAdd(item_counter(p.plan, kCounterPrefill), 1ull);
    fence_mbar_init();
  }
  if (warp == 9 && lane == 0) {
    prefetch_tensormap(tmQ);
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
  }
  if (warp == 8) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // head slot h: S / P at column 256 h, O at 256 h + 128
  auto tS = [&](int h) -> uint32_t { return tmem + 256 * h; };
  auto tO = [&](int h) -> uint32_t { return tmem + 256 * h + 128; };
  auto bS = [&](int h) -> uint32_t { return smem_u32(&bars.s[h]); };
  auto bP = [&](int h) -> uint32_t { return smem_u32(&bars.p[h]); };
  // P V of tile t completes on o[head][t & 1]
  auto bO = [&](int h, uint32_t t) -> uint32_t { return smem_u32(&bars.o[h][t & 1]); };

  const int g = p.H / p.Hkv;
  const int n_items = p.plan.header[2] * p.Hkv * ((g + 1) / 2);
  const float c2 = p.scale_log2;  // > 0 (validated on the host)
  // running use counters, identical in every role: items, K/V ring fills,
  // key tiles done by each head slot
  uint32_t n_item = 0, n_kv = 0, n_t[2] = {0, 0};

  for (;;) {
    const long long item = s_item[n_item & 1];
    if (item >= n_items) break;
    if (threadIdx.x == 0)
      s_item[(n_item + 1) & 1] = (long long)atomicAdd(item_counter(p.plan, kCounterPrefill), 1ull);
    const ItemInfo it = item_info(p, (int)item, g);
    const int nh = 1 + it.has_b;

    if (warp == 9) {
      // ------------------------------ producer ------------------------------
      // Q of this item's heads (the previous item's S products, which read
      // this buffer, all finished before the item boundary)
      if (lane == 0) {
        mbar_expect_tx(bq, nh * L::kQBytes);
        for (int hb = 0; hb < nh; ++hb)
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sQ + hb * L::kQBytes + h * L::kHalfBytes, tmQ, h * 64, it.head0 + hb,
                        it.cu0 + it.tile * kRows, bq);
      }
      for (int kt = 0; kt < it.nkt; ++kt) {
        const uint32_t f = n_kv + kt, st = f % kStages, use = f / kStages;
        const int key0 = kt * kKeys;
        const int nchunk = min(kKeys / kChunk, (it.ctx - key0 + kChunk - 1) / kChunk);
        int blk = 0;  // block id of chunk `lane` (lanes 0..7)
        if (lane < nchunk) {
          blk = p.block_tables[(size_t)it.lane * p.max_blocks + (key0 + lane * kChunk) / p.bs];
          if (blk < 0 || blk >= p.NB) {
            raise_flag(p.status, PA_FLAG_BLOCK_RANGE);
            blk = 0;
          }
        }
        const uint32_t bytes = (uint32_t)nchunk * L::kHalves * kChunk * 128;
        // lane c (< nchunk) copies chunk c: the boxes go out in parallel
        const int tok = blk * p.bs + (key0 + lane * kChunk) % p.bs;
        if (use >= 1 && !wait_or_abort(bke[st], (use - 1) & 1, &s_abort, p.status, p.wait_cycles)) break;
        if (lane == 0) mbar_expect_tx(bkf[st], bytes);
        __syncwarp();
        if (lane < nchunk) {
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sK0 + st * L::kKBytes + h * L::kKHalfBytes + lane * kChunk * 128, tmK,
                        h * 64, it.kvh, tok, bkf[st]);
        }
        if (use >= 1 && !wait_or_abort(bve[st], (use - 1) & 1, &s_abort, p.status, p.wait_cycles)) break;
        if (lane == 0) mbar_expect_tx(bvf[st], bytes);
        __syncwarp();
        if (lane < nchunk) {
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sV0 + st * L::kVBytes + h * L::kKHalfBytes + lane * kChunk * 128, tmV,
                        h * 64, it.kvh, tok, bvf[st]);
        }
      }
    } else if (warp == 8) {
      // ------------------------------ MMA issuer ----------------------------
      constexpr uint32_t idS = umma_idesc_bf16(kRows, kKeys, 0, 0);
      constexpr uint32_t idPV = umma_idesc_bf16(kRows, D, 0, 1);
      // S of key tile j for head slot hb: A = Q tile, B = K tile (both smem)
      auto issue_s = [&](int hb, int j) {
        const uint32_t st = (n_kv + j) % kStages;
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_q = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
            const uint32_t off_k = (kk >> 2) * L::kKHalfBytes + (kk & 3) * 32;
            const uint64_t ad = umma_desc_sw128(sQ + hb * L::kQBytes + off_q, 16, 1024);
            const uint64_t bd = umma_desc_sw128(sK0 + st * L::kKBytes + off_k, 16, 1024);
            umma_bf16(tS(hb), ad, bd, idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(bS(hb));
        }
        __syncwarp();
      };
      bool ok = true;
      // first S of the item, once Q is in TMEM and K tile 0 has landed
      {
        const uint32_t f = n_kv, st = f % kStages;
        ok = wait_or_abort(bkf[st], (f / kStages) & 1, &s_abort, p.status, p.wait_cycles) &&
             wait_or_abort(bq, n_item & 1, &s_abort, p.status, p.wait_cycles);
        for (int hb = 0; ok && hb < nh; ++hb) {
          tc_fence_after();
          issue_s(hb, 0);
        }
        if (ok && lane == 0) umma_commit(bke[st]);
        __syncwarp();
      }
      for (int kt = 0; ok && kt < it.nkt; ++kt) {
        const uint32_t f = n_kv + kt, st = f % kStages;
        const bool next = kt + 1 < it.nkt;
        const uint32_t f1 = f + 1, st1 = f1 % kStages;
        if (!wait_or_abort(bvf[st], (f / kStages) & 1, &s_abort, p.status, p.wait_cycles)) break;
        const int key0 = kt * kKeys;
        if (key0 + kKeys > it.ctx) {
          // keys past the lane's end: zero their V rows (stale bytes must not
          // meet p = 0 as 0 * NaN)
          const int first = max(0, it.ctx - key0);
          const int n16 = (kKeys - first) * 8 * L::kHalves;
          for (int i = lane; i < n16; i += 32) {
            const int c16 = i & 7, rest = i >> 3;
            const int h = rest % L::kHalves, r = first + rest / L::kHalves;
            const uint32_t a = sV0 + st * L::kVBytes + h * L::kKHalfBytes + r * 128 + c16 * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        for (int hb = 0; hb < nh; ++hb) {
          const uint32_t th = n_t[hb] + kt;
          // P V of tile kt, once this head's softmax has written P
          if (!wait_or_abort(bP(hb), th & 1, &s_abort, p.status, p.wait_cycles)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kKeys / 16; ++k) {
              const uint64_t bd = umma_desc_sw128(sV0 + st * L::kVBytes + k * 16 * 128,
                                                  L::kKHalfBytes, 1024);
              umma_bf16_tmem_a(tO(hb), tS(hb) + k * 8, bd, idPV, (kt > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(bO(hb, th));
          }
          __syncwarp();
          if (next) {
            // S of tile kt + 1 needs its K tile, and it overwrites P of tile
            // kt: wait for that P V
            if (hb == 0 && !wait_or_abort(bkf[st1], (f1 / kStages) & 1, &s_abort, p.status, p.wait_cycles)) {
              ok = false;
              break;
            }
            if (!wait_or_abort(bO(hb, th), (th >> 1) & 1, &s_abort, p.status, p.wait_cycles)) { ok = false; break; }
            tc_fence_after();
            issue_s(hb, kt + 1);
          }
        }
        if (!ok) break;
        if (lane == 0) {
          umma_commit(bve[st]);
          if (next) umma_commit(bke[st1]);
        }
        __syncwarp();
      }
    } else if (warp < 4 || it.has_b) {
      // ------------------------------ softmax rows --------------------------
      const int hb = warp >> 2;         // head slot of this group
      const int r = threadIdx.x & 127;  // row within the tile == TMEM lane
      const int pos = it.p_first + min(r, it.nrows - 1);
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tOr = tO(hb) + lane_off;
      const uint32_t tSr = tS(hb) + lane_off;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
#pragma unroll 1
      for (int kt = 0; kt < it.nkt; ++kt) {
        const uint32_t th = n_t[hb] + kt;
        if (!wait_or_abort(bS(hb), th & 1, &s_abort, p.status, p.wait_cycles)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[kKeys];
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c)
          tmem_ld32(tSr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
        tmem_wait_ld();
        const int lim = pos - kt * kKeys;  // columns c <= lim are visible to this row
        const bool full = __all_sync(0xffffffffu, lim >= kKeys - 1);
        // max of the visible raw scores (the scale is positive), eight
        // independent running maxima folded by a fixed tree
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = -INFINITY;
        if (full) {
#pragma unroll
          for (int i = 0; i < kKeys; i += 2)
            m8[(i >> 1) & 7] =
                fmax3(m8[(i >> 1) & 7], __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < kKeys; ++i)
            m8[i & 7] = fmaxf(m8[i & 7], i <= lim ? __uint_as_float(sv[i]) : -INFINITY);
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) m8[j] = fmaxf(m8[j], m8[j + w]);
        const float mx = m8[0] * c2;
        const bool grow = kt == 0 || mx > m + kRescaleLog2;
        const float mn = grow ? fmaxf(m, mx) : m;
        const float alpha = grow ? ex2_approx(m - mn) : 1.f;
        m = mn;
        const float neg = -mn;
        // p = 2^(s c2 - m) rounded to bf16, written over S as P (two per
        // column, 32 columns at a time); l adds the p before rounding, in
        // four independent pairs of partial sums folded by a fixed tree.
        // The scaling runs on packed fp32 pairs (lane by lane the same fmaf).
        const uint64_t c2x2 = f32x2(c2, c2), negx2 = f32x2(neg, neg);
        uint64_t r4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) r4[j] = f32x2(0.f, 0.f);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[kKeys / 4];
#pragma unroll
          for (int i = 0; i < kKeys / 4; ++i) {
            const int c0 = hh * (kKeys / 2) + 2 * i;
            float t0, t1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[c0]), __uint_as_float(sv[c0 + 1])),
                                  c2x2, negx2),
                        t0, t1);
            float e0 = ex2_approx(t0);
            float e1 = ex2_approx(t1);
            if (!full) {
              e0 = (c0 <= lim) ? e0 : 0.f;
              e1 = (c0 + 1 <= lim) ? e1 : 0.f;
            }
            pk[i] = pack_bf16x2(e0, e1);
            r4[i & 3] = add_f32x2(r4[i & 3], f32x2(e0, e1));
          }
          tmem_st16(tSr + hh * 32, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
          tmem_st16(tSr + hh * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
        }
        r4[0] = add_f32x2(r4[0], r4[2]);
        r4[1] = add_f32x2(r4[1], r4[3]);
        r4[0] = add_f32x2(r4[0], r4[1]);
        float rlo, rhi;
        f32x2_split(r4[0], rlo, rhi);
        const float rs = rlo + rhi;
        tmem_wait_st();
        l = fmaf(l, alpha, rs);
        // O is rescaled after P V of the previous tile has finished (it has:
        // S of this tile was issued after it); P V completions alternate
        // between two barriers by tile parity, so a barrier is never more
        // than one phase away from any wait on it even when tiles without a
        // rescale skip the wait.
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!wait_or_abort(bO(hb, th - 1), ((th - 1) >> 1) & 1, &s_abort, p.status, p.wait_cycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tOr + c * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tOr + c * 32, ov);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(bP(hb));
      }
      const uint32_t last = n_t[hb] + it.nkt - 1;
      if (ok && wait_or_abort(bO(hb, last), (last >> 1) & 1, &s_abort, p.status, p.wait_cycles)) {
        tc_fence_after();
        const bool valid = r < it.nrows;
        const float inv_l = 1.f / l;  // one division per row; out = O * (1 / l)
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) +
                             ((size_t)(it.cu0 + it.tile * kRows + r) * p.H + it.head0 + hb) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tOr + c * 32, ov);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(ov[i]) * inv_l, __uint_as_float(ov[i + 1]) * inv_l);
              v.y = pack_bf16x2(__uint_as_float(ov[i + 2]) * inv_l, __uint_as_float(ov[i + 3]) * inv_l);
              v.z = pack_bf16x2(__uint_as_float(ov[i + 4]) * inv_l, __uint_as_float(ov[i + 5]) * inv_l);
              v.w = pack_bf16x2(__uint_as_float(ov[i + 6]) * inv_l, __uint_as_float(ov[i + 7]) * inv_l);
              *reinterpret_cast<uint4*>(out + c * 32 + i) = v;
            }
          }
        }
        tc_fence_before();
      }
    }
    n_kv += it.nkt;
    n_t[0] += it.nkt;
    if (it.has_b) n_t[1] += it.nkt;
    ++n_item;
    __syncthreads();
    if (s_abort) break;
  }
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace pftc
}  // namespace pa
