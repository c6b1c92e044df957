// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05), bf16.
//
// A lane with q_len >= 2 is a causal prefill chunk ("P3: native paged-KV
// continuous-batching sampler", Design, engine.py: prefill chunks and decode
// tokens share one flat step; Evidence, mutant "prefill causal mask off by
// one"): its row j sits at position ctx - q_len + j and attends keys
// 0..position. Work item = (128-row q tile of one lane, a pair of query heads
// that read the same kv head). Per item, key tiles of 64 keys go in ascending
// order; for each head of the pair and each key tile:
//   S = Q K^T           tcgen05.mma, M = 128 rows, N = 64 keys, K = D, fp32 in TMEM
//   m, p, l             one thread per row: running max, p = 2^(t - m) rounded
//                       to bf16 and written back over S in TMEM, l += sum of
//                       the rounded p -- all within the thread
//   O = O * alpha + P V tcgen05.mma with A = P read from TMEM, B = V (MN-major
//                       smem), O in TMEM
// and finally out = O / l. The running max moves only when a tile's max
// exceeds it by more than 8 (log2 units), so O is rescaled rarely. A row's
// arithmetic depends on its q row, its keys and the fixed 64-key tiling from
// key 0 -- never on other lanes.
//
// Warp roles (320 threads): warps 0-3 and 4-7 are two softmax groups (one per
// head of the pair; thread r of a group owns row r = TMEM lane r), warp 8
// issues the MMAs (one elected thread), warp 9 streams Q / K / V in by TMA
// (K / V through the block table, 16 keys per box) into 4-deep K and V rings
// shared by both heads. Each head has two S/P buffers, so S of tile f + 1 is
// computed while the softmax works on tile f and P V of tile f - 1 runs; the
// tensor core also alternates between the two heads. TMEM (512 columns):
// S/P buffers 0 and 1 and O of head A, then the same for head B. Every wait
// is bounded (timeout -> PA_FLAG_TIMEOUT). No parity wait ever meets a barrier
// more than one phase away from the awaited one, ahead or behind (see the P V
// barriers, which alternate by tile parity for that reason).
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kRows = 128;  // query rows per item (M)
constexpr int kKeys = 64;   // keys per tile (N of S, K of PV)
constexpr int kStages = 4;  // depth of the K and V rings
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct PfLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kRows * 128;         // Q: 128 rows x 128 bytes
  static constexpr int kKHalfBytes = kKeys * 128;        // K / V: 64 keys x 128 bytes
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
  uint64_t q, kfull[kStages], kempty[kStages], vfull[kStages], vempty[kStages];
  uint64_t s[2][2], p[2][2], o[2][2];  // [head][buffer / tile parity]
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
                                                volatile int* abort_flag, int* status) {
  if (*abort_flag) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      raise_flag(status, PA_FLAG_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Every lane of the warp waits; the verdict is made warp-uniform.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int* status) {
  return __all_sync(0xffffffffu, wait_or_abort_1(bar, parity, abort_flag, status));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const StepParams p, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using L = PfLayout<D>;
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

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
    mbar_init(bq, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bkf[i], 1);
      mbar_init(bke[i], 1);
      mbar_init(bvf[i], 1);
      mbar_init(bve[i], 1);
    }
    for (int h = 0; h < 2; ++h) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(smem_u32(&bars.s[h][b]), 1);
        mbar_init(smem_u32(&bars.p[h][b]), kRows);
      }
      mbar_init(smem_u32(&bars.o[h][0]), 1);
      mbar_init(smem_u32(&bars.o[h][1]), 1);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 9 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == 8) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // S / P buffer b of head slot h at column 256 h + 64 b; O of head slot h at 256 h + 128
  auto tS = [&](int h, uint32_t b) -> uint32_t { return tmem + 256 * h + kKeys * b; };
  auto tO = [&](int h) -> uint32_t { return tmem + 256 * h + 128; };
  auto bS = [&](int h, uint32_t b) -> uint32_t { return smem_u32(&bars.s[h][b]); };
  auto bP = [&](int h, uint32_t b) -> uint32_t { return smem_u32(&bars.p[h][b]); };
  // P V of tile t completes on o[head][t & 1]
  auto bO = [&](int h, uint32_t t) -> uint32_t { return smem_u32(&bars.o[h][t & 1]); };

  const int g = p.H / p.Hkv;
  const int n_items = p.plan.header[2] * p.Hkv * ((g + 1) / 2);
  const float c2 = p.scale_log2;  // > 0 (validated on the host)
  // running use counters, identical in every role: K/V ring fills, and key
  // tiles done by each head slot
  uint32_t n_item = 0, n_kv = 0, n_t[2] = {0, 0};

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const ItemInfo it = item_info(p, item, g);

    if (warp == 9) {
      // ------------------------------ producer ------------------------------
      if (lane == 0) {
        mbar_expect_tx(bq, (it.has_b ? 2 : 1) * L::kQBytes);
        for (int hb = 0; hb < 1 + it.has_b; ++hb)
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sQ + hb * L::kQBytes + h * L::kHalfBytes, &tmQ, h * 64, it.head0 + hb,
                        it.cu0 + it.tile * kRows, bq);
      }
      for (int kt = 0; kt < it.nkt; ++kt) {
        const uint32_t f = n_kv + kt, st = f % kStages, use = f / kStages;
        const int key0 = kt * kKeys;
        const int nchunk = min(kKeys / kChunk, (it.ctx - key0 + kChunk - 1) / kChunk);
        int blk = 0;  // block id of chunk `lane` (lanes 0..3)
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
        if (use >= 1 && !wait_or_abort(bke[st], (use - 1) & 1, &s_abort, p.status)) break;
        if (lane == 0) mbar_expect_tx(bkf[st], bytes);
        __syncwarp();
        if (lane < nchunk) {
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sK0 + st * L::kKBytes + h * L::kKHalfBytes + lane * kChunk * 128, &tmK,
                        h * 64, it.kvh, tok, bkf[st]);
        }
        if (use >= 1 && !wait_or_abort(bve[st], (use - 1) & 1, &s_abort, p.status)) break;
        if (lane == 0) mbar_expect_tx(bvf[st], bytes);
        __syncwarp();
        if (lane < nchunk) {
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sV0 + st * L::kVBytes + h * L::kKHalfBytes + lane * kChunk * 128, &tmV,
                        h * 64, it.kvh, tok, bvf[st]);
        }
      }
    } else if (warp == 8) {
      // ------------------------------ MMA issuer ----------------------------
      constexpr uint32_t idS = umma_idesc_bf16(kRows, kKeys, 0, 0);
      constexpr uint32_t idPV = umma_idesc_bf16(kRows, D, 0, 1);
      const int nh = 1 + it.has_b;
      bool ok = wait_or_abort(bq, n_item & 1, &s_abort, p.status);
      // P V of key tile j (both heads), once its P and V are there
      auto issue_pv = [&](int j) -> bool {
        const uint32_t f = n_kv + j, st = f % kStages;
        if (!wait_or_abort(bvf[st], (f / kStages) & 1, &s_abort, p.status)) return false;
        const int key0 = j * kKeys;
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
          const uint32_t th = n_t[hb] + j;
          if (!wait_or_abort(bP(hb, th & 1), (th >> 1) & 1, &s_abort, p.status)) return false;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kKeys / 16; ++k) {
              const uint64_t bd = umma_desc_sw128(sV0 + st * L::kVBytes + k * 16 * 128,
                                                  L::kKHalfBytes, 1024);
              umma_bf16_tmem_a(tO(hb), tS(hb, th & 1) + k * 8, bd, idPV,
                               (j > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(bO(hb, th));
          }
          __syncwarp();
        }
        if (lane == 0) umma_commit(bve[st]);
        __syncwarp();
        return true;
      };
      for (int kt = 0; ok && kt < it.nkt; ++kt) {
        const uint32_t f = n_kv + kt, st = f % kStages;
        if (!wait_or_abort(bkf[st], (f / kStages) & 1, &s_abort, p.status)) break;
        for (int hb = 0; hb < nh; ++hb) {
          const uint32_t th = n_t[hb] + kt;
          // buffer th & 1 last held P of tile kt - 2: its P V must be done
          if (kt >= 2 && !wait_or_abort(bO(hb, th - 2), ((th - 2) >> 1) & 1, &s_abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off_q = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
              const uint32_t off_k = (kk >> 2) * L::kKHalfBytes + (kk & 3) * 32;
              const uint64_t ad = umma_desc_sw128(sQ + hb * L::kQBytes + off_q, 16, 1024);
              const uint64_t bd = umma_desc_sw128(sK0 + st * L::kKBytes + off_k, 16, 1024);
              umma_bf16(tS(hb, th & 1), ad, bd, idS, kk > 0 ? 1u : 0u);
            }
            umma_commit(bS(hb, th & 1));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) umma_commit(bke[st]);
        __syncwarp();
        if (kt >= 1 && !issue_pv(kt - 1)) break;
      }
      if (__all_sync(0xffffffffu, s_abort == 0)) issue_pv(it.nkt - 1);
    } else if (warp < 4 || it.has_b) {
      // ------------------------------ softmax rows --------------------------
      const int hb = warp >> 2;         // head slot of this group
      const int r = threadIdx.x & 127;  // row within the tile == TMEM lane
      const int pos = it.p_first + min(r, it.nrows - 1);
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tOr = tO(hb) + lane_off;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
#pragma unroll 1
      for (int kt = 0; kt < it.nkt; ++kt) {
        const uint32_t th = n_t[hb] + kt, b = th & 1;
        const uint32_t tSr = tS(hb, b) + lane_off;
        if (!wait_or_abort(bS(hb, b), (th >> 1) & 1, &s_abort, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[kKeys];
        tmem_ld32(tSr, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(tSr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
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
          for (int i = 0; i < kKeys; ++i) m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(sv[i]));
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
        // column); their sum in eight independent partial sums folded by a
        // fixed tree
        float r8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) r8[j] = 0.f;
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int i = 0; i < kKeys / 2; ++i) {
          float e0 = ex2_approx(fmaf(__uint_as_float(sv[2 * i]), c2, neg));
          float e1 = ex2_approx(fmaf(__uint_as_float(sv[2 * i + 1]), c2, neg));
          if (!full) {
            e0 = (2 * i <= lim) ? e0 : 0.f;
            e1 = (2 * i + 1 <= lim) ? e1 : 0.f;
          }
          pk[i] = pack_bf16x2(e0, e1);
          r8[i & 7] += bf16_lo(pk[i]) + bf16_hi(pk[i]);
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) r8[j] += r8[j + w];
        const float rs = r8[0];
        tmem_st16(tSr, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        tmem_st16(tSr + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
        tmem_wait_st();
        l = fmaf(l, alpha, rs);
        // P V of the previous tile must be done before O is rescaled. P V
        // completions alternate between two barriers by tile parity, so a
        // barrier is never more than one phase away from any wait on it even
        // when tiles without a rescale skip the wait (S of this tile was
        // issued after P V of tile th - 2 finished, and P V of tile th + 1
        // needs this tile's P).
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!wait_or_abort(bO(hb, th - 1), ((th - 1) >> 1) & 1, &s_abort, p.status)) {
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
        mbar_arrive(bP(hb, b));
      }
      const uint32_t last = n_t[hb] + it.nkt - 1;
      if (ok && wait_or_abort(bO(hb, last), (last >> 1) & 1, &s_abort, p.status)) {
        tc_fence_after();
        const bool valid = r < it.nrows;
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
              v.x = pack_bf16x2(finish_div(__uint_as_float(ov[i]), l),
                                finish_div(__uint_as_float(ov[i + 1]), l));
              v.y = pack_bf16x2(finish_div(__uint_as_float(ov[i + 2]), l),
                                finish_div(__uint_as_float(ov[i + 3]), l));
              v.z = pack_bf16x2(finish_div(__uint_as_float(ov[i + 4]), l),
                                finish_div(__uint_as_float(ov[i + 5]), l));
              v.w = pack_bf16x2(finish_div(__uint_as_float(ov[i + 6]), l),
                                finish_div(__uint_as_float(ov[i + 7]), l));
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

template <int D>
cudaError_t launch_d(const StepParams& p, const CUtensorMap& q, const CUtensorMap& k,
                     const CUtensorMap& v, int grid, cudaStream_t s) {
  auto kern = prefill_tc_kernel<D>;
  static unsigned long long done = 0;
  cudaError_t e = smem_opt_in(kern, PfLayout<D>::kSmemBytes, &done);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, PfLayout<D>::kSmemBytes, s>>>(p, q, k, v);
  return cudaGetLastError();
}

}  // namespace

int num_sms();

// max_items: an upper bound on (q tile, kv head, head pair) items of the step.
cudaError_t launch_prefill_tc(const StepParams& p, const CUtensorMap& q, const CUtensorMap& k,
                              const CUtensorMap& v, long long max_items, cudaStream_t s) {
  long long cap = num_sms();
  int grid = (int)(max_items < cap ? max_items : cap);
  if (grid < 1) grid = 1;
  return p.D == 128 ? launch_d<128>(p, q, k, v, grid, s) : launch_d<64>(p, q, k, v, grid, s);
}

}  // namespace pa
