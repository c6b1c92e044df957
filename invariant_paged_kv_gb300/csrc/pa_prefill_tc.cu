// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05), bf16.
//
// A lane with q_len >= 2 is a causal prefill chunk ("P3: native paged-KV
// continuous-batching sampler", Design, engine.py: prefill chunks and decode
// tokens share one flat step; Evidence, mutant "prefill causal mask off by
// one"): its row j sits at position ctx - q_len + j and attends keys
// 0..position. Work item = (128-row q tile of one lane, query head). Per
// item, key tiles of 128 keys go in ascending order, each through
//   S = Q K^T          (tcgen05.mma, M = 128 rows, N = 128 keys, K = D, fp32 in TMEM)
//   m, p, l            (one thread per row: row max, p = 2^(t - m) rounded to
//                       bf16, l += sum of the rounded p, all within the thread)
//   O = O * alpha + P V (P written to shared memory as the A operand,
//                       V read MN-major as the B operand, O kept in TMEM)
// and finally out = O / l. A row's arithmetic depends on its q row, its keys
// and the fixed 128-key tiling from key 0 -- never on other lanes.
//
// Warp roles (192 threads): warps 0-3 own the 128 rows (TMEM lanes), warp 4
// issues the MMAs (one elected thread), warp 5 streams Q / K / V tiles in by
// TMA (through the block table, 16 keys per box) into 2-deep K and V rings.
// TMEM: two S buffers (2 x 128 columns) and O (D columns) in one 512-column
// allocation. Every wait is bounded; a timeout raises PA_FLAG_TIMEOUT.
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kRows = 128;       // query rows per item (M)
constexpr int kKeys = 128;       // keys per tile (N of S, K of PV)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct PfLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kRows * 128;        // 128 rows x 128 bytes
  static constexpr int kQBytes = kHalves * kHalfBytes;  // Q tile
  static constexpr int kKBytes = kHalves * kHalfBytes;  // one K tile
  static constexpr int kVBytes = kHalves * kHalfBytes;  // one V tile
  static constexpr int kPBytes = 2 * kHalfBytes;        // P: 128 rows x 128 keys bf16
  static constexpr int kQ = 0;
  static constexpr int kK0 = kQ + kQBytes;
  static constexpr int kV0 = kK0 + 2 * kKBytes;
  static constexpr int kP = kV0 + 2 * kVBytes;
  static constexpr int kEnd = kP + kPBytes;
  // + alignment slack; at least 116 KB so one CTA (and one 512-column TMEM
  // allocation) per SM
  static constexpr int kSmemBytes = (kEnd + 1024) > 118784 ? (kEnd + 1024) : 118784;
};

struct Bars {
  uint64_t q, kfull[2], kempty[2], vfull[2], vempty[2], s[2], sfree[2], p, o;
};

struct ItemInfo {
  int lane, tile, head, cu0, q_len, ctx, nrows, p_first, nkt;
};

__device__ __forceinline__ ItemInfo item_info(const StepParams& p, int item) {
  ItemInfo it;
  const int t = item / p.H;
  it.head = item - t * p.H;
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
__device__ __forceinline__ bool wait_or_abort_1(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              int* status) {
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
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              int* status) {
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
  const uint32_t sQ = base + L::kQ, sK0 = base + L::kK0, sV0 = base + L::kV0, sP = base + L::kP;
  const uint32_t bq = smem_u32(&bars.q), bp = smem_u32(&bars.p), bo = smem_u32(&bars.o);
  uint32_t bkf[2], bke[2], bvf[2], bve[2], bs[2], bsf[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    bkf[i] = smem_u32(&bars.kfull[i]);
    bke[i] = smem_u32(&bars.kempty[i]);
    bvf[i] = smem_u32(&bars.vfull[i]);
    bve[i] = smem_u32(&bars.vempty[i]);
    bs[i] = smem_u32(&bars.s[i]);
    bsf[i] = smem_u32(&bars.sfree[i]);
  }
  if (threadIdx.x == 0) {
    mbar_init(bq, 1);
    mbar_init(bp, kRows);
    mbar_init(bo, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bkf[i], 1);
      mbar_init(bke[i], 1);
      mbar_init(bvf[i], 1);
      mbar_init(bve[i], 1);
      mbar_init(bs[i], 1);
      mbar_init(bsf[i], kRows);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 4) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t tS[2] = {tmem, tmem + kKeys};
  const uint32_t tO = tmem + 2 * kKeys;

  const int g = p.H / p.Hkv;
  const int n_items = p.plan.header[2] * p.H;
  // running use counters (identical in every role)
  uint32_t n_item = 0;  // items done by this CTA
  uint32_t n_tile = 0;  // key tiles done by this CTA

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const ItemInfo it = item_info(p, item);
    const int kvh = it.head / g;

    if (warp == 5) {
      // ------------------------------ producer ------------------------------
      if (lane == 0) {
        mbar_expect_tx(bq, L::kQBytes);
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h)
          tma_load_3d(sQ + h * L::kHalfBytes, &tmQ, h * 64, it.head, it.cu0 + it.tile * kRows, bq);
      }
      for (int kt = 0; kt < it.nkt; ++kt) {
        const uint32_t f = n_tile + kt, st = f & 1;
        const int key0 = kt * kKeys;
        const int nchunk = min(kKeys / kChunk, (it.ctx - key0 + kChunk - 1) / kChunk);
        // block id of chunk `lane` (lanes 0..7)
        int blk = 0;
        if (lane < nchunk) {
          blk = p.block_tables[(size_t)it.lane * p.max_blocks + (key0 + lane * kChunk) / p.bs];
          if (blk < 0 || blk >= p.NB) {
            raise_flag(p.status, PA_FLAG_BLOCK_RANGE);
            blk = 0;
          }
        }
        const uint32_t bytes = (uint32_t)nchunk * L::kHalves * kChunk * 128;
        // K tile
        if (f >= 2 && !wait_or_abort(bke[st], ((f - 2) >> 1) & 1, &s_abort, p.status)) break;
        if (lane == 0) mbar_expect_tx(bkf[st], bytes);
        __syncwarp();
        for (int c = 0; c < nchunk; ++c) {
          const int b = __shfl_sync(0xffffffffu, blk, c);
          if (lane == 0) {
            const int tok = b * p.bs + (key0 + c * kChunk) % p.bs;
#pragma unroll
            for (int h = 0; h < L::kHalves; ++h)
              tma_load_3d(sK0 + st * L::kKBytes + h * L::kHalfBytes + c * kChunk * 128, &tmK,
                          h * 64, kvh, tok, bkf[st]);
          }
        }
        // V tile
        if (f >= 2 && !wait_or_abort(bve[st], ((f - 2) >> 1) & 1, &s_abort, p.status)) break;
        if (lane == 0) mbar_expect_tx(bvf[st], bytes);
        __syncwarp();
        for (int c = 0; c < nchunk; ++c) {
          const int b = __shfl_sync(0xffffffffu, blk, c);
          if (lane == 0) {
            const int tok = b * p.bs + (key0 + c * kChunk) % p.bs;
#pragma unroll
            for (int h = 0; h < L::kHalves; ++h)
              tma_load_3d(sV0 + st * L::kVBytes + h * L::kHalfBytes + c * kChunk * 128, &tmV,
                          h * 64, kvh, tok, bvf[st]);
          }
        }
      }
    } else if (warp == 4) {
      // ------------------------------ MMA issuer ----------------------------
      constexpr uint32_t idS = umma_idesc_bf16(kRows, kKeys, 0, 0);
      constexpr uint32_t idPV = umma_idesc_bf16(kRows, D, 0, 1);
      bool ok = wait_or_abort(bq, n_item & 1, &s_abort, p.status);
      auto issue_pv = [&](int j) -> bool {
        const uint32_t f = n_tile + j, st = f & 1;
        if (!wait_or_abort(bvf[st], (f >> 1) & 1, &s_abort, p.status)) return false;
        const int key0 = j * kKeys;
        if (key0 + kKeys > it.ctx) {
          // keys past the lane's end: zero their V rows (stale bytes must not
          // meet p = 0 as 0 * NaN)
          const int first = max(0, it.ctx - key0);
          const int n16 = (kKeys - first) * 8 * L::kHalves;
          for (int i = lane; i < n16; i += 32) {
            const int c16 = i & 7, rest = i >> 3;
            const int h = rest % L::kHalves, r = first + rest / L::kHalves;
            const uint32_t a = sV0 + st * L::kVBytes + h * L::kHalfBytes + r * 128 + c16 * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (!wait_or_abort(bp, (n_tile + j) & 1, &s_abort, p.status)) return false;
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k) {
            const uint64_t ad = umma_desc_sw128(sP + (k >> 2) * L::kHalfBytes + (k & 3) * 32, 16, 1024);
            const uint64_t bd = umma_desc_sw128(sV0 + st * L::kVBytes + k * 16 * 128,
                                                L::kHalfBytes, 1024);
            umma_bf16(tO, ad, bd, idPV, (j > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(bo);
          umma_commit(bve[st]);
        }
        __syncwarp();
        return true;
      };
      for (int kt = 0; ok && kt < it.nkt; ++kt) {
        const uint32_t f = n_tile + kt, st = f & 1;
        if (!wait_or_abort(bkf[st], (f >> 1) & 1, &s_abort, p.status)) break;
        const uint32_t sb = f & 1;
        if (f >= 2 && !wait_or_abort(bsf[sb], ((f - 2) >> 1) & 1, &s_abort, p.status)) break;
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::kHalfBytes + (kk & 3) * 32;
            const uint64_t ad = umma_desc_sw128(sQ + off, 16, 1024);
            const uint64_t bd = umma_desc_sw128(sK0 + st * L::kKBytes + off, 16, 1024);
            umma_bf16(tS[sb], ad, bd, idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(bs[sb]);
          umma_commit(bke[st]);
        }
        __syncwarp();
        if (kt >= 1 && !issue_pv(kt - 1)) break;
      }
      if (__all_sync(0xffffffffu, s_abort == 0)) issue_pv(it.nkt - 1);
    } else {
      // ------------------------------ softmax rows --------------------------
      const int r = threadIdx.x;  // row within the tile == TMEM lane
      const int pos = it.p_first + min(r, it.nrows - 1);
      const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int kt = 0; kt < it.nkt; ++kt) {
        const uint32_t f = n_tile + kt, sb = f & 1;
        if (!wait_or_abort(bs[sb], (f >> 1) & 1, &s_abort, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[kKeys / 32][32];
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c) tmem_ld32(tS[sb] + lane_off + c * 32, sv[c]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bsf[sb]);
        const int key0 = kt * kKeys;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          const float t =
              (key0 + c <= pos) ? __uint_as_float(sv[c >> 5][c & 31]) * p.scale_log2 : -INFINITY;
          sv[c >> 5][c & 31] = __float_as_uint(t);
          mx = fmaxf(mx, t);
        }
        const float mn = fmaxf(m, mx);
        const float alpha = ex2_approx(m - mn);
        m = mn;
        float rs = 0.f;
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int c = 0; c < kKeys / 2; ++c) {
          pk[c] = pack_bf16x2(ex2_approx(__uint_as_float(sv[c >> 4][(2 * c) & 31]) - mn),
                              ex2_approx(__uint_as_float(sv[c >> 4][(2 * c + 1) & 31]) - mn));
          rs += bf16_lo(pk[c]);
          rs += bf16_hi(pk[c]);
        }
        l = fmaf(l, alpha, rs);
        if (kt > 0) {  // PV of the previous tile must be done: P buffer and O are ours again
          if (!wait_or_abort(bo, (n_tile + kt - 1) & 1, &s_abort, p.status)) { ok = false; break; }
          tc_fence_after();
        }
        // P row -> shared (A operand of P V: K-major, 128-byte swizzle)
#pragma unroll
        for (int c = 0; c < kKeys / 8; ++c) {
          const int half = c >> 3, c16 = c & 7;
          const uint32_t a = sP + half * L::kHalfBytes + (r >> 3) * 1024 + (r & 7) * 128 +
                             ((c16 ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[4 * c]),
                       "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                       : "memory");
        }
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + lane_off + c * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tO + lane_off + c * 32, ov);
          }
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bp);
      }
      if (ok && wait_or_abort(bo, (n_tile + it.nkt - 1) & 1, &s_abort, p.status)) {
        tc_fence_after();
        const bool valid = r < it.nrows;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) +
                             ((size_t)(it.cu0 + it.tile * kRows + r) * p.H + it.head) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tO + lane_off + c * 32, ov);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              v.x = pack_bf16x2(finish_div(__uint_as_float(ov[i]), l), finish_div(__uint_as_float(ov[i + 1]), l));
              v.y = pack_bf16x2(finish_div(__uint_as_float(ov[i + 2]), l), finish_div(__uint_as_float(ov[i + 3]), l));
              v.z = pack_bf16x2(finish_div(__uint_as_float(ov[i + 4]), l), finish_div(__uint_as_float(ov[i + 5]), l));
              v.w = pack_bf16x2(finish_div(__uint_as_float(ov[i + 6]), l), finish_div(__uint_as_float(ov[i + 7]), l));
              *reinterpret_cast<uint4*>(out + c * 32 + i) = v;
            }
          }
        }
        tc_fence_before();
      }
    }
    n_tile += it.nkt;
    ++n_item;
    __syncthreads();
    if (s_abort) break;
  }
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const StepParams& p, const CUtensorMap& q, const CUtensorMap& k,
                     const CUtensorMap& v, int grid, cudaStream_t s) {
  auto kern = prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PfLayout<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, PfLayout<D>::kSmemBytes, s>>>(p, q, k, v);
  return cudaGetLastError();
}

}  // namespace

int num_sms();

cudaError_t launch_prefill_tc(const StepParams& p, const CUtensorMap& q, const CUtensorMap& k,
                              const CUtensorMap& v, long long max_items, cudaStream_t s) {
  long long cap = num_sms();
  int grid = (int)(max_items < cap ? max_items : cap);
  if (grid < 1) grid = 1;
  return p.D == 128 ? launch_d<128>(p, q, k, v, grid, s) : launch_d<64>(p, q, k, v, grid, s);
}

}  // namespace pa
