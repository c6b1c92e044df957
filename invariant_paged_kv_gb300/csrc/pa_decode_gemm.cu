// Batch-invariant decode GEMM at a fixed token width ("ninfer" issue 80,
// Proposal: opt-in fixed decode width -- every GEMM-class decode op runs at a
// fixed token width T_pad, activations padded, so the kernel and its internal
// schedule are the same for every real token count t <= T_pad; columns never
// mix, so padding columns cannot disturb real ones).
//
// y[t, n] = sum_k x[t, k] W[n, k] for t < T_pad (bf16 in, fp32 accumulate,
// bf16 out). The product is taken in swapped form on tcgen05: M = 128 weight
// rows, N = T_pad tokens, accumulators in TMEM (one fp32 column per token).
// A CTA owns one 128-row tile of W and one range of K; both come from a plan
// that depends on (N, K) alone: the split-K count S makes about kTargetCtas
// CTAs, independent of t, of T_pad and of the device. With S > 1 the CTAs
// write fp32 partials and a second kernel adds them in split order 0..S-1.
// W is read exactly once (the weights dominate the bytes: the op is bound by
// HBM bandwidth, the tensor pipe idles most of the time).
//
// Pipeline per CTA (128 threads): thread 0 issues TMA loads of 64-element K
// slices of the W tile and of x (128-byte swizzle) into a 4-deep ring; thread
// 32 issues 4 tcgen05.mma (K = 16) per slice and frees the slice with a
// tcgen05.commit; after the last slice the four warps read their 32 TMEM lanes
// (weight rows) and store the tokens' outputs. Every wait is bounded
// (PA_FLAG_TIMEOUT), and a CTA that gives up lets its copies land first.
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kRowsW = 128;      // weight rows per tile (mma M)
constexpr int kKc = 64;          // K elements per stage: one 128-byte swizzled row
constexpr int kStagesG = 4;
constexpr int kThreadsG = 128;
constexpr int kTargetCtas = 296; // split-K target, a constant: the plan depends on (N, K) only

template <int TP>
struct GLayout {
  static constexpr int kWBytes = kRowsW * kKc * 2;  // 16 KiB
  static constexpr int kXBytes = TP * kKc * 2;
  static constexpr int kStage = kWBytes + kXBytes;
  static constexpr int kSmem = kStagesG * kStage + 1024;
  static constexpr uint32_t kTmemCols = TP <= 32 ? 32 : (TP <= 64 ? 64 : (TP <= 128 ? 128 : 256));
};

struct GemmParams {
  void* y;        // [T_pad, N] bf16 (S == 1)
  float* part;    // [S, T_pad, N] fp32 (S > 1)
  int N, K, S, chunks_per_split;
  int* status;
};

__device__ __forceinline__ bool wait_g(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int* status) {
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

template <int TP>
__global__ void __launch_bounds__(kThreadsG, 2)
    decode_gemm_kernel(const GemmParams g, const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX) {
  using L = GLayout<TP>;
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full[kStagesG], empty[kStagesG], done;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesG; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(&done), 1);
    s_abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX);
  }
  if (warp == 1) tmem_alloc(smem_u32(&s_tmem), L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  const int n0 = blockIdx.x * kRowsW;
  const int nchunks_total = g.K / kKc;
  const int c0 = blockIdx.y * g.chunks_per_split;
  const int nch = min(g.chunks_per_split, nchunks_total - c0);

  if (threadIdx.x == 0) {
    // ---- producer ----
    int issued = 0;
    for (int i = 0; i < nch; ++i) {
      const int st = i % kStagesG;
      if (i >= kStagesG &&
          !wait_g(smem_u32(&empty[st]), ((i / kStagesG) - 1) & 1, &s_abort, g.status))
        break;
      const uint32_t sW = base + st * L::kStage, sX = sW + L::kWBytes;
      mbar_expect_tx(smem_u32(&full[st]), L::kStage);
      const int k = (c0 + i) * kKc;
      tma_load_2d(sW, &tmW, k, n0, smem_u32(&full[st]));
      tma_load_2d(sX, &tmX, k, 0, smem_u32(&full[st]));
      ++issued;
    }
    // let every copy this CTA started land before anyone can leave (only
    // the last kStagesG can still be in flight; their barriers are at most
    // one phase from the awaited one)
    for (int j = max(0, issued - kStagesG); j < issued; ++j) {
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&full[j % kStagesG]), (j / kStagesG) & 1))
        if (clock64() - t0 > kWaitCycles) break;
    }
  } else if (threadIdx.x == 32) {
    // ---- MMA issuer ----
    constexpr uint32_t idesc = umma_idesc_bf16(kRowsW, TP, 0, 0);
    bool ok = true;
    for (int i = 0; i < nch; ++i) {
      const int st = i % kStagesG;
      if (!wait_g(smem_u32(&full[st]), (i / kStagesG) & 1, &s_abort, g.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sW = base + st * L::kStage, sX = sW + L::kWBytes;
#pragma unroll
      for (int kk = 0; kk < kKc / 16; ++kk) {
        const uint64_t ad = umma_desc_sw128(sW + kk * 32, 16, 1024);
        const uint64_t bd = umma_desc_sw128(sX + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(smem_u32(&empty[st]));
    }
    if (ok) umma_commit(smem_u32(&done));
  }
  __syncwarp();

  // ---- epilogue: warp w reads TMEM lanes 32 w .. 32 w + 31 (weight rows) ----
  const bool ok = nch > 0 && wait_g(smem_u32(&done), 0, &s_abort, g.status);
  if (__all_sync(0xffffffffu, ok)) {
    tc_fence_after();
    const int n = n0 + 32 * warp + lane;
    const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
    for (int c = 0; c < TP; c += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c, r);
      tmem_wait_ld();
      if (g.S == 1) {
        __nv_bfloat16* y = static_cast<__nv_bfloat16*>(g.y);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          y[(size_t)(c + j) * g.N + n] = __float2bfloat16_rn(__uint_as_float(r[j]));
      } else {
        float* part = g.part + (size_t)blockIdx.y * TP * g.N;
#pragma unroll
        for (int j = 0; j < 32; ++j) part[(size_t)(c + j) * g.N + n] = __uint_as_float(r[j]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// y[t, n] = sum over splits s = 0, 1, ..., S - 1 of part[s, t, n], in that order.
__global__ void __launch_bounds__(256) splitk_sum_kernel(const float* part, __nv_bfloat16* y,
                                                         long long per_split, int S) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < per_split;
       i += (long long)gridDim.x * blockDim.x) {
    float a = part[i];
    for (int s = 1; s < S; ++s) a += part[(size_t)s * per_split + i];
    y[i] = __float2bfloat16_rn(a);
  }
}

template <int TP>
cudaError_t launch_tp(const GemmParams& g, const CUtensorMap& w, const CUtensorMap& x,
                      cudaStream_t s) {
  auto kern = decode_gemm_kernel<TP>;
  static unsigned long long done = 0;
  cudaError_t e = smem_opt_in(kern, GLayout<TP>::kSmem, &done);
  if (e != cudaSuccess) return e;
  dim3 grid(g.N / kRowsW, g.S);
  kern<<<grid, kThreadsG, GLayout<TP>::kSmem, s>>>(g, w, x);
  return cudaGetLastError();
}

}  // namespace

// Split-K plan of an N x K weight: a function of (N, K) only.
void decode_gemm_plan(int N, int K, int* S, int* chunks_per_split) {
  const int tiles = N / kRowsW;
  const int chunks = K / kKc;
  int s = (kTargetCtas + tiles - 1) / tiles;
  const int max_s = chunks / 4 > 0 ? chunks / 4 : 1;  // at least 4 slices per split
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  int cps = (chunks + s - 1) / s;
  *chunks_per_split = cps;
  *S = (chunks + cps - 1) / cps;
}

int num_sms();

cudaError_t launch_decode_gemm(void* y, float* part, int T_pad, int N, int K, int S, int cps,
                               int* status, const CUtensorMap& w, const CUtensorMap& x,
                               cudaStream_t s) {
  GemmParams g;
  g.y = y;
  g.part = part;
  g.N = N;
  g.K = K;
  g.S = S;
  g.chunks_per_split = cps;
  g.status = status;
  cudaError_t e;
  switch (T_pad) {
    case 32: e = launch_tp<32>(g, w, x, s); break;
    case 64: e = launch_tp<64>(g, w, x, s); break;
    case 96: e = launch_tp<96>(g, w, x, s); break;
    case 128: e = launch_tp<128>(g, w, x, s); break;
    case 192: e = launch_tp<192>(g, w, x, s); break;
    case 256: e = launch_tp<256>(g, w, x, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || S == 1) return e;
  const long long per = (long long)T_pad * N;
  long long blocks = (per + 255) / 256;
  const long long cap = 4LL * num_sms();
  splitk_sum_kernel<<<(int)(blocks < cap ? blocks : cap), 256, 0, s>>>(
      part, static_cast<__nv_bfloat16*>(y), per, S);
  return cudaGetLastError();
}

}  // namespace pa
