// Steps that mix decode rows and prefill chunks (bf16 caches, the
// batch-invariant mode): the split-KV decode work is bound by HBM bandwidth
// and the tensor-core prefill by the tensor pipe, and on their own they run
// one after the other. Here one launch runs both on disjoint SMs: every CTA
// (one per SM: the prefill's shared memory admits one) takes one role -- the
// prefill CTA of pa_prefill_tc.cuh, or 8 independent decode warps of
// pa_decode_bf16.cuh -- so the two kinds of work overlap. Each role takes its
// items from its own counter, and an item's arithmetic is the same whichever
// CTA computes it, so every output bit is the one the two kernels give on
// their own.
//
// The row-invariant mode has the same shape -- its decode rows on the split
// kernel, its prefill rows on the prefill-row kernel (mma.sync, bound by its
// dependency latency) -- and row_mixed_kernel pairs those two the same way.
//
// The number of prefill CTAs, which balances the two roles' times, comes
// from the plan builder (prefill_role_ctas); a prefill CTA that runs out of
// prefill items then takes decode items, so the launch ends close to the
// point where both kinds of work are done even when that estimate is off.
// Neither decides any result.
#include "pa_decode_bf16.cuh"
#include "pa_prefill_tc.cuh"
#include "pa_rows_bf16.cuh"

namespace pa {

namespace {

constexpr int kDecWarps = 8;  // decode warps of a decode-role CTA

template <int D, int NT>
__global__ void __launch_bounds__(pftc::kThreads, 1)
    mixed_kernel(const StepParams p, const __grid_constant__ CUtensorMap tmQ,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t dsmem[];
  if ((int)blockIdx.x < p.plan.header[kHeaderPrefillCtas]) {
    pftc::prefill_tc_cta<D>(p, &tmQ, &tmK, &tmV, dsmem);
    // out of prefill items (its copies landed, its products finished, its
    // TMEM released): help with whatever decode items are left
    if (threadIdx.x < kDecWarps * 32) decode_bf16_warps<D, NT, false, kDecWarps>(p, &tmK, &tmV, dsmem);
  } else if (threadIdx.x < kDecWarps * 32) {
    decode_bf16_warps<D, NT, false, kDecWarps>(p, &tmK, &tmV, dsmem);
  }
}

template <int D, int NT>
cudaError_t launch_m(const StepParams& p, const CUtensorMap& q, const CUtensorMap& k,
                     const CUtensorMap& v, int grid, cudaStream_t s) {
  constexpr int a = pftc::PfLayout<D>::kSmemBytes, b = DecTile<D>::smem_bytes(kDecWarps);
  constexpr int smem = a > b ? a : b;
  auto kern = mixed_kernel<D, NT>;
  static unsigned long long done = 0;
  cudaError_t e = smem_opt_in(kern, smem, &done);
  if (e != cudaSuccess) return e;
  kern<<<grid, pftc::kThreads, smem, s>>>(p, q, k, v);
  return cudaGetLastError();
}

// Row-invariant mode: prefill-row CTAs (pa_rows_bf16.cuh) and decode CTAs.
template <int D, int NT>
__global__ void __launch_bounds__(rows::kRThreads, 1)
    row_mixed_kernel(const StepParams p, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t dsmem[];
  if ((int)blockIdx.x < p.plan.header[kHeaderPrefillCtas]) {
    rows::rows_bf16_cta<D>(p, &tmK, &tmV, dsmem);
    // out of prefill-row items: once every copy of that role has landed
    // (its TMA warp waits for them before it returns), its shared memory
    // serves decode items
    __syncthreads();
    if (threadIdx.x < kDecWarps * 32) decode_bf16_warps<D, NT, false, kDecWarps>(p, &tmK, &tmV, dsmem);
  } else if (threadIdx.x < kDecWarps * 32) {
    decode_bf16_warps<D, NT, false, kDecWarps>(p, &tmK, &tmV, dsmem);
  }
}

template <int D, int NT>
cudaError_t launch_rm(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v, int grid,
                      cudaStream_t s) {
  static_assert(rows::kRThreads >= kDecWarps * 32, "decode warps fit the CTA");
  constexpr int a = rows::RTile<D>::kSmemBytes, b = DecTile<D>::smem_bytes(kDecWarps);
  constexpr int smem = a > b ? a : b;
  auto kern = row_mixed_kernel<D, NT>;
  static unsigned long long done = 0;
  cudaError_t e = smem_opt_in(kern, smem, &done);
  if (e != cudaSuccess) return e;
  kern<<<grid, rows::kRThreads, smem, s>>>(p, k, v);
  return cudaGetLastError();
}

}  // namespace

// Rows per group of the prefill-row role for a GQA group of g heads: as many
// rows as fill a CTA's rows::kCols (row, head) columns; 0 (no grouping: the
// rows take the decode path) when one row's heads do not fit.
int rows_group_size(int g) { return g >= 1 && g <= rows::kCols ? rows::kCols / g : 0; }

// One CTA per SM (row-invariant mode, steps with prefill rows).
cudaError_t launch_row_mixed(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v,
                             cudaStream_t s) {
  const int grid = p.sm_count;
  const int g = p.H / p.Hkv;
  if (p.group_rows != rows_group_size(g) || p.group_rows < 1) return cudaErrorInvalidValue;
  if (p.D == 128) return g <= 8 ? launch_rm<128, 1>(p, k, v, grid, s) : launch_rm<128, 2>(p, k, v, grid, s);
  return g <= 8 ? launch_rm<64, 1>(p, k, v, grid, s) : launch_rm<64, 2>(p, k, v, grid, s);
}

// One CTA per SM.
cudaError_t launch_mixed(const StepParams& p, const CUtensorMap& q, const CUtensorMap& k,
                         const CUtensorMap& v, cudaStream_t s) {
  const int grid = p.sm_count;
  const int g = p.H / p.Hkv;
  if (p.D == 128) return g <= 8 ? launch_m<128, 1>(p, q, k, v, grid, s) : launch_m<128, 2>(p, q, k, v, grid, s);
  return g <= 8 ? launch_m<64, 1>(p, q, k, v, grid, s) : launch_m<64, 2>(p, q, k, v, grid, s);
}

}  // namespace pa
