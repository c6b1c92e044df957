// Fixed-order combine of split partials.
//
// For every row with n >= 2 splits and every (head, dim): fold the partials
// (m_i, l_i, acc_i) of splits i = 0, 1, ..., n-1 strictly left to right in
// fp32 -- M = m_0, L = l_0, A = acc_0; then M' = max(M, m_i),
// L = L 2^(M - M') + l_i 2^(m_i - M'), A likewise, M = M' -- and write
// A / L rounded to the output type. The order is the ordered fp32 fold of
// "Numerics envelopes" (The hierarchy, collectives.deterministic: partials
// 0..W-1 left to right in fp32, one rounding; Layout invariance of QCP:
// combine_attention_partials with the ordered fold), applied to splits
// instead of ranks. n depends only on the row's own key count, so the fold is
// the same whatever else is in the step.
#include "pa_common.cuh"

namespace pa {

namespace {

__global__ void __launch_bounds__(128) combine_kernel(const StepParams p) {
  const int row = blockIdx.x;
  const int4 info = p.plan.row_info[row];
  if (info.w < 0 || info.z <= 1) return;  // not on the split path, or written directly
  const int n = info.z;
  const int nfull = info.y >= 0 ? n - 1 : n;
  const int D4 = p.D / 4;
  const int hpc = blockDim.x / D4;  // heads per CTA
  const int h = blockIdx.y * hpc + threadIdx.x / D4;
  if (h >= p.H) return;
  const int d4 = threadIdx.x - (threadIdx.x / D4) * D4;
  const float4* acc = reinterpret_cast<const float4*>(p.plan.acc);

  Fold f;
  float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int i = 0; i < n; ++i) {
    const int pair = i < nfull ? info.x + i : info.y;
    const float2 ml = p.plan.ml[(size_t)pair * p.H + h];
    const float4 a = acc[((size_t)pair * p.H + h) * D4 + d4];
    if (i == 0) {
      f.first(ml.x, ml.y);
      A = a;
    } else {
      float ea, eb;
      f.next(ml.x, ml.y, ea, eb);
      A.x = fmaf(A.x, ea, a.x * eb);
      A.y = fmaf(A.y, ea, a.y * eb);
      A.z = fmaf(A.z, ea, a.z * eb);
      A.w = fmaf(A.w, ea, a.w * eb);
    }
  }
  const size_t o = ((size_t)row * p.H + h) * p.D + 4 * d4;
  const float r0 = finish_div(A.x, f.L), r1 = finish_div(A.y, f.L);
  const float r2 = finish_div(A.z, f.L), r3 = finish_div(A.w, f.L);
  if (p.elem_bytes == 4) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) = make_float4(r0, r1, r2, r3);
  } else {
    uint2 v;
    v.x = pack_bf16x2(r0, r1);
    v.y = pack_bf16x2(r2, r3);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + o) = v;
  }
}

}  // namespace

cudaError_t launch_combine(const StepParams& p, cudaStream_t s) {
  if (p.T <= 0) return cudaSuccess;
  const int D4 = p.D / 4;
  const int hpc = 128 / D4;
  dim3 grid(p.T, (p.H + hpc - 1) / hpc);
  combine_kernel<<<grid, 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
