// Split-KV decode partials, bf16 caches: the kernel of 4 independent warps
// per CTA (see pa_decode_bf16.cuh for the work itself) and its launcher.
#include "pa_decode_bf16.cuh"

namespace pa {

namespace {

constexpr int kWarps = 4;

template <int D, int NT, bool kOwner>
__global__ void __launch_bounds__(kWarps * 32, 2)
    decode_bf16_kernel(const StepParams p, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t dsmem[];
  decode_bf16_warps<D, NT, kOwner, kWarps>(p, &tmK, &tmV, dsmem);
}

template <int D, int NT, bool kOwner>
cudaError_t launch_o(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v, int grid,
                     cudaStream_t s) {
  auto kern = decode_bf16_kernel<D, NT, kOwner>;
  static unsigned long long done = 0;
  cudaError_t e = smem_opt_in(kern, DecTile<D>::smem_bytes(kWarps), &done);
  if (e != cudaSuccess) return e;
  kern<<<grid, kWarps * 32, DecTile<D>::smem_bytes(kWarps), s>>>(p, k, v);
  return cudaGetLastError();
}

// The KV-parallel owner variant (partials to canonical entries, never a
// direct write) is a separate instantiation so ordinary steps run the plain
// kernel; both share every line of the arithmetic.
template <int D, int NT>
cudaError_t launch_t(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v, int grid,
                     cudaStream_t s) {
  return p.partials_mode ? launch_o<D, NT, true>(p, k, v, grid, s)
                         : launch_o<D, NT, false>(p, k, v, grid, s);
}

}  // namespace

int num_sms();

// Upper bound on items -> grid of up to two CTAs per SM (each 4 independent warps).
cudaError_t launch_decode_bf16(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v,
                               long long max_items, cudaStream_t s) {
  long long want = (max_items + kWarps - 1) / kWarps;
  const long long cap = 2LL * num_sms();
  int grid = (int)(want < cap ? want : cap);
  if (grid < 1) grid = 1;
  const int g = p.H / p.Hkv;
  if (p.D == 128) return g <= 8 ? launch_t<128, 1>(p, k, v, grid, s) : launch_t<128, 2>(p, k, v, grid, s);
  return g <= 8 ? launch_t<64, 1>(p, k, v, grid, s) : launch_t<64, 2>(p, k, v, grid, s);
}

}  // namespace pa
