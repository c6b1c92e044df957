// Split-KV partials for fp32 caches on the CUDA cores (plain FMA; no TF32,
// which "Numerics envelopes", The hierarchy, kernels.deterministic rules out).
//
// Same work decomposition as the bf16 decode kernel -- item = (row, split,
// kv head), one warp per item, the same split points -- but every row of the
// step takes this path, prefill rows included. Lanes of the warp own D / 32
// dims each; per key the g scores are full-warp butterfly sums (every lane
// ends with the same bits), then the running max, the rescale and the
// accumulation follow key by key in ascending order.
#include "pa_common.cuh"

namespace pa {

namespace {

constexpr int kWarps = 4;

template <int D, int GMAX>
__global__ void __launch_bounds__(kWarps * 32) split_f32_kernel(const StepParams p) {
  constexpr int DPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.H / p.Hkv;
  const long long n_items = (long long)p.plan.header[0] * p.Hkv;
  const int nfull = p.plan.header[1];
  const long long nw = (long long)gridDim.x * kWarps;
  const float* qg = static_cast<const float*>(p.q);
  const float* kc = static_cast<const float*>(p.k_cache);
  const float* vc = static_cast<const float*>(p.v_cache);

#pragma unroll 1
  for (long long item = (long long)blockIdx.x * kWarps + warp; item < n_items; item += nw) {
    const int k = (int)(item / p.Hkv);
    const int kvh = (int)(item - (long long)k * p.Hkv);
    const int pair = pair_slot(p.plan, k, nfull);
    const int4 pr = p.plan.pairs[pair];
    const int row = pr.x, lane_b = pr.z, keys = pr.w;
    const int sl = split_len(keys);
    const int t0 = pr.y * sl;
    const int t1 = min(t0 + sl, keys);
    const size_t head0 = (size_t)row * p.H + (size_t)kvh * g;

    float qv[GMAX][DPL], acc[GMAX][DPL], m[GMAX], l[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        qv[h][i] = h < g ? qg[(head0 + h) * D + lane + 32 * i] : 0.f;
        acc[h][i] = 0.f;
      }
    }
#pragma unroll 1
    for (int t = t0; t < t1; ++t) {
      int blk = p.block_tables[(size_t)lane_b * p.max_blocks + t / p.bs];
      if (blk < 0 || blk >= p.NB) {
        if (lane == 0) raise_flag(p.status, PA_FLAG_BLOCK_RANGE);
        blk = 0;
      }
      const size_t off = (((size_t)blk * p.bs + t % p.bs) * p.Hkv + kvh) * D;
      float kv[DPL], vv[DPL];
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        kv[i] = kc[off + lane + 32 * i];
        vv[i] = vc[off + lane + 32 * i];
      }
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (h < g) {
          float part = 0.f;
#pragma unroll
          for (int i = 0; i < DPL; ++i) part = fmaf(qv[h][i], kv[i], part);
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
          const float tt = part * p.scale_log2;
          const float mn = fmaxf(m[h], tt);
          const float al = ex2_approx(m[h] - mn);
          const float pp = ex2_approx(tt - mn);
          m[h] = mn;
          l[h] = fmaf(l[h], al, pp);
#pragma unroll
          for (int i = 0; i < DPL; ++i) acc[h][i] = fmaf(acc[h][i], al, pp * vv[i]);
        }
      }
    }
    float* out = static_cast<float*>(p.out);
    const bool single = keys <= sl && !p.partials_mode;
    const size_t ph0 = (size_t)partial_entry(p, pair, row, pr.y) * p.H + (size_t)kvh * g;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      if (h < g) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          if (single)
            out[(head0 + h) * D + lane + 32 * i] = finish_div(acc[h][i], l[h]);
          else
            st_hint(p.plan.acc + (ph0 + h) * D + lane + 32 * i, acc[h][i], l2_evict_last());
        }
        if (!single && lane == 0) st_hint(p.plan.ml + ph0 + h, make_float2(m[h], l[h]), l2_evict_last());
      }
    }
  }
}

template <int D>
cudaError_t launch_d(const StepParams& p, int grid, cudaStream_t s) {
  const int g = p.H / p.Hkv;
  if (g <= 4)
    split_f32_kernel<D, 4><<<grid, kWarps * 32, 0, s>>>(p);
  else if (g <= 8)
    split_f32_kernel<D, 8><<<grid, kWarps * 32, 0, s>>>(p);
  else
    split_f32_kernel<D, 16><<<grid, kWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

int num_sms();

cudaError_t launch_split_f32(const StepParams& p, long long max_items, cudaStream_t s) {
  long long want = (max_items + kWarps - 1) / kWarps;
  const long long cap = 8LL * num_sms();
  int grid = (int)(want < cap ? want : cap);
  if (grid < 1) grid = 1;
  return p.D == 128 ? launch_d<128>(p, grid, s) : launch_d<64>(p, grid, s);
}

}  // namespace pa
