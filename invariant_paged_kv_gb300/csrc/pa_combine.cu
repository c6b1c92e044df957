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
// the same whatever else is in the step. The quotient is multiplied by
// out_scale (the V scale of e4m3 caches; 1, an exact no-op, otherwise).
//
// The split kernels store the partials with an evict-last L2 policy and read
// keys evict-first, so the partials are still in L2 here; once folded, an
// ordinary step's partials are dead, and the fold discards their L2 lines so
// they are never written back to HBM (the next step's split kernel then
// streams its keys without those write-backs).
#include <type_traits>

#include "pa_common.cuh"

namespace pa {

namespace {

constexpr int kWarps = 8;  // heads per CTA (one warp per (row, head))

// One warp folds the splits of one (row, head); lane l owns dims 4l .. 4l+3
// (D = 128) or 2l .. 2l+1 (D = 64). The loads of kAhead splits are issued
// before their fold so the memory system sees many requests at once; the fold
// itself runs strictly in split order, so kAhead changes no bit.
// info: the row's row_info (its lane is read only when merging owners).
template <int D, int kAhead>
__device__ __forceinline__ void fold_row_head(const StepParams& p, int row, int4 info, int h,
                                              int lane) {
  constexpr int VPL = D / 32;  // values per lane
  using Vec = typename std::conditional<VPL == 4, float4, float2>::type;
  if (info.w < 0) return;                                  // not on the split path
  if (p.partials_mode != 2 && info.z <= 1) return;         // written directly
  const int n = info.z;
  const int nfull = info.y >= 0 ? n - 1 : n;
  const Vec* acc = reinterpret_cast<const Vec*>(p.plan.acc);
  // merge of KV-parallel owners: split i comes from the owner whose key
  // range holds its first key; its entry is info.x + i in that owner's buffer
  const int sl = p.partials_mode == 2 ? split_len(info.y) : 0;
  auto owner_of = [&](int i) {
    int w = 0;
    const long long k0 = (long long)i * sl;
    while (w + 1 < p.owners && p.key_bounds[(size_t)(w + 1) * p.B + info.w] <= k0) ++w;
    return w;
  };

  if (p.partials_mode != 2 && n > 16 && n > kAhead) {
    // a long row: ask L2 for the partials of its later splits now, so the
    // batches after the first find them there (the fold order is unchanged)
    for (int i = kAhead + lane; i < n; i += 32) {
      const int pair = i < nfull ? info.x + i : info.y;
      const size_t e = (size_t)pair * p.H + h;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.plan.acc + e * D),
                   "r"((uint32_t)(D * sizeof(float)))
                   : "memory");
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.plan.ml + e) : "memory");
    }
  }
  Fold f;
  float A[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) A[j] = 0.f;
  for (int i0 = 0; i0 < n; i0 += kAhead) {
    float2 ml[kAhead];
    Vec a[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int i = i0 + u;
      if (i < n) {
        if (p.partials_mode == 2) {
          const long long e = (long long)info.x + i;
          const size_t off = (size_t)owner_of(i) * (size_t)p.owner_stride;
          const float2* mlw = reinterpret_cast<const float2*>(
              reinterpret_cast<const char*>(p.plan.ml) + off);
          const Vec* accw = reinterpret_cast<const Vec*>(
              reinterpret_cast<const char*>(p.plan.acc) + off);
          ml[u] = mlw[(size_t)e * p.H + h];
          a[u] = accw[((size_t)e * p.H + h) * 32 + lane];
        } else {
          const int pair = i < nfull ? info.x + i : info.y;
          ml[u] = p.plan.ml[(size_t)pair * p.H + h];
          a[u] = acc[((size_t)pair * p.H + h) * 32 + lane];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int i = i0 + u;
      if (i < n) {
        const float* av = reinterpret_cast<const float*>(&a[u]);
        if (i == 0) {
          f.first(ml[u].x, ml[u].y);
#pragma unroll
          for (int j = 0; j < VPL; ++j) A[j] = av[j];
        } else {
          float ea, eb;
          f.next(ml[u].x, ml[u].y, ea, eb);
#pragma unroll
          for (int j = 0; j < VPL; ++j) A[j] = fmaf(A[j], ea, av[j] * eb);
        }
      }
    }
  }
  const size_t o = ((size_t)row * p.H + h) * D + VPL * lane;
  float r[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) r[j] = finish_div(A[j], f.L) * p.out_scale;
  if (p.elem_bytes == 4) {
    float* out = static_cast<float*>(p.out) + o;
#pragma unroll
    for (int j = 0; j < VPL; ++j) out[j] = r[j];
  } else {
    uint32_t* out = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + o);
#pragma unroll
    for (int j = 0; j < VPL; j += 2) out[j / 2] = pack_bf16x2(r[j], r[j + 1]);
  }
  // an ordinary step's partials are dead once folded: drop their L2 lines
  // without writing them back (each (split, head) row of D floats is this
  // warp's alone, and every lane has used its loads)
  if (p.partials_mode == 0) {
    __syncwarp();
    constexpr int kLines = D * (int)sizeof(float) / 128;
    for (int i = lane / kLines; i < n; i += 32 / kLines) {
      const int pair = i < nfull ? info.x + i : info.y;
      const float* line = p.plan.acc + ((size_t)pair * p.H + h) * D + (lane % kLines) * (128 / sizeof(float));
      asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
    }
  }
}

// One CTA per (row of the plan's combine list, group of kWarps heads); CTAs
// past the list's length (the host sizes the grid by an upper bound) return
// at once, and the hardware hands out CTAs as SMs free up. kRowMajor: a 1-D
// grid ordered row by row over the list sorted by split count -- the head
// groups of a row are adjacent, so every long row starts in the first wave.
// Otherwise (prefill rows of a few splits each on the split path) a 2-D
// grid over the flat rows themselves, x the row and y the head group, which
// measured faster there.
template <int D, int kAhead, bool kRowMajor>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(const StepParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (kRowMajor) {
    const int hg_n = (p.H + kWarps - 1) / kWarps;
    const int k = blockIdx.x / hg_n, hg = blockIdx.x - k * hg_n;
    // the entry is read before the list's length is known (k < the grid's
    // row bound <= T entries, so in bounds; used only if k is listed): the
    // two loads travel together
    const int4 c = p.plan.crows[k];
    if (k >= p.plan.header[kHeaderCombineRows]) return;
    const int h = hg * kWarps + warp;
    if (h >= p.H) return;
    const int w = p.partials_mode == 2 ? p.plan.row_info[c.x].w : 0;
    fold_row_head<D, kAhead>(p, c.x, make_int4(c.y, c.z, c.w, w), h, lane);
  } else {
    // every flat row in order (no list: one dependent load less per CTA;
    // rows that need no fold return in fold_row_head); row_info is only
    // this call's when the plan is (the listed path needs no such test:
    // a refused plan lists no rows)
    if (!plan_ok(p)) return;
    const int h = blockIdx.y * kWarps + warp;
    if (h < p.H) fold_row_head<D, kAhead>(p, blockIdx.x, p.plan.row_info[blockIdx.x], h, lane);
  }
}

template <int D, int kAhead>
void launch_c(const StepParams& p, long long max_rows, bool row_order, cudaStream_t s) {
  const int hg_n = (p.H + kWarps - 1) / kWarps;
  if (max_rows <= 0) return;
  if (row_order)
    combine_kernel<D, kAhead, false><<<dim3((unsigned)max_rows, hg_n), kWarps * 32, 0, s>>>(p);
  else
    combine_kernel<D, kAhead, true><<<(unsigned)(max_rows * hg_n), kWarps * 32, 0, s>>>(p);
}

}  // namespace

// Load depth per warp against resident warps: decode rows with long split
// lists go faster with 8 splits in flight; when prefill rows take the split
// path (the row-invariant mode), most folded rows have a few splits and a
// depth of 2 goes faster: 32 registers a thread admit 8 CTAs per SM where
// depth 8 admits 3.
// Rows that can need a fold: when only decode lanes take the split path, at
// most one row per lane; otherwise every row. When prefill rows take the
// split path the grid walks the flat rows, else the plan's sorted list.
cudaError_t launch_combine(const StepParams& p, cudaStream_t s) {
  if (p.T <= 0) return cudaSuccess;
  const long long max_rows = (p.split_all_rows || p.partials_mode) ? p.T : (p.B < p.T ? p.B : p.T);
  const bool row_order = p.split_all_rows && p.max_q_len >= 2 && !p.partials_mode;
  const bool shallow = p.split_all_rows && p.max_q_len >= 2;
  if (p.D == 128) {
    if (shallow)
      launch_c<128, 2>(p, max_rows, row_order, s);
    else
      launch_c<128, 8>(p, max_rows, row_order, s);
  } else {
    if (shallow)
      launch_c<64, 2>(p, max_rows, row_order, s);
    else
      launch_c<64, 8>(p, max_rows, row_order, s);
  }
  return cudaGetLastError();
}

}  // namespace pa
