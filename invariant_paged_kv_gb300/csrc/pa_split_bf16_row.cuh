// The per-row arithmetic of the bf16 decode split kernel (one row per warp).
// The prefill-row kernel of the row-invariant mode repeats it column by
// column, operation for operation, so a row's bits are the same whichever of
// the two computes it.
//
// A row's state for one (split, kv head): the g query heads of the group on
// the N side of mma.sync (n tile nt holds heads 8 nt .. 8 nt + 7), this thread
// holding keys gid and gid + 8 of each 16-key chunk for heads 2 tig and
// 2 tig + 1: running max m and sum l per head (base-2 domain), O^T fragments
// (16 dims x 8 heads per m tile), and the q fragments (B operand of
// S^T = K Q^T).
#pragma once

#include "pa_common.cuh"

namespace pa {

// Shared address of 16-byte chunk c16 (0 .. D/8-1) of key row `tok` inside a
// 16-key tile written by TMA with 128-byte swizzle: one 2 KiB box per 64
// elements, chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t bf16_tile_addr(uint32_t base, int tok, int c16) {
  const int half = c16 >> 3, chunk = c16 & 7;
  return base + half * (kChunk * 128) + tok * 128 + ((chunk ^ (tok & 7)) << 4);
}

template <int D, int NT>
struct RowAcc {
  static constexpr int KS = D / 16;
  float m[NT][2], l[NT][2];
  float o[KS][NT][4];
  uint32_t qf[NT][KS][2];

  // q of `row`, heads kvh * g + (0 .. g-1); heads past g are zero columns
  __device__ __forceinline__ void init(const StepParams& p, int row, int kvh, int gid, int tig) {
    const int g = p.H / p.Hkv;
    const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(p.q);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hl = nt * 8 + gid;
      const bool hv = hl < g;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          qbase + ((size_t)row * p.H + (size_t)kvh * g + (hv ? hl : 0)) * D);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qf[nt][kk][0] = hv ? qrow[(kk * 16 + 2 * tig) >> 1] : 0u;
        qf[nt][kk][1] = hv ? qrow[(kk * 16 + 8 + 2 * tig) >> 1] : 0u;
      }
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    }
  }

  // Online softmax over one 16-key chunk whose scores are s (accumulator
  // layout of S^T, keys gid / gid + 8), nvalid keys of it real: running max,
  // p = 2^(t - m) rounded to bf16, l from the rounded p, O rescaled; returns
  // P^T moved to the B-operand layout (k = keys, n = heads) for O^T += V^T P^T.
  __device__ __forceinline__ void softmax(const float (&s)[NT][4], int nvalid, int gid,
                                          float scale_log2, uint32_t (&pbt)[NT][2]) {
    const bool va = gid < nvalid, vb = gid + 8 < nvalid;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float pa[2], pc[2], alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float ta = va ? __fmul_rn(s[nt][e], scale_log2) : -INFINITY;
        const float tb = vb ? __fmul_rn(s[nt][2 + e], scale_log2) : -INFINITY;
        float mx = fmaxf(ta, tb);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m[nt][e], mx);
        alpha[e] = ex2_approx(m[nt][e] - mn);
        m[nt][e] = mn;
        pa[e] = ex2_approx(ta - mn);
        pc[e] = ex2_approx(tb - mn);
      }
      const uint32_t pb0 = pack_bf16x2(pa[0], pa[1]);  // key gid,     heads 2tig, 2tig+1
      const uint32_t pb1 = pack_bf16x2(pc[0], pc[1]);  // key gid + 8, heads 2tig, 2tig+1
      l[nt][0] = fmaf(l[nt][0], alpha[0], bf16_lo(pb0) + bf16_lo(pb1));
      l[nt][1] = fmaf(l[nt][1], alpha[1], bf16_hi(pb0) + bf16_hi(pb1));
      // o * 1 == o exactly: the rescale is skipped when no head's max moved
      if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[mt][nt][0] *= alpha[0];
          o[mt][nt][1] *= alpha[1];
          o[mt][nt][2] *= alpha[0];
          o[mt][nt][3] *= alpha[1];
        }
      }
      pbt[nt][0] = movmatrix_trans(pb0);
      pbt[nt][1] = movmatrix_trans(pb1);
    }
  }

  // After the split's last chunk: l summed over the warp's key lanes, then
  // either the normalised output (a row with one split) or the partial
  // (m, l, acc) at entry `entry` of the plan's ml / acc.
  __device__ __forceinline__ void finish(const StepParams& p, int row, int kvh, bool single,
                                         long long entry, int gid, int tig) {
    const int g = p.H / p.Hkv;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l[nt][e];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        l[nt][e] = v;
      }
    }
    const size_t head0 = (size_t)row * p.H + (size_t)kvh * g;  // first head of the group
    if (single) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int hl = nt * 8 + 2 * tig + (r & 1);
          if (hl < g) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              const int d = mt * 16 + gid + (r >> 1) * 8;
              out[(head0 + hl) * D + d] = __float2bfloat16_rn(finish_div(o[mt][nt][r], l[nt][r & 1]));
            }
          }
        }
    } else {
      const size_t ph0 = (size_t)entry * p.H + (size_t)kvh * g;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int hl = nt * 8 + 2 * tig + (r & 1);
          if (hl < g) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              const int d = mt * 16 + gid + (r >> 1) * 8;
              // kept in L2 for the combine, which reads them soon after
              st_hint(p.plan.acc + (ph0 + hl) * D + d, o[mt][nt][r], l2_evict_last());
            }
          }
        }
      if (gid == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int hl = nt * 8 + 2 * tig + e;
            if (hl < g) st_hint(p.plan.ml + ph0 + hl, make_float2(m[nt][e], l[nt][e]), l2_evict_last());
          }
      }
    }
  }
};

}  // namespace pa
