// Prefill rows of the row-invariant mode, bf16 caches ("Numerics envelopes",
// Prefix hits resume at any token: a query row depends only on the K/V rows it
// attends, so chunking must not change its bits).
//
// In that mode every row takes the split path with the split partition of its
// own key count. The rows of a prefill lane share their keys, so instead of
// one warp per (row, split) streaming the split privately -- the decode
// kernel's item -- a CTA takes a group of consecutive rows of one lane with
// the same split length, one split and one kv head: a producer warp streams
// the split's 16-key K / V tiles once (TMA, 128-byte swizzle) into an 8-stage
// ring that 8 consumer warps read.
//
// The decode kernel puts the g query heads of one row on the N side of its
// mma.sync products (S^T = K Q^T, O^T = V^T P^T), one column per head, and
// pads a short group with empty columns. Every output column of those
// products, and every step of the online softmax (a max and a sum over keys,
// per column), depends on its own column alone. So here the columns are
// (row, head) pairs packed densely across rows: column k of the group is row
// k / g, head k % g, and warp w owns columns 16 w .. 16 w + 15 (two N tiles).
// Each column goes through exactly the decode kernel's sequence of
// operations -- the same 16-key chunks in the same order, the same products,
// the same max / exp2 / bf16 rounding / sum / rescale, the same finish -- so
// its bits are those of its row computed as a decode row. A column whose row
// has no keys left in a chunk skips the chunk's update (its max, sum and
// rescale factor stay as they are, its p values are zero).
// Every wait is bounded (PA_FLAG_TIMEOUT).
//
// The work is written as the code of one CTA (rows_bf16_cta): it runs as the
// prefill-row role of the row-mode mixed kernel (pa_mixed.cu), which gives
// every CTA this role when a step has no decode rows.
#pragma once

#include "pa_split_bf16_row.cuh"

namespace pa {
namespace rows {


constexpr int kRW = kRowWarps;  // consumer warps
constexpr int kNTW = 2;         // 8-column N tiles per consumer warp
constexpr int kCols = kRW * kNTW * 8;
constexpr int kRStages = 8;
constexpr int kRThreads = (kRW + 1) * 32;

template <int D>
struct RTile {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kChunk * 128;  // one 16-key x 64-element box
  static constexpr int kBytes = kChunk * D * 2;    // one K (or V) chunk
  static constexpr int kStageBytes = 2 * kBytes;
  static constexpr int kSmemBytes = kRStages * kStageBytes + 1024;
};

struct Group {
  int r0, nrows, split, lane, keys0;
};

__device__ __forceinline__ Group group_at(const StepParams& p, int k) {
  const int4 e = p.plan.pairs[p.plan.header[1] + k];
  Group gr;
  gr.r0 = e.x;
  gr.nrows = e.y & 255;
  gr.split = e.y >> 8;
  gr.lane = e.z;
  gr.keys0 = e.w;
  return gr;
}

__device__ __forceinline__ bool wait_r(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int* status, long long limit) {
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

// The state of one warp's 16 columns for one (group, split, kv head). This
// thread holds keys gid and gid + 8 of each chunk for columns 2 tig and
// 2 tig + 1 of each N tile (index e), and the q fragment of column gid.
template <int D>
struct ColAcc {
  static constexpr int KS = D / 16;
  float m[kNTW][2], l[kNTW][2];
  float o[KS][kNTW][4];
  uint32_t qf[kNTW][KS][2];

  __device__ __forceinline__ void init(const StepParams& p, const Group& gr, int kvh, int col0,
                                       int g, int gid, int tig) {
    const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(p.q);
#pragma unroll
    for (int nt = 0; nt < kNTW; ++nt) {
      const int c = col0 + nt * 8 + gid;
      const int j = c / g, h = c - j * g;
      const bool cv = j < gr.nrows;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          qbase + ((size_t)(gr.r0 + (cv ? j : 0)) * p.H + (size_t)kvh * g + (cv ? h : 0)) * D);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qf[nt][kk][0] = cv ? qrow[(kk * 16 + 2 * tig) >> 1] : 0u;
        qf[nt][kk][1] = cv ? qrow[(kk * 16 + 8 + 2 * tig) >> 1] : 0u;
      }
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    }
  }

  // One chunk: s in the accumulator layout of S^T (keys gid / gid + 8),
  // nvalid[nt][e] keys of it real for column (nt, e) (<= 0: the column sits
  // the chunk out). For a column that takes part, the same operations in the
  // same order as the decode kernel's row.
  __device__ __forceinline__ void softmax(const float (&s)[kNTW][4], const int (&nvalid)[kNTW][2],
                                          int gid, float scale_log2,
                                          uint32_t (&pbt)[kNTW][2]) {
#pragma unroll
    for (int nt = 0; nt < kNTW; ++nt) {
      float pa[2], pc[2], alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool va = gid < nvalid[nt][e], vb = gid + 8 < nvalid[nt][e];
        const float ta = va ? __fmul_rn(s[nt][e], scale_log2) : -INFINITY;
        const float tb = vb ? __fmul_rn(s[nt][2 + e], scale_log2) : -INFINITY;
        float mx = fmaxf(ta, tb);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const bool act = nvalid[nt][e] > 0;
        const float mn = act ? fmaxf(m[nt][e], mx) : m[nt][e];
        alpha[e] = act ? ex2_approx(m[nt][e] - mn) : 1.f;
        m[nt][e] = mn;
        pa[e] = act ? ex2_approx(ta - mn) : 0.f;
        pc[e] = act ? ex2_approx(tb - mn) : 0.f;
      }
      const uint32_t pb0 = pack_bf16x2(pa[0], pa[1]);  // key gid,     columns 2tig, 2tig+1
      const uint32_t pb1 = pack_bf16x2(pc[0], pc[1]);  // key gid + 8, columns 2tig, 2tig+1
      // l * 1 + 0 == l: a column sitting out keeps its sum
      l[nt][0] = fmaf(l[nt][0], alpha[0], bf16_lo(pb0) + bf16_lo(pb1));
      l[nt][1] = fmaf(l[nt][1], alpha[1], bf16_hi(pb0) + bf16_hi(pb1));
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
};

// The work of one CTA of kRThreads threads (see above); dsmem holds
// RTile<D>::kSmemBytes bytes.
template <int D>
__device__ __forceinline__ void rows_bf16_cta(const StepParams& p, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, uint8_t* dsmem) {
  using TL = RTile<D>;
  constexpr int KS = D / 16;
  // zeroed[st]: warp 0 has zeroed the V rows past the group's keys in stage
  // st (a group's last, partial chunk); one phase per such use of the stage,
  // and the stage is reused only after every consumer released it, so a
  // waiter never meets the barrier more than one phase away
  __shared__ __align__(8) uint64_t full[kRStages], empty[kRStages], zeroed[kRStages];
  __shared__ volatile int s_abort;
  // The producer takes items from the prefill-row item counter in list order
  // and writes the CTA's k-th into s_q[k % kQueue] before it starts the
  // item's first chunk; consumers read it once that chunk's full barrier has
  // completed (release by the producer's arrive, acquire by the wait). An
  // index past the end goes out the same way with a plain arrive and no
  // copy: the consumers' stop token. The producer runs at most kRStages
  // chunks -- so at most kRStages items -- ahead.
  constexpr int kQueue = 2 * kRStages;
  __shared__ long long s_q[kQueue];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int g = p.H / p.Hkv;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kRW);
      mbar_init(smem_u32(&zeroed[i]), 1);
    }
    s_abort = 0;
    fence_mbar_init();
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
  }
  __syncthreads();

  const long long n_items = (long long)p.plan.header[3] * p.Hkv;
  uint32_t f = 0;      // running chunk counter, identical in every role
  uint32_t zbits = 0;  // consumers: parity of zeroed[st] uses, bit st

  if (warp == kRW) {
    // -------------------------------- producer --------------------------------
    if (lane == 0) {
      bool ok = true;
      for (long long k = 0; ok; ++k) {
        const long long item = (long long)atomicAdd(item_counter(p.plan, kCounterRows), 1ull);
        const bool stop = item >= n_items;
        Group gr{};
        int kvh = 0, t0 = 0, nch = 1;
        if (!stop) {
          gr = group_at(p, (int)(item / p.Hkv));
          kvh = (int)(item % p.Hkv);
          const int sl = split_len(gr.keys0);
          t0 = gr.split * sl;
          const int len_max = min(sl, gr.keys0 + gr.nrows - 1 - t0);  // the last row's share
          nch = (len_max + kChunk - 1) / kChunk;
        }
        for (int ch = 0; ch < nch; ++ch, ++f) {
          const uint32_t st = f % kRStages;
          if (f >= kRStages &&
              !wait_r(smem_u32(&empty[st]), ((f / kRStages) - 1) & 1, &s_abort, p.status, p.wait_cycles)) {
            ok = false;
            break;
          }
          if (ch == 0) s_q[k % kQueue] = item;
          if (stop) {
            mbar_arrive(smem_u32(&full[st]));
            ++f;
            ok = false;  // done
            break;
          }
          const int key = t0 + ch * kChunk;
          int blk = p.block_tables[(size_t)gr.lane * p.max_blocks + key / p.bs];
          if (blk < 0 || blk >= p.NB) {
            raise_flag(p.status, PA_FLAG_BLOCK_RANGE);
            blk = 0;
          }
          const int tok = blk * p.bs + key % p.bs;
          const uint32_t ks = base + st * TL::kStageBytes, vs = ks + TL::kBytes;
          mbar_expect_tx(smem_u32(&full[st]), TL::kStageBytes);
#pragma unroll
          for (int h = 0; h < TL::kHalves; ++h) {
            tma_load_3d(ks + h * TL::kHalfBytes, tmK, h * 64, kvh, tok, smem_u32(&full[st]));
            tma_load_3d(vs + h * TL::kHalfBytes, tmV, h * 64, kvh, tok, smem_u32(&full[st]));
          }
        }
      }
    }
  } else {
    // ---------------------- consumer: 16 (row, head) columns ----------------
    const int col0 = warp * (kNTW * 8);
    for (long long k = 0;; ++k) {
      // the stage of the item's first chunk (or of the stop token)
      if (!__all_sync(0xffffffffu, wait_r(smem_u32(&full[f % kRStages]), (f / kRStages) & 1,
                                          &s_abort, p.status, p.wait_cycles)))
        break;
      const long long item = s_q[k % kQueue];
      if (item >= n_items) break;
      const Group gr = group_at(p, (int)(item / p.Hkv));
      const int kvh = (int)(item % p.Hkv);
      const int sl = split_len(gr.keys0);
      const int t0 = gr.split * sl;
      const int len_max = min(sl, gr.keys0 + gr.nrows - 1 - t0);  // the last row's share
      const int nch = (len_max + kChunk - 1) / kChunk;
      // keys of this split for the columns this thread holds in the softmax
      // layout (<= 0: the column's row lacks the split, or no such row)
      int len[kNTW][2];
      int len_w = 0;
#pragma unroll
      for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = (col0 + nt * 8 + 2 * tig + e) / g;
          len[nt][e] = j < gr.nrows ? min(sl, gr.keys0 + j - t0) : 0;
          len_w = max(len_w, len[nt][e]);
        }
      len_w = __reduce_max_sync(0xffffffffu, len_w);
      const int nch_w = (len_w + kChunk - 1) / kChunk;  // chunks any column of the warp needs
      ColAcc<D> ca;
      if (nch_w > 0) ca.init(p, gr, kvh, col0, g, gid, tig);
      bool ok = true;
      for (int ch = 0; ch < nch; ++ch, ++f) {
        const uint32_t st = f % kRStages;
        if (ch > 0 && !__all_sync(0xffffffffu, wait_r(smem_u32(&full[st]), (f / kRStages) & 1,
                                                      &s_abort, p.status, p.wait_cycles))) {
          ok = false;
          break;
        }
        const uint32_t ks = base + st * TL::kStageBytes, vs = ks + TL::kBytes;
        const int nvalid_max = min(kChunk, len_max - ch * kChunk);
        if (nvalid_max < kChunk) {
          // keys past the group's last row: zero their V rows (stale bytes
          // must not meet p = 0 as 0 * NaN); warp 0 writes, the others wait
          if (warp == 0) {
            const int nz = (kChunk - nvalid_max) * TL::kHalves * 8;
            for (int i = lane; i < nz; i += 32) {
              const int c16 = i & 7, rest = i >> 3;
              const int half = rest % TL::kHalves, tok = nvalid_max + rest / TL::kHalves;
              const uint32_t a = vs + half * TL::kHalfBytes + tok * 128 + c16 * 16;
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&zeroed[st]));
          } else if (!__all_sync(0xffffffffu, wait_r(smem_u32(&zeroed[st]), (zbits >> st) & 1,
                                                     &s_abort, p.status, p.wait_cycles))) {
            ok = false;
            break;
          }
          zbits ^= 1u << st;
        }
        if (ch < nch_w) {
          // S^T = K Q^T : 16 keys x 8 columns per N tile
          float s[kNTW][4];
#pragma unroll
          for (int nt = 0; nt < kNTW; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
          {
            const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(bf16_tile_addr(ks, tok, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < kNTW; ++nt)
                mma_bf16_16816(s[nt], a0, a1, a2, a3, ca.qf[nt][kk][0], ca.qf[nt][kk][1]);
            }
          }
          int nvalid[kNTW][2];
#pragma unroll
          for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) nvalid[nt][e] = min(kChunk, len[nt][e] - ch * kChunk);
          uint32_t pbt[kNTW][2];
          ca.softmax(s, nvalid, gid, p.scale_log2, pbt);
          // O^T += V^T P^T : 16 dims x 8 columns per (m tile, N tile)
          {
            const int tok = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4_trans(bf16_tile_addr(vs, tok, mt * 2 + ((lane >> 3) & 1)), a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < kNTW; ++nt)
                mma_bf16_16816(ca.o[mt][nt], a0, a1, a2, a3, pbt[nt][0], pbt[nt][1]);
            }
          }
        }
        __syncwarp();  // every lane is done reading this stage
        if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
      }
      if (ok && nch_w > 0) {
        // finish: l summed over the warp's key lanes, then per column either
        // the normalised output (a row with one split) or the partial
#pragma unroll
        for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float v = ca.l[nt][e];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            ca.l[nt][e] = v;
          }
#pragma unroll
        for (int nt = 0; nt < kNTW; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            if (len[nt][e] <= 0) continue;
            const int c = col0 + nt * 8 + 2 * tig + e;
            const int j = c / g, h = c - j * g;
            const int r = gr.r0 + j;
            const int keys = gr.keys0 + j;
            const size_t head = (size_t)r * p.H + (size_t)kvh * g + h;
            if ((keys + sl - 1) / sl == 1) {  // one split: the output itself
              __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
              for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                  const int d = mt * 16 + gid + hi * 8;
                  out[head * D + d] = __float2bfloat16_rn(finish_div(ca.o[mt][nt][hi * 2 + e], ca.l[nt][e]));
                }
            } else {
              const size_t ph = ((size_t)p.plan.row_info[r].x + gr.split) * p.H +
                                (size_t)kvh * g + h;
#pragma unroll
              for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                  const int d = mt * 16 + gid + hi * 8;
                  p.plan.acc[ph * D + d] = ca.o[mt][nt][hi * 2 + e];
                }
              if (gid == 0) p.plan.ml[ph] = make_float2(ca.m[nt][e], ca.l[nt][e]);
            }
          }
      }
      if (!ok) break;
    }
  }
  // copies this CTA started land before it leaves
  if (warp == kRW && lane == 0) {
    for (uint32_t j = f > kRStages ? f - kRStages : 0; j < f; ++j) {
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&full[j % kRStages]), (j / kRStages) & 1))
        if (clock64() - t0 > p.wait_cycles) break;
    }
  }
}

}  // namespace rows
}  // namespace pa
