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
// ring that 8 consumer warps read. Consumer warp w carries RPW adjacent rows
// (RPW = 2 when the GQA group fits one mma N tile, else 1), each with exactly
// the decode kernel's per-row code (RowAcc: the same S^T and O^T products over
// the same 16-key chunks in the same order, the same online softmax, the same
// finish); the rows of a warp share the K / V fragments of a chunk and give
// the warp independent mma chains. A row never touches a chunk past its own
// key count (it skips the rest of the group's chunks), so its bits are those
// it would have as a decode row. Every wait is bounded (PA_FLAG_TIMEOUT).
#include "pa_split_bf16_row.cuh"

namespace pa {

namespace {

constexpr int kRW = kRowWarps;  // consumer warps
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

// One 16-key chunk for rows FIRST .. RPW-1 of the warp (the rows still inside
// their key range; the later a row, the more keys it has): the K fragments
// feed every row's S^T chain, the V fragments every row's O^T update.
template <int D, int NT, int RPW, int FIRST>
__device__ __forceinline__ void chunk_rows(RowAcc<D, NT> (&ra)[RPW], const int (&nvalid)[RPW],
                                           uint32_t ks, uint32_t vs, int lane, int gid,
                                           float scale_log2) {
  constexpr int KS = D / 16;
  // S^T = K Q^T : 16 keys x 8 heads per n tile
  float s[RPW][NT][4];
#pragma unroll
  for (int i = FIRST; i < RPW; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[i][nt][0] = s[i][nt][1] = s[i][nt][2] = s[i][nt][3] = 0.f;
  {
    const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(bf16_tile_addr(ks, tok, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
      for (int i = FIRST; i < RPW; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_bf16_16816(s[i][nt], a0, a1, a2, a3, ra[i].qf[nt][kk][0], ra[i].qf[nt][kk][1]);
    }
  }
  uint32_t pbt[RPW][NT][2];
#pragma unroll
  for (int i = FIRST; i < RPW; ++i) ra[i].softmax(s[i], nvalid[i], gid, scale_log2, pbt[i]);
  // O^T += V^T P^T : 16 dims x 8 heads per (m tile, n tile)
  {
    const int tok = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(bf16_tile_addr(vs, tok, mt * 2 + ((lane >> 3) & 1)), a0, a1, a2, a3);
#pragma unroll
      for (int i = FIRST; i < RPW; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_bf16_16816(ra[i].o[mt][nt], a0, a1, a2, a3, pbt[i][nt][0], pbt[i][nt][1]);
    }
  }
}

template <int D, int NT, int RPW>
__global__ void __launch_bounds__(kRThreads, 1)
    rows_bf16_kernel(const StepParams p, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
  using TL = RTile<D>;
  static_assert(RPW == 1 || RPW == 2, "rows per warp");
  extern __shared__ uint8_t dsmem[];
  // zeroed[st]: warp 0 has zeroed the V rows past the group's keys in stage
  // st (a group's last, partial chunk); one phase per such use of the stage,
  // and the stage is reused only after every consumer released it, so a
  // waiter never meets the barrier more than one phase away
  __shared__ __align__(8) uint64_t full[kRStages], empty[kRStages], zeroed[kRStages];
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kRW);
      mbar_init(smem_u32(&zeroed[i]), 1);
    }
    s_abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();

  const int n_items = p.plan.header[3] * p.Hkv;
  uint32_t f = 0;      // running chunk counter, identical in every role
  uint32_t zbits = 0;  // consumers: parity of zeroed[st] uses, bit st

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const Group gr = group_at(p, item / p.Hkv);
    const int kvh = item % p.Hkv;
    const int sl = split_len(gr.keys0);
    const int t0 = gr.split * sl;
    const int len_max = min(sl, gr.keys0 + gr.nrows - 1 - t0);  // the last row's share
    const int nch = (len_max + kChunk - 1) / kChunk;

    if (warp == kRW) {
      // ------------------------------ producer ------------------------------
      if (lane == 0) {
        for (int ch = 0; ch < nch; ++ch, ++f) {
          const uint32_t st = f % kRStages;
          if (f >= kRStages &&
              !wait_r(smem_u32(&empty[st]), ((f / kRStages) - 1) & 1, &s_abort, p.status))
            break;
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
            tma_load_3d(ks + h * TL::kHalfBytes, &tmK, h * 64, kvh, tok, smem_u32(&full[st]));
            tma_load_3d(vs + h * TL::kHalfBytes, &tmV, h * 64, kvh, tok, smem_u32(&full[st]));
          }
        }
      }
      f = __shfl_sync(0xffffffffu, f, 0);
    } else {
      // ------------------------- consumer: RPW rows -------------------------
      RowAcc<D, NT> ra[RPW];
      int len[RPW], my_nch[RPW];
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        const int j = warp * RPW + i;  // row of the group
        len[i] = (j < gr.nrows) ? min(sl, gr.keys0 + j - t0) : 0;  // <= 0: no such split
        my_nch[i] = len[i] > 0 ? (len[i] + kChunk - 1) / kChunk : 0;
        if (my_nch[i] > 0) ra[i].init(p, gr.r0 + j, kvh, gid, tig);
      }
      bool ok = true;
      for (int ch = 0; ch < nch; ++ch, ++f) {
        const uint32_t st = f % kRStages;
        if (!__all_sync(0xffffffffu, wait_r(smem_u32(&full[st]), (f / kRStages) & 1, &s_abort,
                                            p.status))) {
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
                                                     &s_abort, p.status))) {
            ok = false;
            break;
          }
          zbits ^= 1u << st;
        }
        int nvalid[RPW];
#pragma unroll
        for (int i = 0; i < RPW; ++i) nvalid[i] = min(kChunk, len[i] - ch * kChunk);
        // the rows inside their key range at this chunk form a suffix of the
        // warp's rows (my_nch grows with the row)
        if (ch < my_nch[0]) {
          chunk_rows<D, NT, RPW, 0>(ra, nvalid, ks, vs, lane, gid, p.scale_log2);
        } else if (RPW == 2 && ch < my_nch[RPW - 1]) {
          chunk_rows<D, NT, RPW, RPW - 1>(ra, nvalid, ks, vs, lane, gid, p.scale_log2);
        }
        __syncwarp();  // every lane is done reading this stage
        if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
      }
      if (ok) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          if (my_nch[i] > 0) {
            const int r = gr.r0 + warp * RPW + i;
            const int keys = gr.keys0 + warp * RPW + i;
            const int n = (keys + sl - 1) / sl;  // this row's splits
            ra[i].finish(p, r, kvh, n == 1, (long long)p.plan.row_info[r].x + gr.split, gid, tig);
          }
        }
      }
    }
    if (s_abort) break;
  }
  // copies this CTA started land before it leaves
  if (warp == kRW && lane == 0) {
    for (uint32_t j = f > kRStages ? f - kRStages : 0; j < f; ++j) {
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(&full[j % kRStages]), (j / kRStages) & 1))
        if (clock64() - t0 > kWaitCycles) break;
    }
  }
}

template <int D, int NT, int RPW>
cudaError_t launch_r(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v, int grid,
                     cudaStream_t s) {
  auto kern = rows_bf16_kernel<D, NT, RPW>;
  static unsigned long long done = 0;
  cudaError_t e = smem_opt_in(kern, RTile<D>::kSmemBytes, &done);
  if (e != cudaSuccess) return e;
  kern<<<grid, kRThreads, RTile<D>::kSmemBytes, s>>>(p, k, v);
  return cudaGetLastError();
}

}  // namespace

int num_sms();

// Rows per group for a GQA group of g heads: two rows per consumer warp when
// the group fits one mma N tile (g <= 8), else one.
int rows_group_size(int g) { return kRW * (g <= 8 ? 2 : 1); }

// max_items: an upper bound on (group, split, kv head) items of the step.
cudaError_t launch_rows_bf16(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v,
                             long long max_items, cudaStream_t s) {
  long long cap = num_sms();
  int grid = (int)(max_items < cap ? max_items : cap);
  if (grid < 1) grid = 1;
  const int g = p.H / p.Hkv;
  if (p.group_rows != rows_group_size(g)) return cudaErrorInvalidValue;
  if (p.D == 128) return g <= 8 ? launch_r<128, 1, 2>(p, k, v, grid, s) : launch_r<128, 2, 1>(p, k, v, grid, s);
  return g <= 8 ? launch_r<64, 1, 2>(p, k, v, grid, s) : launch_r<64, 2, 1>(p, k, v, grid, s);
}

}  // namespace pa
