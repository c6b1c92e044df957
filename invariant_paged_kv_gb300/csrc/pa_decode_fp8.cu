// Split-KV partials for e4m3 caches with per-tensor scales ("P3: native
// paged-KV continuous-batching sampler", Review (adversarial pass), kv_dtype:
// K/V dequantised on read; fp8 KV needs per-tensor scales).
//
// Same work decomposition and schedule as the bf16 split kernel -- item =
// (row, split, kv head) taken from the item counter in list order, one warp
// per item, chunks of keys through a private
// ring of TMA-filled shared-memory stages, online softmax in ascending key
// order -- with three differences:
//  * a chunk is 32 keys of 1-byte codes (the bytes of a 16-key bf16 chunk):
//    its two 16-key halves give two independent S^T products per k step, and
//    the running max, the rescale and the stage wait happen once per 32 keys;
//  * the products run in f16: one cvt turns two codes into two f16 values
//    exactly, and q is carried in f16 after an exact power-of-two prescale
//    2^-k that brings the item's largest |q| below 2^15 (k is folded back
//    into the score scale, so the scores are those of the unscaled q);
//    the softmax weights are rounded to f16 for the second product;
//  * the scales are applied outside the products: the score scale carries
//    k_scale and every normalised output is multiplied by v_scale.
// Register fragments are built straight from the code tiles: for S^T = K Q^T
// the 16 dims of a k step are a fixed permutation of the head dims (the same
// one on the q side), and for O^T = V^T P^T the 16 dims of an m tile are a
// fixed permutation of the output dims (undone when the result is stored),
// so every thread reads whole 16-byte runs of a key row. A row's arithmetic
// depends only on its own q and keys.
#include "pa_split_items.cuh"

namespace pa {

namespace {

constexpr int kWarps = 4;
constexpr int kStages = 2;  // x 8 KB per warp; 3 CTAs per SM
constexpr int kKeys = 2 * kChunk;  // keys per stage: two 16-key mma tiles

template <int D>
struct Tile8 {
  static constexpr int kBytes = kKeys * D;            // one K (or V) chunk of codes
  static constexpr int kStageBytes = 2 * kBytes;      // K + V
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kWarps * kWarpBytes + 1024;  // + alignment slack
  static constexpr int kBPT = D / 8;                  // V bytes one thread reads per key
};

// Swizzled shared offset of logical byte offset `off` in a tile written by
// TMA: 128-byte swizzle for D = 128 (16-byte chunk index ^= line index mod 8),
// 64-byte swizzle for D = 64 (chunk bits 4-5 ^= bits 7-8).
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  if (D == 128) return off ^ (((off >> 7) & 7u) << 4);
  return off ^ (((off >> 7) & 3u) << 4);
}

template <int D, int NT, bool kOwner>
__global__ void __launch_bounds__(kWarps * 32, 3)
    decode_fp8_kernel(const StepParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using TL = Tile8<D>;
  constexpr int KS = D / 16;   // k steps of S^T (and m tiles of O^T)
  constexpr int SEG = D / 64;  // 16-byte K runs a thread reads per key row
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  __shared__ long long s_items[kWarps][kItemSlots];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t wbase = base + warp * TL::kWarpBytes;
  uint32_t bar[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) bar[s] = smem_u32(&bars[warp][s]);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(bar[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncwarp();

  const int g = p.H / p.Hkv;
  const long long n_items = (long long)p.plan.header[0] * p.Hkv;
  const int nfull = p.plan.header[1];
  static_assert(kStages < kItemSlots, "item slots");
  long long* const wq = s_items[warp];

  // ---- producer cursor: runs up to kStages chunks ahead of the consumer ----
  long long p_k = 0;
  long long p_item = take_item(p, lane);
  if (lane == 0) wq[0] = p_item;
  int p_chunk = 0, p_w0 = 0;
  Item pi;
  int p_blk = 0;
  if (p_item < n_items) {
    pi = load_item(p, p_item, nfull);
    p_blk = load_blocks(p, pi, 0, lane);
  }
  uint32_t issued = 0;
  auto nchunks_of = [](const Item& x) { return (x.len + kKeys - 1) / kKeys; };
  auto produce = [&]() {
    if (p_item >= n_items) return;
    const int stage = issued % kStages;
    const int off = p_chunk * kKeys;  // key offset inside the split (a multiple of 32)
    if (off / p.bs - p_w0 >= 32) {    // next window of block ids
      p_w0 += 32;
      p_blk = load_blocks(p, pi, p_w0, lane);
    }
    // the two 16-key boxes of the chunk (one block for bs = 32, two for
    // bs = 16; off / bs is even then, so both stay inside the window)
    int blk[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) blk[h] = __shfl_sync(0xffffffffu, p_blk, (off + h * kChunk) / p.bs - p_w0);
    if (lane == 0) {
      const uint32_t ks = wbase + stage * TL::kStageBytes;
      mbar_expect_tx(bar[stage], TL::kStageBytes);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        int b = blk[h];
        if (b < 0 || b >= p.NB) {
          raise_flag(p.status, PA_FLAG_BLOCK_RANGE);
          b = 0;
        }
        const int tok = b * p.bs + (pi.t0 + off + h * kChunk) % p.bs;
        tma_load_3d(ks + h * kChunk * D, &tmK, 0, pi.kvh, tok, bar[stage]);
        tma_load_3d(ks + TL::kBytes + h * kChunk * D, &tmV, 0, pi.kvh, tok, bar[stage]);
      }
    }
    ++issued;
    if (++p_chunk == nchunks_of(pi)) {
      p_chunk = 0;
      p_w0 = 0;
      p_item = take_item(p, lane);
      if (lane == 0) wq[++p_k & (kItemSlots - 1)] = p_item;
      if (p_item < n_items) {
        pi = load_item(p, p_item, nfull);
        p_blk = load_blocks(p, pi, 0, lane);
      }
    }
  };
#pragma unroll 1
  for (int s = 0; s < kStages; ++s) produce();

  uint32_t consumed = 0;
  const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(p.q);

#pragma unroll 1
  for (long long c_k = 0;; ++c_k) {
    __syncwarp();
    const long long c_item = wq[c_k & (kItemSlots - 1)];
    if (c_item >= n_items) break;
    const Item it = load_item(p, c_item, nfull);

    // q of the group's heads, k step kk = 4 s + j: this thread's four dims
    // 64 s + 16 tig + 4 j + {0, 1, 2, 3} (B operand rows 2tig, 2tig+1,
    // 2tig+8, 2tig+9 of the step)
    float qv[NT][KS][4];
    float amax = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int hl = nt * 8 + gid;
      const bool hv = hl < g;
      const __nv_bfloat16* qrow =
          qbase + ((size_t)it.row * p.H + (size_t)it.kvh * g + (hv ? hl : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const int d0 = 64 * (kk >> 2) + 16 * tig + 4 * (kk & 3);
        uint2 w = hv ? *reinterpret_cast<const uint2*>(qrow + d0) : make_uint2(0u, 0u);
        qv[nt][kk][0] = bf16_lo(w.x);
        qv[nt][kk][1] = bf16_hi(w.x);
        qv[nt][kk][2] = bf16_lo(w.y);
        qv[nt][kk][3] = bf16_hi(w.y);
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qv[nt][kk][e]));
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // 2^-k brings amax below 2^15 (f16 holds up to 65504); the score scale
    // takes 2^k back, exactly
    const int ebits = (int)((__float_as_uint(amax) >> 23) & 0xffu);
    const int kx = max(0, ebits - 141);
    const float qscale = __uint_as_float((uint32_t)(127 - kx) << 23);
    const float sl2 = p.scale_log2 * __uint_as_float((uint32_t)(127 + kx) << 23);
    uint32_t qf[NT][KS][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qf[nt][kk][0] = pack_f16x2(qv[nt][kk][0] * qscale, qv[nt][kk][1] * qscale);
        qf[nt][kk][1] = pack_f16x2(qv[nt][kk][2] * qscale, qv[nt][kk][3] * qscale);
      }

    float m[NT][2], l[NT][2];
    float o[KS][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    }

#pragma unroll 1
    for (int ch = 0; ch < nchunks_of(it); ++ch) {
      const int stage = consumed % kStages;
      const uint32_t parity = (consumed / kStages) & 1u;
      const bool landed = __all_sync(0xffffffffu, mbar_wait_bounded(bar[stage], parity, p.wait_cycles));
      if (!landed) {
        if (lane == 0) raise_flag(p.status, PA_FLAG_TIMEOUT);
        for (uint32_t c = consumed + 1; c < issued; ++c)
          mbar_wait_bounded(bar[c % kStages], (c / kStages) & 1u, p.wait_cycles);
        return;
      }
      const uint32_t ks = wbase + stage * TL::kStageBytes;
      const uint32_t vs = ks + TL::kBytes;
      const int nvalid = min(kKeys, it.len - ch * kKeys);
      if (nvalid < kKeys) {
        // keys past the end: zero their V codes (a key row is one contiguous
        // run of D bytes whatever the swizzle) so 0 * stale code stays 0
        const int nz = (kKeys - nvalid) * (D / 16);
        for (int i = lane; i < nz; i += 32) {
          const uint32_t a = vs + nvalid * D + i * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

      // S^T = K Q^T for the two 16-key tiles: A rows 16 t + gid and
      // 16 t + gid + 8, 16-byte run 4 sg + tig
      float s[2][NT][4];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) s[t][nt][0] = s[t][nt][1] = s[t][nt][2] = s[t][nt][3] = 0.f;
#pragma unroll
      for (int sg = 0; sg < SEG; ++sg) {
        uint32_t w[2][2][4];  // [tile][row gid / gid + 8][word]
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const uint4 v = lds128(ks + swz<D>((16 * t + gid + 8 * hr) * D + 16 * (4 * sg + tig)));
            w[t][hr][0] = v.x; w[t][hr][1] = v.y; w[t][hr][2] = v.z; w[t][hr][3] = v.w;
          }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint32_t a0 = e4m3x2_to_f16x2(w[t][0][j]), a2 = e4m3x2_to_f16x2(w[t][0][j] >> 16);
            const uint32_t a1 = e4m3x2_to_f16x2(w[t][1][j]), a3 = e4m3x2_to_f16x2(w[t][1][j] >> 16);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_f16_16816(s[t][nt], a0, a1, a2, a3, qf[nt][4 * sg + j][0], qf[nt][4 * sg + j][1]);
          }
      }

      // online softmax over the 32 keys; this thread holds keys 16 t + gid
      // and 16 t + gid + 8 (t = 0, 1) for heads 2 tig and 2 tig + 1
      bool vk[2][2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        vk[t][0] = 16 * t + gid < nvalid;
        vk[t][1] = 16 * t + gid + 8 < nvalid;
      }
      uint32_t pb[2][NT][2];  // [tile][n tile][key gid / gid + 8]
      float alpha[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pr[2][2][2];  // [tile][key half][head]
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float tv[2][2];
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
              tv[t][hr] = vk[t][hr] ? __fmul_rn(s[t][nt][2 * hr + e], sl2) : -INFINITY;
          float mx = fmaxf(fmaxf(tv[0][0], tv[0][1]), fmaxf(tv[1][0], tv[1][1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m[nt][e], mx);
          alpha[nt][e] = ex2_approx(m[nt][e] - mn);
          m[nt][e] = mn;
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) pr[t][hr][e] = ex2_approx(tv[t][hr] - mn);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) pb[t][nt][hr] = pack_f16x2(pr[t][hr][0], pr[t][hr][1]);
        // the chunk's weights in a fixed order: tile 0 (gid, gid + 8), tile 1
        const float s0 = (f16_lo(pb[0][nt][0]) + f16_lo(pb[0][nt][1])) +
                         (f16_lo(pb[1][nt][0]) + f16_lo(pb[1][nt][1]));
        const float s1 = (f16_hi(pb[0][nt][0]) + f16_hi(pb[0][nt][1])) +
                         (f16_hi(pb[1][nt][0]) + f16_hi(pb[1][nt][1]));
        l[nt][0] = fmaf(l[nt][0], alpha[nt][0], s0);
        l[nt][1] = fmaf(l[nt][1], alpha[nt][1], s1);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[mt][nt][0] *= alpha[nt][0];
          o[mt][nt][1] *= alpha[nt][1];
          o[mt][nt][2] *= alpha[nt][0];
          o[mt][nt][3] *= alpha[nt][1];
        }
      }

      // O^T += V^T P^T, one 16-key tile (k step) after the other: m tile mt,
      // row gid + 8 h is output dim kBPT * gid + 2 mt + h; this thread reads
      // those kBPT bytes of keys 16 t + {2tig, 2tig+1, 2tig+8, 2tig+9}
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        uint32_t pbt[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          pbt[nt][0] = movmatrix_trans(pb[t][nt][0]);
          pbt[nt][1] = movmatrix_trans(pb[t][nt][1]);
        }
        uint32_t vw[4][TL::kBPT / 4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int key = 16 * t + 2 * tig + (r & 1) + 8 * (r >> 1);
          const uint32_t a = vs + swz<D>(key * D + TL::kBPT * gid);
          if constexpr (TL::kBPT == 16) {
            const uint4 v = lds128(a);
            vw[r][0] = v.x; vw[r][1] = v.y; vw[r][2] = v.z; vw[r][3] = v.w;
          } else {
            const uint2 v = lds64(a);
            vw[r][0] = v.x; vw[r][1] = v.y;
          }
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
          const uint32_t y01 = prmt(vw[0][mt >> 1], vw[1][mt >> 1], sel);
          const uint32_t y89 = prmt(vw[2][mt >> 1], vw[3][mt >> 1], sel);
          const uint32_t a0 = e4m3x2_to_f16x2(y01), a1 = e4m3x2_to_f16x2(y01 >> 16);
          const uint32_t a2 = e4m3x2_to_f16x2(y89), a3 = e4m3x2_to_f16x2(y89 >> 16);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16_16816(o[mt][nt], a0, a1, a2, a3, pbt[nt][0], pbt[nt][1]);
        }
      }
      __syncwarp();  // every lane is done reading this stage
      ++consumed;
      produce();
    }

    // ---- finish the item ----
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
    const size_t head0 = (size_t)it.row * p.H + (size_t)it.kvh * g;
    if (it.single && !kOwner) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int hl = nt * 8 + 2 * tig + (r & 1);
          if (hl < g) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              const int d = TL::kBPT * gid + 2 * mt + (r >> 1);
              out[(head0 + hl) * D + d] =
                  __float2bfloat16_rn(finish_div(o[mt][nt][r], l[nt][r & 1]) * p.out_scale);
            }
          }
        }
    } else {
      const size_t ph0 =
          (size_t)(kOwner ? (long long)p.plan.row_info[it.row].x + it.t0 / split_len(it.keys)
                          : (long long)it.pair) * p.H +
          (size_t)it.kvh * g;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int hl = nt * 8 + 2 * tig + (r & 1);
          if (hl < g) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              const int d = TL::kBPT * gid + 2 * mt + (r >> 1);
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
}

template <int D, int NT, bool kOwner>
cudaError_t launch_o(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v, int grid,
                     cudaStream_t s) {
  auto kern = decode_fp8_kernel<D, NT, kOwner>;
  static unsigned long long done = 0;
  cudaError_t e = smem_opt_in(kern, Tile8<D>::kSmemBytes, &done);
  if (e != cudaSuccess) return e;
  kern<<<grid, kWarps * 32, Tile8<D>::kSmemBytes, s>>>(p, k, v);
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

cudaError_t launch_decode_fp8(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v,
                              long long max_items, cudaStream_t s) {
  long long want = (max_items + kWarps - 1) / kWarps;
  const long long cap = 3LL * num_sms();  // 3 CTAs (12 independent warps) per SM
  int grid = (int)(want < cap ? want : cap);
  if (grid < 1) grid = 1;
  const int g = p.H / p.Hkv;
  if (p.D == 128) return g <= 8 ? launch_t<128, 1>(p, k, v, grid, s) : launch_t<128, 2>(p, k, v, grid, s);
  return g <= 8 ? launch_t<64, 1>(p, k, v, grid, s) : launch_t<64, 2>(p, k, v, grid, s);
}

}  // namespace pa
