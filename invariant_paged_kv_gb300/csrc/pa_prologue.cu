// Prologue of one step: the KV append (new rows copied into their slots) and
// the split plan of the step, in one launch. CTA 0 builds the plan; the other
// CTAs copy rows. The two jobs touch disjoint memory.
//
// KV append: "P3: native paged-KV continuous-batching sampler", Design
// (paged.py): PagedKVCache's copy-free append scatters each new row into
// (block, offset) = (slot / block_size, slot % block_size) in place. Rows of
// the cache are contiguous [Hkv, D] runs, so a slot names the flat row
// `slot` of the [num_blocks * block_size, Hkv, D] view; the copy moves 16-byte
// vectors and never converts.
//
// Split plan: every row on the split path attends keys 0..position and is cut
// into ranges [kSplit * i, kSplit * (i + 1)) -- a function of its own key
// count only ("Numerics envelopes", The hierarchy, invariance.batch: no split
// count that scales with batch or occupancy). The plan lists one pair
// (row, split) per range, full ranges first.
#include "pa_common.cuh"

namespace pa {

namespace {

// Sum over k = 0..n of floor(k / kSplit), for n >= -1.
__device__ __forceinline__ long long floor_sum(long long n) {
  if (n < 0) return 0;
  const long long t = n / kSplit, r = n % kSplit;
  return kSplit * t * (t - 1) / 2 + t * (r + 1);
}

// Validates lane b (raising status flags when `report`) and returns whether
// it is well formed; q, c, cu0 are its q_len, ctx_len and first row.
__device__ bool lane_valid(const StepParams& p, int b, bool report, int& q, int& c, int& cu0) {
  cu0 = p.cu_seqlens[b];
  const int cu1 = p.cu_seqlens[b + 1];
  c = p.ctx_lens[b];
  q = cu1 - cu0;
  int bad = 0;
  if (cu0 < 0 || cu1 < cu0 || cu1 > p.T || (b == 0 && cu0 != 0) || (b == p.B - 1 && cu1 != p.T))
    bad = PA_FLAG_CU_SEQLENS;
  else if (c < 0 || (long long)c > (long long)p.max_blocks * p.bs)
    bad = PA_FLAG_CTX_RANGE;
  else if (q > c)
    bad = PA_FLAG_QLEN_RANGE;
  else if (q > p.max_q_len || c > p.max_ctx_len)
    bad = PA_FLAG_HOST_BOUND;
  if (bad && report) raise_flag(p.status, bad);
  return bad == 0;
}

// Lane b's contribution to the split plan: the number of full and tail split
// ranges over its rows (zero when the lane is not on the split path).
__device__ bool lane_plan(const StepParams& p, int b, bool report, int& q, int& c, int& cu0,
                          long long& nfull, long long& ntail) {
  nfull = ntail = 0;
  if (!lane_valid(p, b, report, q, c, cu0)) return false;
  const bool on_split = q >= 1 && (p.split_all_rows || q == 1);
  if (!on_split) return false;
  // rows attend k = c - q + 1 .. c keys
  nfull = floor_sum(c) - floor_sum((long long)c - q);
  ntail = q - ((long long)c / kSplit - ((long long)c - q) / kSplit);
  return true;
}

// Exclusive block-wide scan of two counters; returns the block totals.
__device__ void block_scan2(long long a, long long b, long long& ea, long long& eb,
                            long long& ta, long long& tb) {
  __shared__ long long sa[32], sb[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long ia = a, ib = b;  // inclusive within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long xa = __shfl_up_sync(0xffffffffu, ia, o);
    const long long xb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += xa;
      ib += xb;
    }
  }
  if (lane == 31) {
    sa[warp] = ia;
    sb[warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    long long va = lane < nw ? sa[lane] : 0, vb = lane < nw ? sb[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long xa = __shfl_up_sync(0xffffffffu, va, o);
      const long long xb = __shfl_up_sync(0xffffffffu, vb, o);
      if (lane >= o) {
        va += xa;
        vb += xb;
      }
    }
    if (lane < nw) {
      sa[lane] = va;  // inclusive over warps
      sb[lane] = vb;
    }
  }
  __syncthreads();
  const long long wa = warp ? sa[warp - 1] : 0, wb = warp ? sb[warp - 1] : 0;
  ea = wa + ia - a;
  eb = wb + ib - b;
  ta = sa[nw - 1];
  tb = sb[nw - 1];
  __syncthreads();
}

// Tensor-core prefill tiles: 128-row tiles of every lane with q_len >= 2
// (when those lanes do not take the split path), ordered heaviest first (by
// the position of the tile's last row; ties by list order) when there are at
// most 1024 of them. The order only decides which CTA runs a tile first.
__device__ void build_prefill_tiles(const StepParams& p) {
  __shared__ int s_work[1024];
  const int tid = threadIdx.x, nth = blockDim.x;
  const SplitPlan& pl = p.plan;
  long long total = 0;
  if (!p.split_all_rows) {
    for (int base = 0; base < p.B; base += nth) {
      const int b = base + tid;
      int q = 0, c = 0, cu0 = 0;
      long long nt = 0;
      if (b < p.B && lane_valid(p, b, false, q, c, cu0) && q >= 2)
        nt = (q + kPrefillRows - 1) / kPrefillRows;
      long long e0, e1, t0, t1;
      block_scan2(nt, 0, e0, e1, t0, t1);
      if (nt > 0 && total + e0 + nt <= pl.ptile_capacity) {
        for (int t = 0; t < nt; ++t) {
          const int last = min(q, (t + 1) * kPrefillRows) - 1;
          pl.ptiles_tmp[total + e0 + t] = make_int4(b, t, c - q + last, 0);
        }
      }
      total += t0;
    }
  }
  if (total > pl.ptile_capacity) {
    if (tid == 0) raise_flag(p.status, PA_FLAG_WORKSPACE);
    total = 0;
  }
  __syncthreads();
  const int n = (int)total;
  if (n <= nth) {
    if (tid < n) s_work[tid] = pl.ptiles_tmp[tid].z;
    __syncthreads();
    if (tid < n) {
      const int w = s_work[tid];
      int rank = 0;
      for (int j = 0; j < n; ++j) {
        const int x = s_work[j];
        rank += (x > w) || (x == w && j < tid);
      }
      pl.ptiles[rank] = pl.ptiles_tmp[tid];
    }
  } else {
    for (int i = tid; i < n; i += nth) pl.ptiles[i] = pl.ptiles_tmp[i];
  }
  if (tid == 0) pl.header[2] = n;
}

__device__ void build_plan(const StepParams& p) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const SplitPlan& pl = p.plan;
  for (int r = tid; r < p.T; r += nth) pl.row_info[r] = make_int4(0, -1, 0, -1);

  long long tot_full = 0, tot_tail = 0;
  for (int base = 0; base < p.B; base += nth) {
    const int b = base + tid;
    int q, c, cu0;
    long long f = 0, t = 0;
    if (b < p.B) lane_plan(p, b, true, q, c, cu0, f, t);
    long long ef, et, tf, tt;
    block_scan2(f, t, ef, et, tf, tt);
    tot_full += tf;
    tot_tail += tt;
  }
  __syncthreads();
  if (tot_full + tot_tail > pl.capacity) {
    if (tid == 0) {
      raise_flag(p.status, PA_FLAG_WORKSPACE);
      pl.header[0] = 0;
      pl.header[1] = 0;
    }
    build_prefill_tiles(p);
    return;
  }
  long long carry_full = 0, carry_tail = 0;
  for (int base = 0; base < p.B; base += nth) {
    const int b = base + tid;
    int q = 0, c = 0, cu0 = 0;
    long long f = 0, t = 0;
    bool on = false;
    if (b < p.B) on = lane_plan(p, b, false, q, c, cu0, f, t);
    long long ef, et, tf, tt;
    block_scan2(f, t, ef, et, tf, tt);
    if (on) {
      long long fb = carry_full + ef;
      long long tb = tot_full + carry_tail + et;
      for (int j = 0; j < q; ++j) {
        const int keys = c - q + j + 1;
        const int nf = keys / kSplit;
        const bool has_tail = (keys % kSplit) != 0;
        const int row = cu0 + j;
        pl.row_info[row] = make_int4((int)fb, has_tail ? (int)tb : -1, nf + (has_tail ? 1 : 0), b);
        for (int i = 0; i < nf; ++i) pl.pairs[fb + i] = make_int4(row, i, b, keys);
        fb += nf;
        if (has_tail) {
          pl.pairs[tb] = make_int4(row, nf, b, keys);
          ++tb;
        }
      }
    }
    carry_full += tf;
    carry_tail += tt;
  }
  if (tid == 0) {
    pl.header[0] = (int)(tot_full + tot_tail);
    pl.header[1] = (int)tot_full;
  }
  build_prefill_tiles(p);
}

__device__ void write_rows(const StepParams& p, int cta, int ncta) {
  const int n16 = p.Hkv * p.D * p.elem_bytes / 16;  // 16-byte vectors per row
  const long long nslots = (long long)p.NB * p.bs;
  const long long total = (long long)p.T * n16;
  const uint4* kn = static_cast<const uint4*>(p.k_new);
  const uint4* vn = static_cast<const uint4*>(p.v_new);
  uint4* kc = static_cast<uint4*>(const_cast<void*>(p.k_cache));
  uint4* vc = static_cast<uint4*>(const_cast<void*>(p.v_cache));
  for (long long i = (long long)cta * blockDim.x + threadIdx.x; i < total;
       i += (long long)ncta * blockDim.x) {
    const long long t = i / n16;
    const int v = (int)(i - t * n16);
    const long long slot = p.slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= nslots) {
      if (v == 0) raise_flag(p.status, PA_FLAG_SLOT_RANGE);
      continue;
    }
    kc[slot * n16 + v] = kn[t * n16 + v];
    vc[slot * n16 + v] = vn[t * n16 + v];
  }
}

__global__ void __launch_bounds__(1024) prologue_kernel(const StepParams p, int do_plan) {
  if (do_plan && blockIdx.x == 0) {
    build_plan(p);
    return;
  }
  const int first = do_plan ? 1 : 0;
  write_rows(p, blockIdx.x - first, gridDim.x - first);
}

}  // namespace

int num_sms();

cudaError_t launch_prologue(const StepParams& p, bool plan, bool write, cudaStream_t s) {
  int write_ctas = 0;
  if (write && p.T > 0) {
    const long long vecs = (long long)p.T * (p.Hkv * p.D * p.elem_bytes / 16);
    long long want = (vecs + 1023) / 1024;
    const long long cap = 4LL * num_sms();
    write_ctas = (int)(want < cap ? want : cap);
  }
  const int grid = (plan ? 1 : 0) + write_ctas;
  if (grid == 0) return cudaSuccess;
  prologue_kernel<<<grid, 1024, 0, s>>>(p, plan ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace pa
