// Prologue of one step: the KV append (new rows copied into their slots) and
// the split plan of the step, in one launch. CTA 0 builds the plan; the other
// CTAs copy rows. The two jobs touch disjoint memory.
//
// KV append: "P3: native paged-KV continuous-batching sampler", Design
// (paged.py): PagedKVCache's copy-free append scatters each new row into
// (block, offset) = (slot / block_size, slot % block_size) in place. Rows of
// the cache are contiguous [Hkv, D] runs, so a slot names the flat row
// `slot` of the [num_blocks * block_size, Hkv, D] view; the copy moves 16-byte
// vectors and never converts, except into e4m3 caches, where each element is
// quantised under its tensor's scale on the way in.
//
// Split plan: every row on the split path attends keys 0..position and is cut
// into ranges [S i, S (i + 1)) with S = split_len(its key count) -- a function
// of its own key count only ("Numerics envelopes", The hierarchy,
// invariance.batch: no split count that scales with batch or occupancy). The plan lists one pair
// (row, split) per range: full ranges from the front of the list (longer
// splits first), tail ranges from its back.
#include "pa_common.cuh"

namespace pa {

namespace {

// KV-parallel key ranges of lane b (ctx c): this owner's [key_lo, key_hi)
// in mode 1, the owners' partition in mode 2. Interior bounds must be
// multiples of split_len(c), the split length of the lane's longest row (a
// multiple of every shorter row's), so no split straddles two owners.
__device__ bool owner_ranges_bad(const StepParams& p, int b, int c) {
  const int sl = split_len(c > 0 ? c : 1);
  auto aligned = [&](long long x) { return x >= c || x % sl == 0; };
  if (p.partials_mode == 1) {
    const long long lo = p.key_lo[b], hi = p.key_hi[b];
    return lo < 0 || hi < lo || !aligned(lo) || !aligned(hi);
  }
  const int W = p.owners;
  long long prev = p.key_bounds[b];
  if (prev != 0) return true;
  for (int w = 1; w <= W; ++w) {
    const long long x = p.key_bounds[(size_t)w * p.B + b];
    if (x < prev || !aligned(x)) return true;
    prev = x;
  }
  return prev < c;
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

// Counters of the plan scan (see row_counts).
constexpr int kCounters = 5;

// Exclusive block-wide scan of the plan's counters; returns the block totals.
__device__ void block_scan(const long long (&v)[kCounters], long long (&ex)[kCounters],
                           long long (&tot)[kCounters]) {
  __shared__ long long sm[kCounters][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long inc[kCounters];  // inclusive within the warp
#pragma unroll
  for (int k = 0; k < kCounters; ++k) inc[k] = v[k];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < kCounters; ++k) {
      const long long x = __shfl_up_sync(0xffffffffu, inc[k], o);
      if (lane >= o) inc[k] += x;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int k = 0; k < kCounters; ++k) sm[k][warp] = inc[k];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < kCounters; ++k) {
      long long x = lane < nw ? sm[k][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane < nw) sm[k][lane] = x;  // inclusive over warps
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kCounters; ++k) {
    ex[k] = (warp ? sm[k][warp - 1] : 0) + inc[k] - v[k];
    tot[k] = sm[k][nw - 1];
  }
  __syncthreads();
}

// Splits [i0, i1) of a row (split length sl, n splits) this call computes:
// all of them in an ordinary step, the ones whose first key lies in
// [key_lo, key_hi) for a KV-parallel owner, none for the merge.
__device__ __forceinline__ void owned_splits(const StepParams& p, int b, int sl, int n, int& i0,
                                             int& i1) {
  if (p.partials_mode == 0) {
    i0 = 0;
    i1 = n;
  } else if (p.partials_mode == 1) {
    const long long lo = p.key_lo[b], hi = p.key_hi[b];
    i0 = (int)min((long long)n, (lo + sl - 1) / sl);
    i1 = (int)min((long long)n, (hi + sl - 1) / sl);
  } else {
    i0 = i1 = 0;
  }
}

// Steps of up to kLaneCache lanes keep cu_seqlens_q, ctx_lens and each lane's
// validity in shared memory while the plan is built; larger ones read global
// memory.
constexpr int kLaneCache = 1024;
struct LaneCache {
  int cu[kLaneCache + 1];
  int ctx[kLaneCache];
  unsigned char ok[kLaneCache];
};

// Lane of flat row r: the b with cu[b] <= r < cu[b + 1] (binary search over
// cu_seqlens_q), or -1 when cu_seqlens_q is not ordered around r.
__device__ int lane_of_row(const StepParams& p, const LaneCache* lc, int r) {
  const int* cu = lc ? lc->cu : p.cu_seqlens;
  int lo = 0, hi = p.B - 1;  // the last b with cu[b] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= r) lo = mid;
    else hi = mid - 1;
  }
  return (cu[lo] <= r && r < cu[lo + 1]) ? lo : -1;
}

// What one flat row contributes to the plan. Counters: full split pairs of
// rows with splits longer than kSplit ("long"), full kSplit pairs ("short"),
// tail pairs, [3] -- prefill tiles of the row's lane (counted at its first
// row) or, in the KV-parallel modes and for grouped prefill rows, the row's
// entries -- and [4], the records of the prefill-row group the row starts.
// In the KV-parallel modes the entries depend on q_len and ctx_len alone
// (every owner and the merge lay them out alike); malformed owner ranges only
// empty this owner's share (mode 1) or take the rows out of the merge (mode 2).
struct RowPlan {
  int b, q, c, cu0, j, keys, sl, nf, n, i0, i1, g1;
  bool split, tiles, owner_ok;
};

// A unit of the plan is a flat row when every row takes the split path, else
// a lane (whose split path has at most its one decode row; a prefill lane
// only adds its tiles). Returns the unit's row in r.
__device__ bool row_counts(const StepParams& p, const LaneCache* lc, int u, int& r,
                           long long (&cnt)[kCounters], RowPlan& rp) {
  for (int k = 0; k < kCounters; ++k) cnt[k] = 0;
  rp.split = rp.tiles = false;
  rp.owner_ok = true;
  const bool by_row = p.split_all_rows;
  if (u >= (by_row ? p.T : p.B)) return false;
  rp.b = by_row ? lane_of_row(p, lc, u) : u;
  if (rp.b < 0) return false;
  if (lc) {
    if (!lc->ok[rp.b]) return false;
    rp.cu0 = lc->cu[rp.b];
    rp.q = lc->cu[rp.b + 1] - rp.cu0;
    rp.c = lc->ctx[rp.b];
  } else if (!lane_valid(p, rp.b, false, rp.q, rp.c, rp.cu0)) {
    return false;
  }
  if (p.partials_mode && owner_ranges_bad(p, rp.b, rp.c)) rp.owner_ok = false;
  r = by_row ? u : rp.cu0;
  rp.j = r - rp.cu0;
  rp.split = rp.q >= 1 && (p.split_all_rows || rp.q == 1);
  rp.tiles = !p.split_all_rows && rp.q >= 2;
  if (rp.split) {  // row j attends c - q + j + 1 keys
    rp.keys = rp.c - rp.q + rp.j + 1;
    rp.sl = split_len(rp.keys);
    rp.nf = rp.keys / rp.sl;
    rp.n = rp.nf + ((rp.keys % rp.sl) != 0);
    if (p.partials_mode) cnt[3] = rp.n;  // canonical entries (no prefill tiles here)
    if (p.group_rows && rp.q >= 2) {     // a grouped prefill row: entries only
      cnt[3] = rp.n;
      rp.i0 = rp.i1 = 0;                 // no pairs of its own
      // The lane's rows with split length sl form one run (split_len grows
      // with the key count: sl = kSplit up to kSplit * kMaxSplits keys, else
      // sl covers (sl / 2 * kMaxSplits, sl * kMaxSplits]); groups of
      // group_rows rows start at the run's first row. A group has one record
      // per split of its last row: {first row, rows | split << 8, lane, keys
      // of the first row}.
      const long long kmin = rp.sl == kSplit ? 1 : (long long)(rp.sl / 2) * kMaxSplits + 1;
      const long long kmax = (long long)rp.sl * kMaxSplits;
      const long long key0 = (long long)rp.c - rp.q + 1;  // keys of the lane's row 0
      const int js = (int)max(0LL, kmin - key0);
      const int je = (int)min((long long)rp.q, kmax - key0 + 1);
      if ((rp.j - js) % p.group_rows == 0) {
        rp.g1 = min(rp.j + p.group_rows, je);
        const int keys_last = rp.c - rp.q + rp.g1;
        cnt[4] = (keys_last + rp.sl - 1) / rp.sl;
      }
      return true;
    }
    owned_splits(p, rp.b, rp.sl, rp.n, rp.i0, rp.i1);
    if (!rp.owner_ok) rp.i0 = rp.i1 = 0;
    cnt[rp.sl > kSplit ? 0 : 1] = max(0, min(rp.i1, rp.nf) - rp.i0);
    cnt[2] = (rp.n > rp.nf && rp.n - 1 >= rp.i0 && rp.n - 1 < rp.i1);
  }
  // tensor-core prefill items pair two consecutive 128-row q tiles of a lane
  if (rp.tiles && rp.j == 0) cnt[3] = (rp.q + 2 * kPrefillRows - 1) / (2 * kPrefillRows);
  return true;
}

// Prefill-role CTAs of a mixed kernel out of nctas (one per SM): the split
// that balances the two roles' times, from the step's work totals and per-SM
// rates measured on this part with the roles running side by side -- the
// decode role streams ~66 GB/s per SM up to ~6760 GB/s in all; the prefill
// role runs pf_rate flop/s per SM (7.0 TFLOP/s for the tensor-core prefill,
// 0.9 TFLOP/s for the row-invariant mode's prefill rows on mma.sync: the
// values that gave the shortest launch in sweeps on the mixed step, a little
// under the roles' own rates because a prefill CTA that runs out of work
// takes decode items while a decode CTA cannot help the prefill). fp32
// (the part's fp64 rate is low); it decides only where work runs, never its
// result.
__device__ int prefill_role_ctas(const StepParams& p, long long split_keys, long long pf_work,
                                 long long pf_items, float pf_rate, int nctas) {
  if (pf_work <= 0 || pf_items <= 0 || nctas <= 1) return 0;
  if (split_keys <= 0) return nctas;
  const float kDecPerSm = 66e9f, kDecMax = 6760e9f, kPfPerSm = pf_rate;
  const float a = 4.f * p.D * p.H * (float)pf_work / kPfPerSm;               // prefill SM-seconds
  const float b = (float)split_keys * p.Hkv * p.D * 2.f * p.elem_bytes;      // decode bytes
  auto t = [&](int m) {  // the later of the two roles with m prefill CTAs
    return fmaxf(b / fminf(kDecMax, kDecPerSm * (nctas - m)), a / m);
  };
  // the two times cross where a / m = b / (kDecPerSm (nctas - m)) while the
  // decode role is below its cap, or where a / m = b / kDecMax once it is
  // not; the nearest integers around both crossings are the candidates
  const float m1 = nctas * a / (a + b / kDecPerSm), m2 = a * kDecMax / b;
  int best = 1;
  float best_t = t(1);
  const float cand[2] = {m1, m2};
  for (int c = 0; c < 2; ++c)
    for (int d = -1; d <= 1; ++d) {
      // (the crossing can lie far outside [1, nctas - 1]: clamp before the
      // conversion to int)
      const int m = min(nctas - 1, max(1, (int)fminf(fmaxf(cand[c], 0.f), (float)nctas) + d));
      const float tm = t(m);
      if (tm < best_t) {
        best_t = tm;
        best = m;
      }
    }
  return (int)(best < pf_items ? best : pf_items);
}

// The plan is built over units (blockDim at a time, two passes): pass 1
// counts and scans, pass 2 scans again and writes -- long full pairs from the
// front of the list, short full pairs after all long ones, tail pairs from the
// back, prefill tiles to a scratch list. Units are in lane order, so the list
// order is lane-major, row by row; when every row takes the split path each
// row (of a 4000-row chunk as of a decode lane) is handled by its own thread. Lanes are validated (and their
// flags raised) in a pass of their own. Totals are checked against the
// workspace; on overflow nothing runs.
__device__ void build_plan(const StepParams& p) {
  __shared__ int s_work[1024];
  __shared__ LaneCache s_lanes;
  const int tid = threadIdx.x, nth = blockDim.x;
  const SplitPlan& pl = p.plan;
  const LaneCache* lc = p.B <= kLaneCache ? &s_lanes : nullptr;
  for (int r = tid; r < p.T; r += nth) pl.row_info[r] = make_int4(0, -1, 0, -1);
  for (int b = tid; b < p.B; b += nth) {
    int q, c, cu0;
    const bool ok = lane_valid(p, b, true, q, c, cu0);
    if (ok && p.partials_mode && owner_ranges_bad(p, b, c))
      raise_flag(p.status, PA_FLAG_OWNER_RANGE);
    if (lc) {
      s_lanes.cu[b] = p.cu_seqlens[b];
      s_lanes.ctx[b] = p.ctx_lens[b];
      s_lanes.ok[b] = ok ? 1 : 0;
      if (b == p.B - 1) s_lanes.cu[p.B] = p.cu_seqlens[p.B];
    }
  }
  __syncthreads();

  const int units = p.split_all_rows ? p.T : p.B;
  long long total[kCounters] = {0, 0, 0, 0, 0};
  // work totals for the mixed kernels' role split (steps with prefill rows
  // only): keys of the split-path decode rows, (row, key) pairs of the
  // prefill rows -- rows j = 0 .. q-1 of a lane attend c - q + j + 1 keys
  __shared__ long long s_mix[2];
  const bool mixed = (!p.split_all_rows || p.group_rows) && p.max_q_len >= 2;
  if (tid < 2) s_mix[tid] = 0;
  __syncthreads();
  for (int base = 0; base < units; base += nth) {
    long long cnt[kCounters];
    RowPlan rp;
    int r;
    const bool ok0 = row_counts(p, lc, base + tid, r, cnt, rp);
    if (mixed) {
      const bool grouped = ok0 && p.group_rows && rp.q >= 2;  // a prefill row, row mode
      long long w[2] = {ok0 && rp.split && !grouped ? (long long)rp.keys : 0,
                        grouped ? (long long)rp.keys : 0};
      if (ok0 && rp.tiles && rp.j == 0)
        w[1] = (long long)rp.q * (rp.c - rp.q) + (long long)rp.q * (rp.q + 1) / 2;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) w[k] += __shfl_xor_sync(0xffffffffu, w[k], o);
        if ((tid & 31) == 0 && w[k]) atomicAdd(reinterpret_cast<unsigned long long*>(&s_mix[k]),
                                               (unsigned long long)w[k]);
      }
    }
    long long ex[kCounters], tot[kCounters];
    block_scan(cnt, ex, tot);
#pragma unroll
    for (int k = 0; k < kCounters; ++k) total[k] += tot[k];
  }
  const int cap = pl.capacity;
  const long long nfull = total[0] + total[1];
  const bool overflow =
      nfull + total[2] + (p.group_rows ? total[3] : 0) > cap ||
      (!p.group_rows &&
       total[3] > (p.partials_mode ? pl.entry_capacity : (long long)pl.ptile_capacity));
  if (overflow && tid == 0) raise_flag(p.status, PA_FLAG_WORKSPACE);
  __syncthreads();

  if (!overflow) {
    long long carry[kCounters] = {0, 0, 0, 0, 0};
    for (int base = 0; base < units; base += nth) {
      long long cnt[kCounters];
      RowPlan rp;
      int r = 0;
      const bool ok = row_counts(p, lc, base + tid, r, cnt, rp);
      long long ex[kCounters], tot[kCounters];
      block_scan(cnt, ex, tot);
      if (ok && rp.split) {
        const long long lb = carry[0] + ex[0];             // long full pairs
        const long long sb = total[0] + carry[1] + ex[1];  // short full pairs
        const long long tb = carry[2] + ex[2];             // tail pair k sits at cap - 1 - k
        const long long eb = carry[3] + ex[3];             // KV-parallel: the row's first entry
        const long long fb = rp.sl > kSplit ? lb : sb;
        const bool has_tail = rp.n > rp.nf;
        const long long tslot = cap - 1 - tb;
        if (p.group_rows && rp.q >= 2) {  // its entries follow the full pairs
          pl.row_info[r] = make_int4((int)(nfull + eb), -1, rp.n, rp.b);
          // the records of the group it starts, after the full pairs too
          // (never more records than grouped entries: each holds a row's split)
          long long k = nfull + carry[4] + ex[4];
          for (int i = 0; i < cnt[4]; ++i)
            pl.pairs[k++] = make_int4(r, (rp.g1 - rp.j) | (i << 8), rp.b, rp.keys);
        } else if (p.partials_mode) {
          pl.row_info[r] = make_int4((int)eb, rp.keys, rp.n, rp.owner_ok ? rp.b : -1);
        } else {
          pl.row_info[r] = make_int4((int)fb, has_tail ? (int)tslot : -1, rp.n, rp.b);
        }
        long long f = fb;
        for (int i = rp.i0; i < min(rp.i1, rp.nf); ++i) pl.pairs[f++] = make_int4(r, i, rp.b, rp.keys);
        if (has_tail && rp.n - 1 >= rp.i0 && rp.n - 1 < rp.i1)
          pl.pairs[tslot] = make_int4(r, rp.nf, rp.b, rp.keys);  // none for grouped rows
      }
      if (ok && rp.tiles && rp.j == 0) {
        const long long t0 = carry[3] + ex[3];
        for (int t = 0; t < cnt[3]; ++t) {  // tiles 2 t and 2 t + 1
          const int last = min(rp.q, (2 * t + 2) * kPrefillRows) - 1;
          pl.ptiles_tmp[t0 + t] = make_int4(rp.b, t, rp.c - rp.q + last, 0);
        }
      }
#pragma unroll
      for (int k = 0; k < kCounters; ++k) carry[k] += tot[k];
    }
  }
  const int n = (overflow || p.partials_mode || p.group_rows) ? 0 : (int)total[3];
  __syncthreads();
  // prefill tile pairs heaviest first (position of the pair's last row; ties
  // by list order) when there are at most blockDim of them: the order only
  // decides which CTA takes a tile first
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
  // rows the combine folds, the most splits first (decode rows: the
  // batch-invariant mode, e4m3 and fp32 decode steps, KV-parallel merges), by
  // a counting sort over the split counts, so every long row's fold starts in
  // the combine's first wave. (When prefill rows take the split path the
  // combine walks the flat rows instead and no list is kept.) The order
  // decides only when a fold runs, never its bits: each (row, head) is folded
  // by one warp in split order.
  __shared__ int s_bucket[kMaxSplits + 1];
  __shared__ int s_ncomb;
  const int min_n = p.partials_mode == 2 ? 1 : 2;  // merging owners folds every split row
  // when only decode lanes take the split path, a lane's one candidate is
  // its row 0 (if q_len == 1): walk lanes instead of rows
  const bool by_lane = !p.split_all_rows && !p.partials_mode;
  const int nunits = by_lane ? p.B : p.T;
  auto row_of = [&](int u) -> int {
    if (!by_lane) return u;
    if (lc && !lc->ok[u]) return -1;
    const int c0 = lc ? lc->cu[u] : p.cu_seqlens[u];
    const int c1 = lc ? lc->cu[u + 1] : p.cu_seqlens[u + 1];
    return (c1 - c0 == 1 && c0 >= 0 && c0 < p.T) ? c0 : -1;
  };
  auto bucket_of = [&](int r) -> int {
    if (r < 0) return -1;
    const int4 ri = pl.row_info[r];
    return (!overflow && ri.w >= 0 && ri.z >= min_n) ? min(ri.z, kMaxSplits) : -1;
  };
  const bool listed = !(p.split_all_rows && p.max_q_len >= 2 && !p.partials_mode);
  if (listed) {  // (uniform across the CTA)
    for (int i = tid; i <= kMaxSplits; i += nth) s_bucket[i] = 0;
    __syncthreads();  // (also orders every row_info write above before the reads below)
    for (int u = tid; u < nunits; u += nth) {
      const int b = bucket_of(row_of(u));
      if (b >= 0) atomicAdd(&s_bucket[b], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // exclusive scan over the buckets in descending order: lane l holds
      // positions 5 l .. 5 l + 4 of that order (bucket kMaxSplits - position)
      constexpr int kPer = (kMaxSplits + 1 + 31) / 32;
      int v[kPer], sum = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int pos = tid * kPer + j;
        v[j] = pos <= kMaxSplits ? s_bucket[kMaxSplits - pos] : 0;
        sum += v[j];
      }
      int inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, inc, o);
        if (tid >= o) inc += x;
      }
      int run = inc - sum;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int pos = tid * kPer + j;
        if (pos <= kMaxSplits) s_bucket[kMaxSplits - pos] = run;
        run += v[j];
      }
      if (tid == 31) s_ncomb = inc;
    }
    __syncthreads();
    for (int u = tid; u < nunits; u += nth) {
      const int r = row_of(u), b = bucket_of(r);
      if (b >= 0) {
        const int4 ri = pl.row_info[r];
        pl.crows[atomicAdd(&s_bucket[b], 1)] = make_int4(r, ri.x, ri.y, ri.z);
      }
    }
  }
  if (tid < kFingerprintInts) pl.header[kHeaderFingerprint + tid] = plan_fingerprint(p, tid);
  if (tid == 0) {
    pl.header[kHeaderPlanOk] = 1;
    pl.header[kHeaderCombineRows] = listed ? s_ncomb : 0;
    pl.header[0] = overflow ? 0 : (int)(nfull + total[2]);
    pl.header[1] = overflow ? 0 : (int)nfull;
    pl.header[2] = n;
    pl.header[3] = overflow ? 0 : (int)total[4];
    for (int c = 0; c < kItemCounters; ++c) *item_counter(pl, c) = 0ull;
    *header_total(pl, kHeaderSplitKeys) = overflow ? 0 : s_mix[0];
    *header_total(pl, kHeaderPrefillWork) = overflow ? 0 : s_mix[1];
    pl.header[kHeaderPrefillCtas] =
        (overflow || !mixed) ? 0
        : p.group_rows ? prefill_role_ctas(p, s_mix[0], s_mix[1], total[4] * p.Hkv, 0.9e12f,
                                           p.sm_count)
                       : prefill_role_ctas(p, s_mix[0], s_mix[1], (long long)n * p.H,
                                           7.0e12f, p.sm_count);
  }
}

// e4m3 caches: each new bf16 row is quantised on the way in, code =
// RN-even(x / scale) with the quotient in fp32 and saturation to +-448 (the
// per-tensor scaling the kv_dtype item of "P3: native paged-KV
// continuous-batching sampler", Review (adversarial pass), asks for). A thread
// converts 8 elements: one 16-byte load, one 8-byte store.
__device__ void write_rows_fp8(const StepParams& p, int cta, int ncta) {
  const int n8 = p.Hkv * p.D / 8;  // 8-element groups per row
  const long long nslots = (long long)p.NB * p.bs;
  const long long total = (long long)p.T * n8;
  const uint4* kn = static_cast<const uint4*>(p.k_new);
  const uint4* vn = static_cast<const uint4*>(p.v_new);
  uint2* kc = static_cast<uint2*>(const_cast<void*>(p.k_cache));
  uint2* vc = static_cast<uint2*>(const_cast<void*>(p.v_cache));
  for (long long i = (long long)cta * blockDim.x + threadIdx.x; i < total;
       i += (long long)ncta * blockDim.x) {
    const long long t = i / n8;
    const int v = (int)(i - t * n8);
    const long long slot = p.slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= nslots) {
      if (v == 0) raise_flag(p.status, PA_FLAG_SLOT_RANGE);
      continue;
    }
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const uint4 x = (kv ? vn : kn)[t * n8 + v];
      const float sc = kv ? p.v_scale : p.k_scale;
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        c[e] = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(w[e]), sc), __fdiv_rn(bf16_hi(w[e]), sc));
      (kv ? vc : kc)[slot * n8 + v] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
  }
}

__device__ void write_rows(const StepParams& p, int cta, int ncta) {
  if (p.kv_fp8) {
    write_rows_fp8(p, cta, ncta);
    return;
  }
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

// A call that reuses the plan already in the workspace: the plan is valid
// for it when the sizes it was built for match this call's; then only the
// item counters, which the kernels consume, are reset. On a mismatch the
// kernels after the prologue do nothing and PA_FLAG_PLAN_MISMATCH is raised.
__device__ void check_plan(const StepParams& p) {
  const SplitPlan& pl = p.plan;
  const int tid = threadIdx.x;
  const bool same = tid >= kFingerprintInts ||
                    pl.header[kHeaderFingerprint + tid] == plan_fingerprint(p, tid);
  const int ok = __syncthreads_and(same ? 1 : 0);
  if (tid == 0) {
    pl.header[kHeaderPlanOk] = ok;
    if (!ok) {
      // a refused plan offers the kernels after the prologue no work: every
      // item count and the combine list are emptied (the split, prefill and
      // prefill-row kernels find nothing to take; the combine walking flat
      // rows tests kHeaderPlanOk)
      raise_flag(p.status, PA_FLAG_PLAN_MISMATCH);
      for (int i = 0; i < 4; ++i) pl.header[i] = 0;
      pl.header[kHeaderPrefillCtas] = 0;
      pl.header[kHeaderCombineRows] = 0;
      // and it matches no later call either (B >= 1 in every call that
      // reaches the device) until a call without the reuse bit plans again
      pl.header[kHeaderFingerprint] = -1;
    }
    for (int c = 0; c < kItemCounters; ++c) *item_counter(pl, c) = 0ull;
  }
}

// plan_mode: 0 no plan (the write alone), 1 build it, 2 check the one in
// the workspace (CTA 0 in modes 1 and 2; the other CTAs write the new rows)
__global__ void __launch_bounds__(1024) prologue_kernel(const StepParams p, int plan_mode) {
  if (plan_mode && blockIdx.x == 0) {
    if (plan_mode == 1)
      build_plan(p);
    else
      check_plan(p);
    return;
  }
  const int first = plan_mode ? 1 : 0;
  write_rows(p, blockIdx.x - first, gridDim.x - first);
}

}  // namespace

int num_sms();

cudaError_t launch_prologue(const StepParams& p, int plan_mode, bool write, cudaStream_t s) {
  int write_ctas = 0;
  if (write && p.T > 0) {
    const long long vecs = (long long)p.T * (p.Hkv * p.D * p.elem_bytes / 16);  // 16-byte loads
    long long want = (vecs + 1023) / 1024;
    const long long cap = 4LL * num_sms();
    write_ctas = (int)(want < cap ? want : cap);
  }
  const int grid = (plan_mode ? 1 : 0) + write_ctas;
  if (grid == 0) return cudaSuccess;
  prologue_kernel<<<grid, 1024, 0, s>>>(p, plan_mode);
  return cudaGetLastError();
}

}  // namespace pa
