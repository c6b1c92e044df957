// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05), bf16.
//
// A lane with q_len >= 2 is a causal prefill chunk ("P3: native paged-KV
// continuous-batching sampler", Design, engine.py: prefill chunks and decode
// tokens share one flat step; Evidence, mutant "prefill causal mask off by
// one"): its row j sits at position ctx - q_len + j and attends keys
// 0..position. Work item = (query head, pair of consecutive 128-row q tiles
// of one lane): two streams that read the same key tiles. Per item, key tiles
// of 128 keys go in ascending order; for each stream s and key tile:
//   S = Q K^T           tcgen05.mma, M = 128 rows, N = 128 keys, K = D, fp32 in TMEM
//   m, p, l             one thread per row: running max, p = 2^(t - m) rounded
//                       to bf16 and written back over S in TMEM, l += sum of
//                       the p (fp32, before rounding) -- all within the thread
//   O = O * alpha + P V tcgen05.mma with A = P read from TMEM, B = V (MN-major
//                       smem), O in TMEM
// and finally out = O * (1 / l). The running max moves only when a tile's max
// exceeds it by more than 8 (log2 units), so O is rescaled rarely. A row's
// arithmetic depends on its q row, its keys and the fixed 128-key tiling from
// key 0 -- never on other lanes, other heads, or the other stream. (N = 128
// keys: a 128 x 128 x 16 product runs at the tensor core's full rate, where
// a 128 x 64 x 16 one reaches ~70%.) The second tile of a pair may need one
// key tile more than the first (causal); the first stream skips it.
//
// Warp roles (320 threads): warps 0-3 and 4-7 are the two streams' softmax
// groups (thread r of a group owns row r = TMEM lane r), warp 8 issues the
// MMAs (one elected lane of the converged warp), warp 9 streams Q / K / V in
// by TMA (K / V through the block table, 16 keys per box) into 2-deep K and
// V rings shared by both streams. TMEM per stream (256 of the 512 columns): S / P (128), O (128).
// The issuing warp is stalled while the tensor pipe's queue is full, so its
// order is the pipe's order: per key tile and stream, P V of tile t and then
// S of tile t + 1 (which overwrites P of tile t in TMEM, so it waits for
// that P V to finish); the streams alternate, so one stream's softmax runs
// while the tensor core serves the other.
//
// Every wait is bounded (timeout -> PA_FLAG_TIMEOUT); before the CTA leaves,
// the MMA warp waits for its products and the TMA warp for its copies. No
// parity wait ever meets a barrier more than one phase away from the awaited
// one, ahead or behind (the P V barriers alternate by tile parity for that
// reason).
//
// The work is written as the code of one CTA (prefill_tc_cta): it runs as the
// prefill role of the mixed-step kernel (pa_mixed.cu), which gives every CTA
// this role when a step has no decode rows.
#pragma once

#include "pa_tcgen05.cuh"

namespace pa {
namespace pftc {


constexpr int kRows = 128;  // query rows per tile (M)
constexpr int kKeys = 128;  // keys per tile (N of S, K of PV)
constexpr int kStages = 2;  // depth of the K and V rings
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct PfLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kRows * 128;         // Q: 128 rows x 128 bytes
  static constexpr int kKHalfBytes = kKeys * 128;        // K / V: 128 keys x 128 bytes
  static constexpr int kQBytes = kHalves * kHalfBytes;   // one Q tile
  static constexpr int kKBytes = kHalves * kKHalfBytes;  // one K tile
  static constexpr int kVBytes = kHalves * kKHalfBytes;  // one V tile
  static constexpr int kQ = 0;                           // Q of stream 0, then stream 1
  static constexpr int kK0 = kQ + 2 * kQBytes;
  static constexpr int kV0 = kK0 + kStages * kKBytes;
  static constexpr int kEnd = kV0 + kStages * kVBytes;
  // + alignment slack; at least 116 KB so one CTA (and one 512-column TMEM
  // allocation) per SM
  static constexpr int kSmemBytes = (kEnd + 1024) > 118784 ? (kEnd + 1024) : 118784;
};

struct Bars {
  uint64_t kfull[kStages], kempty[kStages], vfull[kStages], vempty[kStages];
  // vtail[stage]: a tail tile (keys past ctx) in that V stage is zeroed; one
  // barrier per stage, so a fill can never complete a second phase of it
  // before the first is consumed (the stage's next fill waits for that)
  uint64_t q, qempty, vtail[kStages], fin, s[2], p[2], o[2][2];  // [stream] ([tile parity] for o)
};

struct ItemInfo {
  int lane, head, kvh, cu0, q_len, ctx, nst, nkt;
  int row0[2], nrows[2], p_first[2], nkt_s[2];
};

// Item = (pair entry t, head): consecutive items share a pair and walk its
// heads in order, so the g heads of a kv head follow each other.
__device__ __forceinline__ ItemInfo item_info(const StepParams& p, int item) {
  ItemInfo it;
  const int t = item / p.H;
  it.head = item - t * p.H;
  it.kvh = it.head / (p.H / p.Hkv);
  const int4 e = p.plan.ptiles[t];
  it.lane = e.x;
  it.cu0 = p.cu_seqlens[it.lane];
  it.q_len = p.cu_seqlens[it.lane + 1] - it.cu0;
  it.ctx = p.ctx_lens[it.lane];
  it.nst = 0;
  it.nkt = 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    it.row0[s] = (2 * e.y + s) * kRows;
    it.nrows[s] = min(kRows, it.q_len - it.row0[s]);
    it.p_first[s] = it.ctx - it.q_len + it.row0[s];
    it.nkt_s[s] = it.nrows[s] > 0 ? (it.p_first[s] + it.nrows[s] - 1) / kKeys + 1 : 0;
    if (it.nrows[s] > 0) it.nst = s + 1;
    it.nkt = max(it.nkt, it.nkt_s[s]);
  }
  return it;
}

// Wait with the CTA-wide abort flag: returns false (and sets the flag) on
// timeout. The fast path is one try_wait: the flag lives in shared memory,
// and a shared load waits behind the tensor core's operand reads (~140
// cycles while products stream), so it is read only in the slow loop.
__device__ __forceinline__ bool wait_or_abort_1(uint32_t bar, uint32_t parity,
                                                volatile int* abort_flag, int* status,
                                                long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 7) == 7) {
      if (*abort_flag) return false;
      if (clock64() - t0 > limit) {
        *abort_flag = 1;
        raise_flag(status, PA_FLAG_TIMEOUT);
        return false;
      }
    }
  }
}

// Every lane of the warp waits; the outcome is made warp-uniform.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int* status,
                                              long long limit) {
  return __all_sync(0xffffffffu, wait_or_abort_1(bar, parity, abort_flag, status, limit));
}

// The work of one CTA of kThreads threads (see the roles above); dsmem
// holds PfLayout<D>::kSmemBytes bytes. Each role runs its own loop over the
// CTA's items (no CTA-wide barrier between items): the TMA warp takes item
// indices from the prefill counter and publishes them through a 4-slot queue
// (slot n % 4 for the CTA's n-th item, freed when all nine consumer warps
// have read it), and the rings, the Q buffer and the TMEM regions carry the
// handoffs from one item to the next.
template <int D>
__device__ __forceinline__ void prefill_tc_cta(const StepParams& p, const CUtensorMap* tmQ,
                                               const CUtensorMap* tmK, const CUtensorMap* tmV,
                                               uint8_t* dsmem) {
  using L = PfLayout<D>;
  constexpr int kSlots = 4;
  __shared__ __align__(8) Bars bars;
  __shared__ __align__(8) uint64_t item_full[kSlots], item_free[kSlots];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ long long s_items[kSlots];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sQ = base + L::kQ, sK0 = base + L::kK0, sV0 = base + L::kV0;
  const uint32_t bq = smem_u32(&bars.q), bqe = smem_u32(&bars.qempty);
  auto bvt = [&](uint32_t st) -> uint32_t { return smem_u32(&bars.vtail[st]); };
  // ring barriers by stage: address arithmetic, not arrays (an array
  // indexed by a run-time stage lives in local memory, and every local load
  // waits ~150 cycles behind the tensor core's shared-memory reads)
  const uint32_t bkf0 = smem_u32(&bars.kfull[0]), bke0 = smem_u32(&bars.kempty[0]);
  const uint32_t bvf0 = smem_u32(&bars.vfull[0]), bve0 = smem_u32(&bars.vempty[0]);
  auto bkf = [&](uint32_t i) -> uint32_t { return bkf0 + 8u * i; };
  auto bke = [&](uint32_t i) -> uint32_t { return bke0 + 8u * i; };
  auto bvf = [&](uint32_t i) -> uint32_t { return bvf0 + 8u * i; };
  auto bve = [&](uint32_t i) -> uint32_t { return bve0 + 8u * i; };
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bkf(i), 1);
      mbar_init(bke(i), 1);
      mbar_init(bvf(i), 1);
      mbar_init(bve(i), 1);
    }
    mbar_init(bq, 1);
    mbar_init(bqe, 1);
    for (int i = 0; i < kStages; ++i) mbar_init(bvt(i), 1);
    mbar_init(smem_u32(&bars.fin), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&bars.s[h]), 1);
      mbar_init(smem_u32(&bars.p[h]), kRows);
      mbar_init(smem_u32(&bars.o[h][0]), 1);
      mbar_init(smem_u32(&bars.o[h][1]), 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_u32(&item_full[i]), 1);
      mbar_init(smem_u32(&item_free[i]), 9);  // 8 softmax warps + the MMA warp
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 9 && lane == 0) {
    prefetch_tensormap(tmQ);
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
  }
  if (warp == 8) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // stream s: S / P at column 256 s, O at 256 s + 128
  auto tS = [&](int s) -> uint32_t { return tmem + 256 * s; };
  auto tO = [&](int s) -> uint32_t { return tmem + 256 * s + 128; };
  auto bS = [&](int s) -> uint32_t { return smem_u32(&bars.s[s]); };
  auto bP = [&](int s) -> uint32_t { return smem_u32(&bars.p[s]); };
  // P V of tile t completes on o[stream][t & 1]
  auto bO = [&](int s, uint32_t t) -> uint32_t { return smem_u32(&bars.o[s][t & 1]); };
  volatile int* ab = &s_abort;
  const long long lim = p.wait_cycles;
  // the CTA's n-th item, as the TMA warp published it (a consumer warp:
  // wait for the slot, read it, free it); false on abort
  auto read_item = [&](uint32_t n, long long& item) -> bool {
    if (!wait_or_abort(smem_u32(&item_full[n % kSlots]), (n / kSlots) & 1, ab, p.status, lim))
      return false;
    item = s_items[n % kSlots];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&item_free[n % kSlots]));
    return true;
  };

  const int n_items = p.plan.header[2] * p.H;
  const float c2 = p.scale_log2;  // > 0 (validated on the host)
  // running use counters, identical in every role: K/V ring fills, key tiles
  // of each stream, items with a tail key tile
  // (n_t0 / n_t1: key tiles of stream 0 / 1; tail_par: bit st = parity of
  // the next tail use of V stage st)
  uint32_t n_item = 0, n_kv = 0, n_t0 = 0, n_t1 = 0, tail_par = 0;

  if (warp == 9) {
    // -------------------------------- producer ------------------------------
    for (;; ++n_item) {
      const uint32_t n = n_item;
      // slot n % 4 is free once every consumer has read item n - 4
      if (n >= kSlots &&
          !wait_or_abort(smem_u32(&item_free[n % kSlots]), ((n / kSlots) - 1) & 1, ab, p.status, lim))
        break;
      long long item = 0;
      if (lane == 0) {
        item = (long long)atomicAdd(item_counter(p.plan, kCounterPrefill), 1ull);
        s_items[n % kSlots] = item;
        mbar_arrive(smem_u32(&item_full[n % kSlots]));
      }
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item >= n_items) break;
      const ItemInfo it = item_info(p, (int)item);
      const bool tail = it.nkt * kKeys > it.ctx;  // only the last key tile can run past ctx
      // block ids of key tile kt (lane c < 8: chunk c), loaded one tile ahead
      // so the global load's latency passes while the ring waits and copies
      auto load_blk = [&](int kt) -> int {
        const int key0 = kt * kKeys;
        const int nch = min(kKeys / kChunk, (it.ctx - key0 + kChunk - 1) / kChunk);
        return lane < nch ? p.block_tables[(size_t)it.lane * p.max_blocks + (key0 + lane * kChunk) / p.bs]
                          : 0;
      };
      int blk_next = load_blk(0);
      // Q of this item's streams, once every S product of the previous item
      // (which read this buffer) has finished
      if (n >= 1 && !wait_or_abort(bqe, (n - 1) & 1, ab, p.status, lim)) break;
      if (lane == 0) {
        mbar_expect_tx(bq, it.nst * L::kQBytes);
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (s < it.nst) {
#pragma unroll
            for (int h = 0; h < L::kHalves; ++h)
              tma_load_3d(sQ + s * L::kQBytes + h * L::kHalfBytes, tmQ, h * 64, it.head,
                          it.cu0 + it.row0[s], bq);
          }
      }
      bool ok = true;
      for (int kt = 0; ok && kt < it.nkt; ++kt) {
        const uint32_t f = n_kv + kt, st = f % kStages, use = f / kStages;
        const int key0 = kt * kKeys;
        const int nchunk = min(kKeys / kChunk, (it.ctx - key0 + kChunk - 1) / kChunk);
        int blk = blk_next;  // block id of chunk `lane` (lanes 0..7)
        if (kt + 1 < it.nkt) blk_next = load_blk(kt + 1);
        if (lane < nchunk && (blk < 0 || blk >= p.NB)) {
          raise_flag(p.status, PA_FLAG_BLOCK_RANGE);
          blk = 0;
        }
        const uint32_t bytes = (uint32_t)nchunk * L::kHalves * kChunk * 128;
        // lane c (< nchunk) copies chunk c: the boxes go out in parallel
        const int tok = blk * p.bs + (key0 + lane * kChunk) % p.bs;
        ok = use < 1 || wait_or_abort(bke(st), (use - 1) & 1, ab, p.status, lim);
        if (!ok) break;
        if (lane == 0) mbar_expect_tx(bkf(st), bytes);
        __syncwarp();
        if (lane < nchunk) {
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sK0 + st * L::kKBytes + h * L::kKHalfBytes + lane * kChunk * 128, tmK,
                        h * 64, it.kvh, tok, bkf(st));
        }
        ok = use < 1 || wait_or_abort(bve(st), (use - 1) & 1, ab, p.status, lim);
        if (!ok) break;
        if (lane == 0) mbar_expect_tx(bvf(st), bytes);
        __syncwarp();
        if (lane < nchunk) {
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h)
            tma_load_3d(sV0 + st * L::kVBytes + h * L::kKHalfBytes + lane * kChunk * 128, tmV,
                        h * 64, it.kvh, tok, bvf(st));
        }
        if (kt == it.nkt - 1 && tail) {
          // keys past the lane's end: once the tile has landed, zero their V
          // rows (stale bytes must not meet p = 0 as 0 * NaN); the MMA warp
          // takes this tile from the vtail barrier
          ok = wait_or_abort(bvf(st), use & 1, ab, p.status, lim);
          if (!ok) break;
          const int first = it.ctx - key0;
          const int n16 = (kKeys - first) * 8 * L::kHalves;
          for (int i = lane; i < n16; i += 32) {
            const int c16 = i & 7, rest = i >> 3;
            const int h = rest % L::kHalves, r = first + rest / L::kHalves;
            const uint32_t a = sV0 + st * L::kVBytes + h * L::kKHalfBytes + r * 128 + c16 * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bvt(st));
        }
      }
      if (!ok) break;
      n_kv += it.nkt;
    }
  } else if (warp == 8) {
    // -------------------------------- MMA issuer ----------------------------
    // the whole warp runs the loop with warp-uniform operands; one elected
    // lane issues each product and commit. Descriptors of each operand tile
    // are built once and stepped by constant offsets (14-bit address field,
    // in 16-byte units).
    constexpr uint32_t idS = umma_idesc_bf16(kRows, kKeys, 0, 0);
    constexpr uint32_t idPV = umma_idesc_bf16(kRows, D, 0, 1);
    const uint64_t dQ0 = umma_desc_sw128(sQ, 16, 1024);
    const uint64_t dK0 = umma_desc_sw128(sK0, 16, 1024);
    const uint64_t dV0 = umma_desc_sw128(sV0, L::kKHalfBytes, 1024);
    // S of key tile j of the current item for stream s: A = Q tile, B = K tile
    auto issue_s = [&](int s, int j) {
      const uint32_t st = (n_kv + j) % kStages;
      const uint64_t dq = dQ0 + (uint64_t)((s * L::kQBytes) >> 4);
      const uint64_t dk = dK0 + (uint64_t)((st * L::kKBytes) >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t oq = ((kk >> 2) * L::kHalfBytes + (kk & 3) * 32) >> 4;
        const uint32_t ok = ((kk >> 2) * L::kKHalfBytes + (kk & 3) * 32) >> 4;
        umma_bf16_w(tS(s), dq + oq, dk + ok, idS, kk > 0 ? 1u : 0u);
      }
      umma_commit_w(bS(s));
    };
    auto issue_pv = [&](int s, int j, uint32_t ts) {
      const uint32_t st = (n_kv + j) % kStages;
      const uint64_t dv = dV0 + (uint64_t)((st * L::kVBytes) >> 4);
#pragma unroll
      for (int k = 0; k < kKeys / 16; ++k)
        umma_bf16_tmem_a_w(tO(s), tS(s) + k * 8, dv + (uint64_t)((k * 16 * 128) >> 4), idPV,
                           (j > 0 || k > 0) ? 1u : 0u);
      umma_commit_w(bO(s, ts));
    };
    for (;; ++n_item) {
      long long item;
      if (!read_item(n_item, item) || item >= n_items) break;
      const ItemInfo it = item_info(p, (int)item);
      const bool tail = it.nkt * kKeys > it.ctx;
      bool ok = true;
      // first S of the item for each stream, once Q and K tile 0 have landed
      // and the stream's last P V (of an earlier item), which reads the P
      // this S overwrites, has finished
      {
        const uint32_t f = n_kv, st = f % kStages;
        ok = wait_or_abort(bkf(st), (f / kStages) & 1, ab, p.status, lim) &&
             wait_or_abort(bq, n_item & 1, ab, p.status, lim);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (!ok || s >= it.nst) break;
          const uint32_t nts = s ? n_t1 : n_t0;
          if (nts > 0) ok = wait_or_abort(bO(s, nts - 1), ((nts - 1) >> 1) & 1, ab, p.status, lim);
          if (!ok) break;
          tc_fence_after();
          issue_s(s, 0);
        }
        if (!ok) break;
        umma_commit_w(bke(st));
        if (it.nkt == 1) umma_commit_w(bqe);  // every S of the item issued
      }
      for (int kt = 0; ok && kt < it.nkt; ++kt) {
        const uint32_t f = n_kv + kt, st = f % kStages;
        const bool next = kt + 1 < it.nkt;
        const uint32_t f1 = f + 1, st1 = f1 % kStages;
        // V of tile kt (the tail tile once its stale rows are zeroed)
        if (kt == it.nkt - 1 && tail) {
          ok = wait_or_abort(bvt(st), (tail_par >> st) & 1, ab, p.status, lim);
          tail_par ^= 1u << st;
        } else {
          ok = wait_or_abort(bvf(st), (f / kStages) & 1, ab, p.status, lim);
        }
        if (!ok) break;
        // per stream: P V of tile kt, once its softmax has written P, then S
        // of tile kt + 1, which overwrites P of tile kt in TMEM and so waits
        // for that P V to finish; the streams alternate, so one stream's
        // softmax runs while the tensor core serves the other
        bool k_ready = false;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (!ok || s >= it.nst) break;
          if (kt >= it.nkt_s[s]) continue;
          const uint32_t ts = (s ? n_t1 : n_t0) + kt;
          ok = wait_or_abort(bP(s), ts & 1, ab, p.status, lim);
          if (!ok) break;
          tc_fence_after();
          issue_pv(s, kt, ts);
          if (kt + 1 >= it.nkt_s[s]) continue;
          if (!k_ready) {
            ok = wait_or_abort(bkf(st1), (f1 / kStages) & 1, ab, p.status, lim);
            k_ready = true;
          }
          ok = ok && wait_or_abort(bO(s, ts), (ts >> 1) & 1, ab, p.status, lim);
          if (!ok) break;
          tc_fence_after();
          issue_s(s, kt + 1);
        }
        if (!ok) break;
        // Q is free once the item's last S products finish (tile nkt - 1's)
        if (kt + 2 == it.nkt) umma_commit_w(bqe);
        umma_commit_w(bve(st));
        if (next) umma_commit_w(bke(st1));
      }
      if (!ok) break;
      n_kv += it.nkt;
      n_t0 += it.nkt_s[0];
      n_t1 += it.nkt_s[1];
    }
  } else {
    // -------------------------------- softmax rows --------------------------
    const int s = warp >> 2;          // stream of this group
    const int r = threadIdx.x & 127;  // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tOr = tO(s) + lane_off;
    const uint32_t tSr = tS(s) + lane_off;
    for (;; ++n_item) {
      long long item;
      if (!read_item(n_item, item) || item >= n_items) break;
      const ItemInfo it = item_info(p, (int)item);
      if (s >= it.nst) continue;  // the pair has no second tile
      // this stream's values as scalars (selects, not a run-time index)
      const int nkt_s = s ? it.nkt_s[1] : it.nkt_s[0];
      const int nrows = s ? it.nrows[1] : it.nrows[0];
      const int row0 = s ? it.row0[1] : it.row0[0];
      const uint32_t nts = s ? n_t1 : n_t0;
      const int pos = (s ? it.p_first[1] : it.p_first[0]) + min(r, nrows - 1);
      float m = -INFINITY, l = 0.f;
      bool ok = true;
#pragma unroll 1
      for (int kt = 0; kt < nkt_s; ++kt) {
        const uint32_t th = nts + kt;
        if (!wait_or_abort(bS(s), th & 1, ab, p.status, lim)) { ok = false; break; }
        tc_fence_after();
        const int lim_c = pos - kt * kKeys;  // columns c <= lim_c are visible to this row
        const bool full = __all_sync(0xffffffffu, lim_c >= kKeys - 1);
        // pass 1: max of the visible raw scores (the scale is positive), in
        // 32-column chunks two at a time; eight independent running maxima
        // folded by a fixed tree
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = -INFINITY;
#pragma unroll
        for (int c2p = 0; c2p < kKeys / 64; ++c2p) {
          uint32_t a[32], b[32];
          tmem_ld32(tSr + 64 * c2p, a);
          tmem_ld32(tSr + 64 * c2p + 32, b);
          tmem_wait_ld();
          if (full) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              m8[(i >> 1) & 3] = fmax3(m8[(i >> 1) & 3], __uint_as_float(a[i]), __uint_as_float(a[i + 1]));
              m8[4 + ((i >> 1) & 3)] =
                  fmax3(m8[4 + ((i >> 1) & 3)], __uint_as_float(b[i]), __uint_as_float(b[i + 1]));
            }
          } else {
            const int c0 = 64 * c2p;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              m8[i & 3] = fmaxf(m8[i & 3], c0 + i <= lim_c ? __uint_as_float(a[i]) : -INFINITY);
              m8[4 + (i & 3)] =
                  fmaxf(m8[4 + (i & 3)], c0 + 32 + i <= lim_c ? __uint_as_float(b[i]) : -INFINITY);
            }
          }
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int j = 0; j < w; ++j) m8[j] = fmaxf(m8[j], m8[j + w]);
        const float mx = m8[0] * c2;
        const bool grow = kt == 0 || mx > m + kRescaleLog2;
        const float mn = grow ? fmaxf(m, mx) : m;
        const float alpha = grow ? ex2_approx(m - mn) : 1.f;
        m = mn;
        const float neg = -mn;
        // pass 2: p = 2^(s c2 - m) rounded to bf16, written over S as P (two
        // per column: chunk c of 32 scores becomes P columns 16 c .. 16 c + 15,
        // all of them already read); the next chunk's scores are loaded while
        // this one is computed. l adds the p before rounding, in four
        // independent pairs of partial sums folded by a fixed tree. The
        // scaling runs on packed fp32 pairs (lane by lane the same fmaf).
        const uint64_t c2x2 = f32x2(c2, c2), negx2 = f32x2(neg, neg);
        uint64_t r4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) r4[j] = f32x2(0.f, 0.f);
        uint32_t cur[32], nxt[32];
        tmem_ld32(tSr, cur);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c) {
          if (c + 1 < kKeys / 32) tmem_ld32(tSr + 32 * (c + 1), nxt);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = 32 * c + 2 * i;
            float t0, t1;
            f32x2_split(fma_f32x2(f32x2(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])),
                                  c2x2, negx2),
                        t0, t1);
            float e0 = ex2_approx(t0);
            float e1 = ex2_approx(t1);
            if (!full) {
              e0 = (col <= lim_c) ? e0 : 0.f;
              e1 = (col + 1 <= lim_c) ? e1 : 0.f;
            }
            pk[i] = pack_bf16x2(e0, e1);
            r4[i & 3] = add_f32x2(r4[i & 3], f32x2(e0, e1));
          }
          tmem_st16(tSr + 16 * c, pk);
          if (c + 1 < kKeys / 32) {
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) cur[i] = nxt[i];
          }
        }
        r4[0] = add_f32x2(r4[0], r4[2]);
        r4[1] = add_f32x2(r4[1], r4[3]);
        r4[0] = add_f32x2(r4[0], r4[1]);
        float rlo, rhi;
        f32x2_split(r4[0], rlo, rhi);
        const float rs = rlo + rhi;
        tmem_wait_st();
        l = fmaf(l, alpha, rs);
        // O is rescaled after P V of the previous tile has finished (it has:
        // S of this tile was issued after it); P V completions alternate
        // between two barriers by tile parity, so a barrier is never more
        // than one phase away from any wait on it even when tiles without a
        // rescale skip the wait.
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!wait_or_abort(bO(s, th - 1), ((th - 1) >> 1) & 1, ab, p.status, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tOr + c * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tOr + c * 32, ov);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(bP(s));
      }
      if (!ok) break;
      // the row's output once its last P V has finished; the next item's
      // first P V (which restarts O) waits for this group's first P of that
      // item, which comes after these reads
      const uint32_t last = nts + nkt_s - 1;
      if (!wait_or_abort(bO(s, last), (last >> 1) & 1, ab, p.status, lim)) break;
      tc_fence_after();
      const bool valid = r < nrows;
      const float inv_l = 1.f / l;  // one division per row; out = O * (1 / l)
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) +
                           ((size_t)(it.cu0 + row0 + r) * p.H + it.head) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tOr + c * 32, ov);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(ov[i]) * inv_l, __uint_as_float(ov[i + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(ov[i + 2]) * inv_l, __uint_as_float(ov[i + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(ov[i + 4]) * inv_l, __uint_as_float(ov[i + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(ov[i + 6]) * inv_l, __uint_as_float(ov[i + 7]) * inv_l);
            *reinterpret_cast<uint4*>(out + c * 32 + i) = v;
          }
        }
      }
      tc_fence_before();
      if (s) n_t1 += nkt_s; else n_t0 += nkt_s;
    }
  }
  // before TMEM is released and the CTA leaves: every product the MMA warp
  // issued has completed (a commit tracks all of them), and every copy the
  // TMA warp issued has landed (on an abort some may still be in flight; on
  // a normal exit the waits return at once)
  if (warp == 8) {
    umma_commit_w(smem_u32(&bars.fin));
    mbar_wait_bounded(smem_u32(&bars.fin), 0, lim);
  }
  if (warp == 9 && lane == 0) {
    if (n_item > 0) mbar_wait_bounded(bq, (n_item - 1) & 1, lim);
    for (uint32_t f = n_kv > kStages ? n_kv - kStages : 0; f < n_kv; ++f) {
      mbar_wait_bounded(bkf(f % kStages), (f / kStages) & 1, lim);
      mbar_wait_bounded(bvf(f % kStages), (f / kStages) & 1, lim);
    }
  }
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace pftc
}  // namespace pa
