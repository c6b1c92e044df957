// Shared device-side definitions of libpa: launch parameters, the split plan
// stored in the caller's workspace, and thin wrappers over the PTX
// instructions the kernels issue (mbarrier, TMA, ldmatrix, mma, movmatrix).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Split-KV partition of a row with K keys: ranges of split_len(K) keys,
// split_len(K) = kSplit * 2^j for the smallest j giving at most kMaxSplits
// ranges. A function of K alone, so a row's split points never depend on
// what else is in the step (rows up to 65536 keys use 512-key splits).
constexpr int kSplit = 512;
constexpr int kMaxSplits = 128;

__host__ __device__ __forceinline__ int split_len(int keys) {
  int s = kSplit;
  while ((keys + s - 1) / s > kMaxSplits) s <<= 1;
  return s;
}
// Keys per pipeline stage of the split kernels (one mma M tile).
constexpr int kChunk = 16;
// Bounded waits give up after this many SM clock cycles (about 1 s) unless
// a step carries another limit (StepParams::wait_cycles).
constexpr long long kWaitCycles = 2000000000LL;

// ---------------------------------------------------------------------------
// Split plan, built on the device by the prologue kernel from cu_seqlens_q and
// ctx_lens, stored in the workspace:
//   header[0] = number of (row, split) pairs, header[1] = number of full pairs,
//   header[2] = number of prefill q-tile pairs, header[3] = number of prefill-row
//   group records, header[4 + 2 c .. 5 + 2 c] = item counter c (64-bit,
//   zeroed with the plan): c = 0 the split kernels, 1 the tensor-core
//   prefill, 2 the prefill-row kernel; header[kHeaderSplitKeys],
//   header[kHeaderPrefillWork] (64-bit) = the step's work totals
//   (full pairs of rows with longer splits come first, then full 512-key
//   pairs, then tails: roughly largest first, the order items are taken in)
//   (pair k < header[1] sits at pairs[k]; tail pair k >= header[1] at
//   pairs[capacity - 1 - (k - header[1])], see pair_slot)
//   row_info[r] = {first full pair, tail pair or -1, number of splits, lane or -1}
//   pairs[k]    = {row, split index, lane, key count of the row}
//   crows[k]    = {row, first full pair, tail pair or -1, number of splits}
//                 of the k-th row the combine folds (rows with 2 or more
//                 splits -- every split row when merging KV-parallel
//                 owners), most splits first; header[kHeaderCombineRows] of
//                 them (not kept when prefill rows take the split path).
//                 The entry repeats the row's row_info so a combine warp
//                 reaches its partials with one dependent load less.
//   ptiles[i]   = {lane, index t of the pair of 128-row q tiles 2 t and
//                 2 t + 1, position of the pair's last row, 0}, heaviest
//                 first (tensor-core prefill path)
// Full pairs (exactly kSplit keys) come first, lane-major; tail pairs after.
// row_info.y holds the tail pair's slot itself.
// Partial results of pair k: ml[k * H + h] = {m (log2 domain), l},
// acc[(k * H + h) * D + d].
// ---------------------------------------------------------------------------
struct SplitPlan {
  int* header;
  int4* row_info;
  int4* ptiles;
  int4* ptiles_tmp;  // unsorted list, scratch of the plan
  int4* pairs;
  int4* crows;  // rows whose splits the combine folds, most splits first
  float2* ml;
  float* acc;
  int capacity;        // pairs the workspace holds
  int ptile_capacity;  // prefill tiles the workspace holds
  long long entry_capacity;  // KV-parallel modes: entries the partial buffer holds
};

// Item counters: each worker (a warp of the split kernels, a CTA of the
// prefill kernels) takes its next item from one, in list order.
constexpr int kCounterSplit = 0, kCounterPrefill = 1, kCounterRows = 2, kItemCounters = 3;
// 64-bit work totals of the step, for the mixed-step kernel's role split:
// keys of the rows on the split path, and the (row, key) pairs the prefill
// tiles' rows attend
constexpr int kHeaderSplitKeys = 4 + 2 * kItemCounters;
constexpr int kHeaderPrefillWork = kHeaderSplitKeys + 2;
// prefill-role CTAs of the mixed-step kernel, chosen by the plan builder
constexpr int kHeaderPrefillCtas = kHeaderPrefillWork + 2;
// rows the combine folds (the length of crows)
constexpr int kHeaderCombineRows = kHeaderPrefillCtas + 1;
// 1 when the plan in the workspace was built for this call's sizes (the
// builder sets it; a call that reuses the plan sets it from the fingerprint
// check, and on a mismatch also empties the plan's item counts and combine
// list, so the kernels after the prologue find no work)
constexpr int kHeaderPlanOk = kHeaderCombineRows + 1;
// the sizes the plan was built for (plan_fingerprint), compared by calls
// that reuse it
constexpr int kHeaderFingerprint = kHeaderPlanOk + 1;
constexpr int kFingerprintInts = 14;
__device__ __forceinline__ long long* header_total(const SplitPlan& pl, int at) {
  return reinterpret_cast<long long*>(pl.header + at);
}
__device__ __forceinline__ unsigned long long* item_counter(const SplitPlan& pl, int c) {
  return reinterpret_cast<unsigned long long*>(pl.header + 4 + 2 * c);
}

// Slot of the k-th pair in work order: full pairs from the front of the
// list, tail pairs from its back.
__device__ __forceinline__ int pair_slot(const SplitPlan& pl, int k, int nfull) {
  return k < nfull ? k : pl.capacity - 1 - (k - nfull);
}

// Query rows per tile of the tensor-core prefill path.
constexpr int kPrefillRows = 128;
// Consumer warps of the row-invariant prefill-row kernel; a group holds
// kRowWarps rows per row a warp carries.
constexpr int kRowWarps = 8;

struct StepParams {
  const void* q;
  void* out;
  const void* k_cache;
  const void* v_cache;
  const int* block_tables;
  const int* cu_seqlens;
  const int* ctx_lens;
  const int64_t* slot_mapping;
  const void* k_new;
  const void* v_new;
  int* status;
  int max_blocks;
  int B, T, H, Hkv, D, bs, NB;
  int max_q_len, max_ctx_len;
  int elem_bytes;
  int split_all_rows;  // 1: every row takes the split path; 0: lanes with q_len == 1 only
  int kv_fp8;          // 1: caches hold e4m3 codes (q, out and new rows stay bf16)
  float scale;
  float scale_log2;  // scale * log2(e) (* k_scale for e4m3 caches): base-2 score domain
  float k_scale, v_scale;  // per-tensor scales of e4m3 caches (1 otherwise)
  float out_scale;   // factor on every normalised output: v_scale for e4m3, else 1
  // KV-parallel page owners: 0 = an ordinary step; 1 = this owner's partials
  // (splits whose first key lies in [key_lo, key_hi) of the lane) written to
  // canonical entries row_info[row].x + split of the plan's ml / acc;
  // 2 = merge: fold every row's splits, split i read from the owner whose
  // range [key_bounds[w][lane], key_bounds[w + 1][lane]) holds its first key.
  // In modes 1 and 2 row_info[row] = {first entry, key count, splits, lane}.
  // bf16 row-invariant steps: the rows of lanes with q_len >= 2 are computed
  // in groups of up to group_rows consecutive rows sharing key tiles (their
  // partials at row_info[row].x + split, the group records after the full
  // pairs: pairs[header[1] + k], header[3] of them); decode lanes as usual.
  // 0: no grouping.
  int group_rows;
  int sm_count;  // SMs of the device (the mixed-step kernel's grid)
  int partials_mode;
  // every bounded wait of the step's kernels gives up after this many SM
  // clock cycles (kWaitCycles unless a test shortened it)
  long long wait_cycles;
  // test hook, -1 normally: the split kernel's producer issues no copy for
  // the first chunk of this item, so the consumer's bounded wait on it runs
  // out (PA_FLAG_TIMEOUT) -- how the tests make a wait expire without any
  // fault
  long long skip_item;
  const int* key_lo;
  const int* key_hi;
  const int* key_bounds;        // [owners + 1][B]
  int owners;
  long long owner_stride;       // bytes between owners' buffers
  SplitPlan plan;
};

// Whether the plan in the workspace belongs to this call (see kHeaderPlanOk);
// uniform across the grid, so a kernel tests it once at entry.
__device__ __forceinline__ bool plan_ok(const StepParams& p) {
  return p.plan.header[kHeaderPlanOk] != 0;
}

// Entry i < kFingerprintInts of the sizes a split plan depends on (besides
// the contents of cu_seqlens_q and ctx_lens, which a caller that reuses the
// plan vouches for).
__device__ __forceinline__ int plan_fingerprint(const StepParams& p, int i) {
  switch (i) {
    case 0: return p.B;
    case 1: return p.T;
    case 2: return p.H;
    case 3: return p.Hkv;
    case 4: return p.D;
    case 5: return p.bs;
    case 6: return p.elem_bytes;
    case 7: return p.split_all_rows;
    case 8: return p.group_rows;
    case 9: return p.max_q_len;
    case 10: return p.max_ctx_len;
    case 11: return p.plan.capacity;
    case 12: return p.sm_count;
    default: return p.partials_mode * 4 + p.kv_fp8;
  }
}

// Canonical partial entry of (row, split) in the KV-parallel modes, else the
// pair's own slot.
__device__ __forceinline__ long long partial_entry(const StepParams& p, int pair, int row,
                                                   int split) {
  return p.partials_mode ? (long long)p.plan.row_info[row].x + split : (long long)pair;
}

// Opt a kernel in to `bytes` of dynamic shared memory once per device (the
// attribute is per device and sticky; later calls only read a flag).
template <typename Kernel>
inline cudaError_t smem_opt_in(Kernel kern, int bytes, unsigned long long* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
  return e;
}

__device__ __forceinline__ void raise_flag(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Normalised output of one (row, head, dim): shared by the single-split
// direct write and the combine so both round the same quotient.
__device__ __forceinline__ float finish_div(float acc, float l) { return acc / l; }

// Left fold of one more split (m_i, l_i, a_i) into (M, L, A), fp32.
struct Fold {
  float M, L;
  __device__ __forceinline__ void first(float m, float l) { M = m; L = l; }
  // Returns the two rescale factors for the accumulators.
  __device__ __forceinline__ void next(float m, float l, float& ea, float& eb) {
    const float Mn = fmaxf(M, m);
    ea = exp2f(M - Mn);
    eb = exp2f(m - Mn);
    L = fmaf(L, ea, l * eb);
    M = Mn;
  }
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most `limit`
// SM cycles. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// 3-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// L2 eviction policies (createpolicy): keys streamed once go first, split
// partials that the combine reads soon after stay longest.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 int z, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void st_hint(float* ptr, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint(float2* ptr, float2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(ptr), "f"(v.x), "f"(v.y),
               "l"(pol)
               : "memory");
}

// 2-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two fp32 values rounded to f16 (RN), lo in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float f16_lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// Two e4m3 codes (low byte -> low half) to f16x2; exact: every e4m3 value
// is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  const unsigned short h = (unsigned short)(two_codes & 0xffffu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}

// Two fp32 values to e4m3 codes (RN, finite overflow and infinities
// saturate to +-448, NaN stays NaN); lo goes to the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Store an fp32 value as the output element type.
__device__ __forceinline__ void store_out(void* out, size_t idx, float v, int elem_bytes) {
  if (elem_bytes == 4) {
    static_cast<float*>(out)[idx] = v;
  } else {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  }
}

}  // namespace pa
