// C ABI of libpa: host-side validation, workspace layout, tensor-map encoding
// and launch sequencing. Declarations and contracts are in include/pa.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pa_common.cuh"
#include "pa_test.h"

namespace pa {

cudaError_t launch_prologue(const StepParams& p, int plan_mode, bool write, cudaStream_t s);
cudaError_t launch_decode_bf16(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v,
                               long long max_items, cudaStream_t s);
cudaError_t launch_decode_fp8(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v,
                              long long max_items, cudaStream_t s);
cudaError_t launch_split_f32(const StepParams& p, long long max_items, cudaStream_t s);
int rows_group_size(int g);
cudaError_t launch_combine(const StepParams& p, cudaStream_t s);
cudaError_t launch_mixed(const StepParams& p, const CUtensorMap& q, const CUtensorMap& k,
                         const CUtensorMap& v, cudaStream_t s);
cudaError_t launch_row_mixed(const StepParams& p, const CUtensorMap& k, const CUtensorMap& v,
                             cudaStream_t s);

void decode_gemm_plan(int N, int K, int* S, int* chunks_per_split);
cudaError_t launch_decode_gemm(void* y, float* part, int T_pad, int N, int K, int S, int cps,
                               int* status, const CUtensorMap& w, const CUtensorMap& x,
                               cudaStream_t s);

static std::atomic<long long> g_launches{0};

// Test hooks (include/pa_test.h): the wait limit every step's kernels get,
// and the split item whose first copy is never issued (-1: none).
static std::atomic<long long> g_wait_cycles{kWaitCycles};
static std::atomic<long long> g_skip_item{-1};

void apply_test_hooks(StepParams& p) {
  p.wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
  p.skip_item = g_skip_item.load(std::memory_order_relaxed);
}

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Bytes of a q / out / new-row element (bf16 for e4m3 caches).
int elem_bytes_of(pa_dtype d) { return d == PA_F32 ? 4 : 2; }

bool scales_ok(float k_scale, float v_scale) {
  return std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f;
}

pa_status check_geometry(int32_t H, int32_t Hkv, int32_t D, int32_t block_size, pa_dtype dtype) {
  if (H <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
  if (H % Hkv != 0 || H / Hkv > 16) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// Every row takes the split path for fp32 (CUDA-core FMA, no TF32), for
// e4m3 caches and in the row-invariant mode. Otherwise (bf16) only decode
// lanes (q_len == 1) do; lanes with q_len >= 2 go to the tensor-core prefill
// kernel.
bool split_all_rows(pa_dtype dtype, pa_mode mode) {
  return dtype != PA_BF16 || mode == PA_MODE_ROW_INVARIANT;
}

// The invariance mode of a pa_mode value (the PA_MODE_REUSE_PLAN bit taken off).
pa_mode invariance_of(pa_mode mode) {
  return static_cast<pa_mode>(static_cast<int>(mode) & ~static_cast<int>(PA_MODE_REUSE_PLAN));
}
bool reuses_plan(pa_mode mode) {
  return (static_cast<int>(mode) & static_cast<int>(PA_MODE_REUSE_PLAN)) != 0;
}
bool mode_known(pa_mode mode) {
  const pa_mode m = invariance_of(mode);
  return m == PA_MODE_BATCH_INVARIANT || m == PA_MODE_ROW_INVARIANT;
}

// Prefill tiles a step can hold: sum over lanes of ceil(q_len / 128).
long long max_prefill_tiles(int32_t B, int32_t T) { return (long long)T / kPrefillRows + B + 1; }

struct Layout {
  size_t header, row_info, ptiles, ptiles_tmp, crows, pairs, fixed, per_pair;
  int ptile_capacity;
};

Layout layout_for(int32_t B, int32_t T, int32_t H, int32_t D) {
  Layout L;
  L.ptile_capacity = (int)max_prefill_tiles(B, T);
  L.header = 0;
  L.row_info = kAlign;
  L.ptiles = L.row_info + align_up((size_t)T * sizeof(int4));
  L.ptiles_tmp = L.ptiles + align_up((size_t)L.ptile_capacity * sizeof(int4));
  L.crows = L.ptiles_tmp + align_up((size_t)L.ptile_capacity * sizeof(int4));
  L.pairs = L.crows + align_up((size_t)T * sizeof(int4));
  L.fixed = L.pairs;
  L.per_pair = sizeof(int4) + (size_t)H * sizeof(float2) + (size_t)H * D * sizeof(float);
  return L;
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Upper bound on (row, split) pairs of a step (split_len(K) >= kSplit, so a
// row of K keys has at most ceil(K / kSplit) splits).
long long max_pairs(int32_t B, int32_t T, int32_t max_ctx_len, int64_t total_ctx,
                    pa_dtype dtype, pa_mode mode) {
  const long long per_row = ceil_div(max_ctx_len > 0 ? max_ctx_len : 1, kSplit);
  if (split_all_rows(dtype, mode)) return (long long)T * per_row;
  long long loose = (long long)(B < T ? B : T) * per_row;
  if (total_ctx >= 0) {
    const long long tight = total_ctx / kSplit + B;
    if (tight < loose) loose = tight;
  }
  return loose;
}

size_t bytes_for_pairs(int32_t B, int32_t T, int32_t H, int32_t D, long long pairs) {
  const Layout L = layout_for(B, T, H, D);
  // pairs, ml and acc as three arrays, each 256-byte aligned
  return L.fixed + align_up((size_t)pairs * sizeof(int4)) +
         align_up((size_t)pairs * H * sizeof(float2)) +
         align_up((size_t)pairs * H * D * sizeof(float));
}

int capacity_of(size_t bytes, int32_t B, int32_t T, int32_t H, int32_t D) {
  const Layout L = layout_for(B, T, H, D);
  if (bytes <= L.fixed) return 0;
  long long cap = (long long)((bytes - L.fixed) / L.per_pair);
  while (cap > 0 && bytes_for_pairs(B, T, H, D, cap) > bytes) --cap;
  if (cap > 0x7fffffffLL) cap = 0x7fffffffLL;
  return (int)cap;
}

SplitPlan carve(void* ws, int cap, int32_t B, int32_t T, int32_t H, int32_t D) {
  const Layout L = layout_for(B, T, H, D);
  char* b = static_cast<char*>(ws);
  SplitPlan pl;
  pl.header = reinterpret_cast<int*>(b + L.header);
  pl.row_info = reinterpret_cast<int4*>(b + L.row_info);
  pl.ptiles = reinterpret_cast<int4*>(b + L.ptiles);
  pl.ptiles_tmp = reinterpret_cast<int4*>(b + L.ptiles_tmp);
  pl.ptile_capacity = L.ptile_capacity;
  pl.crows = reinterpret_cast<int4*>(b + L.crows);
  size_t off = L.pairs;
  pl.pairs = reinterpret_cast<int4*>(b + off);
  off += align_up((size_t)cap * sizeof(int4));
  pl.ml = reinterpret_cast<float2*>(b + off);
  off += align_up((size_t)cap * H * sizeof(float2));
  pl.acc = reinterpret_cast<float*>(b + off);
  pl.capacity = cap;
  return pl;
}

// ---- KV-parallel partial buffers ----
// Entries of a step's partial buffer: every row has at most
// ceil(max_ctx_len / kSplit) splits.
long long partial_entries(int32_t T, int32_t max_ctx_len) {
  return (long long)T * ceil_div(max_ctx_len > 0 ? max_ctx_len : 1, kSplit);
}

size_t partials_ml_bytes(long long entries, int32_t H) {
  return align_up((size_t)entries * H * sizeof(float2));
}

size_t partials_bytes_for(int32_t T, int32_t max_ctx_len, int32_t H, int32_t D) {
  const long long e = partial_entries(T, max_ctx_len);
  return partials_ml_bytes(e, H) + align_up((size_t)e * H * D * sizeof(float));
}

// Workspace of the KV-parallel calls: the plan's fixed part and one pair
// record per split this owner may compute (no partials: those go to the
// caller's buffer).
size_t partials_ws_bytes(int32_t B, int32_t T, int32_t max_ctx_len) {
  const Layout L = layout_for(B, T, 1, 1);
  return L.fixed + align_up((size_t)partial_entries(T, max_ctx_len) * sizeof(int4));
}

SplitPlan carve_partials(void* ws, size_t ws_bytes, void* partials, int32_t B, int32_t T,
                         int32_t H, int32_t max_ctx_len) {
  const Layout L = layout_for(B, T, 1, 1);
  char* b = static_cast<char*>(ws);
  SplitPlan pl;
  pl.header = reinterpret_cast<int*>(b + L.header);
  pl.row_info = reinterpret_cast<int4*>(b + L.row_info);
  pl.ptiles = reinterpret_cast<int4*>(b + L.ptiles);
  pl.ptiles_tmp = reinterpret_cast<int4*>(b + L.ptiles_tmp);
  pl.ptile_capacity = L.ptile_capacity;
  pl.crows = reinterpret_cast<int4*>(b + L.crows);
  pl.pairs = reinterpret_cast<int4*>(b + L.pairs);
  long long cap = ws_bytes > L.fixed ? (long long)((ws_bytes - L.fixed) / sizeof(int4)) : 0;
  pl.capacity = (int)(cap > 0x7fffffffLL ? 0x7fffffffLL : cap);
  const long long e = partial_entries(T, max_ctx_len);
  char* pb = static_cast<char*>(partials);
  pl.ml = reinterpret_cast<float2*>(pb);
  pl.acc = reinterpret_cast<float*>(pb + partials_ml_bytes(e, H));
  pl.entry_capacity = e;
  return pl;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [NB * bs tokens, Hkv, D] bf16 cache; box = 64 elements x 1 head x 16 tokens,
// 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* cache, int NB, int bs, int Hkv, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)NB * (cuuint64_t)bs};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kChunk};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(cache), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [NB * bs tokens, Hkv, D] e4m3 code cache; box = D bytes x 1 head x 16
// tokens, 128-byte swizzle for D = 128 and 64-byte swizzle for D = 64 (the
// box row is the whole swizzle span either way).
bool encode_code_map(CUtensorMap* map, const void* cache, int NB, int bs, int Hkv, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)NB * (cuuint64_t)bs};
  cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)Hkv * D};
  cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)kChunk};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(cache), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major [rows, K] bf16 matrix; box = 64 elements x box_rows rows, 128-byte swizzle.
bool encode_rows_map(CUtensorMap* map, const void* ptr, int rows, int K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool gemm_shape_ok(int32_t T_pad, int32_t N, int32_t K) {
  const bool tp = T_pad == 32 || T_pad == 64 || T_pad == 96 || T_pad == 128 || T_pad == 192 ||
                  T_pad == 256;
  return tp && N > 0 && K > 0 && N % 128 == 0 && K % 64 == 0 && (long long)N * K < (1LL << 40);
}

// q [T, H, D] bf16; box = 64 elements x 1 head x 128 rows, 128-byte swizzle.
bool encode_q_map(CUtensorMap* map, const void* q, int T, int H, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kPrefillRows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Record a phase event. Under stream capture it becomes an event-record node
// of the graph (recorded at every replay) rather than a capture dependency.
pa_status record(void* const* events, int32_t n_events, int idx, cudaStream_t s) {
  if (events && idx < n_events && events[idx]) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return PA_ERR_CUDA;
    const cudaEvent_t ev = static_cast<cudaEvent_t>(events[idx]);
    const cudaError_t e = cs == cudaStreamCaptureStatusActive
                              ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                              : cudaEventRecord(ev, s);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
  }
  return "PA_ERR_UNKNOWN";
}

int64_t pa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t pa_split_tokens(void) { return kSplit; }

pa_status pa_write_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int32_t T, int32_t num_blocks,
                      int32_t block_size, int32_t Hkv, int32_t D, pa_dtype dtype,
                      int32_t* status, void* stream) {
  if (dtype == PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;  // needs the scales
  return pa_write_kv_scaled(k_new, v_new, k_cache, v_cache, slot_mapping, T, num_blocks,
                            block_size, Hkv, D, dtype, 1.f, 1.f, status, stream);
}

pa_status pa_write_kv_scaled(const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, const int64_t* slot_mapping, int32_t T,
                             int32_t num_blocks, int32_t block_size, int32_t Hkv, int32_t D,
                             pa_dtype dtype, float k_scale, float v_scale, int32_t* status,
                             void* stream) {
  if (T < 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  pa_status g = check_geometry(Hkv, Hkv, D, block_size, dtype);
  if (g != PA_OK) return g;
  const bool fp8 = dtype == PA_FP8_E4M3;
  if (fp8 && !scales_ok(k_scale, v_scale)) return PA_ERR_INVALID_ARG;
  if (T == 0) return PA_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  StepParams p;
  std::memset(&p, 0, sizeof(p));
  apply_test_hooks(p);
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_new = k_new;
  p.v_new = v_new;
  p.slot_mapping = slot_mapping;
  p.status = status;
  p.T = T;
  p.Hkv = Hkv;
  p.H = Hkv;
  p.D = D;
  p.bs = block_size;
  p.NB = num_blocks;
  p.elem_bytes = elem_bytes_of(dtype);
  p.kv_fp8 = fp8 ? 1 : 0;
  p.k_scale = fp8 ? k_scale : 1.f;
  p.v_scale = fp8 ? v_scale : 1.f;
  cudaError_t e = launch_prologue(p, 0, true, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  return PA_OK;
}

size_t pa_attention_workspace_bytes_ex(int32_t B, int32_t T, int32_t max_q_len,
                                       int32_t max_ctx_len, int64_t total_ctx, int32_t H,
                                       int32_t Hkv, int32_t D, int32_t block_size,
                                       pa_dtype dtype, pa_mode mode) {
  if (B < 0 || T < 0 || max_q_len < 0 || max_ctx_len < 0 || !mode_known(mode)) return 0;
  mode = invariance_of(mode);
  if (check_geometry(H, Hkv, D, block_size, dtype) != PA_OK) return 0;
  const long long pairs = max_pairs(B, T, max_ctx_len, total_ctx, dtype, mode);
  return bytes_for_pairs(B, T, H, D, pairs > 0 ? pairs : 1);
}

size_t pa_attention_workspace_bytes(int32_t B, int32_t T, int32_t max_q_len,
                                    int32_t max_ctx_len, int64_t total_ctx, int32_t H,
                                    int32_t Hkv, int32_t D, int32_t block_size,
                                    pa_dtype dtype) {
  return pa_attention_workspace_bytes_ex(B, T, max_q_len, max_ctx_len, total_ctx, H, Hkv, D,
                                         block_size, dtype, PA_MODE_BATCH_INVARIANT);
}

pa_status pa_attention_ex(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                          const int64_t* slot_mapping, const void* k_new, const void* v_new,
                          void* out, int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t D,
                          int32_t block_size, int32_t num_blocks, int32_t max_q_len,
                          int32_t max_ctx_len, float scale, pa_dtype dtype, void* workspace,
                          size_t workspace_bytes, int32_t* status, void* stream,
                          float k_scale, float v_scale, pa_mode mode, void* const* events,
                          int32_t n_events) {
  // ---- host validation: nothing below touches CUDA until it all passes ----
  if (B < 0 || T < 0 || num_blocks <= 0 || max_q_len < 0 || max_ctx_len < 0 || n_events < 0 ||
      !mode_known(mode))
    return PA_ERR_INVALID_ARG;
  const bool reuse = reuses_plan(mode);
  mode = invariance_of(mode);
  pa_status g = check_geometry(H, Hkv, D, block_size, dtype);
  if (g != PA_OK) return g;
  if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
  const bool fp8 = dtype == PA_FP8_E4M3;
  if (fp8 && !scales_ok(k_scale, v_scale)) return PA_ERR_INVALID_ARG;
  const bool with_write = slot_mapping || k_new || v_new;
  if (with_write && !(slot_mapping && k_new && v_new)) return PA_ERR_INVALID_ARG;
  if ((long long)num_blocks * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  if (T > 0 && B == 0) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0 || B == 0) {
    // nothing to compute; still honour the phase events
    for (int i = 0; i < n_events && i < 5; ++i)
      if (record(events, n_events, i, s) != PA_OK) return PA_ERR_CUDA;
    return PA_OK;
  }
  if (!q || !k_cache || !v_cache || !block_tables || !cu_seqlens_q || !ctx_lens || !out)
    return PA_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_INVALID_ARG;
  if (with_write && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
    return PA_ERR_WORKSPACE;
  const int cap = capacity_of(workspace_bytes, B, T, H, D);
  if (cap <= 0) return PA_ERR_WORKSPACE;

  StepParams p;
  std::memset(&p, 0, sizeof(p));
  apply_test_hooks(p);
  p.q = q;
  p.out = out;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.cu_seqlens = cu_seqlens_q;
  p.ctx_lens = ctx_lens;
  p.slot_mapping = slot_mapping;
  p.k_new = k_new;
  p.v_new = v_new;
  p.status = status;
  p.max_blocks = max_blocks_per_seq;
  p.B = B;
  p.T = T;
  p.H = H;
  p.Hkv = Hkv;
  p.D = D;
  p.bs = block_size;
  p.NB = num_blocks;
  p.max_q_len = max_q_len;
  p.max_ctx_len = max_ctx_len;
  p.elem_bytes = elem_bytes_of(dtype);
  p.split_all_rows = split_all_rows(dtype, mode) ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.kv_fp8 = fp8 ? 1 : 0;
  p.k_scale = fp8 ? k_scale : 1.f;
  p.v_scale = fp8 ? v_scale : 1.f;
  p.out_scale = p.v_scale;
  if (fp8) p.scale_log2 *= k_scale;
  p.plan = carve(workspace, cap, B, T, H, D);
  p.sm_count = num_sms();
  const bool prefill_tc = !p.split_all_rows && max_q_len >= 2;
  // row-invariant bf16 steps: prefill rows in groups sharing key tiles
  p.group_rows = (dtype == PA_BF16 && mode == PA_MODE_ROW_INVARIANT && max_q_len >= 2)
                     ? rows_group_size(H / Hkv)
                     : 0;

  CUtensorMap tmK, tmV, tmQ;
  if (fp8) {
    if (!encode_code_map(&tmK, k_cache, num_blocks, block_size, Hkv, D) ||
        !encode_code_map(&tmV, v_cache, num_blocks, block_size, Hkv, D))
      return PA_ERR_CUDA;
  } else if (dtype == PA_BF16) {
    if (!encode_cache_map(&tmK, k_cache, num_blocks, block_size, Hkv, D) ||
        !encode_cache_map(&tmV, v_cache, num_blocks, block_size, Hkv, D))
      return PA_ERR_CUDA;
    if (prefill_tc && !encode_q_map(&tmQ, q, T, H, D)) return PA_ERR_CUDA;
  }
  long long items = max_pairs(B, T, max_ctx_len, -1, dtype, mode);
  if (items > cap) items = cap;
  items *= Hkv;

  if (record(events, n_events, 0, s) != PA_OK) return PA_ERR_CUDA;
  if (launch_prologue(p, reuse ? 2 : 1, with_write, s) != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  if (record(events, n_events, 1, s) != PA_OK) return PA_ERR_CUDA;
  // steps with prefill chunks on the tensor cores run decode and prefill in
  // one launch on disjoint SMs (the phase events then see it all as the
  // split phase)
  cudaError_t e = prefill_tc    ? launch_mixed(p, tmQ, tmK, tmV, s)
                  : p.group_rows ? launch_row_mixed(p, tmK, tmV, s)
                  : fp8          ? launch_decode_fp8(p, tmK, tmV, items, s)
                  : dtype == PA_BF16 ? launch_decode_bf16(p, tmK, tmV, items, s)
                                     : launch_split_f32(p, items, s);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  if (record(events, n_events, 2, s) != PA_OK) return PA_ERR_CUDA;
  if (record(events, n_events, 3, s) != PA_OK) return PA_ERR_CUDA;
  if (launch_combine(p, s) != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  if (record(events, n_events, 4, s) != PA_OK) return PA_ERR_CUDA;
  return PA_OK;
}

pa_status pa_attention(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                       const int64_t* slot_mapping, const void* k_new, const void* v_new,
                       void* out, int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t D,
                       int32_t block_size, int32_t num_blocks, int32_t max_q_len,
                       int32_t max_ctx_len, float scale, pa_dtype dtype, void* workspace,
                       size_t workspace_bytes, int32_t* status, void* stream) {
  if (dtype == PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;  // needs the scales
  return pa_attention_ex(q, k_cache, v_cache, block_tables, max_blocks_per_seq, cu_seqlens_q,
                         ctx_lens, slot_mapping, k_new, v_new, out, B, T, H, Hkv, D, block_size,
                         num_blocks, max_q_len, max_ctx_len, scale, dtype, workspace,
                         workspace_bytes, status, stream, 1.f, 1.f, PA_MODE_BATCH_INVARIANT,
                         nullptr, 0);
}

size_t pa_partials_bytes(int32_t T, int32_t max_ctx_len, int32_t H, int32_t D) {
  if (T < 0 || max_ctx_len < 0 || H <= 0 || (D != 64 && D != 128)) return 0;
  return partials_bytes_for(T > 0 ? T : 1, max_ctx_len, H, D);
}

size_t pa_partials_workspace_bytes(int32_t B, int32_t T, int32_t max_ctx_len) {
  if (B < 0 || T < 0 || max_ctx_len < 0) return 0;
  return partials_ws_bytes(B, T, max_ctx_len);
}

pa_status pa_attention_partials(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                const int32_t* key_lo, const int32_t* key_hi, int32_t B,
                                int32_t T, int32_t H, int32_t Hkv, int32_t D,
                                int32_t block_size, int32_t num_blocks, int32_t max_q_len,
                                int32_t max_ctx_len, float scale, pa_dtype dtype, float k_scale,
                                float v_scale, void* partials, size_t partials_bytes,
                                void* workspace, size_t workspace_bytes, int32_t* status,
                                void* stream) {
  if (B < 0 || T < 0 || num_blocks <= 0 || max_q_len < 0 || max_ctx_len < 0)
    return PA_ERR_INVALID_ARG;
  pa_status g = check_geometry(H, Hkv, D, block_size, dtype);
  if (g != PA_OK) return g;
  if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
  const bool fp8 = dtype == PA_FP8_E4M3;
  if (fp8 && !scales_ok(k_scale, v_scale)) return PA_ERR_INVALID_ARG;
  if ((long long)num_blocks * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  if (T > 0 && B == 0) return PA_ERR_INVALID_ARG;
  if (T == 0 || B == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !cu_seqlens_q || !ctx_lens || !key_lo ||
      !key_hi || max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
  if (!partials || (reinterpret_cast<uintptr_t>(partials) & (kAlign - 1)) ||
      partials_bytes < partials_bytes_for(T, max_ctx_len, H, D))
    return PA_ERR_WORKSPACE;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) ||
      workspace_bytes < partials_ws_bytes(B, T, max_ctx_len))
    return PA_ERR_WORKSPACE;

  StepParams p;
  std::memset(&p, 0, sizeof(p));
  apply_test_hooks(p);
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.cu_seqlens = cu_seqlens_q;
  p.ctx_lens = ctx_lens;
  p.status = status;
  p.max_blocks = max_blocks_per_seq;
  p.B = B;
  p.T = T;
  p.H = H;
  p.Hkv = Hkv;
  p.D = D;
  p.bs = block_size;
  p.NB = num_blocks;
  p.max_q_len = max_q_len;
  p.max_ctx_len = max_ctx_len;
  p.elem_bytes = elem_bytes_of(dtype);
  p.split_all_rows = 1;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.kv_fp8 = fp8 ? 1 : 0;
  p.k_scale = fp8 ? k_scale : 1.f;
  p.v_scale = fp8 ? v_scale : 1.f;
  p.out_scale = p.v_scale;
  if (fp8) p.scale_log2 *= k_scale;
  p.partials_mode = 1;
  p.key_lo = key_lo;
  p.key_hi = key_hi;
  p.plan = carve_partials(workspace, workspace_bytes, partials, B, T, H, max_ctx_len);

  CUtensorMap tmK, tmV;
  if (fp8) {
    if (!encode_code_map(&tmK, k_cache, num_blocks, block_size, Hkv, D) ||
        !encode_code_map(&tmV, v_cache, num_blocks, block_size, Hkv, D))
      return PA_ERR_CUDA;
  } else if (dtype == PA_BF16) {
    if (!encode_cache_map(&tmK, k_cache, num_blocks, block_size, Hkv, D) ||
        !encode_cache_map(&tmV, v_cache, num_blocks, block_size, Hkv, D))
      return PA_ERR_CUDA;
  }
  long long items = partial_entries(T, max_ctx_len);
  if (items > p.plan.capacity) items = p.plan.capacity;
  items *= Hkv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_prologue(p, 1, false, s) != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  cudaError_t e = fp8 ? launch_decode_fp8(p, tmK, tmV, items, s)
                      : dtype == PA_BF16 ? launch_decode_bf16(p, tmK, tmV, items, s)
                                         : launch_split_f32(p, items, s);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  return PA_OK;
}

pa_status pa_merge_partials(const void* partials, size_t partials_bytes, int32_t W,
                            const int32_t* key_bounds, const int32_t* cu_seqlens_q,
                            const int32_t* ctx_lens, void* out, int32_t B, int32_t T, int32_t H,
                            int32_t D, int32_t max_q_len, int32_t max_ctx_len, pa_dtype dtype,
                            float v_scale, void* workspace, size_t workspace_bytes,
                            int32_t* status, void* stream) {
  if (B < 0 || T < 0 || W <= 0 || max_q_len < 0 || max_ctx_len < 0) return PA_ERR_INVALID_ARG;
  pa_status g = check_geometry(H, H, D, 16, dtype);
  if (g != PA_OK) return g;
  const bool fp8 = dtype == PA_FP8_E4M3;
  if (fp8 && !scales_ok(1.f, v_scale)) return PA_ERR_INVALID_ARG;
  if (T > 0 && B == 0) return PA_ERR_INVALID_ARG;
  if (T == 0 || B == 0) return PA_OK;
  if (!partials || !key_bounds || !cu_seqlens_q || !ctx_lens || !out) return PA_ERR_INVALID_ARG;
  if (!aligned16(out)) return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(partials) & (kAlign - 1)) || (partials_bytes & (kAlign - 1)) ||
      partials_bytes < partials_bytes_for(T, max_ctx_len, H, D))
    return PA_ERR_WORKSPACE;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) ||
      workspace_bytes < partials_ws_bytes(B, T, max_ctx_len))
    return PA_ERR_WORKSPACE;

  StepParams p;
  std::memset(&p, 0, sizeof(p));
  apply_test_hooks(p);
  p.out = out;
  p.cu_seqlens = cu_seqlens_q;
  p.ctx_lens = ctx_lens;
  p.status = status;
  p.max_blocks = 0x7fffffff / 32;  // no block table here; the ctx range check is moot
  p.B = B;
  p.T = T;
  p.H = H;
  p.Hkv = H;
  p.D = D;
  p.bs = 32;
  p.max_q_len = max_q_len;
  p.max_ctx_len = max_ctx_len;
  p.elem_bytes = elem_bytes_of(dtype);
  p.split_all_rows = 1;
  p.out_scale = fp8 ? v_scale : 1.f;
  p.partials_mode = 2;
  p.key_bounds = key_bounds;
  p.owners = W;
  p.owner_stride = (long long)partials_bytes;
  p.plan = carve_partials(workspace, workspace_bytes, const_cast<void*>(partials), B, T, H,
                          max_ctx_len);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_prologue(p, 1, false, s) != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  if (launch_combine(p, s) != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  return PA_OK;
}

int32_t pa_decode_gemm_splits(int32_t N, int32_t K) {
  if (N <= 0 || K <= 0 || N % 128 || K % 64) return 0;
  int S, cps;
  decode_gemm_plan(N, K, &S, &cps);
  return S;
}

size_t pa_decode_gemm_workspace_bytes(int32_t T_pad, int32_t N, int32_t K) {
  if (!gemm_shape_ok(T_pad, N, K)) return 0;
  const int S = pa_decode_gemm_splits(N, K);
  return S > 1 ? align_up((size_t)S * T_pad * N * sizeof(float)) : 0;
}

pa_status pa_decode_gemm(const void* x, const void* w, void* y, int32_t T_pad, int32_t N,
                         int32_t K, void* workspace, size_t workspace_bytes, int32_t* status,
                         void* stream) {
  if (!gemm_shape_ok(T_pad, N, K)) return PA_ERR_UNSUPPORTED;
  if (!x || !w || !y || !aligned16(x) || !aligned16(w) || !aligned16(y)) return PA_ERR_INVALID_ARG;
  int S, cps;
  decode_gemm_plan(N, K, &S, &cps);
  const size_t need = pa_decode_gemm_workspace_bytes(T_pad, N, K);
  if (need && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) ||
               workspace_bytes < need))
    return PA_ERR_WORKSPACE;
  CUtensorMap tmW, tmX;
  if (!encode_rows_map(&tmW, w, N, K, 128) || !encode_rows_map(&tmX, x, T_pad, K, T_pad))
    return PA_ERR_CUDA;
  if (launch_decode_gemm(y, static_cast<float*>(workspace), T_pad, N, K, S, cps, status, tmW,
                         tmX, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  count_launches(S > 1 ? 2 : 1);
  return PA_OK;
}

pa_status pa_read_status(int32_t* status, void* stream, int32_t* flags_out, int32_t clear) {
  if (!status || !flags_out) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ERR_CUDA;
  if (clear && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  *flags_out = v;
  return PA_OK;
}

}  // extern "C"

extern "C" void pa_test_set_wait_cycles(int64_t cycles) {
  pa::g_wait_cycles.store(cycles > 0 ? (long long)cycles : pa::kWaitCycles,
                          std::memory_order_relaxed);
}

extern "C" void pa_test_skip_split_item(int64_t item) {
  pa::g_skip_item.store(item >= 0 ? (long long)item : -1LL, std::memory_order_relaxed);
}
