// pa_attention_static_scratch: pa_attention with the split-KV scratch taken
// from a fixed array compiled into the library instead of a caller buffer.
//
// Who needs it: code that cannot call cudaMalloc on the path that runs a
// step -- for instance a plugin loaded into a host framework that gives it no
// device allocator, a process whose memory pool has already claimed all free
// device memory up front, or a latency-critical loop that cannot afford the
// device-wide synchronisation cudaMalloc / cudaFree may imply. Such a caller
// still passes its inputs and outputs; only the scratch is built in.
//
// The array below is a file-scope __device__ object. It lives in this
// file's own device module, which CUDA loads on a device when the module is
// first used there (lazy module loading is the default): here, at the
// cudaGetSymbolAddress of the first call on that device. That is when the
// device memory for the array is taken; the device then holds
// PA_STATIC_SCRATCH_BYTES of it until the process exits. In host code the
// array's name is only a host-side stand-in, never a device address, so the
// host looks the address up with cudaGetSymbolAddress, once per device, with
// that device current, and passes the looked-up pointer on. The address
// belongs to the device's context of that moment: after a cudaDeviceReset
// the entry point must not be called again in the same process.
#include <mutex>

#include "pa_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device (set up on first use).
pa_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return PA_ERR_CUDA;
  if (dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_attention_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
    const int64_t* slot_mapping, const void* k_new, const void* v_new, void* out, int32_t B,
    int32_t T, int32_t H, int32_t Hkv, int32_t D, int32_t block_size, int32_t num_blocks,
    int32_t max_q_len, int32_t max_ctx_len, int64_t total_ctx, float scale, pa_dtype dtype,
    int32_t* status, void* stream) {
  // Argument and size checks first, on the host, before any CUDA call:
  // negative sizes are the caller's error, as in pa_attention.
  if (B < 0 || T < 0 || max_q_len < 0 || max_ctx_len < 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  const size_t need = pa_attention_workspace_bytes(B, T, max_q_len, max_ctx_len, total_ctx, H,
                                                   Hkv, D, block_size, dtype);
  if (need == 0) return PA_ERR_UNSUPPORTED;
  if (need > (size_t)PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const pa_status st = scratch_on_current_device(&scratch);
  if (st != PA_OK) return st;
  // Nothing in the scratch has to start at zero: the step's plan and partial
  // results are rewritten in full by every call before they are read.
  return pa_attention(q, k_cache, v_cache, block_tables, max_blocks_per_seq, cu_seqlens_q,
                      ctx_lens, slot_mapping, k_new, v_new, out, B, T, H, Hkv, D, block_size,
                      num_blocks, max_q_len, max_ctx_len, scale, dtype, scratch,
                      (size_t)PA_STATIC_SCRATCH_BYTES, status, stream);
}
