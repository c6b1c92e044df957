"""ctypes binding of libpa.so (include/pa.h). Argument marshalling only.

Every function takes torch tensors, checks dtype / shape / device, passes raw
device pointers and the current CUDA stream to the C ABI, and raises
``PaError`` on a non-zero status. No arithmetic of the method runs here, and
there is no fallback: if the library is missing, importing the functions
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libpa.so")

PA_F32, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
FP8_CACHE_DTYPES = (torch.uint8, torch.float8_e4m3fn)  # e4m3 code caches
MODES = {"batch": 0, "row": 1}  # pa_mode: PA_MODE_BATCH_INVARIANT, PA_MODE_ROW_INVARIANT
REUSE_PLAN = 0x100  # PA_MODE_REUSE_PLAN, OR-ed into a mode
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
                3: "PA_ERR_WORKSPACE", 4: "PA_ERR_CUDA"}
FLAGS = {
    "SLOT_RANGE": 0x01, "BLOCK_RANGE": 0x02, "CTX_RANGE": 0x04, "QLEN_RANGE": 0x08,
    "CU_SEQLENS": 0x10, "WORKSPACE": 0x20, "HOST_BOUND": 0x40, "TIMEOUT": 0x80,
    "OWNER_RANGE": 0x100, "PLAN_MISMATCH": 0x200,
}

EXPORTS = ("pa_write_kv", "pa_write_kv_scaled", "pa_attention_workspace_bytes",
           "pa_attention_workspace_bytes_ex",
           "pa_attention", "pa_attention_ex", "pa_read_status", "pa_status_string",
           "pa_kernel_launches", "pa_split_tokens", "pa_attention_static_scratch",
           "pa_partials_bytes", "pa_partials_workspace_bytes", "pa_attention_partials",
           "pa_merge_partials", "pa_decode_gemm_splits", "pa_decode_gemm_workspace_bytes",
           "pa_decode_gemm")
# test hooks declared in include/pa_test.h (not part of the attention boundary)
TEST_EXPORTS = ("pa_test_set_wait_cycles", "pa_test_skip_split_item")


class PaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")
        self.code = code


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libpa.so (built by ``invariant_paged_kv_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"libpa.so not built ({_LIB_PATH}); run `python -m invariant_paged_kv_gb300.build`")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    L.pa_write_kv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
    L.pa_write_kv.restype = ctypes.c_int
    L.pa_write_kv_scaled.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, f32,
                                     vp, vp]
    L.pa_write_kv_scaled.restype = ctypes.c_int
    L.pa_attention_workspace_bytes.argtypes = [i32, i32, i32, i32, i64, i32, i32, i32, i32, i32]
    L.pa_attention_workspace_bytes.restype = sz
    L.pa_attention_workspace_bytes_ex.argtypes = [i32, i32, i32, i32, i64, i32, i32, i32, i32,
                                                  i32, i32]
    L.pa_attention_workspace_bytes_ex.restype = sz
    att = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
           i32, i32, f32, i32, vp, sz, vp, vp]
    L.pa_attention.argtypes = att
    L.pa_attention.restype = ctypes.c_int
    L.pa_attention_ex.argtypes = att + [f32, f32, i32, ctypes.POINTER(vp), i32]
    L.pa_attention_ex.restype = ctypes.c_int
    L.pa_read_status.argtypes = [vp, vp, ctypes.POINTER(i32), i32]
    L.pa_read_status.restype = ctypes.c_int
    L.pa_status_string.argtypes = [ctypes.c_int]
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_kernel_launches.argtypes = []
    L.pa_kernel_launches.restype = i64
    L.pa_split_tokens.argtypes = []
    L.pa_split_tokens.restype = i32
    L.pa_attention_static_scratch.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, i32,
                                              i32, i32, i32, i32, i32, i32, i32, i32, i64, f32,
                                              i32, vp, vp]
    L.pa_attention_static_scratch.restype = ctypes.c_int
    L.pa_partials_bytes.argtypes = [i32, i32, i32, i32]
    L.pa_partials_bytes.restype = sz
    L.pa_partials_workspace_bytes.argtypes = [i32, i32, i32]
    L.pa_partials_workspace_bytes.restype = sz
    L.pa_attention_partials.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32,
                                        i32, i32, i32, i32, i32, f32, i32, f32, f32, vp, sz, vp,
                                        sz, vp, vp]
    L.pa_attention_partials.restype = ctypes.c_int
    L.pa_merge_partials.argtypes = [vp, sz, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                    i32, f32, vp, sz, vp, vp]
    L.pa_merge_partials.restype = ctypes.c_int
    L.pa_decode_gemm_splits.argtypes = [i32, i32]
    L.pa_decode_gemm_splits.restype = i32
    L.pa_decode_gemm_workspace_bytes.argtypes = [i32, i32, i32]
    L.pa_decode_gemm_workspace_bytes.restype = sz
    L.pa_decode_gemm.argtypes = [vp, vp, vp, i32, i32, i32, vp, sz, vp, vp]
    L.pa_decode_gemm.restype = ctypes.c_int
    L.pa_test_set_wait_cycles.argtypes = [i64]
    L.pa_test_set_wait_cycles.restype = None
    L.pa_test_skip_split_item.argtypes = [i64]
    L.pa_test_skip_split_item.restype = None
    _lib = L
    return L


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _cache_code(k_cache: torch.Tensor, q_dtype: torch.dtype) -> int:
    """Element-type code of a step from its cache (e4m3 codes) or q."""
    if k_cache.dtype in FP8_CACHE_DTYPES:
        if q_dtype != torch.bfloat16:
            raise TypeError("e4m3 caches take bf16 queries and new rows")
        return PA_FP8_E4M3
    if k_cache.dtype != q_dtype:
        raise TypeError("caches and queries must share a dtype (or the caches hold e4m3 codes)")
    return PA_F32 if q_dtype == torch.float32 else PA_BF16


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, what: str):
    if code != 0:
        raise PaError(code, what)


def split_tokens() -> int:
    return int(load().pa_split_tokens())


def kernel_launches() -> int:
    return int(load().pa_kernel_launches())


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_status(status: torch.Tensor, stream=None, clear: bool = True) -> int:
    out = ctypes.c_int32(0)
    _check(load().pa_read_status(_ptr(status), _stream(stream), ctypes.byref(out),
                                 1 if clear else 0), "pa_read_status")
    return int(out.value)


def write_kv(k_new, v_new, k_cache, v_cache, slot_mapping, status=None, stream=None,
             k_scale: float = 1.0, v_scale: float = 1.0):
    """pa_write_kv_scaled: scatter new rows [T, Hkv, D] into caches
    [NB, bs, Hkv, D] (quantised under k_scale / v_scale into e4m3 caches)."""
    NB, bs, Hkv, D = k_cache.shape
    T = k_new.shape[0]
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    _check(load().pa_write_kv_scaled(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(slot_mapping), T, NB, bs, Hkv, D,
                                     _cache_code(k_cache, k_new.dtype), float(k_scale),
                                     float(v_scale), _ptr(status), _stream(stream)),
           "pa_write_kv_scaled")


def _mode_code(mode: str) -> int:
    if mode not in MODES:
        raise ValueError(f"mode must be one of {sorted(MODES)}")
    return MODES[mode]


def workspace_bytes(B, T, max_q_len, max_ctx_len, total_ctx, H, Hkv, D, block_size,
                    dtype: torch.dtype, mode: str = "batch") -> int:
    """pa_attention_workspace_bytes_ex for ``mode`` ("batch" or "row");
    ``dtype`` is the cache dtype (uint8 / float8_e4m3fn for e4m3 codes)."""
    code = PA_FP8_E4M3 if dtype in FP8_CACHE_DTYPES else (
        PA_F32 if dtype == torch.float32 else PA_BF16)
    n = int(load().pa_attention_workspace_bytes_ex(B, T, max_q_len, max_ctx_len, total_ctx, H,
                                                   Hkv, D, block_size, code, _mode_code(mode)))
    if n == 0:
        raise PaError(2, "pa_attention_workspace_bytes_ex")
    return n


def attention(q, k_cache, v_cache, block_tables, cu_seqlens_q, ctx_lens, out, *,
              max_q_len: int, max_ctx_len: int, scale: float, workspace: torch.Tensor,
              slot_mapping=None, k_new=None, v_new=None, status=None, stream=None,
              events: Optional[Sequence[torch.cuda.Event]] = None, mode: str = "batch",
              k_scale: float = 1.0, v_scale: float = 1.0, reuse_plan: bool = False):
    """pa_attention, or pa_attention_ex when ``events``, mode="row", e4m3
    caches (uint8 / float8_e4m3fn, with k_scale and v_scale) or
    ``reuse_plan`` are given.

    mode "batch": a row's bits depend only on its own lane. mode "row": also
    not on its lane's q_len (every row takes the split-KV path); the
    workspace must then be sized with ``workspace_bytes(..., mode="row")``.
    reuse_plan: the workspace holds the plan an earlier call built for this
    very step (PA_MODE_REUSE_PLAN) -- the later layers of a step.
    """
    T, H, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    B = ctx_lens.shape[0]
    if block_tables.dtype != torch.int32 or cu_seqlens_q.dtype != torch.int32 \
            or ctx_lens.dtype != torch.int32:
        raise TypeError("block_tables, cu_seqlens_q and ctx_lens must be int32")
    if workspace.dtype != torch.uint8:
        raise TypeError("workspace must be a uint8 tensor")
    mb = block_tables.shape[1] if block_tables.dim() == 2 else 0
    args = [_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mb, _ptr(cu_seqlens_q),
            _ptr(ctx_lens), _ptr(slot_mapping), _ptr(k_new), _ptr(v_new), _ptr(out), B, T, H,
            Hkv, D, bs, NB, int(max_q_len), int(max_ctx_len), float(scale),
            _cache_code(k_cache, q.dtype), _ptr(workspace), workspace.numel(), _ptr(status),
            _stream(stream)]
    L = load()
    code = _mode_code(mode) | (REUSE_PLAN if reuse_plan else 0)
    if events is None and code == 0 and k_cache.dtype not in FP8_CACHE_DTYPES:
        _check(L.pa_attention(*args), "pa_attention")
        return
    arr, n = None, 0
    if events:
        for e in events:  # torch creates events lazily; recording once creates them
            if not e.cuda_event:
                e.record(stream)
        arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        n = len(events)
    _check(L.pa_attention_ex(*args, float(k_scale), float(v_scale), code, arr, n),
           "pa_attention_ex")


def attention_static_scratch(q, k_cache, v_cache, block_tables, cu_seqlens_q, ctx_lens, out, *,
                             max_q_len: int, max_ctx_len: int, total_ctx: int, scale: float,
                             slot_mapping=None, k_new=None, v_new=None, status=None,
                             stream=None):
    """pa_attention_static_scratch: like ``attention`` but without a workspace.

    For callers that cannot allocate device memory: the split scratch is an
    array built into the library (``PA_STATIC_SCRATCH_BYTES`` per GPU). Steps
    that need more raise PaError(PA_ERR_WORKSPACE). Calls overlapping on the
    GPU share that array and must be serialised by the caller.
    """
    T, H, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    B = ctx_lens.shape[0]
    if block_tables.dtype != torch.int32 or cu_seqlens_q.dtype != torch.int32 \
            or ctx_lens.dtype != torch.int32:
        raise TypeError("block_tables, cu_seqlens_q and ctx_lens must be int32")
    mb = block_tables.shape[1] if block_tables.dim() == 2 else 0
    _check(load().pa_attention_static_scratch(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mb, _ptr(cu_seqlens_q),
        _ptr(ctx_lens), _ptr(slot_mapping), _ptr(k_new), _ptr(v_new), _ptr(out), B, T, H, Hkv,
        D, bs, NB, int(max_q_len), int(max_ctx_len), int(total_ctx), float(scale),
        _dtype_code(q), _ptr(status), _stream(stream)), "pa_attention_static_scratch")


# ---------------------------------------------------------------------------
# KV-parallel page owners
# ---------------------------------------------------------------------------

def partials_bytes(T: int, max_ctx_len: int, H: int, D: int) -> int:
    """pa_partials_bytes: one owner's partial buffer."""
    n = int(load().pa_partials_bytes(T, max_ctx_len, H, D))
    if n == 0:
        raise PaError(1, "pa_partials_bytes")
    return n


def partials_workspace_bytes(B: int, T: int, max_ctx_len: int) -> int:
    return int(load().pa_partials_workspace_bytes(B, T, max_ctx_len))


def attention_partials(q, k_cache, v_cache, block_tables, cu_seqlens_q, ctx_lens, key_lo,
                       key_hi, partials, *, max_q_len: int, max_ctx_len: int, scale: float,
                       workspace: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0,
                       status=None, stream=None):
    """pa_attention_partials: this owner's split partials into ``partials``
    (a uint8 tensor of partials_bytes(...)); key_lo / key_hi int32 [B]."""
    T, H, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    B = ctx_lens.shape[0]
    for t in (block_tables, cu_seqlens_q, ctx_lens, key_lo, key_hi):
        if t.dtype != torch.int32:
            raise TypeError("tables, lengths and key ranges must be int32")
    mb = block_tables.shape[1] if block_tables.dim() == 2 else 0
    _check(load().pa_attention_partials(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), mb, _ptr(cu_seqlens_q),
        _ptr(ctx_lens), _ptr(key_lo), _ptr(key_hi), B, T, H, Hkv, D, bs, NB, int(max_q_len),
        int(max_ctx_len), float(scale), _cache_code(k_cache, q.dtype), float(k_scale),
        float(v_scale), _ptr(partials), partials.numel(), _ptr(workspace), workspace.numel(),
        _ptr(status), _stream(stream)), "pa_attention_partials")


def merge_partials(gathered, owners: int, key_bounds, cu_seqlens_q, ctx_lens, out, *,
                   max_q_len: int, max_ctx_len: int, workspace: torch.Tensor,
                   kv_dtype: torch.dtype = None, v_scale: float = 1.0, status=None,
                   stream=None):
    """pa_merge_partials: fold the owners' gathered buffers (uint8,
    owners x partials_bytes, back to back) into out [T, H, D];
    key_bounds int32 [owners + 1, B]; kv_dtype is the caches' dtype."""
    T, H, D = out.shape
    B = ctx_lens.shape[0]
    if key_bounds.dtype != torch.int32 or tuple(key_bounds.shape) != (owners + 1, B):
        raise TypeError("key_bounds must be int32 [owners + 1, B]")
    if gathered.numel() % owners:
        raise ValueError("gathered buffer is not owners equal parts")
    code = PA_FP8_E4M3 if kv_dtype in FP8_CACHE_DTYPES else (
        PA_F32 if out.dtype == torch.float32 else PA_BF16)
    _check(load().pa_merge_partials(
        _ptr(gathered), gathered.numel() // owners, owners, _ptr(key_bounds),
        _ptr(cu_seqlens_q), _ptr(ctx_lens), _ptr(out), B, T, H, D, int(max_q_len),
        int(max_ctx_len), code, float(v_scale), _ptr(workspace), workspace.numel(),
        _ptr(status), _stream(stream)), "pa_merge_partials")


# ---------------------------------------------------------------------------
# batch-invariant decode GEMM at a fixed token width
# ---------------------------------------------------------------------------

def decode_gemm_splits(N: int, K: int) -> int:
    return int(load().pa_decode_gemm_splits(N, K))


def decode_gemm_workspace(T_pad: int, N: int, K: int, device=None) -> torch.Tensor:
    n = int(load().pa_decode_gemm_workspace_bytes(T_pad, N, K))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def decode_gemm(x, w, y, workspace=None, status=None, stream=None):
    """pa_decode_gemm: y [T_pad, N] = x [T_pad, K] w [N, K]^T (bf16, fp32
    accumulate) with a schedule fixed by (N, K); x's padding rows reach only
    their own rows of y."""
    T_pad, K = x.shape
    N = w.shape[0]
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or y.dtype != torch.bfloat16:
        raise TypeError("decode_gemm takes bf16 x, w and y")
    if tuple(w.shape) != (N, K) or tuple(y.shape) != (T_pad, N):
        raise ValueError("shapes: x [T_pad, K], w [N, K], y [T_pad, N]")
    if workspace is None:
        workspace = decode_gemm_workspace(T_pad, N, K, x.device)
    _check(load().pa_decode_gemm(_ptr(x), _ptr(w), _ptr(y), T_pad, N, K, _ptr(workspace),
                                 workspace.numel(), _ptr(status), _stream(stream)),
           "pa_decode_gemm")
