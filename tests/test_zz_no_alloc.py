"""pa_attention_static_scratch: attention for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run a step: a plugin whose
host framework gives it no device allocator, a process whose memory pool has
already claimed all free device memory, a loop that cannot take the
device-wide synchronisation cudaMalloc may cause. The entry point uses scratch
compiled into the library instead of a caller workspace. Through the C ABI this
file checks that:
  * after its set-up call (B = T = 0), two calls in a row give outputs bitwise
    equal to pa_attention's with a caller workspace (the same plan and
    kernels run, so not one bit may differ);
  * a smaller step run right after a bigger one -- the array still holds the
    bigger step's plan and partials -- is bitwise equal to the workspace entry
    point and within the oracle's parity bound;
  * a warm call takes no device memory;
  * a step too big for the built-in array is refused.
It is named to be collected last, so a run that stops at its first failure
has run every other test before it.
"""
import numpy as np
import pytest
import torch

import oracle.paged_attention as opa
from gpu_harness import (check_parity, device_step, oracle_attention, rows_of, to_cpu,
                         workspace_for)
from invariant_paged_kv_gb300 import build, pa, workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    pa.load()


def _setup_call():
    """B = T = 0: only the per-device set-up (the array's address)."""
    L = pa.load()
    code = L.pa_attention_static_scratch(None, None, None, None, 1, None, None, None, None,
                                         None, None, 0, 0, 8, 2, 128, 16, 1, 0, 0, 0, 0.088,
                                         1, None, None)
    assert code == 0


def _args(step, t):
    dev = device_step(step)
    common = dict(max_q_len=step.max_q_len, max_ctx_len=step.max_ctx_len,
                  scale=opa.default_scale(step.geom.D), slot_mapping=dev["slot_mapping"],
                  k_new=t["k_new"][0], v_new=t["v_new"][0])
    args = (t["q"][0], t["k_cache"][0], t["v_cache"][0], dev["block_tables"],
            dev["cu_seqlens_q"], dev["ctx_lens"])
    return args, common


def _static(step, t, args, common):
    got = torch.full_like(t["q"][0], float("nan"))
    st = pa.new_status()
    pa.attention_static_scratch(*args, got, total_ctx=int(step.ctx_lens.sum()), status=st,
                                **common)
    assert pa.read_status(st) == 0
    return got


def _workspace(step, t, args, common):
    ref = torch.full_like(t["q"][0], float("nan"))
    st = pa.new_status()
    pa.attention(*args, ref, workspace=workspace_for(step), status=st, **common)
    assert pa.read_status(st) == 0
    return ref


def _bits(x):
    return x.view(torch.int32 if x.dtype == torch.float32 else torch.int16)


def _fresh(step, seed):
    """Tensors of the step; the caches are copied back before each call, so
    every call attends the same keys after writing the same new rows."""
    t = wl.make_tensors(step, seed, "cuda")
    k0, v0 = t["k_cache"][0].clone(), t["v_cache"][0].clone()

    def reset():
        t["k_cache"][0].copy_(k0)
        t["v_cache"][0].copy_(v0)
    return t, reset


def test_two_calls_in_a_row_match_workspace_entry_bitwise():
    _setup_call()
    # first: decode rows with several splits each; second: a different step
    # (prefill chunk + decode rows, other geometry) over the same array
    s1 = wl.decode_batch(0, lanes=24)
    rng = np.random.default_rng(8)
    s2 = wl.build_step(wl.Geometry(16, 4, 64, 32, "bf16"), [1, 1, 37, 1],
                       [1300, 9, 700, 2600], 200, rng)
    runs = []
    for step, seed in ((s1, 61), (s2, 62)):
        t, reset = _fresh(step, seed)
        args, common = _args(step, t)
        reset()
        got = _static(step, t, args, common)
        runs.append((step, seed, t, reset, args, common, got))
    for step, seed, t, reset, args, common, got in runs:
        reset()
        ref = _workspace(step, t, args, common)
        assert torch.equal(_bits(ref), _bits(got)), f"{step.geom}: not bitwise equal"


def test_smaller_step_after_bigger_one_matches_oracle():
    _setup_call()
    big = wl.decode_batch(1, lanes=40)
    tb, resetb = _fresh(big, 64)
    argsb, commonb = _args(big, tb)
    small = wl.decode_batch(2, lanes=6)
    ts, resets = _fresh(small, 65)
    argss, commons = _args(small, ts)
    resetb()
    _static(big, tb, argsb, commonb)
    resets()
    got = _static(small, ts, argss, commons)
    resets()
    ref = _workspace(small, ts, argss, commons)
    assert torch.equal(_bits(ref), _bits(got))
    resets()
    rows = list(range(small.T))
    oref, _, _, terms = oracle_attention(small, to_cpu(ts), rows=rows, terms=True)
    check_parity(got, oref, rows_of(terms, rows), small.row_positions(), small.geom,
                 "static scratch, small step after a big one")


def test_fp32_step_matches_workspace_entry_bitwise():
    _setup_call()
    step = wl.tiny_f32(2)
    t, reset = _fresh(step, 63)
    args, common = _args(step, t)
    reset()
    got = _static(step, t, args, common)
    reset()
    ref = _workspace(step, t, args, common)
    assert torch.equal(_bits(ref), _bits(got))


def test_warm_call_takes_no_device_memory():
    _setup_call()
    step = wl.decode_batch(3, lanes=16)
    t, reset = _fresh(step, 66)
    args, common = _args(step, t)
    got = torch.empty_like(t["q"][0])
    st = pa.new_status()
    kw = dict(total_ctx=int(step.ctx_lens.sum()), status=st, **common)
    pa.attention_static_scratch(*args, got, **kw)  # warm: kernels loaded
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        pa.attention_static_scratch(*args, got, **kw)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert pa.read_status(st) == 0


def test_step_beyond_the_limit_is_refused():
    step = wl.long_tail(0, pool_bytes_per_layer=1e8)  # descriptor only
    g = step.geom
    need = pa.workspace_bytes(step.B, step.T, step.max_q_len, step.max_ctx_len,
                              int(step.ctx_lens.sum()), g.H, g.Hkv, g.D, g.block_size,
                              torch.bfloat16)
    assert need > 32 * 1024 * 1024
    L = pa.load()
    code = L.pa_attention_static_scratch(
        None, None, None, None, step.max_blocks_per_seq, None, None, None, None, None, None,
        step.B, step.T, g.H, g.Hkv, g.D, g.block_size, step.num_blocks, step.max_q_len,
        step.max_ctx_len, int(step.ctx_lens.sum()), 0.088, 1, None, None)
    assert code == 3  # PA_ERR_WORKSPACE, refused before any CUDA work
