"""pa_attention_static_scratch: attention for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run a step (a plugin with no
device allocator, a process whose pool already holds all free memory, a loop
that cannot take cudaMalloc's synchronisation). The entry point uses scratch
compiled into the library instead of a caller workspace. This file checks,
through the C ABI, that two calls in a row give the same outputs as
pa_attention with a caller workspace, and that a step too big for the built-in
array is refused. It is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle.paged_attention as opa
from gpu_harness import TOL, device_step, workspace_for
from invariant_paged_kv_gb300 import build, pa, workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    pa.load()


def _both(step, seed):
    """Outputs of the workspace entry point and of the static-scratch one."""
    t = wl.make_tensors(step, seed, "cuda")
    dev = device_step(step)
    g = step.geom
    scale = opa.default_scale(g.D)
    common = dict(max_q_len=step.max_q_len, max_ctx_len=step.max_ctx_len, scale=scale,
                  slot_mapping=dev["slot_mapping"], k_new=t["k_new"][0], v_new=t["v_new"][0])
    args = (t["q"][0], t["k_cache"][0], t["v_cache"][0], dev["block_tables"],
            dev["cu_seqlens_q"], dev["ctx_lens"])
    ref = torch.full_like(t["q"][0], float("nan"))
    st = pa.new_status()
    pa.attention(*args, ref, workspace=workspace_for(step), status=st, **common)
    assert pa.read_status(st) == 0
    got = torch.full_like(t["q"][0], float("nan"))
    pa.attention_static_scratch(*args, got, total_ctx=int(step.ctx_lens.sum()), status=st,
                                **common)
    assert pa.read_status(st) == 0
    return ref, got


def _close(ref, got, dtype):
    a = ref.double().cpu().numpy()
    b = got.double().cpu().numpy()
    assert not np.isnan(b).any()
    assert np.max(np.abs(a - b)) <= TOL[dtype]


def test_two_calls_in_a_row_match_workspace_entry():
    # first: decode rows with several splits each; second: a different step
    # (prefill chunk + decode rows, other geometry) over the same array
    s1 = wl.decode_batch(0, lanes=24)
    rng = np.random.default_rng(8)
    s2 = wl.build_step(wl.Geometry(16, 4, 64, 32, "bf16"), [1, 1, 37, 1],
                       [1300, 9, 700, 2600], 200, rng)
    for step, seed in ((s1, 61), (s2, 62)):
        ref, got = _both(step, seed)
        _close(ref, got, step.geom.dtype)


def test_fp32_step_matches_workspace_entry():
    step = wl.tiny_f32(2)
    ref, got = _both(step, 63)
    _close(ref, got, "f32")


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
