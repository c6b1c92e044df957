"""PA_MODE_REUSE_PLAN: the layers of one step attend over the same lanes, so
only the first layer's call builds the split plan and the others reuse it
("P3: native paged-KV continuous-batching sampler", Design: one flat step
description serves every layer). Reusing it changes no output bit and no
cache byte; a plan built for other sizes is refused on the device
(PA_FLAG_PLAN_MISMATCH, no output written) and the next ordinary call is
right again.
"""
import numpy as np
import pytest
import torch

from gpu_harness import device_step, run_attention, workspace_for
from invariant_paged_kv_gb300 import build, pa, workload as wl

pytestmark = pytest.mark.gpu

LAYERS = 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    pa.load()


def _bits(x):
    return x.contiguous().view(torch.uint8)


CASES = {
    "decode bf16": (lambda: wl.decode_batch(0, lanes=24), "batch"),
    "decode e4m3": (lambda: wl.decode_batch(1, lanes=16, dtype="fp8"), "batch"),
    "decode f32": (lambda: wl.decode_batch(2, lanes=12, dtype="f32"), "batch"),
    "mixed bf16": (lambda: wl.mixed_step(0, chunks=2, chunk_len=300, decodes=12), "batch"),
    "mixed bf16 row mode": (lambda: wl.mixed_step(1, chunks=2, chunk_len=200, decodes=8), "row"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_reused_plan_gives_the_same_bits(name):
    make, mode = CASES[name]
    step = make()
    dev = device_step(step)
    fresh = wl.make_tensors(step, 321, "cuda", layers=LAYERS)
    reused = wl.make_tensors(step, 321, "cuda", layers=LAYERS)
    ws = workspace_for(step, mode)
    for layer in range(LAYERS):
        # every layer planned on its own (a fresh workspace each time) ...
        ref, f0 = run_attention(step, fresh, layer=layer, dev=dev, mode=mode,
                                workspace=workspace_for(step, mode))
        # ... against one workspace whose plan the first layer builds
        got, f1 = run_attention(step, reused, layer=layer, dev=dev, mode=mode, workspace=ws,
                                reuse_plan=layer > 0)
        assert f0 == 0 and f1 == 0, (f0, f1)
        assert torch.equal(_bits(got), _bits(ref)), f"{name}: layer {layer} output differs"
        for c in ("k_cache", "v_cache"):
            assert torch.equal(_bits(reused[c][layer]), _bits(fresh[c][layer])), (name, layer, c)


def test_plan_of_other_sizes_is_refused():
    a = wl.decode_batch(0, lanes=24)
    b = wl.decode_batch(3, lanes=20)
    ws_bytes = max(workspace_for(a).numel(), workspace_for(b).numel())
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ta = wl.make_tensors(a, 5, "cuda")
    tb = wl.make_tensors(b, 6, "cuda")
    _, fa = run_attention(a, ta, workspace=ws)  # builds a's plan
    assert fa == 0
    out_b, fb = run_attention(b, tb, workspace=ws, write=False, reuse_plan=True)
    assert fb == pa.FLAGS["PLAN_MISMATCH"], f"flags {fb:#x}"
    assert torch.isnan(out_b.float()).all(), "a refused call wrote output"
    # the refusal discarded a's plan: reusing it for a is refused as well
    out_a, fa2 = run_attention(a, ta, workspace=ws, write=False, reuse_plan=True)
    assert fa2 == pa.FLAGS["PLAN_MISMATCH"], f"flags {fa2:#x}"
    assert torch.isnan(out_a.float()).all(), "a refused call wrote output"
    # the next ordinary call plans again and matches a fresh workspace
    got, f2 = run_attention(b, tb, workspace=ws, write=False)
    ref, f3 = run_attention(b, tb, write=False)
    assert f2 == 0 and f3 == 0
    assert torch.equal(_bits(got), _bits(ref))
    # and its plan is reusable
    again, f4 = run_attention(b, tb, workspace=ws, write=False, reuse_plan=True)
    assert f4 == 0 and torch.equal(_bits(again), _bits(ref))
