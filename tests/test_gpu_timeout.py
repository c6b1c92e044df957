"""A bounded device wait that runs out is reported and leaves the library usable.

Every wait inside libpa's kernels gives up after a limit ("P3: native paged-KV
continuous-batching sampler", Review (adversarial pass): a failure must surface
as an error the caller sees, not wedge the engine). Here the test hooks of
include/pa_test.h shorten the limit to about a millisecond and make the bf16
split kernel skip the copy of one chunk, so the warp that owns it waits for
data that never comes. Nothing faults or hangs: that warp gives up, raises
PA_FLAG_TIMEOUT, lets its other copies land and returns; the call completes;
and the next ordinary call in the same process gives the oracle's answer.
"""
import numpy as np
import pytest
import torch

from gpu_harness import check_parity, oracle_attention, rows_of, run_attention, to_cpu
from invariant_paged_kv_gb300 import build, pa, workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    pa.load()


def test_split_wait_runs_out_then_next_call_is_right():
    L = pa.load()
    step = wl.decode_batch(0, lanes=16)
    t = wl.make_tensors(step, 81, "cuda")
    before = to_cpu(t)  # caches before the step's write
    try:
        L.pa_test_set_wait_cycles(2_000_000)  # about a millisecond of SM clock
        L.pa_test_skip_split_item(0)          # item 0 is always taken first
        _, flags = run_attention(step, t)     # returns: read_status synchronises
    finally:
        L.pa_test_skip_split_item(-1)
        L.pa_test_set_wait_cycles(0)
    assert flags & pa.FLAGS["TIMEOUT"], f"flags {flags:#x}"
    assert not flags & ~pa.FLAGS["TIMEOUT"], f"flags {flags:#x}"
    # an ordinary call in the same process: no flag, the oracle's output (the
    # write stores the same rows again, so the caches match the oracle's)
    out, flags = run_attention(step, t)
    assert flags == 0, f"flags {flags:#x}"
    rows = list(range(step.T))
    ref, kc, _, terms = oracle_attention(step, before, rows=rows, terms=True)
    check_parity(out, ref, rows_of(terms, rows), step.row_positions(), step.geom,
                 "after a timed-out call")
    assert np.array_equal(t["k_cache"][0].cpu().view(torch.int16).numpy().view(np.uint16), kc)
