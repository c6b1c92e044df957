"""Batch invariance on the GPU: a fixed target row keeps its output bits in
every step composition (GPU).

The target is a decode row at ctx 4096 ("Numerics envelopes", The contract,
item 2 and Acceptance: the same request alone and packed with random
co-batches must give identical bits). Neighbours are random decode rows and
256-row prefill chunks; up to 7 siblings share the target's first 255 full
blocks read-only (GRPO samples of one prompt, prefix sharing as in "P3:
native paged-KV continuous-batching sampler", Design, engine.py). The target
lane's index and the physical ids of its blocks change with the composition.
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


@pytest.fixture(scope="module")
def target():
    g = torch.Generator(device="cuda").manual_seed(4242)
    C = wl.INVARIANCE_TARGET_CTX
    mk = lambda *s: torch.randn(*s, generator=g, device="cuda", dtype=torch.bfloat16)
    return dict(k=mk(C, 8, 128), v=mk(C, 8, 128), q=mk(32, 128))


def _compose(t, target):
    step, trow = wl.invariance_step(t)
    tens = wl.make_tensors(step, 4000 + t, "cuda")
    lane = int(step.row_lane()[trow])
    bs = step.geom.block_size
    C = wl.INVARIANCE_TARGET_CTX
    pos = np.arange(C)
    flat = step.block_tables[lane, pos // bs].astype(np.int64) * bs + pos % bs
    idx = torch.from_numpy(flat).cuda()
    for name, src in (("k_cache", "k"), ("v_cache", "v")):
        tens[name][0].view(-1, 8, 128)[idx[:-1]] = target[src][:-1]
    # the last key arrives as this step's new row
    tens["k_new"][0][trow] = target["k"][-1]
    tens["v_new"][0][trow] = target["v"][-1]
    tens["q"][0][trow] = target["q"]
    return step, trow, tens


def test_target_matches_oracle_alone(target):
    step, trow, tens = _compose(1, target)
    out, flags = run_attention(step, tens)
    assert flags == 0
    ref, _, _, terms = oracle_attention(step, to_cpu(tens), rows=[trow], terms=True)
    check_parity(out[trow:trow + 1], ref[trow:trow + 1], rows_of(terms, [trow]),
                 step.row_positions()[[trow]], step.geom, "invariance target alone")


def test_target_bitwise_across_compositions(target):
    ref_bits = None
    seen_pos = set()
    for t in range(1, 65):
        step, trow, tens = _compose(t, target)
        out, flags = run_attention(step, tens)
        assert flags == 0, (t, flags)
        bits = out[trow].view(torch.int16).cpu()
        if ref_bits is None:
            ref_bits = bits
        else:
            assert torch.equal(bits, ref_bits), f"target row changed in the {t}-lane step"
        seen_pos.add(int(step.row_lane()[trow]))
        del tens
    assert len(seen_pos) > 10  # the target really moved around the step


def test_shared_blocks_untouched(target):
    """Blocks with refcount > 1 are read-only: the step's write leaves them unchanged."""
    step, trow, tens = _compose(8, target)
    shared = torch.from_numpy(step.shared_blocks).cuda()
    before = tens["k_cache"][0].index_select(0, shared).clone()
    run_attention(step, tens)
    after = tens["k_cache"][0].index_select(0, shared)
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))


def test_block_relabelling_bitwise():
    """Moving every block to a new physical id changes no output bit."""
    step = wl.decode_batch(0, lanes=24)
    tens = wl.make_tensors(step, 77, "cuda")
    a, _ = run_attention(step, {k: [v[0].clone()] for k, v in tens.items()})
    rng = np.random.default_rng(5)
    perm = rng.permutation(step.num_blocks)
    moved = wl.Step(step.geom, step.num_blocks, step.q_lens, step.ctx_lens,
                    np.where(step.block_tables >= 0, perm[np.maximum(step.block_tables, 0)],
                             -1).astype(np.int32),
                    (perm[step.slot_mapping // 16] * 16 + step.slot_mapping % 16).astype(np.int64))
    pt = torch.from_numpy(perm).cuda()
    t2 = {k: [v[0].clone()] for k, v in tens.items()}
    for name in ("k_cache", "v_cache"):
        t2[name][0][pt] = tens[name][0]
    b, _ = run_attention(moved, t2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_poisoned_tails_do_not_leak():
    """NaN in every non-key cache position: outputs finite and bit-identical."""
    step = wl.decode_batch(1, lanes=32)
    clean = wl.make_tensors(step, 99, "cuda", poison=False)
    dirty = {k: [v[0].clone()] for k, v in clean.items()}
    mask = torch.from_numpy(~wl.key_mask(step)).cuda()
    for name in ("k_cache", "v_cache"):
        dirty[name][0].view(step.num_blocks * 16, 8, 128)[mask] = float("nan")
    a, _ = run_attention(step, clean)
    b, _ = run_attention(step, dirty)
    assert not torch.isnan(b.float()).any()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_prefill_rows_bitwise_across_compositions():
    """A fixed 200-row prefill chunk (positions 800..999) keeps its output bits
    whatever lanes surround it and wherever its blocks sit."""
    geom = wl.Geometry(32, 8, 128, 16, "bf16")
    g = torch.Generator(device="cuda").manual_seed(99)
    C, Q = 1000, 200
    mk = lambda *s: torch.randn(*s, generator=g, device="cuda", dtype=torch.bfloat16)
    K, V, q = mk(C, 8, 128), mk(C, 8, 128), mk(Q, 32, 128)
    ref = None
    for t in (1, 2, 5, 17):
        rng = np.random.default_rng(500 + t)
        lanes = [(1, int(rng.integers(1, 5000))) if rng.random() < 0.6 else
                 (int(rng.integers(2, 300)), int(rng.integers(300, 3000))) for _ in range(t - 1)]
        pos = int(rng.integers(0, t))
        lanes.insert(pos, (Q, C))
        ql = [x[0] for x in lanes]
        cl = [x[1] for x in lanes]
        used = sum(-(-c // 16) for c in cl)
        step = wl.build_step(geom, ql, cl, int(used * 1.2) + 4, rng)
        tens = wl.make_tensors(step, 900 + t, "cuda")
        bs = 16
        p_ = np.arange(C)
        flat = torch.from_numpy(step.block_tables[pos, p_ // bs].astype(np.int64) * bs + p_ % bs).cuda()
        r0 = int(step.cu_seqlens_q[pos])
        tens["k_cache"][0].view(-1, 8, 128)[flat[:C - Q]] = K[:C - Q]
        tens["v_cache"][0].view(-1, 8, 128)[flat[:C - Q]] = V[:C - Q]
        tens["k_new"][0][r0:r0 + Q] = K[C - Q:]
        tens["v_new"][0][r0:r0 + Q] = V[C - Q:]
        tens["q"][0][r0:r0 + Q] = q
        out, flags = run_attention(step, tens)
        assert flags == 0
        bits = out[r0:r0 + Q].view(torch.int16).cpu()
        if ref is None:
            ref = bits
            rr = list(range(r0, r0 + Q))
            oref, _, _, terms = oracle_attention(step, to_cpu(tens), rows=rr, terms=True)
            check_parity(out[r0:r0 + Q], oref[rr], rows_of(terms, rr), step.row_positions()[rr],
                         step.geom, "invariance prefill chunk alone")
        else:
            assert torch.equal(bits, ref), f"prefill rows changed in the {t}-lane step"
