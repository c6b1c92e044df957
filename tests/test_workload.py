"""Host-side step descriptors and the block allocator (CPU only)."""
import numpy as np
import pytest

from invariant_paged_kv_gb300 import workload as wl


def test_allocator_property_run():
    """10,000 random events, books checked after every one (P3 Evidence item 4)."""
    rng = np.random.default_rng(0)
    NB = 64
    a = wl.BlockAllocator(NB, order=rng.permutation(NB))
    live = []  # list of block lists, each holding one reference per block
    ooms = shared = 0
    for _ in range(10_000):
        ev = rng.integers(0, 4)
        if ev == 0:  # admit
            n = int(rng.integers(0, 9))
            try:
                live.append(a.alloc(n))
            except wl.AllocatorError:
                ooms += 1
        elif ev == 1 and live:  # share a prefix
            src = live[int(rng.integers(0, len(live)))]
            k = int(rng.integers(0, len(src) + 1))
            a.incref(src[:k])
            live.append(list(src[:k]))
            shared += 1
        elif ev == 2 and live:  # grow
            i = int(rng.integers(0, len(live)))
            try:
                live[i] = live[i] + a.alloc(int(rng.integers(1, 4)))
            except wl.AllocatorError:
                ooms += 1
        elif ev == 3 and live:  # finish
            a.free(live.pop(int(rng.integers(0, len(live)))))
        a.check_consistent()
        counts = np.zeros(NB, dtype=np.int64)
        for blocks in live:
            for b in blocks:
                counts[b] += 1
        assert all(a.refcount(b) == counts[b] for b in range(NB))
    assert ooms > 100 and shared > 100
    for blocks in live:
        a.free(blocks)
    a.check_consistent()
    assert a.num_free == NB


def test_allocator_refusals():
    a = wl.BlockAllocator(4)
    got = a.alloc(3)
    with pytest.raises(wl.AllocatorError):
        a.alloc(2)
    assert a.num_free == 1  # all-or-nothing
    a.free(got[:1])
    with pytest.raises(wl.AllocatorError):
        a.free(got[:1])  # double free
    with pytest.raises(wl.AllocatorError):
        a.incref(got[:1])
    a.check_consistent()


def _check_step(step):
    bs = step.geom.block_size
    assert step.block_tables.dtype == np.int32
    assert step.slot_mapping.dtype == np.int64
    assert step.slot_mapping.shape == (step.T,)
    assert len(set(step.slot_mapping.tolist())) == step.T  # unique slots
    pos = step.row_positions()
    lane = step.row_lane()
    for t in range(step.T):
        b, p = lane[t], pos[t]
        blk = step.block_tables[b, p // bs]
        assert step.slot_mapping[t] == blk * bs + p % bs
        assert blk not in set(step.shared_blocks.tolist())  # no write into a shared block
    for b in range(step.B):
        n = -(-int(step.ctx_lens[b]) // bs)
        row = step.block_tables[b]
        assert np.all(row[:n] >= 0) and np.all(row[:n] < step.num_blocks)
        assert np.all(row[n:] == -1)


@pytest.mark.parametrize("make", [wl.tiny_f32, wl.decode_batch, wl.mixed_step])
def test_configs_well_formed(make):
    _check_step(make(0))


def test_config_shapes():
    s = wl.tiny_f32(0)
    assert list(s.ctx_lens) == [3, 9, 17, 40] and s.T == 4 and s.num_blocks == 64
    s = wl.decode_batch(0)
    assert s.B == 64 and s.T == 64 and s.ctx_lens.min() >= 16 and s.ctx_lens.max() <= 16384
    s = wl.mixed_step(0)
    assert s.T == 8 * 512 + 120 and s.B == 128 and s.max_q_len == 512
    s = wl.long_tail(0, pool_bytes_per_layer=1e8)
    assert s.B == 256 and s.T == 256
    assert int((s.ctx_lens >= 16384).sum()) == 26
    assert s.ctx_lens.min() >= 1024 and s.ctx_lens.max() <= 40960


@pytest.mark.parametrize("t", [1, 2, 5, 9, 33, 64])
def test_invariance_compositions(t):
    step, target_row = wl.invariance_step(t)
    _check_step(step)
    assert step.B == t
    lane = step.row_lane()[target_row]
    assert step.ctx_lens[lane] == wl.INVARIANCE_TARGET_CTX and step.q_lens[lane] == 1
    if t > 1:
        assert len(step.shared_blocks) == (wl.INVARIANCE_TARGET_CTX - 1) // 16


def test_poison_marks_only_non_keys():
    step = wl.tiny_f32(0)
    t = wl.make_tensors(step, 3, poison=True)
    kc = t["k_cache"][0].view(-1, step.geom.Hkv, step.geom.D)
    mask = wl.key_mask(step)
    assert not kc[mask].isnan().any()
    assert kc[~mask].isnan().all()
