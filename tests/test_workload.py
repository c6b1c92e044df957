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


def _long_tail_small_pool(sample):
    return wl.long_tail(sample, pool_bytes_per_layer=1e8)  # pool = the used blocks


@pytest.mark.parametrize("make", [wl.tiny_f32, wl.decode_batch, wl.mixed_step,
                                  _long_tail_small_pool])
def test_configs_well_formed(make):
    _check_step(make(0))


def test_mixed_step_recipe():
    """Decode lanes first (q_len 1, ctx in [16, 16384]), then 8 chunks of 512
    new rows after U{0..4096} earlier keys."""
    for sample in range(3):
        s = wl.mixed_step(sample)
        assert list(s.q_lens[:120]) == [1] * 120 and list(s.q_lens[120:]) == [512] * 8
        assert s.ctx_lens[:120].min() >= 16 and s.ctx_lens[:120].max() <= 16384
        offs = s.ctx_lens[120:] - 512
        assert offs.min() >= 0 and offs.max() <= 4096


def test_length_distributions_follow_the_recipe():
    """Seeded lognormal medians (decode_batch 2048, mixed decode rows 3000) and
    the long tail's 90/10 split, over several samples."""
    dec = np.concatenate([wl.decode_batch(k).ctx_lens for k in range(5)])
    assert 1600 <= np.median(dec) <= 2600
    mix = np.concatenate([wl.mixed_step(k).ctx_lens[:120] for k in range(5)])
    assert 2400 <= np.median(mix) <= 3700
    for k in range(3):
        c = wl.long_tail(k, pool_bytes_per_layer=1e8).ctx_lens
        short, long_ = c[c < 16384], c[c >= 16384]
        assert len(short) == 230 and len(long_) == 26
        assert short.min() >= 1024 and short.max() <= 4096
        assert long_.min() >= 16384 and long_.max() <= 40960


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
