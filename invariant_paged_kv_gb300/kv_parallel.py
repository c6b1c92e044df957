"""KV-parallel page owners: key ranges and the gather-and-merge driver.

The keys of every lane are spread over W owners ("Numerics envelopes",
Layout invariance of query context parallelism: the page-sharded KV of the
KV-parallel owners, whose attention partials combine_attention_partials merges
with the ordered fold). Owner w holds keys [bounds[w][b], bounds[w + 1][b]) of
lane b; interior bounds are multiples of the lane's split length, so every
split of every row belongs to one owner. Each owner computes the partials of
its splits (pa_attention_partials), the partial buffers are all-gathered
(data movement only), and every rank folds each row's splits in global split
order (pa_merge_partials): the result is bitwise the single-owner one.
"""
from __future__ import annotations

import numpy as np

SPLIT_TOKENS = 512
MAX_SPLITS = 128


def split_len(keys: int) -> int:
    """Split length of a row with ``keys`` keys (the library's rule, on the host)."""
    s = SPLIT_TOKENS
    while -(-int(keys) // s) > MAX_SPLITS:
        s *= 2
    return s


def owner_bounds(ctx_lens, owners: int) -> np.ndarray:
    """int32 [owners + 1, B]: contiguous, split-aligned shards of each lane's
    keys, as even as whole splits allow (owner w gets splits
    [w n / W, (w + 1) n / W) of a lane with n splits)."""
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    B = ctx.shape[0]
    out = np.zeros((owners + 1, B), dtype=np.int64)
    for b in range(B):
        c = int(ctx[b])
        sl = split_len(max(c, 1))
        n = -(-c // sl)
        for w in range(owners + 1):
            out[w, b] = min(c, (w * n // owners) * sl)
        out[owners, b] = c
    return out.astype(np.int32)


def kv_parallel_attention(partials_fn, merge_fn, local_partials, group=None):
    """One KV-parallel step on this rank: compute this owner's partials into
    ``local_partials`` (a uint8 tensor), all-gather every owner's buffer
    (torch.distributed, back to back in rank order) and merge.

    ``partials_fn(local_partials)`` and ``merge_fn(gathered, owners)`` wrap
    pa.attention_partials / pa.merge_partials with the step's arguments.
    """
    import torch
    import torch.distributed as dist

    W = dist.get_world_size(group)
    partials_fn(local_partials)
    gathered = torch.empty(W * local_partials.numel(), dtype=local_partials.dtype,
                           device=local_partials.device)
    dist.all_gather_into_tensor(gathered, local_partials, group=group)
    return merge_fn(gathered, W)
