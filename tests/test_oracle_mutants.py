"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

The mutant list follows the mutation tests of "P3: native paged-KV
continuous-batching sampler" (Evidence, item 5: gather drops the last key,
slot mapping ignores the block offset, K heads flipped, causal mask off by
one) plus mistakes a from-scratch oracle could make (operands swapped, scale
dropped, unnormalised weights, wrong bf16 widening, row positions counted
from the chunk start).
"""
import numpy as np
import pytest

import oracle.paged_attention as pa
import oracle_pins

_orig_gather = pa.gather
_orig_attend = pa.attend_row


def _gather_drops_last(cache, table_row, ctx_len, block_size):
    return _orig_gather(cache, table_row, max(ctx_len - 1, 0), block_size)


def _slot_ignores_offset(slot, block_size):
    return slot // block_size, 0


def _heads_flipped(h, H, Hkv):
    return h % Hkv


def _causal_plus_one(position):
    return position + 2


def _causal_minus_one(position):
    return max(position, 1)


def _attend_swapped(q_row, K, V, position, scale):
    return _orig_attend(q_row, V, K, position, scale)


def _attend_no_scale(q_row, K, V, position, scale):
    return _orig_attend(q_row, K, V, position, 1.0)


def _unnormalised(scores):
    return np.exp(scores - np.max(scores))


def _widen_wrong(x, dtype):
    x = np.asarray(x)
    if dtype == "bf16":
        return (x.astype(np.uint32) << np.uint32(15)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def _kv_bytes_no_v(layers, kv_heads, head_dim, elem_bytes, tp_degree=1):
    return layers * (kv_heads // tp_degree) * head_dim * elem_bytes


MUTANTS = {
    "gather drops last key": ("gather", _gather_drops_last),
    "slot ignores block offset": ("slot_location", _slot_ignores_offset),
    "K heads flipped": ("kv_head_of", _heads_flipped),
    "causal one too many": ("visible_keys", _causal_plus_one),
    "causal one too few": ("visible_keys", _causal_minus_one),
    "K and V swapped": ("attend_row", _attend_swapped),
    "scale dropped": ("attend_row", _attend_no_scale),
    "weights not normalised": ("softmax_weights", _unnormalised),
    "bf16 widened with the wrong shift": ("widen", _widen_wrong),
    "kv bytes forget V": ("kv_bytes_per_token", _kv_bytes_no_v),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(pa, attr, fn)
    fails = oracle_pins.failures()
    assert fails, f"no pin caught the mutant '{name}'"


def test_control_passes():
    assert oracle_pins.failures() == []
