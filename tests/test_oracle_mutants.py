"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

The mutant list follows the mutation tests of "P3: native paged-KV
continuous-batching sampler" (Evidence, item 5: gather drops the last key,
slot mapping ignores the block offset, K heads flipped, causal mask off by
one) plus mistakes a from-scratch oracle could make (operands swapped, scale
dropped, unnormalised weights, wrong bf16 widening, row positions counted
from the chunk start), and for the e4m3 cache format: exponent bias off by
one, subnormals read as normals, truncation instead of rounding, ties away
from zero, no saturation, the scale ignored or applied the wrong way.
"""
import math

import numpy as np
import pytest

import oracle.decode_gemm as dg
import oracle.e4m3 as e4m3
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


_orig_decode = e4m3.decode
_orig_encode = e4m3.encode


def _decode_bias8(codes):
    v = _orig_decode(codes)
    e = (np.asarray(codes).astype(np.int64) >> 3) & 0xF
    return np.where(e > 0, v / 2.0, v)


def _decode_subnormal_as_normal(codes):
    c = np.asarray(codes).astype(np.int64)
    v = _orig_decode(codes)
    e, m = (c >> 3) & 0xF, (c & 7).astype(np.float64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    return np.where((e == 0) & (m > 0), sign * (1 + m / 8) * 2.0 ** -7, v)


def _encode_truncates(y):
    # round toward zero: pick the code below, then step up only on exact hits
    y = np.asarray(y)
    c = _orig_encode(y)
    back = np.abs(_orig_decode(c))
    over = back > np.abs(y.astype(np.float64))
    return np.where(over & ((c & 0x7F) > 0), c - 1, c).astype(np.uint8)


def _encode_ties_away(y):
    y = np.asarray(y)
    c = _orig_encode(y)
    a = np.abs(y.astype(np.float64))
    nxt = (np.minimum((c & 0x7F) + 1, 126) | (c & 0x80)).astype(np.uint8)
    v_c, v_n = np.abs(_orig_decode(c)), np.abs(_orig_decode(nxt))
    tie = (v_c < a) & (a - v_c == v_n - a)  # a tie that went to the lower code
    return np.where(tie, nxt, c).astype(np.uint8)


def _encode_no_saturation(y):
    y = np.asarray(y)
    c = _orig_encode(y)
    big = np.isfinite(y) & (np.abs(y.astype(np.float64)) > 464)
    return np.where(big, (c & 0x80) | 0x7F, c).astype(np.uint8)


def _dequantize_ignores_scale(codes, scale):
    return _orig_decode(codes)


def _quantize_multiplies(bits, scale):
    return _orig_encode((e4m3.bf16_bits_to_f32(bits) * np.float32(scale)).astype(np.float32))


_orig_fold = pa.fold_partials


def _fold_unordered_max(parts):
    # uses the last partial's max as the reference without rescaling the others
    M = parts[-1][0]
    L = sum(l * math.exp(m - M) for m, l, _ in parts[:-1]) + parts[-1][1]
    A = sum(np.asarray(a) for _, _, a in parts)
    return A / L


def _fold_drops_first(parts):
    return _orig_fold(parts[1:] if len(parts) > 1 else parts)


_orig_terms = pa.attend_row_terms


def _terms_w_not_squared(q_row, K, V, position, scale):
    t = _orig_terms(q_row, K, V, position, scale)
    t["w2v2"] = t["wv"] ** 2  # (sum w |v|)^2 in place of sum w^2 v^2
    return t


def _terms_signed_q(q_row, K, V, position, scale):
    H, D = q_row.shape
    t = _orig_terms(q_row, K, V, position, scale)
    n = position + 1
    for h in range(H):
        kv = h // (H // K.shape[1])
        t["cmax"][h] = np.max(np.abs(K[:n, kv, :] @ q_row[h]))
    return t


def _terms_drop_last_key(q_row, K, V, position, scale):
    t = _orig_terms(q_row, K, V, max(position - 1, 0), scale)
    return t


TERMS_MUTANTS = {
    "bound terms square the weighted mean instead of weighting squares": _terms_w_not_squared,
    "bound terms take |q.k| for sum |q||k|": _terms_signed_q,
    "bound terms drop the last key": _terms_drop_last_key,
}


@pytest.mark.parametrize("name", sorted(TERMS_MUTANTS))
def test_terms_mutant_is_caught(name, monkeypatch):
    monkeypatch.setattr(pa, "attend_row_terms", TERMS_MUTANTS[name])
    assert oracle_pins.failures(), f"no pin caught the mutant '{name}'"


FOLD_MUTANTS = {
    "fold forgets to rescale": ("fold_partials", _fold_unordered_max),
    "fold drops the first partial": ("fold_partials", _fold_drops_first),
}


_orig_linear = dg.linear


def _linear_k_reversed(x_bits, w_bits):
    return dg.widen_bf16(x_bits) @ dg.widen_bf16(w_bits)[:, ::-1].T


def _linear_drops_last_k(x_bits, w_bits):
    return _orig_linear(np.asarray(x_bits)[:, :-1], np.asarray(w_bits)[:, :-1])


def _abs_sum_signed(x_bits, w_bits):
    return np.abs(dg.widen_bf16(x_bits) @ dg.widen_bf16(w_bits).T)


def _linear_wrong_widening(x_bits, w_bits):
    x = (np.asarray(x_bits).astype(np.uint32) << np.uint32(15)).view(np.float32).astype(np.float64)
    return x @ dg.widen_bf16(w_bits).T


GEMM_MUTANTS = {
    "gemm pairs x and w along reversed k": ("linear", _linear_k_reversed),
    "gemm drops the last k": ("linear", _linear_drops_last_k),
    "gemm widens x with the wrong shift": ("linear", _linear_wrong_widening),
    "abs sum takes |sum| instead of sum of |x w|": ("abs_sum", _abs_sum_signed),
}


@pytest.mark.parametrize("name", sorted(GEMM_MUTANTS))
def test_gemm_mutant_is_caught(name, monkeypatch):
    attr, fn = GEMM_MUTANTS[name]
    monkeypatch.setattr(dg, attr, fn)
    assert oracle_pins.failures(), f"no pin caught the mutant '{name}'"


@pytest.mark.parametrize("name", sorted(FOLD_MUTANTS))
def test_fold_mutant_is_caught(name, monkeypatch):
    attr, fn = FOLD_MUTANTS[name]
    monkeypatch.setattr(pa, attr, fn)
    assert oracle_pins.failures(), f"no pin caught the mutant '{name}'"


E4M3_MUTANTS = {
    "e4m3 exponent bias 8": ("decode", _decode_bias8),
    "e4m3 subnormals read as normals": ("decode", _decode_subnormal_as_normal),
    "e4m3 encode truncates": ("encode", _encode_truncates),
    "e4m3 ties away from zero": ("encode", _encode_ties_away),
    "e4m3 no saturation": ("encode", _encode_no_saturation),
    "fp8 scale ignored on read": ("dequantize", _dequantize_ignores_scale),
    "fp8 scale multiplied on write": ("quantize_bf16", _quantize_multiplies),
}


@pytest.mark.parametrize("name", sorted(E4M3_MUTANTS))
def test_e4m3_mutant_is_caught(name, monkeypatch):
    attr, fn = E4M3_MUTANTS[name]
    monkeypatch.setattr(e4m3, attr, fn)
    fails = oracle_pins.failures()
    assert fails, f"no pin caught the mutant '{name}'"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(pa, attr, fn)
    fails = oracle_pins.failures()
    assert fails, f"no pin caught the mutant '{name}'"


def test_control_passes():
    assert oracle_pins.failures() == []
