"""float8 e4m3fn codes and per-tensor scaled quantisation of K/V rows.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import or call this module. It shares
no code with the CUDA library and imports nothing from it.

Why a cache of 8-bit codes with scales: "P3: native paged-KV
continuous-batching sampler", Review (adversarial pass), the kv_dtype item --
K/V are dequantised on read; float8_e4m3fn used without scales was visibly
lossy, so fp8 KV needs per-tensor scales, not only a dtype switch (and the
"Tensor parallelism" Open items repeat that fp8 KV would double the pool).

The format is the one the name float8_e4m3fn stands for (the OCP 8-bit
floating point E4M3 encoding): bit 7 sign, bits 6..3 exponent with bias 7,
bits 2..0 mantissa. Exponent field 0 holds subnormals (m / 8) * 2^-6; fields
1..15 hold normals (1 + m / 8) * 2^(e - 7); the pattern S.1111.111 is NaN and
there is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448.

Readings where the pages stop at "per-tensor scales" (listed in the design
notes of this repository):
  * one float32 scale s per tensor (K and V of a layer each have one);
  * a stored code is RN-even(x / s) with x / s evaluated in float32 (the
    precision in which the device takes the same decision), finite values
    past 448 and infinities saturating to +-448 and NaN staying NaN;
  * a code reads back as decode(code) * s, exactly, in float64.
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0
NAN_CODE = 0x7F


def decode(codes) -> np.ndarray:
    """Exact float64 value of each code (uint8 array); NaN codes give NaN."""
    c = np.asarray(codes)
    if c.dtype != np.uint8:
        raise TypeError("e4m3 codes must be uint8")
    c = c.astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    sub = (m / 8.0) * 2.0 ** -6
    nrm = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    val = np.where(e == 0, sub, nrm)
    val = np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)
    return sign * val


def encode(y) -> np.ndarray:
    """Code of each float32 value: round to nearest, ties to the even code,
    saturating to +-448 (the sign of zero is kept; NaN gives NAN_CODE)."""
    y = np.asarray(y)
    if y.dtype != np.float32:
        raise TypeError("encode takes float32 values")
    a = np.abs(y.astype(np.float64))
    neg = np.signbit(y)
    special = ~np.isfinite(a)
    a = np.where(special, 0.0, a)
    # subnormal grid: step 2^-9 (a value that rounds up to 8 steps is the
    # smallest normal, code 8, so the two branches meet without a seam)
    q_sub = np.rint(np.minimum(a, 1.0) / 2.0 ** -9).astype(np.int64)
    # normal grid: for 2^e <= a < 2^(e+1) the step is 2^(e-3); the mantissa
    # steps q run 8..16 and q = 16 carries into the exponent field
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    e = E.astype(np.int64) - 1
    q_nrm = np.rint(a / np.exp2((e - 3).astype(np.float64))).astype(np.int64)
    mag = np.where(a < 2.0 ** -6, q_sub, (e + 7) * 8 + q_nrm - 8)
    mag = np.where(special | (a > MAX_FINITE), 126, np.minimum(mag, 126))
    code = (mag | np.where(neg, 0x80, 0)).astype(np.uint8)
    return np.where(np.isnan(y), np.uint8(NAN_CODE), code).astype(np.uint8)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) widened exactly to float32."""
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        raise TypeError("bf16 data must be carried as uint16 bit patterns")
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_bf16(bits, scale: float) -> np.ndarray:
    """Codes of bf16 values x under the per-tensor scale s: encode(x / s),
    the division in float32."""
    s = np.float32(scale)
    if not (np.isfinite(s) and s > 0):
        raise ValueError("scale must be finite and > 0")
    with np.errstate(over="ignore", invalid="ignore"):
        y = (bf16_bits_to_f32(bits) / s).astype(np.float32)
    return encode(y)


def dequantize(codes, scale: float) -> np.ndarray:
    """float64 values decode(code) * s."""
    return decode(codes) * float(np.float32(scale))
