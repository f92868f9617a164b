"""Storage formats used by the CSA2 oracle, written from their definitions.

TEST INFRASTRUCTURE ONLY. This module belongs to the CPU oracle: only the
tests, the smoke check and the benchmark's CPU-baseline leg may import it.
The CUDA product path never calls into it and shares no code with it.

Formats (all decoded exactly into float64):

* bf16: 1 sign, 8 exponent (bias 127), 7 fraction bits; the upper half of an
  IEEE binary32. Encoding is round-to-nearest-even from float64.
* e4m3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 fraction bits, no
  infinities, 0x7F/0xFF are NaN, largest finite value 448, subnormals
  m * 2^-9. Encoding is round-to-nearest-even with saturation to +-448.
* ue8m0: an unsigned power-of-two scale 2^(E-127), E in [0, 254].

The block-32 fp8 KV format (one e4m3 code per channel plus one ue8m0 scale
per 32 consecutive channels) follows the page "DeepSeek-V4.1-Flash on WASTE",
section "The shape" (fp8 e4m3 with ue8m0 scales) and the PocketLLM page,
section "The CSA2 attention layers" (window quantized to FP8 over 32
elements). The pages do not state how the scale is chosen; the reading used
here is the smallest power of two that brings the block's largest magnitude
into the e4m3 range: scale = 2^k with k the least integer such that
amax <= 448 * 2^k, and an all-zero block takes E = 0.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
FP8_BLOCK = 32


# ----------------------------------------------------------------------------
# bf16
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16 array) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bf16 (round half to even); returns uint16 bits.

    The value is rounded once, directly from float64: the quantum of the
    binade that holds |x| is 2^(e-8) for |x| in [2^(e-1), 2^e) with 8
    significant bits, and 2^-133 below the smallest normal 2^-126.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_x = x.reshape(-1)
    flat_o = out.reshape(-1)
    ax = np.abs(flat_x)
    sign = np.signbit(flat_x)
    _, e = np.frexp(ax)  # ax = m * 2^e with m in [0.5, 1)
    q_exp = np.maximum(e, -125) - 8
    quantum = np.ldexp(1.0, q_exp)
    rounded = np.rint(ax / quantum) * quantum  # rint: half to even
    with np.errstate(over="ignore"):
        as32 = rounded.astype(np.float32)  # exact: rounded has <= 8 significant bits
    bits = (as32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    # overflow: anything that rounded past the largest finite bf16 is inf
    bits = np.where(rounded >= 2.0 ** 128, np.uint16(0x7F80), bits)
    bits = np.where(np.isnan(flat_x), np.uint16(0x7FC0), bits)
    bits = np.where(sign & ~np.isnan(flat_x), bits | np.uint16(0x8000), bits)
    flat_o[:] = bits
    return out


def round_bf16(x) -> np.ndarray:
    """float64 -> nearest bf16 value (as float64)."""
    return bf16_bits_to_f64(f64_to_bf16_bits(x))


def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 values at |x| (the quantum of x's binade)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(ax)
    return np.ldexp(1.0, np.maximum(e, -125) - 8)


# ----------------------------------------------------------------------------
# e4m3 and ue8m0
# ----------------------------------------------------------------------------

def _e4m3_table() -> np.ndarray:
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = s * m * 2.0 ** -9
        else:
            vals[code] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _e4m3_table()
# non-negative finite codes sorted by value: code c in [0, 126] has value
# E4M3_VALUES[c], strictly increasing in c
_POS_VALUES = E4M3_VALUES[:127]


def e4m3_bits_to_f64(bits) -> np.ndarray:
    return E4M3_VALUES[np.asarray(bits, dtype=np.uint8)]


def f64_to_e4m3_bits(x) -> np.ndarray:
    """Round to e4m3 (half to even), saturating to +-448. NaN is not accepted."""
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN has no e4m3 encoding in this format")
    ax = np.abs(x)
    _, e = np.frexp(ax)  # binade [2^(e-1), 2^e)
    # 3 fraction bits: quantum 2^(e-1-3); subnormal quantum 2^-9 below 2^-6
    quantum = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    r = np.rint(ax / quantum) * quantum
    r = np.minimum(r, E4M3_MAX)
    code = np.searchsorted(_POS_VALUES, r)
    if not np.all(_POS_VALUES[np.minimum(code, 126)] == r):
        raise AssertionError("rounded value is not an e4m3 grid point")
    code = code.astype(np.uint8)
    # the sign survives rounding to zero (a negative value that underflows is -0)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


def ue8m0_to_f64(e) -> np.ndarray:
    e = np.asarray(e, dtype=np.int64)
    return np.ldexp(1.0, e - 127)


def fp8_block_scale_exponent(amax: float) -> int:
    """ue8m0 byte for one block: least k with amax <= 448 * 2^k, E = k + 127."""
    if amax == 0.0:
        return 0
    k = int(np.ceil(np.log2(amax / E4M3_MAX)))
    # settle the rounding of log2 exactly with power-of-two comparisons
    while amax > E4M3_MAX * 2.0 ** k:
        k += 1
    while amax <= E4M3_MAX * 2.0 ** (k - 1):
        k -= 1
    return int(min(max(k + 127, 0), 254))


def fp8_block_scale_exponents(amax) -> np.ndarray:
    """The same rule as fp8_block_scale_exponent, for an array of block maxima.

    With amax = f * 2^e (f in [0.5, 1), from frexp) and 448 = 0.875 * 2^9,
    amax <= 448 * 2^k holds exactly when k >= e - 9 (f <= 0.875) or
    k >= e - 8 (f > 0.875); the least such k is taken.
    """
    amax = np.asarray(amax, dtype=np.float64)
    f, e = np.frexp(amax)
    k = np.where(f <= 0.875, e - 9, e - 8)
    return np.where(amax == 0.0, 0, np.clip(k + 127, 0, 254)).astype(np.uint8)


def fp8_block_quantize(x, block: int = FP8_BLOCK):
    """Quantize rows [n, D] to (codes uint8 [n, D], scale bytes uint8 [n, D/block])."""
    x = np.asarray(x, dtype=np.float64)
    n, d = x.shape
    if d % block:
        raise ValueError("row length must be a multiple of the block")
    xb = x.reshape(n, d // block, block)
    amax = np.abs(xb).max(axis=2)
    exps = fp8_block_scale_exponents(amax)
    scale = ue8m0_to_f64(exps)[:, :, None]
    codes = f64_to_e4m3_bits(xb / scale).reshape(n, d)
    return codes, exps


def fp8_block_dequantize(codes, exps, block: int = FP8_BLOCK) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    n, d = codes.shape
    v = e4m3_bits_to_f64(codes).reshape(n, d // block, block)
    return (v * ue8m0_to_f64(exps)[:, :, None]).reshape(n, d)


# ----------------------------------------------------------------------------
# e2m1 (fp4) blocks
#
# "Reading Notes of DeepSeek-V4.1-Flash", section 3f, C4 (FP4 main KV cache):
# each cached number is a 4-bit E2M1 code times a scale shared by 16
# channels; the grid is {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}, the scale
# s = amax / 6 is an 8-bit E4M3 number, c_i = round_E2M1(x_i / s) and the
# decoded value is s * c_i. The PocketLLM page "DeepSeek-V4.1-Flash", section
# "The op layer", fixes the two details the formula leaves open: the stored
# scale is e4m3(amax / 6), the ratio rounded to E4M3, and the amax is floored
# at 6 * 2^-9 so that an all-zero block still has a nonzero scale. The index
# keys use the MXFP4 variant of the same codes (C2 "Resulting memory"; the
# op-layer page: E8M0 scales over 32 channels), whose scale is
# 2^round(log2(amax / 6)), amax floored at 6 * 2^-126.
#
# Readings where the pages are silent: round_E2M1 is round-to-nearest with
# ties to the even code (mantissa bit 0), saturating at +-6 (x / s can pass 6
# once s is rounded down); the code's sign bit is kept when a negative value
# rounds to 0; round(log2(.)) rounds to nearest (an exact half never occurs
# for a nonzero finite amax / 6 that is not a power of two times sqrt 2).
# Codes are stored two to a byte, the even channel in the low nibble.
# ----------------------------------------------------------------------------

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])  # magnitude of code & 7
E2M1_MAX = 6.0
FP4_BLOCK = 16
MXFP4_BLOCK = 32
FP4_AMAX_FLOOR = 6.0 * 2.0 ** -9
MXFP4_AMAX_FLOOR = 6.0 * 2.0 ** -126


def f64_to_e2m1_codes(x) -> np.ndarray:
    """Nearest E2M1 code (ties to the even code, saturating at +-6); uint8 in [0, 15]."""
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN has no e2m1 encoding")
    ax = np.minimum(np.abs(x), E2M1_MAX)
    hi = np.searchsorted(E2M1_VALUES, ax)          # first magnitude >= ax
    hi = np.minimum(hi, 7)
    lo = np.maximum(hi - 1, 0)
    d_lo = ax - E2M1_VALUES[lo]
    d_hi = E2M1_VALUES[hi] - ax
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(8), code).astype(np.uint8)


def e2m1_codes_to_f64(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    v = E2M1_VALUES[c & 7]
    return np.where(c & 8, -v, v)


def fp4_block_quantize(x, block: int = FP4_BLOCK):
    """Rows [n, D] -> (codes uint8 [n, D], e4m3 scale bytes uint8 [n, D/block])."""
    x = np.asarray(x, dtype=np.float64)
    n, d = x.shape
    if d % block:
        raise ValueError("row length must be a multiple of the block")
    xb = x.reshape(n, d // block, block)
    amax = np.abs(xb).max(axis=2)
    sbits = f64_to_e4m3_bits(np.maximum(amax, FP4_AMAX_FLOOR) / E2M1_MAX)
    s = e4m3_bits_to_f64(sbits)[:, :, None]
    codes = f64_to_e2m1_codes(xb / s).reshape(n, d)
    return codes, sbits


def fp4_block_dequantize(codes, sbits, block: int = FP4_BLOCK) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    n, d = codes.shape
    v = e2m1_codes_to_f64(codes).reshape(n, d // block, block)
    return (v * e4m3_bits_to_f64(sbits)[:, :, None]).reshape(n, d)


def mxfp4_block_quantize(x, block: int = MXFP4_BLOCK):
    """Rows [n, D] -> (codes uint8 [n, D], ue8m0 scale bytes uint8 [n, D/block])."""
    x = np.asarray(x, dtype=np.float64)
    n, d = x.shape
    if d % block:
        raise ValueError("row length must be a multiple of the block")
    xb = x.reshape(n, d // block, block)
    amax = np.maximum(np.abs(xb).max(axis=2), MXFP4_AMAX_FLOOR)
    # round(log2(r)) for r = f * 2^k, f in [0.5, 1): k - 1 when log2 f < -1/2,
    # i.e. f < 2^-1/2, else k (f = 2^-1/2 exactly cannot occur)
    f, k = np.frexp(amax / E2M1_MAX)
    e = np.where(f < 2.0 ** -0.5, k - 1, k).astype(np.int64)
    ebytes = np.clip(e + 127, 0, 254).astype(np.uint8)
    s = ue8m0_to_f64(ebytes)[:, :, None]
    codes = f64_to_e2m1_codes(xb / s).reshape(n, d)
    return codes, ebytes


def mxfp4_block_dequantize(codes, ebytes, block: int = MXFP4_BLOCK) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    n, d = codes.shape
    v = e2m1_codes_to_f64(codes).reshape(n, d // block, block)
    return (v * ue8m0_to_f64(ebytes)[:, :, None]).reshape(n, d)


def pack_e2m1(codes) -> np.ndarray:
    """[n, D] codes -> [n, D/2] bytes, channel 2i in the low nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack_e2m1(packed) -> np.ndarray:
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty((b.shape[0], 2 * b.shape[1]), dtype=np.uint8)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out
