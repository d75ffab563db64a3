"""Low-precision read-copy formats (test infrastructure only).

ReplaySSM keeps the high-precision checkpoint for the recurrence and a
separate low-precision copy that only serves reads, so the copy's rounding
error never re-enters later updates ([ai-jitan] 何がどれだけ速くなったのか,
item 3; [richland] What shipped, the paragraph on quantization).  The pages
name NVFP4 and FP8; the element formats are the OCP ones:

* e4m3 ("FP8 E4M3", no infinities): 1 sign, 4 exponent (bias 7), 3 mantissa
  bits; largest finite 448; subnormals m * 2**-9; code 0x7F/0xFF is NaN.
* e2m1 ("FP4 E2M1"): 1 sign, 2 exponent (bias 1), 1 mantissa bit; values
  0, 0.5, 1, 1.5, 2, 3, 4, 6.

Encoding is round-to-nearest, ties to the even code, saturating to the
largest finite magnitude.  Scales and the scaled values are computed in
float32 (the precision the kernels take these decisions in), then encoded.

Read-copy layouts (one state matrix = one head: R rows x N columns):

* FP8 per-row: codes [..][R][N] uint8, one float32 scale per row,
  scale = amax(row) / 448, code = e4m3(x / scale); amax = 0 gives scale 0 and
  all-zero codes.
* NVFP4: per matrix s = amax / (448 * 6); per 16-element block along N a
  block scale e4m3(amax_blk / (6 * s)); code = e2m1(x / (blockscale * s)),
  two codes per byte (element 2i in the low nibble, 2i+1 in the high nibble).
  A zero divisor gives zero codes.
"""

from __future__ import annotations

import numpy as np


# --- element formats -------------------------------------------------------

def e4m3_decode(code) -> np.ndarray:
    """Value of e4m3 codes (uint8) as float64, from the bit-field definition."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = m * 2.0 ** -9
    val = s * np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, val)


def e2m1_decode(code) -> np.ndarray:
    """Value of e2m1 codes (4-bit, uint8) as float64, from the bit-field definition."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    normal = (1.0 + m / 2.0) * np.exp2(e - 1.0)
    sub = m * 0.5
    return s * np.where(e == 0, sub, normal)


def _rne_encode(x, table_codes, table_vals, max_finite, sign_bit):
    """Nearest table value, ties to the even code, saturating, sign kept."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), max_finite)
    idx = np.searchsorted(table_vals, mag)            # table_vals[idx-1] < mag <= table_vals[idx]
    idx = np.clip(idx, 1, len(table_vals) - 1)
    lo_v = table_vals[idx - 1]
    hi_v = table_vals[idx]
    lo_c = table_codes[idx - 1]
    hi_c = table_codes[idx]
    d_lo = mag - lo_v
    d_hi = hi_v - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi_c % 2 == 0))
    code = np.where(pick_hi, hi_c, lo_c)
    code = np.where(mag == 0.0, 0, code)
    neg = np.signbit(x)
    return (code | np.where(neg, sign_bit, 0)).astype(np.uint8)


_E4M3_CODES = np.arange(0, 0x7F, dtype=np.int64)          # non-negative finite codes 0..126
_E4M3_VALS = e4m3_decode(_E4M3_CODES)
_E2M1_CODES = np.arange(0, 8, dtype=np.int64)
_E2M1_VALS = e2m1_decode(_E2M1_CODES)


def e4m3_encode(x) -> np.ndarray:
    """e4m3 code of each value (round to nearest even, saturate to +-448)."""
    return _rne_encode(x, _E4M3_CODES, _E4M3_VALS, 448.0, 0x80)


def e2m1_encode(x) -> np.ndarray:
    """e2m1 code of each value (round to nearest even, saturate to +-6)."""
    return _rne_encode(x, _E2M1_CODES, _E2M1_VALS, 6.0, 0x8)


# --- read-copy formats -------------------------------------------------------

def _f32(x):
    return np.asarray(x, dtype=np.float32)


def fp8_rows_quantize(S32: np.ndarray):
    """FP8 per-row read copy of float32 matrices [..][R][N].

    Returns (codes uint8 [..][R][N], scales float32 [..][R]).
    """
    S32 = _f32(S32)
    amax = np.max(np.abs(S32), axis=-1)                       # float32
    scale = (amax / np.float32(448.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = (S32 / scale[..., None]).astype(np.float32)
    codes = e4m3_encode(scaled)
    codes = np.where(scale[..., None] == 0, 0, codes).astype(np.uint8)
    return codes, scale


def fp8_rows_dequantize(codes, scales) -> np.ndarray:
    """float64 values of an FP8 per-row read copy."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def nvfp4_quantize(S32: np.ndarray):
    """NVFP4 read copy of float32 matrices [..][R][N] (N a multiple of 16).

    Returns (packed codes uint8 [..][R][N/2], block scales uint8 e4m3
    [..][R][N/16], matrix scales float32 [..]).
    """
    S32 = _f32(S32)
    R, N = S32.shape[-2], S32.shape[-1]
    lead = S32.shape[:-2]
    amax = np.max(np.abs(S32), axis=(-2, -1))                 # float32 [..]
    s = (amax / np.float32(448.0 * 6.0)).astype(np.float32)
    blocks = S32.reshape(lead + (R, N // 16, 16))
    amax_blk = np.max(np.abs(blocks), axis=-1)                 # [..][R][N/16]
    six_s = (np.float32(6.0) * s).astype(np.float32)[..., None, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (amax_blk / six_s).astype(np.float32)
    bs_code = np.where(six_s == 0, 0, e4m3_encode(r)).astype(np.uint8)
    bs_val = e4m3_decode(bs_code).astype(np.float32)
    d = (bs_val * s[..., None, None]).astype(np.float32)       # [..][R][N/16]
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = (blocks / d[..., None]).astype(np.float32)
    codes = np.where(d[..., None] == 0, 0, e2m1_encode(scaled)).astype(np.uint8)
    codes = codes.reshape(lead + (R, N))
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, bs_code, s


def nvfp4_dequantize(packed, bs_code, s) -> np.ndarray:
    """float64 values of an NVFP4 read copy."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 0xF
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (packed.shape[-1] * 2,))
    vals = e2m1_decode(codes)
    R, N = vals.shape[-2], vals.shape[-1]
    blk = e4m3_decode(bs_code)                                 # [..][R][N/16]
    vals = vals.reshape(vals.shape[:-1] + (N // 16, 16)) * blk[..., None]
    vals = vals.reshape(vals.shape[:-2] + (N,))
    return vals * np.asarray(s, dtype=np.float64)[..., None, None]
