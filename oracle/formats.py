"""Number formats of the MSA caches, decoded and encoded from their definitions.

TEST INFRASTRUCTURE (see the package docstring).

* bf16: the upper 16 bits of an IEEE binary32.
* FP8 E4M3 (OCP "E4M3FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
  subnormals when the exponent field is 0; the pattern S.1111.111 is NaN; there
  is no infinity; the largest finite magnitude is 448.
* FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* NVFP4 (the KV format of "MiniMax-M3.1-Flash Day-0 対応", section
  "何が新しいか"): E2M1 values, one E4M3 scale per 16 consecutive values and one
  fp32 scale per tensor; value = e2m1 * e4m3_scale * global.

Encoders round to nearest with ties to the even code and saturate to the
largest finite magnitude ("satfinite"), the rounding used by the GPU's
conversion instructions.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_from_fields(codes: np.ndarray) -> np.ndarray:
    """E4M3 byte -> fp64, by the bit-field definition."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.power(2.0, (e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)
    return sign * mag


def e2m1_from_fields(nibbles: np.ndarray) -> np.ndarray:
    """E2M1 nibble -> fp64, by the bit-field definition (bias 1, 1 mantissa bit)."""
    c = np.asarray(nibbles).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    mag = np.where(e == 0, (m / 2.0) * 2.0 ** 0, (1.0 + m / 2.0) * np.power(2.0, (e - 1).astype(np.float64)))
    return sign * mag


# Decoding large arrays goes through the tables of all codes built from the definitions above.
_E4M3_TABLE = e4m3_from_fields(np.arange(256))
_E2M1_TABLE = e2m1_from_fields(np.arange(16))


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _E4M3_TABLE[np.asarray(codes).astype(np.uint8)]


def e2m1_decode(nibbles: np.ndarray) -> np.ndarray:
    return _E2M1_TABLE[np.asarray(nibbles).astype(np.uint8) & 0xF]


# Non-negative finite values, indexed by code (ascending in value).
_E4M3_POS = e4m3_decode(np.arange(0, 0x7F))   # codes 0x00..0x7E, 0 .. 448
_E2M1_POS = e2m1_decode(np.arange(0, 8))      # codes 0..7, 0 .. 6


def _encode_rne(x: np.ndarray, table: np.ndarray, sign_bit: int) -> np.ndarray:
    """Nearest table entry to |x|, ties to the even code, saturating at the top."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    top = len(table) - 1
    lo = np.clip(np.searchsorted(table, a, side="right") - 1, 0, top)
    hi = np.minimum(lo + 1, top)
    dlo = a - table[lo]
    dhi = table[hi] - a
    pick_hi = (hi != lo) & ((dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0)))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    code = np.where(np.signbit(x), code | sign_bit, code)
    return code.astype(np.uint8)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """fp32/fp64 -> E4M3 byte, round to nearest even, saturating at +-448."""
    return _encode_rne(x, _E4M3_POS, 0x80)


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """fp32/fp64 -> E2M1 nibble (in the low 4 bits), round to nearest even, saturating at +-6."""
    return _encode_rne(x, _E2M1_POS, 0x8)


def nvfp4_unpack(packed: np.ndarray) -> np.ndarray:
    """[..., D/2] bytes -> [..., D] nibbles; the low nibble holds the even element."""
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def nvfp4_pack(nibbles: np.ndarray) -> np.ndarray:
    n = np.asarray(nibbles).astype(np.uint8)
    return (n[..., 0::2] & 0xF) | ((n[..., 1::2] & 0xF) << 4)


def nvfp4_decode(packed: np.ndarray, scales: np.ndarray, global_scale: float) -> np.ndarray:
    """NVFP4 -> fp64: e2m1 * (E4M3 scale of its 16-element group) * global scale."""
    vals = e2m1_decode(nvfp4_unpack(packed))
    sc = e4m3_decode(scales)
    sc = np.repeat(sc, 16, axis=-1)
    return vals * sc * float(np.float32(global_scale))
