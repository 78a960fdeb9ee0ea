"""FP8 (E4M3) KV cache: the oracle's quantiser, dequantiser and cache write.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``): only the
tests, the smoke check and the benchmark's CPU legs use it.

Source: "KV cache & PagedAttention -- vi sao chatbot AI ton bo nho"
(aiwiki.vn), the paragraph on quantisation and offloading: a quantised KV
cache keeps keys and values in a lower-precision representation to cut the
bytes per element, paying a conversion cost and risking numerical error.  The
page names no format and no scaling rule; the readings taken here are:

* the representation is the 8-bit float E4M3 of the OCP FP8 format (sign, 4
  exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
  subnormals m * 2**-9; no infinities; S.1111.111 is NaN; largest finite
  value 448);
* one float32 scale per tensor (one for K, one for V): the code of a value x
  is the E4M3 number nearest to the float32 quotient fl32(x / scale), ties to
  the even code, magnitudes beyond 448 (infinities included) saturating to
  +-448, NaN giving the NaN code 0x7F;
* the value a code stands for is e4m3(code) * scale, and attention over a
  quantised cache is ordinary attention over those values.

Cache layout (codes, one byte each): K is [num_blocks][Hkv][block_size][D]
like the bf16 cache; V is stored transposed inside each block,
[num_blocks][Hkv][D][block_size].
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code, straight from the field definition."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * 2.0 ** (e - 7) * (1.0 + m / 8.0)


# all 256 codes, and the 127 non-negative finite ones in code order (which is
# also increasing value order)
_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
_GRID = _TABLE[:0x7F].copy()


def e4m3_to_float(codes) -> np.ndarray:
    """float64 values of an array of codes (any integer dtype)."""
    return _TABLE[np.asarray(codes).astype(np.int64) & 0xFF]


def float_to_e4m3(x) -> np.ndarray:
    """Round float32 values to E4M3 codes (nearest, ties to even, saturating).

    The rounding decision compares |x| with the midpoint of the two
    neighbouring grid values; both are exact in float64, so the comparison is
    exact for every float32 input.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    nan = np.isnan(x)
    sat = ~nan & (a >= E4M3_MAX)
    a_in = np.where(nan | sat, 0.0, a)
    hi = np.minimum(np.searchsorted(_GRID, a_in, side="left"), len(_GRID) - 1)
    lo = np.maximum(hi - 1, 0)
    mid = (_GRID[lo] + _GRID[hi]) / 2.0  # exact in float64
    code = np.where(_GRID[hi] == a_in, hi,
                    np.where(a_in < mid, lo,
                             np.where(a_in > mid, hi, np.where(lo % 2 == 0, lo, hi))))
    code = np.where(sat, 0x7E, code) | np.where(np.signbit(x), 0x80, 0)
    code = np.where(nan, NAN_CODE, code)
    return code.astype(np.uint8)


def quantize(x, scale: float) -> np.ndarray:
    """Codes of ``x`` under a per-tensor ``scale``: e4m3(fl32(x / scale))."""
    x32 = np.asarray(x, dtype=np.float32)
    q = np.divide(x32, np.float32(scale), dtype=np.float32)
    return float_to_e4m3(q)


def dequantize(codes, scale: float) -> np.ndarray:
    """float64 values e4m3(code) * scale (exact: 4 and 24 significant bits)."""
    return e4m3_to_float(codes) * float(np.float32(scale))


def kv_cache_write_fp8(k_cache, v_cache, k_new, v_new, slot_mapping, block_size, k_scale, v_scale):
    """In place: token t's K codes go to k_cache[slot // B, :, slot % B, :] and
    its V codes to v_cache[slot // B, :, :, slot % B].

    k_cache: uint8 [num_blocks, Hkv, B, D]; v_cache: uint8 [num_blocks, Hkv, D, B];
    k_new, v_new: [T, Hkv, D] (bf16 values given as float32).  A negative slot
    writes nothing.
    """
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        k_cache[blk, :, off, :] = quantize(k_new[t], k_scale)
        v_cache[blk, :, :, off] = quantize(v_new[t], v_scale)
