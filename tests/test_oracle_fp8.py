"""Pins for the FP8 (E4M3) part of the oracle.

The pages fix no 8-bit format, so the pins come from the format's own
definition (landmark values of the OCP E4M3 encoding), from an independent
library routine (PyTorch's float8_e4m3fn conversions, which round to nearest
even and are exact on decode) and from properties every correct rounding has
(round trip of each code, ties to even, the half-spacing error bound).  A
swapped field, a wrong bias, a missed subnormal, a tie rounded the wrong way
or a transposed V block fails one of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle import fp8_e4m3 as f8

FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_landmark_values():
    assert f8.e4m3_value(0x7E) == 448.0
    assert f8.e4m3_value(0xFE) == -448.0
    assert f8.e4m3_value(0x38) == 1.0
    assert f8.e4m3_value(0x01) == 2.0 ** -9       # smallest subnormal
    assert f8.e4m3_value(0x07) == 7 * 2.0 ** -9   # largest subnormal
    assert f8.e4m3_value(0x08) == 2.0 ** -6       # smallest normal
    assert f8.e4m3_value(0x40) == 2.0
    assert f8.e4m3_value(0x3F) == 1.875
    assert f8.e4m3_value(0x00) == 0.0 and not math.copysign(1.0, f8.e4m3_value(0x00)) < 0
    assert f8.e4m3_value(0x80) == 0.0 and math.copysign(1.0, f8.e4m3_value(0x80)) < 0
    assert math.isnan(f8.e4m3_value(0x7F)) and math.isnan(f8.e4m3_value(0xFF))
    assert len(FINITE) == 254
    vals = [f8.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))  # code order is value order


def test_decode_table_matches_library():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = f8.e4m3_to_float(np.arange(256))
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(ours)
    assert np.array_equal(lib[ok], ours[ok])
    assert np.array_equal(np.signbit(lib[ok]), np.signbit(ours[ok]))


def test_every_code_round_trips():
    vals = np.array([f8.e4m3_value(c) for c in FINITE], dtype=np.float32)
    assert f8.float_to_e4m3(vals).tolist() == FINITE


def test_ties_go_to_the_even_code():
    cases = {
        1.0625: 0x38,            # between 1.0 (0x38) and 1.125 (0x39)
        1.1875: 0x3A,            # between 1.125 (0x39) and 1.25 (0x3A)
        2.0 ** -10: 0x00,        # between 0 and the smallest subnormal
        1.5 * 2.0 ** -9: 0x02,   # between subnormals 1 and 2
        7.5 * 2.0 ** -9: 0x08,   # between the largest subnormal and the smallest normal
        -1.0625: 0xB8,
        432.0: 0x7E,             # between 416 (0x7D) and 448 (0x7E)
        3.5 * 2.0 ** -9: 0x04,
    }
    got = f8.float_to_e4m3(np.array(list(cases), dtype=np.float32)).tolist()
    assert got == list(cases.values())


def test_saturation_and_specials():
    x = np.array([448.0, 449.0, 464.0, 1e30, np.inf, -np.inf, -500.0, np.nan, 0.0, -0.0, -1e-30],
                 dtype=np.float32)
    assert f8.float_to_e4m3(x).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F,
                                             0x00, 0x80, 0x80]


def test_rounding_matches_library_inside_the_range():
    rng = np.random.default_rng(5)
    parts = [
        rng.standard_normal(20000) * 40.0,
        rng.uniform(-448.0, 448.0, 5000),
        rng.standard_normal(5000) * 2.0 ** -8,          # subnormal region
        np.ldexp(rng.integers(1, 16, 4000) * 0.5, rng.integers(-12, 8, 4000)),  # near midpoints
    ]
    x = np.concatenate(parts).astype(np.float32)
    x = x[np.abs(x) < 448.0]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(f8.float_to_e4m3(x), lib)


def test_quantization_error_within_half_a_spacing():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(50000).astype(np.float32)
    for scale in (1.0, 1.0 / 64, 0.0137):
        q = np.divide(x, np.float32(scale), dtype=np.float32).astype(np.float64)
        back = f8.e4m3_to_float(f8.quantize(x, scale))
        inside = np.abs(q) <= 448.0
        # spacing of E4M3 at |q|: 2**(e - 3) for normals, 2**-9 for subnormals
        e = np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6)))
        half = np.ldexp(1.0, (e - 4).astype(int))
        assert np.all(np.abs(back - q)[inside] <= half[inside])
        assert np.all(np.abs(back[~inside]) == 448.0)


def test_quantize_divides_in_float32():
    # 1/3 is not a float32: the quotient is rounded to float32 before E4M3
    x = np.array([1.0], dtype=np.float32)
    s = np.float32(3.0)
    q32 = np.float32(x[0] / s)
    assert f8.quantize(x, 3.0).tolist() == f8.float_to_e4m3(np.array([q32])).tolist()
    # by hand: 1/3 = 1.333 * 2**-2 -> exponent field 5, mantissa nearest 3/8 (1.375) -> 0x2B
    assert f8.quantize(x, 3.0).tolist() == [0x2B]
    assert f8.dequantize(f8.quantize(x, 3.0), 3.0)[0] == 0.34375 * 3.0


def test_cache_write_layout_k_rows_v_columns():
    B, Hkv, D, NB = 16, 2, 8, 4
    kc = np.zeros((NB, Hkv, B, D), dtype=np.uint8)
    vc = np.zeros((NB, Hkv, D, B), dtype=np.uint8)
    rng = np.random.default_rng(7)
    k = rng.standard_normal((3, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((3, Hkv, D)).astype(np.float32)
    slots = [2 * B + 5, -1, 3 * B + 15]
    f8.kv_cache_write_fp8(kc, vc, k, v, slots, B, 0.5, 0.25)
    for t, slot in ((0, slots[0]), (2, slots[2])):
        blk, off = divmod(slot, B)
        for h in range(Hkv):
            for d in range(D):
                assert kc[blk, h, off, d] == f8.float_to_e4m3(np.float32(k[t, h, d] / np.float32(0.5)))
                assert vc[blk, h, d, off] == f8.float_to_e4m3(np.float32(v[t, h, d] / np.float32(0.25)))
    # nothing else was written (token 1 had a padding slot)
    assert np.count_nonzero(kc) <= 2 * Hkv * D and np.count_nonzero(vc) <= 2 * Hkv * D
    kc2 = kc.copy()
    kc2[2, :, 5, :] = 0
    kc2[3, :, 15, :] = 0
    assert not kc2.any()


def test_attention_over_dequantized_cache_is_exact_for_representable_values():
    # values already on the scaled E4M3 grid survive the round trip unchanged,
    # so attention over the quantised cache equals attention over the inputs
    import oracle
    rng = np.random.default_rng(8)
    scale = 0.125
    codes = rng.choice(np.array(FINITE[:0x7E]), size=(5, 1, 16))
    k = f8.dequantize(codes, scale)
    assert np.array_equal(f8.dequantize(f8.quantize(k.astype(np.float32), scale), scale), k)
    q = rng.standard_normal((1, 2, 16))
    a = oracle.decode_attention(q, [k], [k], 0.25)
    b = oracle.decode_attention(q, [f8.dequantize(f8.quantize(k.astype(np.float32), scale), scale)],
                                [k], 0.25)
    assert np.array_equal(a, b)
