"""Pins of the oracle's DQ(Q(x)) (bf16 of the exact dequantized value): the
expected bits come from exact rational arithmetic written here from the
definitions (E2M1 grid, E4M3 fields, round to nearest even on the bf16 grid),
not from the oracle.  The cases include exact grid values, bf16 ties, values
just past a tie, products whose fp32 rounding lands on a bf16 midpoint that
the exact value is not on, and bf16 subnormals."""
from fractions import Fraction

import numpy as np
import pytest

import nvfp4_quantized_moe_token_gb300 as nv
import oracle

E2M1 = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def e2m1_value(code):
    v = E2M1[code & 7]
    return -v if code & 8 else v


def e4m3_value(byte):
    e, m = (byte >> 3) & 15, byte & 7
    if e == 0:
        return Fraction(m, 8) * Fraction(1, 2 ** 6)
    return (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def f32_value(x):
    return Fraction(float(np.float32(x)))


def rne_bf16_bits(x, neg=None):
    """Round an exact rational to bf16 (8 significant bits, exponent >= -126,
    subnormal spacing 2^-133), ties to even; returns the 16-bit pattern.  neg
    gives the sign where x is zero (a rational has no -0)."""
    neg = (x < 0) if neg is None else neg
    a = -x if x < 0 else x
    if a == 0:
        return 0x8000 if neg else 0
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    spacing = Fraction(2) ** (e - 7)
    n = a / spacing
    lo = n.numerator // n.denominator
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    val = float(lo * spacing)
    bits = int(np.array([val], np.float32).view(np.uint32)[0]) >> 16
    return bits | (0x8000 if neg else 0)


def run(code_rows, sbyte_rows, sg):
    """codes [rows, 16] (one block per row), block scale byte per row, s_g per row."""
    code_rows = np.asarray(code_rows, np.uint8)
    packed = (code_rows[:, 0::2] | (code_rows[:, 1::2] << 4)).astype(np.uint8)
    sf = np.asarray(sbyte_rows, np.uint8).reshape(-1, 1)
    scale = np.asarray(sg, np.float32)
    return oracle.dequantize_bf16(packed, sf, scale)


def expected(code_rows, sbyte_rows, sg):
    out = np.empty(np.asarray(code_rows).shape, np.uint16)
    for r, (codes, sb, s) in enumerate(zip(code_rows, sbyte_rows, sg)):
        for j, c in enumerate(codes):
            # the sign of the code is the sign of the product (s_b, s_g >= 0), zero included
            out[r, j] = rne_bf16_bits(e2m1_value(int(c)) * e4m3_value(int(sb)) * f32_value(s), neg=bool(int(c) & 8))
    return out


def test_dq_grid_values_exact():
    codes = [list(range(16))]
    got = run(codes, [0x38], [1.0])  # s_b = 1.0
    want = [0x0000, 0x3F00, 0x3F80, 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0,
            0x8000, 0xBF00, 0xBF80, 0xBFC0, 0xC000, 0xC040, 0xC080, 0xC0C0]
    assert got[0].tolist() == want
    assert np.array_equal(got, expected(codes, [0x38], [1.0]))


def test_dq_ties_and_past_ties():
    one = np.float32(1.0)
    sg = [one + np.float32(2.0 ** -8),                                  # 1 + 2^-8: exact tie -> even (1.0)
          np.float32(1.0 + 2.0 ** -8 + 2.0 ** -23),                      # just past the tie -> up
          np.float32(1.0 + 2.0 ** -8 - 2.0 ** -23),                      # just short -> down
          np.float32((1.0 + 2.0 ** -8) / 3.0)]                           # 3 s_g rounds in fp32 onto the tie
    codes = [[2] * 16, [2] * 16, [2] * 16, [5] * 16]                     # q = 1, 1, 1, 3
    got = run(codes, [0x38] * 4, sg)
    want = expected(codes, [0x38] * 4, sg)
    assert np.array_equal(got, want)
    assert got[0, 0] == 0x3F80 and got[1, 0] == 0x3F81 and got[2, 0] == 0x3F80
    # the last row: fp32 rounding of 3 s_g gives exactly the midpoint 1 + 2^-8; the exact
    # product is off it, so a second rounding from fp32 would pick the wrong neighbour
    p32 = np.float32(3.0) * np.float32(sg[3])
    assert float(p32) == 1.0 + 2.0 ** -8
    exact = 3 * f32_value(sg[3])
    assert exact != Fraction(257, 256)
    assert got[3, 0] == (0x3F81 if exact > Fraction(257, 256) else 0x3F80)


def test_dq_subnormal_products():
    sg = [np.float32(2.0 ** -133), np.float32(2.0 ** -120), np.float32(3.0 * 2.0 ** -140), np.float32(2.0 ** -149)]
    codes = [[1, 3, 2, 9, 11, 7, 15, 0] * 2] * 4
    sbytes = [0x4A, 0x01, 0x38, 0x7E]    # 5.0, 2^-9, 1.0, 448
    got = run(codes, sbytes, sg)
    want = expected(codes, sbytes, sg)
    assert np.array_equal(got, want)
    # 0.5 * 5 * 2^-133 = 2.5 * 2^-133: a tie on the subnormal grid -> 2 * 2^-133
    assert got[0, 0] == 0x0002
    # 1.5 * 5 * 2^-133 = 7.5 * 2^-133 -> 8 * 2^-133
    assert got[0, 1] == 0x0008


def test_dq_random_blocks_match_rational_rounding():
    rng = np.random.default_rng(11)
    rows = 64
    codes = rng.integers(0, 16, size=(rows, 16))
    sbytes = rng.integers(0, 0x7F, size=rows)
    sg = (2.0 ** rng.uniform(-140, 10, size=rows) * rng.uniform(1, 2, size=rows)).astype(np.float32)
    assert np.array_equal(run(codes, sbytes, sg), expected(codes, sbytes, sg))


def test_dequantize_rejects_bad_arguments_without_gpu():
    """Argument checks run on the host, before anything touches a device."""
    L = nv.lib()
    import ctypes
    t = nv._Tensor(0, 0, 0, 4, 32)
    assert L.nvfp4_dequantize_rows(ctypes.byref(t), 0, None, None, 0, None, 32, None) == -1  # null buffers
    t = nv._Tensor(16, 16, 16, 4, 24)
    assert L.nvfp4_dequantize_rows(ctypes.byref(t), 0, None, None, 0, 16, 32, None) == -2  # cols % 16
    t = nv._Tensor(16, 16, 16, 4, 32)
    assert L.nvfp4_dequantize_rows(ctypes.byref(t), 0, None, None, 0, 16, 30, None) == -3  # ldy % 8
    assert L.nvfp4_dequantize_rows(ctypes.byref(t), 0, 16, None, 4, 16, 32, None) == -1  # one offset array
    assert L.nvfp4_dequantize_rows(ctypes.byref(t), 0, 16, 16, 0, 16, 32, None) == -2  # groups
    assert L.nvfp4_dequantize_rows(ctypes.byref(t), 64, None, None, 0, 16, 32, None) == -1  # scale mode
