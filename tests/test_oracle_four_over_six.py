"""Pins of the oracle's four-over-six quantizer ('The 4-bitter Lesson',
Four-Over-Six for RL Weights and Activations): hand-worked blocks, the
pages' 1/6-versus-1/8 closed form, the definition restated by brute force in
fp64 on random rows, and invariants (power-of-two scaling, negation,
per-tensor mode, scale range)."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def unpack(codes, cols):
    out = np.empty((codes.shape[0], cols), np.uint8)
    out[:, 0::2] = codes & 15
    out[:, 1::2] = codes >> 4
    return out


def _cases():
    with open(os.path.join(GOLDEN, "four_over_six_blocks.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("err", ["mse", "mae"])
@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_worked_blocks(case, err):
    x = workloads.to_bf16_bits(np.array([case["row"]], np.float32))
    assert np.array_equal(workloads.bf16_bits_to_f32(x)[0], np.array(case["row"], np.float32))
    codes, sf, scale, choice = oracle.quantize_46(x, err, with_choice=True)
    want = case[err]
    assert unpack(codes, x.shape[1])[0].tolist() == want["codes"]
    assert sf[0].tolist() == want["sf"]
    assert choice[0].tolist() == want["choice"]
    assert int(scale.view(np.uint32)[0]) == case["s_g_bits"]


def test_pages_closed_form_on_decoded_values():
    """A value at 5/6 of the block max is off by 1/6 of the max when the max maps
    to 6 and by at most 1/8 when it maps to 4; four-over-six keeps the latter."""
    x = workloads.to_bf16_bits(np.array([[1.5] + [1.25] * 15], np.float32))
    c6 = oracle.dequantize(*oracle.quantize(x))  # plain rule: max -> 6
    c46 = oracle.dequantize(*oracle.quantize_46(x, "mse"))
    assert abs(c6[0, 1] - 1.25) == pytest.approx(1.5 / 6, rel=1e-2)
    assert abs(c46[0, 1] - 1.25) <= 1.5 / 8


def _nearest_code(v):
    """E2M1 code of v by definition: nearest grid value, ties to the even code, |v| > 6 -> 6."""
    a = abs(v)
    d = np.abs(GRID - a)
    best = min(range(8), key=lambda i: (d[i], i % 2))
    if a > 6.0:
        best = 7
    return (8 if np.signbit(v) else 0) | best


def _candidate(xb, s_g, c):
    """Max -> c candidate of one block in fp64 from the definition: the block
    scale by the (pinned) E4M3 encoder of fp32 u = bmax / (c s_g), then codes of
    the exact quotients x / (s_b s_g); error sum in units of s_g."""
    t = np.float32(np.float32(c) * s_g)
    u = np.float32(np.float32(np.abs(xb).max()) / t)
    sb = oracle.e4m3_encode(float(u))
    sbv = oracle.e4m3_decode(sb)
    if sb == 0:
        codes = [0] * 16
        near_tie = False
    else:
        d = sbv * float(s_g)
        v = xb.astype(np.float64) / d
        codes = [_nearest_code(vi) for vi in v]
        ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
        near_tie = bool(np.any(np.abs(np.abs(v)[:, None] - ties[None, :]) < 1e-5))
    dq = np.array([oracle.e2m1_decode(q) for q in codes]) * sbv
    diff = dq - xb.astype(np.float64) / float(s_g)
    return sb, codes, float((diff ** 2).sum()), float(np.abs(diff).sum()), near_tie


@pytest.mark.parametrize("err", ["mse", "mae"])
def test_brute_force_definition_on_random_rows(err):
    rng = np.random.default_rng(46)
    x = workloads.gaussian_bf16(rng, (48, 256), outlier_frac=0.03, outlier_mult=20.0)
    xf = workloads.bf16_bits_to_f32(x)
    codes, sf, scale, choice = oracle.quantize_46(x, err, with_choice=True)
    cu = unpack(codes, 256)
    checked = skipped = fours = 0
    for r in range(x.shape[0]):
        s_g = np.float32(np.float32(np.abs(xf[r]).max()) / np.float32(1536.0))
        assert scale[r] == s_g
        for b in range(16):
            xb = xf[r, b * 16:(b + 1) * 16]
            sb6, q6, mse6, mae6, tie6 = _candidate(xb, s_g, 6)
            sb4, q4, mse4, mae4, tie4 = _candidate(xb, s_g, 4)
            e6, e4 = (mse6, mse4) if err == "mse" else (mae6, mae4)
            if tie6 or tie4 or abs(e4 - e6) <= 1e-5 * max(e4, e6):
                skipped += 1  # fp32 rounding of v or of the error sums can decide these
                continue
            want = 4 if e4 < e6 else 6
            assert choice[r, b] == want, (r, b, e4, e6)
            assert sf[r, b] == (sb4 if want == 4 else sb6)
            assert cu[r, b * 16:(b + 1) * 16].tolist() == (q4 if want == 4 else q6)
            checked += 1
            fours += want == 4
    assert skipped < 0.05 * (checked + skipped)
    assert 0 < fours < checked  # both outcomes occur


def test_invariants_scaling_negation_per_tensor_scale_range():
    rng = np.random.default_rng(7)
    x = workloads.gaussian_bf16(rng, (32, 128), outlier_frac=0.02)
    base = oracle.quantize_46(x, "mse", with_choice=True)
    # every block scale within E4M3 without saturation: s_b <= 384 (0x7C)
    assert base[1].max() <= 0x7C
    # power-of-two scaling of the row: same codes, scales and choices; s_g scaled exactly
    for k in (-3, 5):
        xs = workloads.to_bf16_bits(workloads.bf16_bits_to_f32(x) * np.float32(2.0 ** k))
        sc = oracle.quantize_46(xs, "mse", with_choice=True)
        assert np.array_equal(sc[0], base[0]) and np.array_equal(sc[1], base[1]) and np.array_equal(sc[3], base[3])
        assert np.array_equal(sc[2], base[2] * np.float32(2.0 ** k))
    # negation flips only the sign bits (zeros included: the sign of zero is kept)
    neg = oracle.quantize_46(x ^ np.uint16(0x8000), "mse", with_choice=True)
    assert np.array_equal(neg[0], base[0] ^ np.uint8(0x88))
    assert np.array_equal(neg[1], base[1]) and np.array_equal(neg[3], base[3])
    # per-tensor mode = per-row mode fed the tensor amax
    amax = np.float32(np.abs(workloads.bf16_bits_to_f32(x)).max())
    pt = oracle.quantize_46(x, "mae", per_tensor=True)
    pr = oracle.quantize_46(x, "mae", amax_in=np.full(x.shape[0], amax, np.float32))
    assert np.array_equal(pt[0], pr[0]) and np.array_equal(pt[1], pr[1]) and pt[2][0] == pr[2][0]


def test_never_worse_than_max_to_six_in_fp64():
    """Per block, the chosen encoding's fp64 squared error is no larger than the
    max -> 6 candidate's (up to the fp32 accumulation of the decision)."""
    rng = np.random.default_rng(11)
    x = workloads.gaussian_bf16(rng, (16, 512), outlier_frac=0.05, outlier_mult=30.0)
    xf = workloads.bf16_bits_to_f32(x).astype(np.float64)
    codes, sf, scale = oracle.quantize_46(x, "mse")
    deq = oracle.dequantize(codes, sf, scale)
    for r in range(x.shape[0]):
        s_g = np.float32(np.float32(np.abs(xf[r]).max()) / np.float32(1536.0))
        for b in range(32):
            xb = xf[r, b * 16:(b + 1) * 16].astype(np.float32)
            _, _, mse6, _, _ = _candidate(xb, s_g, 6)
            got = float((((deq[r, b * 16:(b + 1) * 16] - xf[r, b * 16:(b + 1) * 16]) / float(s_g)) ** 2).sum())
            assert got <= mse6 * (1 + 1e-5) + 1e-9
