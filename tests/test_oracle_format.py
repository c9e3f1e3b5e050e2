"""Pins for the oracle's number formats and per-token quantizer (CPU only).

Each test checks the oracle against something other than itself: values
worked by hand from the pages (tests/golden/worked_blocks.json), a library
conversion (torch's float8_e4m3fn and bf16 casts), exact rational
arithmetic, or invariants that hold for any correct implementation.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # "The 4-bitter Lesson", Four-Over-Six


def unpack(codes, cols):
    codes = np.asarray(codes, np.uint8)
    out = np.empty(codes.shape[:-1] + (cols,), np.uint8)
    out[..., 0::2] = codes & 15
    out[..., 1::2] = codes >> 4
    return out


def test_e2m1_decode_matches_grid():
    for c in range(16):
        v = E2M1_GRID[c & 7]
        assert oracle.e2m1_decode(c) == (-v if c & 8 else v)


def test_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert np.isnan(got)
        else:
            assert got == ref[c], c
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne_below_saturation():
    rng = np.random.default_rng(7)
    u = np.concatenate([
        rng.uniform(0, 448, 20000).astype(np.float32),
        np.exp2(rng.uniform(-14, 8.8, 20000)).astype(np.float32),
        # every midpoint between consecutive finite E4M3 values (exact ties)
        np.array([(oracle.e4m3_decode(c) + oracle.e4m3_decode(c + 1)) / 2 for c in range(0, 126)],
                 np.float32),
    ])
    u = u[u <= 448]
    ref = torch.from_numpy(u).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(x) for x in u], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates():
    for u in [448.0, 449.0, 463.9, 464.0, 500.0, 1e30]:
        assert oracle.e4m3_encode(u) == 0x7E


def test_e2m1_encode_is_nearest_with_even_ties():
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(-8, 8, 50000), [0.25 * i for i in range(-30, 31)]]).astype(np.float32)
    for v in vals:
        c = oracle.e2m1_encode(v)
        q = oracle.e2m1_decode(c)
        a = abs(float(v))
        dists = [abs(a - g) for g in E2M1_GRID]
        best = min(dists)
        if a > 6:
            assert c & 7 == 7
        else:
            assert abs(abs(q) - a) == best
            ties = [i for i, d in enumerate(dists) if d == best]
            if len(ties) == 2:
                assert (c & 7) % 2 == 0
        assert (c >> 3) == (1 if np.signbit(v) else 0)


def test_bf16_round_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(1e3),
        np.exp2(rng.uniform(-140, 127, 100000)).astype(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, ref)


def _bf16_exact_nearest(xf):
    """Round a Fraction to bf16 by brute force over the two neighbours."""
    lo = np.float32(float(xf))
    cands = set()
    b = np.array([lo], np.float32).view(np.uint32)[0] >> 16
    for d in (-2, -1, 0, 1, 2):
        h = (int(b) + d) & 0xFFFF
        cands.add(h)
    best = None
    for h in cands:
        v = float((np.array([h << 16], np.uint32)).view(np.float32)[0])
        if not np.isfinite(v):
            continue
        dist = abs(Fraction(v) - xf)
        key = (dist, h & 1)
        if best is None or key < best[0]:
            best = (key, h)
    return best[1]


def test_bf16_round_is_exact_rne_on_fp64_inputs():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, 3000))
    got = oracle.bf16_round(x)
    for xi, g in zip(x, got):
        assert g == _bf16_exact_nearest(Fraction(float(xi))), xi


def _golden_cases():
    with open(os.path.join(GOLDEN, "worked_blocks.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_worked_blocks(case):
    if "row_bits" in case:
        x = np.array([case["row_bits"]], np.uint16)
    else:
        x = workloads.to_bf16_bits(np.array([case["row"]], np.float32))
        assert np.array_equal(workloads.bf16_bits_to_f32(x)[0], np.array(case["row"], np.float32))
    amax = None if "amax_in" not in case else np.array([case["amax_in"]], np.float32)
    codes, sf, scale = oracle.quantize(x, amax_in=amax)
    assert unpack(codes, x.shape[1])[0].tolist() == case["codes"]
    assert sf[0].tolist() == case["sf"]
    if "s_g_bits" in case:
        assert scale.view(np.uint32)[0] == case["s_g_bits"]
    else:
        assert scale[0] == np.float32(case["s_g"])


def test_brute_force_every_bf16_value_in_a_fixed_block():
    """With s_g = 2^-4 and s_b = 1 (d = 2^-4, 1/d exact), every bf16 value
    x with |x| <= 0.375 must encode to the grid value nearest to 16 x (ties
    to the even code), for all 65536 bit patterns that qualify."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = workloads.bf16_bits_to_f32(bits)
    keep = np.isfinite(vals) & (np.abs(vals) <= 0.375)
    bits = bits[keep]
    n = len(bits)
    per_row = 15
    rows = (n + per_row - 1) // per_row
    x = np.zeros((rows, 32), np.uint16)
    x[:, 0] = workloads.to_bf16_bits(np.array([168.0], np.float32))[0]   # s_g = 2^-4
    x[:, 16] = workloads.to_bf16_bits(np.array([0.375], np.float32))[0]  # block max: s_b = 1
    flat = np.zeros(rows * per_row, np.uint16)
    flat[:n] = bits
    x[:, 17:32] = flat.reshape(rows, per_row)
    codes, sf, scale = oracle.quantize(x)
    assert np.all(scale == np.float32(0.0625))
    assert np.all(sf[:, 1] == 0x38)
    q = unpack(codes, 32)[:, 17:32].reshape(-1)[:n]
    v = workloads.bf16_bits_to_f32(bits).astype(np.float64) * 16.0
    grid = np.array(E2M1_GRID)
    d = np.abs(np.abs(v)[:, None] - grid[None, :])
    best = d.min(axis=1)
    mag = q & 7
    assert np.all(d[np.arange(n), mag] == best)
    tie = (d == best[:, None]).sum(axis=1) == 2
    assert np.all(mag[tie] % 2 == 0)
    assert np.all((q >> 3) == np.signbit(workloads.bf16_bits_to_f32(bits)))


def _half_step(qmag):
    # intervals of v mapped to each magnitude index: idx 0..3 -> within 0.25,
    # idx 4 (2) and 5 (3) -> within 0.5, idx 6 (4) and 7 (6, incl. saturation) -> within 1
    return np.where(qmag <= 3, 0.25, np.where(qmag <= 5, 0.5, 1.0))


def test_error_bound_and_max_element_invariants():
    x = workloads.quant_rows(seed=1, rows=512, cols=2048)["x"]
    codes, sf, scale = oracle.quantize(x)
    xf = workloads.bf16_bits_to_f32(x).astype(np.float64)
    xhat = oracle.dequantize(codes, sf, scale)
    q = unpack(codes, 2048)
    sb = np.vectorize(oracle.e4m3_decode)(sf).astype(np.float64)
    d = np.repeat(sb, 16, axis=1) * scale.astype(np.float64)[:, None]
    normal = np.repeat(sb >= 2.0 ** -6, 16, axis=1) & (d >= 2.0 ** -126)
    bound = _half_step(q & 7) * d * (1 + 2.0 ** -20)
    err = np.abs(xf - xhat)
    assert np.all(err[normal] <= bound[normal])
    nz = np.abs(xf).max(axis=1) > 0
    assert (~nz).sum() > 0  # the workload has zero rows
    jmax = np.abs(xf).argmax(axis=1)
    r = np.nonzero(nz)[0]
    assert np.all(q[r, jmax[r]] & 7 == 7)
    assert np.all(sf[r, jmax[r] // 16] == 0x7E)
    assert np.all(codes[~nz] == 0) and np.all(sf[~nz] == 0) and np.all(scale[~nz] == 0)
    m = oracle.error_metrics(xf[nz], xhat[nz])
    assert 0.05 < m["rel_l2"] < 0.2 and m["snr_db"] > 15


def test_power_of_two_scaling_and_negation():
    x = workloads.quant_rows(seed=9, rows=64, cols=256)["x"]
    xf = workloads.bf16_bits_to_f32(x)
    c0, s0, g0 = oracle.quantize(x)
    for j in (-3, 5):
        c1, s1, g1 = oracle.quantize(workloads.to_bf16_bits(xf * np.float32(2.0 ** j)))
        assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
        assert np.array_equal(g1, g0 * np.float32(2.0 ** j))
    cn, sn, gn = oracle.quantize(workloads.to_bf16_bits(-xf))
    assert np.array_equal(s0, sn) and np.array_equal(g0, gn)
    q0, qn = unpack(c0, 256), unpack(cn, 256)
    live = np.repeat(s0 > 0, 16, axis=1)
    assert np.array_equal(q0[live] ^ 8, qn[live])
    assert np.all(qn[~live] == 0)


def test_context_swap_per_token_is_independent_per_tensor_is_not():
    """'miniTE Technical Report' 2.3 / 6.2.1: a row's per-token result does
    not depend on the other rows; the per-tensor scale does."""
    base = workloads.quant_rows(seed=4, rows=32, cols=512)["x"]
    target = base[5:6]
    ct, st, gt = oracle.quantize(target)
    loud = workloads.to_bf16_bits(workloads.bf16_bits_to_f32(base) * np.float32(40.0))
    contexts = [base, loud, np.concatenate([loud[:3], target, base[:7]])]
    changed = 0
    for ctx in contexts:
        rows = np.concatenate([ctx[:11], target, ctx[11:]])
        c, s, g = oracle.quantize(rows)
        assert np.array_equal(c[11], ct[0]) and np.array_equal(s[11], st[0]) and g[11] == gt[0]
        cp, sp, gp = oracle.quantize(rows, per_tensor=True)
        cpt, spt, gpt = oracle.quantize(target, per_tensor=True)
        if not (np.array_equal(cp[11], cpt[0]) and np.array_equal(sp[11], spt[0])):
            changed += 1
    assert changed >= 2


def test_per_tensor_equals_per_row_with_tensor_amax():
    x = workloads.quant_rows(seed=6, rows=48, cols=256)["x"]
    cp, sp, gp = oracle.quantize(x, per_tensor=True)
    amax = np.abs(workloads.bf16_bits_to_f32(x)).max()
    cr, sr, gr = oracle.quantize(x, amax_in=np.full(48, amax, np.float32))
    assert np.array_equal(cp, cr) and np.array_equal(sp, sr)
    assert np.all(gr == gp[0]) and gp[0] == np.float32(amax) / np.float32(2688)


def test_four_over_six_closed_form():
    """'The 4-bitter Lesson': a value at 5/6 of the range has error 1/6 of the
    range on the 0..6 grid; mapping the maximum to 4 gives at most 1/8."""
    assert abs(oracle.e2m1_decode(oracle.e2m1_encode(5.0)) - 5.0) == 1.0
    worst4 = max(abs(oracle.e2m1_decode(oracle.e2m1_encode(v)) - v) for v in np.linspace(0, 4, 4001))
    assert worst4 == 0.5  # 1/8 of the range 4


def test_dequantize_hand_values():
    codes = np.array([[0x72, 0xF1]], np.uint8)  # elements: 1.0, 6, 0.5, -6
    sf = np.array([[0x38]], np.uint8)           # 1.0
    scale = np.array([0.5], np.float32)
    codes16 = np.zeros((1, 8), np.uint8)
    codes16[0, :2] = codes[0]
    out = oracle.dequantize(codes16, sf, scale)
    assert out[0, :4].tolist() == [0.5, 3.0, 0.25, -3.0]


def test_bf16_ulp_is_the_gap_to_the_next_bf16_value():
    """oracle.bf16_ulp, the unit of every bf16 tolerance, against the spacing
    read off consecutive bf16 bit patterns: for every non-negative finite
    pattern, the distance to the next pattern's value (the largest finite
    value takes the gap below it), at the value itself, at points strictly
    inside the gap, and for the negated value."""
    b = np.arange(0, 0x7F80, dtype=np.uint32)  # +0 .. largest finite, as bit patterns
    v = (b << 16).view(np.float32).astype(np.float64)
    nxt = ((b + 1) << 16).view(np.float32).astype(np.float64)  # 0x7F80 is +inf
    gap = nxt - v
    gap[-1] = v[-1] - v[-2]
    assert np.array_equal(oracle.bf16_ulp(v), gap)
    assert np.array_equal(oracle.bf16_ulp(-v), gap)
    inside = v[:-1] + gap[:-1] * 0.75  # strictly between two neighbours (exact in fp64)
    assert np.all((inside > v[:-1]) & (inside < nxt[:-1]))
    assert np.array_equal(oracle.bf16_ulp(inside), gap[:-1])
    # the smallest subnormal spacing holds from zero through the top of the subnormal range
    assert oracle.bf16_ulp(0.0) == 2.0 ** -133 and oracle.bf16_ulp(2.0 ** -126) == 2.0 ** -133
    assert oracle.bf16_ulp(1.0) == 2.0 ** -7 and oracle.bf16_ulp(np.nextafter(2.0, 0.0)) == 2.0 ** -7


def test_error_metrics_closed_forms():
    """rel-L2, SNR (dB) and MAE of a reconstruction ("miniTE Technical Report"
    2.3) on vectors whose values are known in closed form."""
    x = np.array([3.0, 4.0, 0.0, 0.0])
    m = oracle.error_metrics(x, x + np.array([0.0, 0.0, 0.5, -0.5]))
    assert np.isclose(m["rel_l2"], np.sqrt(0.5) / 5.0)
    assert np.isclose(m["snr_db"], 20 * np.log10(5.0 / np.sqrt(0.5)))
    assert np.isclose(m["mae"], 0.25)
    assert oracle.error_metrics(x, x)["snr_db"] == np.inf
