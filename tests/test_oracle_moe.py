"""Pins for the oracle's layout, routing, GEMM, SwiGLU and combine (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit

import oracle
import workloads
from tests.test_oracle_format import unpack


# ---------------------------------------------------------------- scale-factor layout

def test_sf_layout_hand_offsets():
    # 128x4 tiles of 512 bytes, tile-row-major; inside a tile row r%32 is a
    # 16-byte line, (r%128)/32 picks the 4-byte group, c%4 the byte.
    S = 128  # 2048 columns / 16
    cases = {(0, 0): 0, (0, 1): 1, (0, 3): 3, (1, 0): 16, (31, 0): 496, (32, 0): 4,
             (64, 0): 8, (96, 3): 15, (0, 4): 512, (0, 127): 31 * 512 + 3,
             (127, 127): 31 * 512 + 31 * 16 + 12 + 3, (128, 0): 32 * 512, (200, 5): 32 * 512 + 512 + 8 * 16 + 8 + 1}
    for (r, c), off in cases.items():
        assert oracle.sf_offset(r, c, S) == off, (r, c)
    # 48 scale columns (K = 768): 12 tiles per 128-row band
    assert oracle.sf_offset(128, 0, 48) == 12 * 512
    # 3 scale columns pad to 4
    assert oracle.sf_bytes(5, 3) == 128 * 4
    assert oracle.sf_offset(1, 2, 3) == 18


def test_sf_layout_is_a_bijection_onto_the_padded_buffer():
    for rows, sc in [(130, 8), (128, 48), (7, 3)]:
        rp, sp = (rows + 127) // 128 * 128, (sc + 3) // 4 * 4
        offs = {oracle.sf_offset(r, c, sc) for r in range(rp) for c in range(sp)}
        assert len(offs) == rp * sp and min(offs) == 0 and max(offs) == oracle.sf_bytes(rows, sc) - 1


def test_sf_swizzle_roundtrip_with_row_map():
    rng = np.random.default_rng(0)
    sf = rng.integers(0, 127, (20, 8), dtype=np.uint8)
    rm = np.array([3, 4, 5] + list(range(128, 145)), np.int64)
    sw = oracle.sf_swizzle(sf, rm, 256)
    assert np.array_equal(oracle.sf_unswizzle(sw, 20, 8, rm), sf)
    assert sw[oracle.sf_offset(0, 0, 8)] == 0  # unused rows are zero-padded


# ---------------------------------------------------------------- routing

def test_route_matches_stable_argsort_and_full_softmax():
    d = workloads.moe_layer(2, 512, 1.0, with_weights=False)
    ids, w = oracle.route(d["logits"], d["bias"], 8)
    z = d["logits"] + d["bias"][None, :]           # fp32 add, as in the router
    ref = np.argsort(-z, axis=1, kind="stable")[:, :8]
    assert np.array_equal(ids, ref)
    zf = z.astype(np.float64)
    p = np.exp(zf - zf.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)               # softmax over all 128 experts
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_route_tie_goes_to_lower_expert():
    logits = np.zeros((2, 16), np.float32)
    logits[1, [3, 9, 12]] = 1.0
    ids, w = oracle.route(logits, np.zeros(16, np.float32), 4)
    assert ids[0].tolist() == [0, 1, 2, 3]
    assert ids[1].tolist() == [3, 9, 12, 0]
    np.testing.assert_allclose(w[0], 0.25, rtol=0, atol=1e-15)


def test_route_metadata_invariants():
    d = workloads.moe_layer(3, 700, 2.0, with_weights=False)
    ids, _ = oracle.route(d["logits"], d["bias"], 8)
    m = oracle.route_metadata(ids, 128)
    assert np.array_equal(m["cnt"], np.bincount(ids.reshape(-1), minlength=128))
    assert m["cnt"].sum() == 700 * 8 and m["off"][-1] == 700 * 8
    assert np.array_equal(m["perm"], np.argsort(ids.reshape(-1), kind="stable"))
    assert np.array_equal(m["inv"][m["perm"]], np.arange(700 * 8))
    assert np.all(m["poff"] % 128 == 0)
    gap = np.diff(m["poff"]) - m["cnt"]
    assert np.all((gap >= 0) & (gap < 128))
    assert (m["cnt"] == 0).any()  # bias std 2 leaves some experts empty
    assert m["cnt"].max() > 5 * m["cnt"].mean()


# ---------------------------------------------------------------- GEMM

def _exact_gemm(codes_a, sf_a, s_a, codes_b, sf_b, s_b, K):
    qa = unpack(codes_a, K)
    qb = unpack(codes_b, K)
    grid = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]

    def val(q):
        return -grid[q & 7] if q & 8 else grid[q & 7]

    def e4(b):
        return Fraction(oracle.e4m3_decode(int(b)))

    M, N = qa.shape[0], qb.shape[0]
    out = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += val(qa[m, k]) * e4(sf_a[m, k // 16]) * val(qb[n, k]) * e4(sf_b[n, k // 16])
            out[m][n] = acc * Fraction(float(s_a[m])) * Fraction(float(s_b[0]))
    return out


@pytest.mark.parametrize("M,N,K", [(3, 5, 64), (17, 33, 128)])
def test_gemm_against_exact_rational_sum(M, N, K):
    rng = np.random.default_rng(M * N)
    x = workloads.gaussian_bf16(rng, (M, K), outlier_frac=0.05)
    w = workloads.gaussian_bf16(rng, (N, K), std=0.02)
    xq = oracle.quantize(x)
    wq = oracle.quantize(w, per_tensor=True)
    y = oracle.gemm_f64(oracle.dequantize(*xq), oracle.dequantize(*wq, per_tensor=True))
    ex = _exact_gemm(*xq, *wq, K)
    yb = oracle.linear(xq, wq)
    for m in range(M):
        for n in range(N):
            e = ex[m][n]
            assert abs(Fraction(y[m, n]) - e) <= abs(e) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 1000)
            assert yb[m, n] == oracle.bf16_round(np.array([float(e)]))[0]


def test_gemm_one_hot_weights_select_columns():
    """W rows are one-hot (code for 1.0, block scale 1, tensor scale 2^-3):
    Y[m, n] = deq(X)[m, col(n)] / 8 exactly."""
    rng = np.random.default_rng(1)
    M, N, K = 9, 12, 64
    x = workloads.gaussian_bf16(rng, (M, K))
    xq = oracle.quantize(x)
    cols = rng.integers(0, K, N)
    q = np.zeros((N, K), np.uint8)
    q[np.arange(N), cols] = 2                        # E2M1 code of 1.0
    wcodes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    wsf = np.full((N, K // 16), 0x38, np.uint8)      # E4M3 1.0
    wq = (wcodes, wsf, np.array([0.125], np.float32))
    y = oracle.gemm_f64(oracle.dequantize(*xq), oracle.dequantize(*wq, per_tensor=True))
    xd = oracle.dequantize(*xq)
    assert np.array_equal(y, xd[:, cols] / 8.0)


# ---------------------------------------------------------------- SwiGLU / combine

def test_swiglu_matches_expit_closed_form():
    rng = np.random.default_rng(2)
    c = rng.standard_normal((64, 2 * 48)) * 3
    d, amax = oracle.swiglu(c)
    g, u = c[:, :48], c[:, 48:]
    ref = oracle.bf16_round(g * expit(g) * u)
    assert np.array_equal(d, ref)
    assert np.array_equal(amax, np.abs(oracle.bf16_to_f64(d)).max(axis=1).astype(np.float32))
    z, _ = oracle.swiglu(np.zeros((1, 4)))
    assert np.all(z == 0)


def test_combine_special_cases():
    rng = np.random.default_rng(4)
    T, k, H = 6, 3, 16
    y = rng.standard_normal((T * k, H))
    inv = rng.permutation(T * k).astype(np.int32)
    w1 = np.zeros((T, k))
    w1[:, 1] = 1.0
    out = oracle.combine(y, inv, w1)
    assert np.array_equal(out, oracle.bf16_round(y[inv.reshape(T, k)[:, 1]]))
    yc = np.tile(np.full((1, H), 0.75), (T * k, 1))
    wc = np.full((T, k), 1.0 / 3.0)
    assert np.all(oracle.bf16_to_f64(oracle.combine(yc, inv, wc)) == 0.75)


# ---------------------------------------------------------------- MoE composition

def test_moe_forward_matches_per_token_loop():
    """The permuted, grouped formulation equals a direct per-token loop over
    each token's experts (no metadata, no permutation)."""
    T, E, k, H, F = 24, 6, 2, 64, 32
    rng = np.random.default_rng(8)
    x = workloads.gaussian_bf16(rng, (T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = rng.standard_normal(E).astype(np.float32)
    w1 = [oracle.quantize(workloads.gaussian_bf16(rng, (2 * F, H), std=0.02), per_tensor=True) for _ in range(E)]
    w2 = [oracle.quantize(workloads.gaussian_bf16(rng, (H, F), std=0.02), per_tensor=True) for _ in range(E)]
    res = oracle.moe_forward(x, logits, bias, w1, w2, k)
    ids, w = oracle.route(logits, bias, k)
    ref = np.zeros((T, H), np.uint16)
    for t in range(T):
        xq = oracle.quantize(x[t:t + 1])
        acc = np.zeros(H)
        for s in range(k):
            e = ids[t, s]
            c = oracle.gemm_f64(oracle.dequantize(*xq), oracle.dequantize(*w1[e], per_tensor=True))
            dd, am = oracle.swiglu(c)
            q2 = oracle.quantize(dd, amax_in=am)
            y2 = oracle.bf16_to_f64(oracle.bf16_round(
                oracle.gemm_f64(oracle.dequantize(*q2), oracle.dequantize(*w2[e], per_tensor=True))))
            acc += w[t, s] * y2[0]
        ref[t] = oracle.bf16_round(acc)
    assert np.array_equal(res["out"], ref)
    sub = oracle.moe_forward(x, logits, bias, w1, w2, k, rows=[3, 17])
    assert np.array_equal(sub["out"], ref[[3, 17]])
