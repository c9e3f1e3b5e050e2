"""Pins of the oracle's grouped BF16 backward GEMMs (the dequantized
backward: dgrad dx = dy . w_g per row group, wgrad dw_g = dy_g^T . x_g):
exact integer sums on tiny cases, the adjoint identities that tie both to
the forward GEMM, and the grouping rules (empty groups, zero padding rows)."""
import numpy as np

import oracle
import workloads


def _bits(a):
    return workloads.to_bf16_bits(np.asarray(a, np.float32))


def test_exact_integer_sums():
    rng = np.random.default_rng(0)
    poff = [0, 2, 2, 5]  # three groups, the middle one empty
    dy = rng.integers(-7, 8, (5, 3))
    w = rng.integers(-5, 6, (3, 3, 4))
    x = rng.integers(-9, 10, (5, 4))
    dx, _ = oracle.grouped_dgrad(_bits(dy), _bits(w), poff)
    dw, _ = oracle.grouped_wgrad(_bits(dy), _bits(x), poff)
    for g in range(3):
        for r in range(poff[g], poff[g + 1]):
            for k in range(4):
                assert dx[r, k] == sum(int(dy[r, n]) * int(w[g, n, k]) for n in range(3))
        for n in range(3):
            for k in range(4):
                assert dw[g, n, k] == sum(int(dy[r, n]) * int(x[r, k]) for r in range(poff[g], poff[g + 1]))
    assert not dw[1].any()


def test_adjoint_identities_with_the_forward_gemm():
    """For the grouped forward y[r] = x[r] . w_g^T (oracle.gemm_f64), the
    backward must satisfy sum <dy, y> = sum <dgrad(dy), x> = sum_g <wgrad(dy, x)_g, w_g>:
    a transposed operand or a wrong group fails it."""
    rng = np.random.default_rng(1)
    poff = np.array([0, 128, 384, 384, 512])
    rows, nf, kf = 512, 64, 96
    x = workloads.gaussian_bf16(rng, (rows, kf))
    dy = workloads.gaussian_bf16(rng, (rows, nf))
    w = np.stack([workloads.gaussian_bf16(rng, (nf, kf), std=0.02) for _ in range(4)])
    xf, dyf, wf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(dy), oracle.bf16_to_f64(w)
    lhs = 0.0
    for g in range(4):
        lo, hi = poff[g], poff[g + 1]
        lhs += float(np.sum(dyf[lo:hi] * oracle.gemm_f64(xf[lo:hi], wf[g])))
    dx, _ = oracle.grouped_dgrad(dy, w, poff)
    dw, _ = oracle.grouped_wgrad(dy, x, poff)
    assert np.isclose(float(np.sum(dx * xf)), lhs, rtol=1e-12)
    assert np.isclose(float(np.sum(dw * wf)), lhs, rtol=1e-12)


def test_zero_padding_rows_change_nothing():
    rng = np.random.default_rng(2)
    dy = workloads.gaussian_bf16(rng, (10, 32))
    x = workloads.gaussian_bf16(rng, (10, 48))
    w = workloads.gaussian_bf16(rng, (2, 32, 48))
    poff = [0, 4, 10]
    pad_dy = np.zeros((256, 32), np.uint16)
    pad_x = np.zeros((256, 48), np.uint16)
    pad_dy[0:4], pad_dy[128:134] = dy[0:4], dy[4:10]
    pad_x[0:4], pad_x[128:134] = x[0:4], x[4:10]
    ppoff = [0, 128, 256]
    dw, _ = oracle.grouped_wgrad(dy, x, poff)
    dw_p, _ = oracle.grouped_wgrad(pad_dy, pad_x, ppoff)
    assert np.array_equal(dw, dw_p)
    dx, _ = oracle.grouped_dgrad(dy, w, poff)
    dx_p, _ = oracle.grouped_dgrad(pad_dy, w, ppoff)
    assert np.array_equal(dx_p[[0, 1, 2, 3, 128, 129, 130, 131, 132, 133]], dx)
    assert not np.delete(dx_p, [0, 1, 2, 3, 128, 129, 130, 131, 132, 133], axis=0).any()
