"""Shared helpers of the parity tests: moving seeded inputs to the device and
comparing device results with the oracle element by element."""
import numpy as np
import torch

import oracle


def to_dev_bf16(bits):
    """uint16 bf16 bit patterns (numpy) -> CUDA bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def unpack_codes(codes, cols):
    codes = np.asarray(codes, np.uint8)
    out = np.empty(codes.shape[:-1] + (cols,), np.uint8)
    out[..., 0::2] = codes & 15
    out[..., 1::2] = codes >> 4
    return out


def device_sf_linear(sf_dev, rows, cols, row_map=None):
    """Read the valid [rows x cols/16] block scales out of a swizzled device buffer."""
    return oracle.sf_unswizzle(sf_dev.cpu().numpy(), rows, cols // 16, row_map)


def assert_quant_equal(got, ref, rows, cols, row_map=None, what=""):
    """Bit-exact comparison of a device NVFP4Tensor with the oracle's (codes, sf_lin, scale)."""
    codes, sf, scale = ref
    gc = got.codes.cpu().numpy()
    bad = np.nonzero((gc != codes).any(axis=1))[0]
    assert len(bad) == 0, f"{what}: codes differ in {len(bad)} rows, first {bad[:5]}"
    gs = device_sf_linear(got.sf, rows, cols, row_map)
    bad = np.nonzero((gs != sf).any(axis=1))[0]
    assert len(bad) == 0, f"{what}: block scales differ in {len(bad)} rows, first {bad[:5]}"
    gsc = got.scale.cpu().numpy()[:len(scale)]
    assert np.array_equal(gsc.view(np.uint32), scale.view(np.uint32)), f"{what}: outer scales differ"


def gemm_tolerance_check(y_dev_bits, y_exact, abs_sum, what=""):
    """|Y_gpu - Y_oracle| <= ulp_bf16 + 1e-5 * sum_k |a_k b_k| per element, Y_oracle the
    oracle's bf16 rounding of its fp64 result; the ulp is taken at the larger of the
    two magnitudes (a result and its neighbour can sit on two sides of a power of 2)."""
    y_or = oracle.bf16_to_f64(oracle.bf16_round(y_exact))
    y_gpu = oracle.bf16_to_f64(y_dev_bits)
    tol = oracle.bf16_ulp(np.maximum(np.abs(y_gpu), np.abs(y_or))) + 1e-5 * abs_sum
    err = np.abs(y_gpu - y_or)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; first "
                             f"{[(tuple(j), y_gpu[tuple(j)], y_or[tuple(j)], tol[tuple(j)]) for j in i]}")
    return float(err.max()), float((err / np.maximum(tol, 1e-300)).max())
