"""Parity of the dense W4A4 linear (tcgen05 block-scaled GEMM) with the
oracle: quantized operands bit-exact, outputs within 1 bf16 ulp +
1e-5 * sum_k |a_k b_k| per element."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import oracle
import workloads
from tests.helpers import assert_quant_equal, bf16_bits, gemm_tolerance_check, to_dev_bf16

pytestmark = pytest.mark.gpu


def linear_case(x_bits, w_bits, rows=None):
    x, w = to_dev_bf16(x_bits), to_dev_bf16(w_bits)
    xq = nv.quantize_rows(x)
    wq = nv.quantize_rows(w, per_tensor=True)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = nv.linear(xq, wq, err=err)
    torch.cuda.synchronize()
    assert err[0].item() == 0
    sel = np.arange(x_bits.shape[0]) if rows is None else np.asarray(rows)
    xr = oracle.quantize(x_bits[sel])
    wr = oracle.quantize(w_bits, per_tensor=True)
    if rows is None:
        assert_quant_equal(xq, xr, *x_bits.shape, what="x")
    assert_quant_equal(wq, wr, *w_bits.shape, what="w")
    a = oracle.dequantize(*xr)
    b = oracle.dequantize(*wr, per_tensor=True)
    yd = bf16_bits(y)[sel]
    return gemm_tolerance_check(yd, oracle.gemm_f64(a, b), oracle.abs_product_sum(a, b), what="y")


def test_linear_single_small():
    """64 x 256 activations, 256 -> 512 weights, seed 0."""
    d = workloads.linear_small()
    linear_case(d["x"], d["w"])


@pytest.mark.parametrize("M,K,N", [(300, 576, 512), (128, 64, 256), (1, 256, 256), (513, 2048, 768)])
def test_linear_ragged_tiles(M, K, N):
    rng = np.random.default_rng(M + K + N)
    x = workloads.gaussian_bf16(rng, (M, K), outlier_frac=0.01, zero_row_frac=0.02)
    w = workloads.gaussian_bf16(rng, (N, K), std=0.02)
    linear_case(x, w)


def test_linear_attention_projections_sampled():
    """QKV [32768 x 2048] . [5120 x 2048]^T and o_proj [32768 x 4096] .
    [2048 x 4096]^T on the device in full; the oracle checks 384 sampled rows
    (first, last, random) of each output."""
    d = workloads.attn_proj()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 127, 128, 32767], rng.integers(0, 32768, 380)]))
    linear_case(d["x"], d["wqkv"], rows)
    linear_case(d["o"], d["wo"], rows)
