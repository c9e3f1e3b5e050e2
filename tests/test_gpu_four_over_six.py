"""Parity of the device's four-over-six quantizer with the oracle ('The
4-bitter Lesson', Four-Over-Six for RL Weights and Activations): codes,
E4M3 block scales and outer scales bit-exact, in both error modes, for every
kernel shape (8 / 16 / 32 lanes per row, the long-row form), per-tensor
mode, a reused amax, every hand-worked block; and the expert layer with
four-over-six activations and weights, stage by stage."""
import json
import os

import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import oracle
import workloads
from tests.helpers import assert_quant_equal, to_dev_bf16
from tests.test_gpu_moe import check_stagewise, run_device, small_layer

pytestmark = pytest.mark.gpu


def run_both(x_bits, err, per_tensor=False, amax=None):
    am_dev = None if amax is None else torch.from_numpy(np.asarray(amax, np.float32)).cuda()
    got = nv.quantize_rows(to_dev_bf16(x_bits), per_tensor=per_tensor, amax_in=am_dev, four_over_six=err)
    torch.cuda.synchronize()
    return got, oracle.quantize_46(x_bits, err, per_tensor=per_tensor, amax_in=amax)


@pytest.mark.parametrize("err", ["mse", "mae"])
def test_quant_rows_full_size(err):
    """The 16384 x 2048 quantizer workload (1% x50 outliers, 2% zero rows), every byte."""
    x = workloads.quant_rows()["x"]
    got, ref = run_both(x, err)
    assert_quant_equal(got, ref, *x.shape, what=f"4/6 {err} 16384x2048")


@pytest.mark.parametrize("err", ["mse", "mae"])
@pytest.mark.parametrize("rows,cols", [(1, 16), (7, 48), (130, 272), (300, 768), (64, 2048), (9, 5120)])
def test_ragged_shapes_all_kernel_forms(rows, cols, err):
    rng = np.random.default_rng(rows * 31 + cols)
    x = workloads.gaussian_bf16(rng, (rows, cols), outlier_frac=0.03, outlier_mult=20.0, zero_row_frac=0.1)
    got, ref = run_both(x, err)
    assert_quant_equal(got, ref, rows, cols, what=f"4/6 {err} {rows}x{cols}")


@pytest.mark.parametrize("err", ["mse", "mae"])
def test_per_tensor_reused_amax_and_scale_sweep(err):
    rng = np.random.default_rng(5)
    x = workloads.gaussian_bf16(rng, (384, 768), std=0.02)
    got, ref = run_both(x, err, per_tensor=True)
    assert_quant_equal(got, ref, 384, 768, what="per-tensor")
    am = np.abs(workloads.bf16_bits_to_f32(x)).max(axis=1) * np.float32(1.5)
    got, ref = run_both(x, err, amax=am)
    assert_quant_equal(got, ref, 384, 768, what="amax_in")
    # rows scaled by 2^k across the exponent range: every division path, subnormal block scales
    base = rng.standard_normal((2048, 256)).astype(np.float32)
    k = (np.arange(2048) % 250) - 130
    xs = workloads.to_bf16_bits(base * np.exp2(k).astype(np.float32)[:, None])
    got, ref = run_both(xs, err)
    assert_quant_equal(got, ref, 2048, 256, what="scale sweep")


def test_hand_worked_blocks_on_device():
    with open(os.path.join(os.path.dirname(__file__), "golden", "four_over_six_blocks.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x = workloads.to_bf16_bits(np.array([c["row"]], np.float32))
        for err in ("mse", "mae"):
            got, ref = run_both(x, err)
            assert_quant_equal(got, ref, 1, x.shape[1], what=f"{c['name']} {err}")


def test_moe_layer_with_four_over_six_activations_and_weights():
    T, E, k, H, F = 600, 32, 4, 512, 256
    d = small_layer(T, E, k, H, F, seed=46, bias_std=2.0)
    dev = run_device(d, E, k, F, fos="mse", wfos="mae")
    check_stagewise(d, E, k, F, dev)
