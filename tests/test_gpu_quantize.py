"""Parity of the device quantizer with the oracle: bit-exact codes, E4M3
block scales (swizzled layout) and fp32 outer scales."""
import json
import os

import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import oracle
import workloads
from tests.helpers import assert_quant_equal, to_dev_bf16

pytestmark = pytest.mark.gpu


def run_both(x_bits, per_tensor=False, amax=None):
    x = to_dev_bf16(x_bits)
    am_dev = None if amax is None else torch.from_numpy(np.asarray(amax, np.float32)).cuda()
    got = nv.quantize_rows(x, per_tensor=per_tensor, amax_in=am_dev)
    torch.cuda.synchronize()
    ref = oracle.quantize(x_bits, per_tensor=per_tensor, amax_in=amax)
    return got, ref


def test_quant_rows_config_full_size():
    """16384 x 2048, ~N(0,1), 1% x50 outliers, 2% zero rows: every byte."""
    x = workloads.quant_rows()["x"]
    got, ref = run_both(x)
    assert_quant_equal(got, ref, *x.shape, what="quant 16384x2048")


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 48), (130, 272), (257, 2048), (64, 4096), (5, 5120)])
def test_quant_ragged_shapes(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    x = workloads.gaussian_bf16(rng, (rows, cols), outlier_frac=0.02, zero_row_frac=0.1)
    got, ref = run_both(x)
    assert_quant_equal(got, ref, rows, cols, what=f"{rows}x{cols}")


def test_quant_per_tensor_and_external_amax():
    rng = np.random.default_rng(3)
    x = workloads.gaussian_bf16(rng, (384, 768), std=0.02)
    got, ref = run_both(x, per_tensor=True)
    assert_quant_equal(got, ref, 384, 768, what="per-tensor")
    am = np.abs(workloads.bf16_bits_to_f32(x)).max(axis=1) * np.float32(0.75)  # forces saturation
    got, ref = run_both(x, amax=am)
    assert_quant_equal(got, ref, 384, 768, what="amax_in")


def test_quant_worked_blocks_on_device():
    with open(os.path.join(os.path.dirname(__file__), "golden", "worked_blocks.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        if "row_bits" in c:
            x = np.array([c["row_bits"]], np.uint16)
        else:
            x = workloads.to_bf16_bits(np.array([c["row"]], np.float32))
        amax = None if "amax_in" not in c else np.array([c["amax_in"]], np.float32)
        got, ref = run_both(x, amax=amax)
        assert_quant_equal(got, ref, 1, x.shape[1], what=c["name"])


def test_quant_every_bf16_pattern():
    """All finite bf16 values as block members under a fixed row scale, plus
    rows of bf16 subnormals (block scales and d in the subnormal range)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = workloads.bf16_bits_to_f32(bits)
    bits = bits[np.isfinite(vals)]
    n = len(bits)
    rows = (n + 14) // 15
    x = np.zeros((rows, 32), np.uint16)
    x[:, 0] = workloads.to_bf16_bits(np.array([3.0e38], np.float32))[0]
    flat = np.zeros(rows * 15, np.uint16)
    flat[:n] = bits
    x[:, 17:32] = flat.reshape(rows, 15)
    got, ref = run_both(x)
    assert_quant_equal(got, ref, rows, 32, what="all bf16, large row scale")
    # each pattern alone in its row: every amax / s_g / d regime, subnormals included
    y = np.zeros((n, 16), np.uint16)
    y[:, 3] = bits
    y[:, 9] = bits ^ 0x8000
    got, ref = run_both(y)
    assert_quant_equal(got, ref, n, 16, what="all bf16, one per row")


def test_context_swap_on_device():
    base = workloads.quant_rows(seed=4, rows=64, cols=2048)["x"]
    target = base[5:6]
    alone = nv.quantize_rows(to_dev_bf16(target))
    loud = workloads.to_bf16_bits(workloads.bf16_bits_to_f32(base) * np.float32(40.0))
    batch = np.concatenate([loud[:20], target, base[20:]])
    inb = nv.quantize_rows(to_dev_bf16(batch))
    torch.cuda.synchronize()
    assert torch.equal(alone.codes[0].cpu(), inb.codes[20].cpu())
    assert alone.scale[0].item() == inb.scale[20].item()


def test_quant_row_scale_sweep():
    """Rows scaled by 2^k for k across the bf16 exponent range: the per-block
    division bmax / t meets every binade of t (rows with tiny t take the
    plain IEEE division, the rest the FMA division with 1/t)."""
    rng = np.random.default_rng(21)
    rows, cols = 4096, 512
    base = rng.standard_normal((rows, cols)).astype(np.float32)
    base[rng.random((rows, cols)) < 0.05] *= np.float32(37.0)
    base[rng.random((rows, cols)) < 0.2] *= np.float32(1e-3)
    k = (np.arange(rows) % 250) - 130
    x = workloads.to_bf16_bits(base * np.exp2(k).astype(np.float32)[:, None])
    got, ref = run_both(x)
    assert_quant_equal(got, ref, rows, cols, what="scale sweep")


def test_quant_strided_and_offset_rows():
    """Rows read through a row stride of cols + 8 and from a base 16 bytes
    past a 32-byte boundary: the quantizer's 16-byte load path (one 32-byte
    load per block is taken only for 32-byte aligned rows)."""
    rng = np.random.default_rng(29)
    rows, cols = 300, 2048
    x = workloads.gaussian_bf16(rng, (rows, cols), outlier_frac=0.01, zero_row_frac=0.05)
    wide = np.zeros((rows, cols + 8), np.uint16)
    wide[:, :cols] = x
    dev = to_dev_bf16(wide)[:, :cols]
    assert dev.stride(0) == cols + 8
    got = nv.quantize_rows(dev)
    torch.cuda.synchronize()
    assert_quant_equal(got, oracle.quantize(x), rows, cols, what="row stride cols + 8")
    flat = np.zeros(rows * cols + 8, np.uint16)
    flat[8:] = x.reshape(-1)
    dev = to_dev_bf16(flat)[8:].view(rows, cols)
    assert dev.data_ptr() % 32 == 16
    got = nv.quantize_rows(dev)
    torch.cuda.synchronize()
    assert_quant_equal(got, oracle.quantize(x), rows, cols, what="base 16 bytes off a 32-byte boundary")


@pytest.mark.parametrize("fos", [None, "mse"])
def test_quant_grouped_per_tensor_matches_each_group(fos):
    """nvfp4_quantize_grouped: G expert matrices, each with its own per-tensor
    scale (different magnitudes, one all-zero group), bit-identical to the
    oracle's per-tensor quantization of every group."""
    G, N, K = 5, 256, 768
    rng = np.random.default_rng(17)
    ws = [workloads.gaussian_bf16(rng, (N, K), std=s) for s in (0.02, 1.0, 0.0, 3e-5, 40.0)]
    w = np.stack(ws)
    wt = to_dev_bf16(w.reshape(G * N, K)).view(G, N, K)
    got = nv.quantize_grouped_weights(wt, four_over_six=fos)
    torch.cuda.synchronize()
    per = nv.sf_bytes(N, K)
    for g in range(G):
        ref = oracle.quantize(w[g], per_tensor=True) if fos is None else oracle.quantize_46(w[g], err=fos, per_tensor=True)
        sub = nv.NVFP4Tensor(got.codes[g * N:(g + 1) * N], got.sf[g * per:(g + 1) * per], got.scale[g:g + 1], N, K)
        assert_quant_equal(sub, ref, N, K, what=f"group {g} ({fos})")
