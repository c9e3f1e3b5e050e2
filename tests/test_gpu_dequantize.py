"""Parity of the device DQ(Q(x)) (NVFP4 -> bf16 of the exact dequantized
value) with the oracle: bit-exact bf16 over every code x every E4M3 block
scale x a spread of outer scales (fp32 ties, subnormal products), the
16384 x 2048 quantizer workload, per-tensor weights, expert-padded scale
rows and ragged or strided shapes.  Inputs are quantized by the oracle."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import oracle
import workloads
from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu


def device_tensor(codes, sf_swizzled, scale, rows, cols):
    t = nv.NVFP4Tensor(torch.from_numpy(np.ascontiguousarray(codes)).cuda(),
                       torch.from_numpy(np.ascontiguousarray(sf_swizzled)).cuda(),
                       torch.from_numpy(np.ascontiguousarray(scale, np.float32)).cuda(), rows, cols)
    return t


def check(codes, sf_lin, scale, per_tensor=False, ldy=None, what=""):
    rows, cols = codes.shape[0], codes.shape[1] * 2
    t = device_tensor(codes, oracle.sf_swizzle(sf_lin), scale, rows, cols)
    ldy = cols if ldy is None else ldy
    buf = torch.full((max(rows, 1), ldy), -7.0, dtype=torch.bfloat16, device="cuda")
    nv.dequantize_rows(t, per_tensor=per_tensor, out=buf[:rows, :cols] if ldy == cols else
                       torch.as_strided(buf, (rows, cols), (ldy, 1)))
    torch.cuda.synchronize()
    got = bf16_bits(buf)[:rows]
    want = oracle.dequantize_bf16(codes, sf_lin, scale, per_tensor)
    bad = np.nonzero((got[:, :cols] != want).any(axis=1))[0]
    assert len(bad) == 0, f"{what}: {len(bad)} rows differ, first {bad[:5]}"
    if ldy > cols:  # columns past cols untouched
        assert np.all(got[:, cols:] == bf16_bits(torch.tensor([-7.0], dtype=torch.bfloat16))[0]), what


def test_dq_every_code_scale_and_many_outer_scales():
    # block b of every row uses scale byte b (0..126, all finite E4M3 values), codes 0..15
    nb = 127
    rng = np.random.default_rng(5)
    special = [1.0, 1.0 + 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -23, (1.0 + 2.0 ** -8) / 3.0, 2.0 ** -100,
               2.0 ** -100 * (1 - 2.0 ** -24), 2.0 ** -126, 2.0 ** -133, 2.0 ** -149, 3.0 * 2.0 ** -140,
               1.0 / 2688.0, 448.0 / 2688.0, 0.0, 1.5e-45 * 7]
    sg = np.concatenate([np.array(special, np.float32),
                         (2.0 ** rng.uniform(-149, 20, size=114)).astype(np.float32),
                         (rng.uniform(1, 2, size=32) * 2.0 ** -101).astype(np.float32)])
    rows = len(sg)
    codes16 = np.arange(16, dtype=np.uint8)
    packed_block = (codes16[0::2] | (codes16[1::2] << 4)).astype(np.uint8)
    codes = np.tile(packed_block, (rows, nb))
    sf_lin = np.tile(np.arange(nb, dtype=np.uint8), (rows, 1))
    check(codes, sf_lin, sg, what="codes x scales x s_g")


def test_dq_quantizer_workload_full_size():
    x = workloads.quant_rows()["x"]
    codes, sf, scale = oracle.quantize(x)
    check(codes, sf, scale, what="16384x2048")


def test_dq_per_tensor_weights():
    rng = np.random.default_rng(8)
    w = workloads.gaussian_bf16(rng, (384, 768), std=0.02)
    codes, sf, scale = oracle.quantize(w, per_tensor=True)
    check(codes, sf, scale, per_tensor=True, what="per-tensor")


@pytest.mark.parametrize("rows,cols,ldy", [(1, 16, 16), (3, 48, 56), (130, 272, 272), (257, 4096, 4104),
                                           (5, 32768, 32768), (64, 2048, 2048)])
def test_dq_ragged_and_strided(rows, cols, ldy):
    rng = np.random.default_rng(rows * 31 + cols)
    x = workloads.gaussian_bf16(rng, (rows, cols), outlier_frac=0.02, zero_row_frac=0.1)
    codes, sf, scale = oracle.quantize(x)
    check(codes, sf, scale, ldy=ldy, what=f"{rows}x{cols} ldy {ldy}")


def test_dq_expert_padded_scale_rows():
    """Scale rows padded to 128 per group, as in the expert-ordered buffers."""
    counts = np.array([5, 0, 130, 1, 128, 77, 0, 256], np.int64)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    poff = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    R, cols = int(off[-1]), 768
    rng = np.random.default_rng(21)
    x = workloads.gaussian_bf16(rng, (R, cols), outlier_frac=0.01, zero_row_frac=0.05)
    codes, sf_lin, scale = oracle.quantize(x)
    row_map = np.empty(R, np.int64)
    for g in range(len(counts)):
        row_map[off[g]:off[g + 1]] = poff[g] + np.arange(counts[g])
    sw = oracle.sf_swizzle(sf_lin, row_map=row_map, dst_rows=int(poff[-1]))
    t = device_tensor(codes, sw, scale, R, cols)
    y = nv.dequantize_rows(t, group_offsets=torch.from_numpy(off).cuda(), padded_offsets=torch.from_numpy(poff).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(y), oracle.dequantize_bf16(codes, sf_lin, scale))


def test_dq_zero_rows_is_a_no_op():
    dev = "cuda"
    t = nv.NVFP4Tensor(torch.zeros(16, dtype=torch.uint8, device=dev), torch.zeros(16, dtype=torch.uint8, device=dev),
                       torch.zeros(1, dtype=torch.float32, device=dev), 0, 64)
    y = torch.full((1, 64), 3.0, dtype=torch.bfloat16, device=dev)
    nv.dequantize_rows(t, out=y[:0])
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
