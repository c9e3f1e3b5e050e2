"""Parity of the grouped BF16 backward GEMMs (tcgen05 kind::f16) with the
oracle: nvfp4_grouped_dgrad_bf16 (dx = dy . w_g per row group) and
nvfp4_grouped_wgrad_bf16 (dw_g = dy_g^T . x_g), element by element within
the GEMM tolerance (1 bf16 ulp + 1e-5 sum |a b|), on ragged groups of the
128-row-padded layout (an empty group among them), on dense operands of a
row count that is no multiple of the tile, and on the FC1 backward of the
8192-token Qwen3-shaped layer built from the forward pass's own quantized
operands (DQ(Q(x)) written in the padded layout, DQ(Q(W1)) with one scale
per expert)."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import oracle
import workloads
from tests.helpers import bf16_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


def tol_check(got_bits, exact, absum, what):
    g = oracle.bf16_to_f64(got_bits)
    r = oracle.bf16_to_f64(oracle.bf16_round(exact))
    tol = oracle.bf16_ulp(np.maximum(np.abs(g), np.abs(r))) + 1e-5 * absum
    bad = np.abs(g - r) > tol
    assert not bad.any(), (f"{what}: {bad.sum()} / {bad.size} out of tolerance, first "
                           f"{[(tuple(i), g[tuple(i)], r[tuple(i)]) for i in np.argwhere(bad)[:3]]}")


def padded_layout(counts):
    poff = np.zeros(len(counts) + 1, np.int64)
    poff[1:] = np.cumsum([(c + 127) // 128 * 128 for c in counts])
    return poff


def padded_operand(rng, counts, poff, cols, std=1.0):
    a = np.zeros((int(poff[-1]), cols), np.uint16)
    for g, c in enumerate(counts):
        a[poff[g]:poff[g] + c] = workloads.gaussian_bf16(rng, (c, cols), std=std)
    return a


@pytest.mark.parametrize("counts,nf,kf", [([0, 3, 128, 200, 57], 256, 512), ([300, 0, 129], 512, 256),
                                          ([1], 256, 256)])
def test_grouped_dgrad_and_wgrad(counts, nf, kf):
    rng = np.random.default_rng(len(counts) * 7 + nf)
    poff = padded_layout(counts)
    G = len(counts)
    dy = padded_operand(rng, counts, poff, nf)
    x = padded_operand(rng, counts, poff, kf)
    w = workloads.gaussian_bf16(rng, (G, nf, kf), std=0.02)
    po = torch.from_numpy(poff.astype(np.int32)).cuda()
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    dx = nv.grouped_dgrad_bf16(to_dev_bf16(dy), to_dev_bf16(w), po, err=err)
    dw = nv.grouped_wgrad_bf16(to_dev_bf16(dy), to_dev_bf16(x), po, err=err)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    ex, ab = oracle.grouped_dgrad(dy, w, poff)
    tol_check(bf16_bits(dx), ex, ab, "dgrad")
    ew, abw = oracle.grouped_wgrad(dy, x, poff)
    tol_check(bf16_bits(dw), ew, abw, "wgrad")
    assert not bf16_bits(dw)[counts.index(0)].any() if 0 in counts else True


@pytest.mark.parametrize("rows,nf,kf", [(300, 192, 256), (1, 64, 256), (4096, 1536, 768)])
def test_dense_dgrad_and_wgrad(rows, nf, kf):
    """One group of any row count (the dense linear's backward): rows past the end
    are zero-filled on load and dropped on store."""
    rng = np.random.default_rng(rows + nf)
    dy = workloads.gaussian_bf16(rng, (rows, nf))
    x = workloads.gaussian_bf16(rng, (rows, kf))
    w = workloads.gaussian_bf16(rng, (1, nf, kf), std=0.02)
    dx = nv.grouped_dgrad_bf16(to_dev_bf16(dy), to_dev_bf16(w))
    torch.cuda.synchronize()
    ex, ab = oracle.grouped_dgrad(dy, w)
    tol_check(bf16_bits(dx), ex, ab, "dense dgrad")
    if nf % 256 == 0:
        dw = nv.grouped_wgrad_bf16(to_dev_bf16(dy), to_dev_bf16(x))
        torch.cuda.synchronize()
        ew, abw = oracle.grouped_wgrad(dy, x)
        tol_check(bf16_bits(dw), ew, abw, "dense wgrad")


def test_offsets_off_the_128_row_grid_are_refused_on_the_device():
    rng = np.random.default_rng(3)
    dy = to_dev_bf16(workloads.gaussian_bf16(rng, (256, 256)))
    w = to_dev_bf16(workloads.gaussian_bf16(rng, (2, 256, 256), std=0.02))
    po = torch.tensor([0, 100, 256], dtype=torch.int32, device="cuda")
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.full((256, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    nv.grouped_dgrad_bf16(dy, w, po, out=out, err=err)
    torch.cuda.synchronize()
    assert int(err[0]) & nv.DEVERR_BADGROUP
    assert bool((out == 7.0).all()), "nothing may be written"


def test_dequantize_into_the_padded_layout():
    """DQ(Q(x)) rows written at their padded positions, the padding rows zeroed
    (over a buffer full of garbage), and DQ(Q(W)) of stacked weights with one
    scale per group: bit-exact with the oracle."""
    rng = np.random.default_rng(4)
    counts = [5, 0, 130, 128]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    poff = padded_layout(counts).astype(np.int32)
    x = workloads.gaussian_bf16(rng, (int(off[-1]), 256), outlier_frac=0.01)
    # an expert-ordered NVFP4 buffer as the forward pass keeps it: codes and outer scales by
    # row, block scales at the padded rows
    codes, sf_lin, scale = oracle.quantize(x)
    prow = np.concatenate([np.arange(poff[g], poff[g] + counts[g]) for g in range(len(counts))])
    sf_sw = oracle.sf_swizzle(sf_lin, prow, int(poff[-1]))
    t = nv.NVFP4Tensor(torch.from_numpy(codes).cuda(), torch.from_numpy(sf_sw).cuda(),
                       torch.from_numpy(scale).cuda(), int(off[-1]), 256)
    out = torch.full((int(poff[-1]), 256), -3.0, dtype=torch.bfloat16, device="cuda")
    nv.dequantize_rows(t, group_offsets=torch.from_numpy(off).cuda(), padded_offsets=torch.from_numpy(poff).cuda(),
                       out=out, padded_rows=True)
    torch.cuda.synchronize()
    want = np.zeros((int(poff[-1]), 256), np.uint16)
    want[prow] = oracle.dequantize_bf16(codes, sf_lin, scale)
    assert np.array_equal(bf16_bits(out), want)
    # stacked weights, one per-tensor scale per group
    w = workloads.gaussian_bf16(rng, (3, 256, 512), std=0.02)
    wq = nv.quantize_grouped_weights(to_dev_bf16(w))
    goff = torch.tensor([0, 256, 512, 768], dtype=torch.int32, device="cuda")
    y = nv.dequantize_rows(wq, per_tensor=True, group_offsets=goff, padded_offsets=goff)
    torch.cuda.synchronize()
    for g in range(3):
        assert np.array_equal(bf16_bits(y)[g * 256:(g + 1) * 256],
                              oracle.dequantize_bf16(*oracle.quantize(w[g], per_tensor=True), per_tensor=True))


def test_fc1_backward_on_the_8k_layer():
    """The FC1 backward of the 8192-token layer from the forward pass's own
    operands: x^ = DQ(Q(x)) of the permuted, quantized tokens (a1 in the
    workspace) written in the padded layout, w^ = DQ(Q(W1)) per expert, and a
    synthetic gradient dY1 [Rp x 2F] in the same layout.  dgrad and wgrad on
    sampled rows / experts against the oracle."""
    d = workloads.moe_8k()
    T, H = d["x"].shape
    E, k, F = 128, 8, 768
    R = T * k
    w1q = nv.quantize_grouped_weights(to_dev_bf16(d["w1"]))
    w2q = nv.quantize_grouped_weights(to_dev_bf16(d["w2"]))
    out, ws = nv.moe_expert_forward(to_dev_bf16(d["x"]), torch.from_numpy(d["logits"]).cuda(),
                                    torch.from_numpy(d["bias"]).cuda(), w1q, w2q, F, k)
    lay = nv.moe_workspace_layout(T, H, F, E, k)
    off = ws[lay["offsets"]:lay["offsets"] + 4 * (E + 1)].view(torch.int32)
    poff = ws[lay["padded_offsets"]:lay["padded_offsets"] + 4 * (E + 1)].view(torch.int32)
    torch.cuda.synchronize()
    off_h, poff_h = off.cpu().numpy().astype(np.int64), poff.cpu().numpy().astype(np.int64)
    Rp = int(poff_h[-1])
    a1 = nv.NVFP4Tensor(ws[lay["a1_codes"]:lay["a1_codes"] + R * H // 2].view(R, H // 2),
                        ws[lay["a1_sf"]:lay["a1_sf"] + Rp * H // 16],
                        ws[lay["a1_scale"]:lay["a1_scale"] + 4 * R].view(torch.float32), R, H)
    xh = torch.empty((Rp, H), dtype=torch.bfloat16, device="cuda")
    nv.dequantize_rows(a1, group_offsets=off, padded_offsets=poff, out=xh, padded_rows=True)
    gw = torch.arange(0, (E + 1) * 2 * F, 2 * F, dtype=torch.int32, device="cuda")
    wh = nv.dequantize_rows(w1q, per_tensor=True, group_offsets=gw, padded_offsets=gw).view(E, 2 * F, H)
    rng = np.random.default_rng(9)
    counts = np.diff(off_h)
    dy = padded_operand(rng, counts, poff_h, 2 * F, std=1e-3)
    dyd = to_dev_bf16(dy)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    dx = nv.grouped_dgrad_bf16(dyd, wh, poff, err=err)
    dw = nv.grouped_wgrad_bf16(dyd, xh, poff, err=err)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    xh_h, wh_h = bf16_bits(xh), bf16_bits(wh)
    # the operands are the oracle's DQ(Q(.)) of the same tensors
    m = oracle.route_metadata(oracle.route(d["logits"], d["bias"], k)[0], E)
    a1o = oracle.permute(oracle.quantize(d["x"]), m, k)
    prow = oracle.padded_rows(m)
    sample = np.random.default_rng(10).choice(R, 512, replace=False)
    assert np.array_equal(xh_h[prow[sample]], oracle.dequantize_bf16(a1o[0][sample], a1o[1][sample],
                                                                      a1o[2][sample]))
    experts = [int(np.argmax(counts)), int(np.nonzero(counts)[0][0]), 77]
    for e in experts:
        assert np.array_equal(wh_h[e], oracle.dequantize_bf16(*oracle.quantize(d["w1"][e], per_tensor=True),
                                                              per_tensor=True))
    # dgrad on the sampled rows (their experts' weights), wgrad on whole experts
    dx_h = bf16_bits(dx)
    rows = np.sort(prow[sample[:128]])
    grp = np.searchsorted(poff_h, rows, side="right") - 1
    for g in np.unique(grp):
        rr = rows[grp == g]
        ex, ab = oracle.grouped_dgrad(dy[rr], wh_h[g:g + 1])
        tol_check(dx_h[rr], ex, ab, f"dgrad expert {g}")
    dw_h = bf16_bits(dw)
    for e in experts + [int(np.argmin(np.where(counts > 0, counts, 1 << 30)))]:
        lo, hi = int(poff_h[e]), int(poff_h[e + 1])
        ew, abw = oracle.grouped_wgrad(dy[lo:hi], xh_h[lo:hi])
        tol_check(dw_h[e:e + 1], ew, abw, f"wgrad expert {e}")
    for e in np.nonzero(counts == 0)[0][:2]:
        assert not dw_h[e].any()
