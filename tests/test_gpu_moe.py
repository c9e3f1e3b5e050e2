"""Parity of moe_expert_forward with the oracle, stage by stage (each
device stage checked against the oracle applied to the device's previous
stage, since rounding in FC1 can legitimately flip a rare FC2-input code)
and end to end on a reduced layer."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import oracle
import workloads
from tests.helpers import assert_quant_equal, bf16_bits, gemm_tolerance_check, to_dev_bf16

pytestmark = pytest.mark.gpu


def ws_np(ws, lay, field, dtype, n):
    off = lay[field]
    nbytes = n * np.dtype(dtype).itemsize
    return ws[off:off + nbytes].cpu().numpy().view(dtype)


class DevQuant:
    def __init__(self, codes, sf, scale):
        self.codes, self.sf, self.scale = codes, sf, scale


def oq(x, fos, **kw):
    """The oracle quantizer of a mode: plain, or four-over-six by 'mse' / 'mae'."""
    return oracle.quantize(x, **kw) if fos is None else oracle.quantize_46(x, fos, **kw)


def run_device(d, E, k, F, weight_at_fc1=False, fos=None, wfos=None):
    x = to_dev_bf16(d["x"])
    T, H = d["x"].shape
    w1q = nv.quantize_grouped_weights(to_dev_bf16(d["w1"]), four_over_six=wfos)
    w2q = nv.quantize_grouped_weights(to_dev_bf16(d["w2"]), four_over_six=wfos)
    logits = torch.from_numpy(d["logits"]).cuda()
    bias = torch.from_numpy(d["bias"]).cuda()
    R = T * k
    fc1 = torch.empty((R, 2 * F), dtype=torch.float32, device="cuda")
    need = nv.lib().moe_expert_workspace(T, H, F, E, k)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out, ws = nv.moe_expert_forward(x, logits, bias, w1q, w2q, F, k, weight_at_fc1=weight_at_fc1,
                                    ws=ws, fc1_debug=fc1, four_over_six=fos)
    torch.cuda.synchronize()
    return dict(out=bf16_bits(out), ws=ws, fc1=fc1, w1q=w1q, w2q=w2q,
                lay=nv.moe_workspace_layout(T, H, F, E, k), fos=fos, wfos=wfos)


def ws_rows(ws, lay, field, dtype, R, C, rows):
    """Rows `rows` of an [R x C] intermediate in the workspace, fetched on the device."""
    tdt = {np.uint16: torch.int16, np.uint8: torch.uint8, np.float32: torch.float32}[dtype]
    n = R * C * np.dtype(dtype).itemsize
    full = ws[lay[field]:lay[field] + n].view(tdt).view(R, C)
    return full[torch.from_numpy(np.asarray(rows, np.int64)).cuda()].cpu().numpy().view(dtype)


U32 = 2.0 ** -24  # unit roundoff of fp32


def router_weight_bound(logits, bias, ids):
    """Relative error bound of the device's router weights against the oracle's
    fp64 softmax over the k selected z (the same fp32 z = fl(logit + bias) on
    both sides).  The device forms d_s = fl(z_s - z_max) (relative rounding
    error u = 2^-24 of |d_s|, which moves exp(d_s) by a relative |d_s| u),
    e_s = expf(d_s) (at most 2 ulp = 2^-22 relative, CUDA's documented bound
    for expf), S = the k e_s summed in slot order in fp32 (positive terms:
    relative error at most the largest term error plus (k - 1) u), and
    w_s = e_s / S (one more u).  To first order |w_dev - w| / w <= eps_s +
    max_j eps_j + (k - 1) u + u with eps_s = 2^-22 + |d_s| u; 0.1% more covers
    the second-order terms."""
    z = (np.asarray(logits, np.float32) + np.asarray(bias, np.float32)[None, :]).astype(np.float64)
    zs = np.take_along_axis(z, ids.astype(np.int64), axis=1)
    dz = np.abs(zs - zs[:, :1])
    eps = 2.0 ** -22 + dz * U32
    k = ids.shape[1]
    return (eps + eps.max(axis=1, keepdims=True) + k * U32) * 1.001


def check_router_weights(w_dev, w_or, logits, bias, ids):
    bound = router_weight_bound(logits, bias, ids)
    err = np.abs(w_dev.astype(np.float64) - w_or)
    bad = err > bound * w_or + 1e-45
    assert not bad.any(), (f"router weights: {bad.sum()} outside the derived bound, worst relative "
                           f"{(err / w_or).max():.3e} against bound {bound[bad].min():.3e}")


def check_stagewise(d, E, k, F, dev, experts=None, weight_at_fc1=False, token_sample=None):
    T, H = d["x"].shape
    R = T * k
    ws, lay = dev["ws"], dev["lay"]
    assert ws_np(ws, lay, "err", np.uint32, 1)[0] == 0, "device error word set"

    # routing: ids exact, weights within the error bound of their fp32 evaluation
    ids_o, w_o = oracle.route(d["logits"], d["bias"], k)
    ids = ws_np(ws, lay, "ids", np.int32, R).reshape(T, k)
    w = ws_np(ws, lay, "weights", np.float32, R).reshape(T, k)
    assert np.array_equal(ids, ids_o)
    check_router_weights(w, w_o, d["logits"], d["bias"], ids_o)

    # metadata exact
    m = oracle.route_metadata(ids_o, E)
    for f, name, n in [("cnt", "counts", E), ("off", "offsets", E + 1), ("poff", "padded_offsets", E + 1),
                       ("perm", "perm", R), ("inv", "inv", R)]:
        assert np.array_equal(ws_np(ws, lay, name, np.int32, n), m[f]), name

    # per-token quantization of X (block scales row-linear, the permute's input) and the
    # permute (block scales swizzled, padded per expert): exact bytes
    fos, wfos = dev.get("fos"), dev.get("wfos")
    xq_o = oq(d["x"], fos)
    assert np.array_equal(ws_np(ws, lay, "xq_codes", np.uint8, T * H // 2).reshape(T, H // 2), xq_o[0]), "xq codes"
    assert np.array_equal(ws_np(ws, lay, "xq_sf", np.uint8, T * H // 16).reshape(T, H // 16), xq_o[1]), "xq sf"
    assert np.array_equal(ws_np(ws, lay, "xq_scale", np.float32, T).view(np.uint32), xq_o[2].view(np.uint32))
    a1_o = oracle.permute(xq_o, m, k)
    prow = oracle.padded_rows(m)
    Rp = int(m["poff"][-1])
    a1 = DevQuant(ws[lay["a1_codes"]:lay["a1_codes"] + R * H // 2].view(R, H // 2),
                  ws[lay["a1_sf"]:lay["a1_sf"] + Rp * H // 16],
                  ws[lay["a1_scale"]:lay["a1_scale"] + 4 * R].view(torch.float32))
    assert_quant_equal(a1, a1_o, R, H, row_map=prow, what="a1")
    # the padding rows of each expert's last m-tile carry zero block scales
    a1_all = oracle.sf_unswizzle(a1.sf.cpu().numpy(), Rp, H // 16)
    pad = np.ones(Rp, bool)
    pad[prow] = False
    assert not a1_all[pad].any(), "a1 padding rows: nonzero block scales"

    off = m["off"]
    if experts is None:
        experts = [e for e in range(E) if m["cnt"][e] > 0]
    amax2 = ws_np(ws, lay, "amax2", np.float32, R)
    a2s = ws_np(ws, lay, "a2_scale", np.float32, R)
    a2sf = ws[lay["a2_sf"]:lay["a2_sf"] + Rp * ((F // 16 + 3) // 4 * 4)].cpu().numpy()
    w1c = dev["w1q"].codes.cpu().numpy()
    w2c = dev["w2q"].codes.cpu().numpy()
    w1s = dev["w1q"].scale.cpu().numpy()
    w2s = dev["w2q"].scale.cpu().numpy()
    w1sf, w2sf = dev["w1q"].sf.cpu().numpy(), dev["w2q"].sf.cpu().numpy()
    row_w = np.zeros(R)
    row_w[m["inv"]] = w.reshape(-1)  # router weight of each expert-ordered row (device values)
    checked = 0
    for e in experts:
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        rows = np.arange(lo, hi)
        if len(rows) > 256:
            rng = np.random.default_rng(e)
            rows = np.unique(np.concatenate([rows[:64], rows[-64:], rng.choice(rows, 128, replace=False)]))
        # the expert's weights: device quantization bit-exact with the oracle's
        w1e = oq(d["w1"][e], wfos, per_tensor=True)
        w2e = oq(d["w2"][e], wfos, per_tensor=True)
        s1 = oracle.sf_bytes(2 * F, H // 16)
        s2 = oracle.sf_bytes(H, F // 16)
        assert np.array_equal(w1c[e * 2 * F:(e + 1) * 2 * F], w1e[0])
        assert np.array_equal(oracle.sf_unswizzle(w1sf[e * s1:(e + 1) * s1], 2 * F, H // 16), w1e[1])
        assert w1s[e] == w1e[2][0] and w2s[e] == w2e[2][0]
        assert np.array_equal(w2c[e * H:(e + 1) * H], w2e[0])
        assert np.array_equal(oracle.sf_unswizzle(w2sf[e * s2:(e + 1) * s2], H, F // 16), w2e[1])
        # FC1 (fp32 debug output) against the fp64 product of the dequantized operands
        a = oracle.dequantize(a1_o[0][rows], a1_o[1][rows], a1_o[2][rows])
        b = oracle.dequantize(*w1e, per_tensor=True)
        c_ex = oracle.gemm_f64(a, b)
        c_gpu = dev["fc1"][torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
        tol = 2.0 ** -22 * np.abs(c_ex) + 1e-5 * oracle.abs_product_sum(a, b) + 1e-30
        assert np.all(np.abs(c_gpu - c_ex) <= tol), f"fc1 expert {e}"
        # SwiGLU of the device's C: within one bf16 ulp; amax exact
        prob = row_w[rows] if weight_at_fc1 else None
        d_o, _ = oracle.swiglu(c_gpu, prob)
        d_rows = ws_rows(ws, lay, "d", np.uint16, R, F, rows)
        dg = oracle.bf16_to_f64(d_rows)
        do = oracle.bf16_to_f64(d_o)
        assert np.all(np.abs(dg - do) <= oracle.bf16_ulp(np.maximum(np.abs(dg), np.abs(do)))), f"D expert {e}"
        assert np.array_equal(amax2[rows], np.abs(dg).max(axis=1).astype(np.float32)), f"amax2 expert {e}"
        # requant of the device's D with the reused amax: bit-exact
        q2 = oq(d_rows, fos, amax_in=amax2[rows])
        assert np.array_equal(ws_rows(ws, lay, "a2_codes", np.uint8, R, F // 2, rows), q2[0]), f"q2 codes e{e}"
        assert np.array_equal(oracle.sf_unswizzle(a2sf, len(rows), F // 16, prow[rows]), q2[1]), f"q2 sf {e}"
        assert np.array_equal(a2s[rows].view(np.uint32), q2[2].view(np.uint32)), f"q2 scale {e}"
        # FC2 within the GEMM tolerance
        a = oracle.dequantize(*q2)
        b = oracle.dequantize(*w2e, per_tensor=True)
        gemm_tolerance_check(ws_rows(ws, lay, "y2", np.uint16, R, H, rows), oracle.gemm_f64(a, b),
                             oracle.abs_product_sum(a, b), what=f"y2 e{e}")
        checked += len(rows)
    assert checked > 0

    # combine of the device's Y2 (all tokens, or a sample)
    toks = np.arange(T) if token_sample is None else np.asarray(token_sample)
    inv_t = m["inv"].reshape(T, k)[toks]
    y2f = oracle.bf16_to_f64(ws_rows(ws, lay, "y2", np.uint16, R, H, inv_t.reshape(-1)))
    wc = np.ones((len(toks), k)) if weight_at_fc1 else w[toks].astype(np.float64)
    ref = oracle.combine(y2f, np.arange(len(toks) * k, dtype=np.int32), wc)
    got = dev["out"][toks]
    absum = np.einsum("tk,tkh->th", np.abs(wc), np.abs(y2f.reshape(len(toks), k, H)))
    g, r = oracle.bf16_to_f64(got), oracle.bf16_to_f64(ref)
    tol = oracle.bf16_ulp(np.maximum(np.abs(g), np.abs(r))) + 1e-5 * absum
    assert np.all(np.abs(g - r) <= tol), "combine"
    return m


def small_layer(T, E, k, H, F, seed, bias_std=1.0):
    rng = np.random.default_rng(seed)
    return dict(x=workloads.gaussian_bf16(rng, (T, H)),
                logits=rng.standard_normal((T, E), dtype=np.float32),
                bias=(rng.standard_normal(E, dtype=np.float32) * np.float32(bias_std)),
                w1=workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02),
                w2=workloads.gaussian_bf16(rng, (E, H, F), std=0.02))


@pytest.mark.parametrize("T,E,k,H,F", [(1000, 32, 4, 512, 256), (1, 32, 2, 256, 128), (129, 64, 8, 256, 384),
                                         (129, 128, 8, 1024, 128), (33, 128, 8, 2048, 256),
                                         # top-1 (router weight exactly 1), E = 96 (3 logits per lane)
                                         (200, 96, 1, 512, 256),
                                         # the largest E and top-k the library accepts (256, 16): most
                                         # experts get 0-10 rows; the combine's 16-slot instance
                                         (64, 256, 16, 256, 128),
                                         # E = 160 (5 logits per lane), top-16
                                         (40, 160, 16, 256, 128)])
def test_moe_small_full_and_end_to_end(T, E, k, H, F):
    d = small_layer(T, E, k, H, F, seed=T + E)
    dev = run_device(d, E, k, F)
    check_stagewise(d, E, k, F, dev)
    # independent end to end: the oracle's own chain from the same inputs
    w1o = [oracle.quantize(d["w1"][e], per_tensor=True) for e in range(E)]
    w2o = [oracle.quantize(d["w2"][e], per_tensor=True) for e in range(E)]
    ref = oracle.moe_forward(d["x"], d["logits"], d["bias"], w1o, w2o, k)
    g = oracle.bf16_to_f64(dev["out"])
    r = oracle.bf16_to_f64(ref["out"])
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    assert rel <= 2e-3, rel


def test_moe_zero_and_outlier_tokens_and_a_zero_expert():
    """Degenerate rows through the whole layer: all-zero tokens (s_g = 0, zero
    codes and block scales), x50 outlier entries (block scales near E4M3
    saturation), and an expert whose W1 is all zero, so that its rows reach
    the requant with amax 0 (zero codes, scales and outer scale) and FC2 with
    zero operands; those tokens' outputs then sum only their other slots."""
    T, E, k, H, F = 400, 64, 4, 512, 256
    rng = np.random.default_rng(41)
    d = dict(x=workloads.gaussian_bf16(rng, (T, H), outlier_frac=0.02, outlier_mult=50.0, zero_row_frac=0.05),
             logits=rng.standard_normal((T, E), dtype=np.float32),
             bias=rng.standard_normal(E, dtype=np.float32),
             w1=workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02),
             w2=workloads.gaussian_bf16(rng, (E, H, F), std=0.02))
    zero_e = 3
    d["w1"][zero_e] = 0       # bf16 +0.0 everywhere
    d["bias"][zero_e] = 3.0   # route plenty of rows to it
    zero_tok = np.nonzero(~d["x"].any(axis=1))[0]
    assert len(zero_tok) > 0
    dev = run_device(d, E, k, F)
    check_stagewise(d, E, k, F, dev)
    m = oracle.route_metadata(oracle.route(d["logits"], d["bias"], k)[0], E)
    lo, hi = int(m["off"][zero_e]), int(m["off"][zero_e + 1])
    assert hi - lo > 0
    ws, lay = dev["ws"], dev["lay"]
    R = T * k
    assert not ws_np(ws, lay, "amax2", np.float32, R)[lo:hi].any()
    assert not ws_np(ws, lay, "a2_scale", np.float32, R)[lo:hi].any()
    assert not ws_rows(ws, lay, "a2_codes", np.uint8, R, F // 2, np.arange(lo, hi)).any()
    # all-zero tokens: every one of their slots is zero through the layer, output exactly zero
    assert np.all((dev["out"][zero_tok] & 0x7FFF) == 0)
    w1o = [oracle.quantize(d["w1"][e], per_tensor=True) for e in range(E)]
    w2o = [oracle.quantize(d["w2"][e], per_tensor=True) for e in range(E)]
    ref = oracle.moe_forward(d["x"], d["logits"], d["bias"], w1o, w2o, k)
    g = oracle.bf16_to_f64(dev["out"])
    r = oracle.bf16_to_f64(ref["out"])
    assert np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30) <= 2e-3


def test_moe_weight_at_fc1_variant():
    T, E, k, H, F = 300, 32, 4, 512, 256
    d = small_layer(T, E, k, H, F, seed=11)
    dev = run_device(d, E, k, F, weight_at_fc1=True)
    check_stagewise(d, E, k, F, dev, weight_at_fc1=True)
    base = run_device(d, E, k, F)
    g = oracle.bf16_to_f64(dev["out"])
    r = oracle.bf16_to_f64(base["out"])
    # same layer with the weight applied before the bf16 rounding of D: codes of
    # FC2's input can flip, so the two placements agree only to FP4 resolution
    assert np.linalg.norm(g - r) / np.linalg.norm(r) < 0.1


def test_moe_deterministic():
    T, E, k, H, F = 777, 64, 8, 512, 256
    d = small_layer(T, E, k, H, F, seed=5, bias_std=2.0)
    a = run_device(d, E, k, F)
    b = run_device(d, E, k, F)
    assert np.array_equal(a["out"], b["out"])
    lay = a["lay"]
    assert torch.equal(a["ws"][lay["ids"]:lay["y2"]], b["ws"][lay["ids"]:lay["y2"]])


def _pick_experts(m, n_random, seed):
    cnt = m["cnt"]
    nz = np.nonzero(cnt)[0]
    rng = np.random.default_rng(seed)
    pick = {int(nz[np.argmax(cnt[nz])]), int(nz[np.argmin(cnt[nz])]), int(nz[0]), int(nz[-1])}
    pick |= set(int(e) for e in rng.choice(nz, min(n_random, len(nz)), replace=False))
    return sorted(pick)


def test_moe_long_layer_past_the_scan_register_form():
    """70000 tokens: 2188 routing chunks, more than the 8 per thread that the
    scan keeps in registers, so it takes its loop form; top-2 of 32 experts
    (the top-k launched alone). Routing metadata, permute and requant exact,
    the GEMMs and the combine within tolerance, as in the other layers."""
    T, E, k, H, F = 70000, 32, 2, 256, 128
    d = small_layer(T, E, k, H, F, seed=70)
    dev = run_device(d, E, k, F)
    m = oracle.route_metadata(oracle.route(d["logits"], d["bias"], k)[0], E)
    toks = np.random.default_rng(3).choice(T, 2048, replace=False)
    check_stagewise(d, E, k, F, dev, experts=_pick_experts(m, 2, 2), token_sample=toks)


@pytest.mark.parametrize("name", ["moe_8k", "moe_32k"])
def test_moe_qwen3_shapes_stagewise(name):
    """8192 tokens (bias ~N(0,1)) and 32768 tokens (bias ~N(0,4): empty and
    >5x-mean experts) through the full layer H=2048, E=128, top-8, F=768;
    routing, metadata, quantization and permute checked in full, the GEMM
    stages on every row of a sample of experts, the combine on 2048 tokens."""
    d = getattr(workloads, name)()
    E, k, F = 128, 8, 768
    dev = run_device(d, E, k, F)
    ids_o, _ = oracle.route(d["logits"], d["bias"], k)
    m = oracle.route_metadata(ids_o, E)
    if name == "moe_32k":
        assert (m["cnt"] == 0).any() and m["cnt"].max() > 5 * m["cnt"].mean()
    experts = _pick_experts(m, 4, 0)
    toks = np.random.default_rng(1).choice(d["x"].shape[0], 2048, replace=False)
    check_stagewise(d, E, k, F, dev, experts=experts, token_sample=toks)


@pytest.mark.parametrize("E,k", [(128, 8), (96, 6), (256, 16), (32, 4), (160, 9)])
def test_moe_router_ties_and_signed_zeros(E, k):
    """Logits from a handful of values (exact ties everywhere, +0 and -0
    among them): ids must match the oracle's lower-index tie rule exactly
    (-0 and +0 are one value), and the rest of the layer with it.  E = 128
    runs the top-k that shares a launch with the quantization of X; the
    others the top-k launched alone, with 1, 3, 5 and 8 logits per lane (a
    lane's keys are sorted before the rounds, so equal keys inside one lane
    must keep their expert order)."""
    T, H, F = 512, 1024, 128
    rng = np.random.default_rng(17)
    d = small_layer(T, E, k, H, F, seed=17)
    vals = np.array([-1.0, -0.0, 0.0, 0.5, 1.0, 2.0], np.float32)
    d["logits"] = vals[rng.integers(0, len(vals), (T, E))]
    d["bias"] = np.zeros(E, np.float32)
    d["bias"][::7] = np.float32(-0.0)
    dev = run_device(d, E, k, F)
    ids_o, _ = oracle.route(d["logits"], d["bias"], k)
    m = oracle.route_metadata(ids_o, E)
    check_stagewise(d, E, k, F, dev, experts=_pick_experts(m, 3, 2))
