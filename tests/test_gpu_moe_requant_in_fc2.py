"""The FC2 input requantized inside FC2 (moe_options.fc2_requant =
MOE_REQUANT_IN_FC2): FC2 reads D and FC1's row amax, encodes each 128-row A
tile in shared memory and reuses it for all output columns ("miniTE
Technical Report" 5.6, the quantization moved into the consumer GEMM).

The encode is the quantizer's own block encode and the MMAs see the same
operands, so the layer must give the same bits as with the separate
requantization launch, whose stages the other MoE tests check against the
oracle: the output, Y2 and, with moe_debug.requant_copy, the requantized
codes, block scales and row scales in the workspace."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import workloads
from tests.helpers import to_dev_bf16

pytestmark = pytest.mark.gpu


def _layer(d, E, k, F, wfos=None):
    w1q = nv.quantize_grouped_weights(to_dev_bf16(d["w1"]), four_over_six=wfos)
    w2q = nv.quantize_grouped_weights(to_dev_bf16(d["w2"]), four_over_six=wfos)
    x = to_dev_bf16(d["x"])
    lg = torch.from_numpy(d["logits"]).cuda()
    bs = torch.from_numpy(d["bias"]).cuda()
    T, H = d["x"].shape

    def run(**kw):
        ws = torch.zeros(int(nv.lib().moe_expert_workspace(T, H, F, E, k)), dtype=torch.uint8, device="cuda")
        out, ws = nv.moe_expert_forward(x, lg, bs, w1q, w2q, F, k, ws=ws, **kw)
        torch.cuda.synchronize()
        return out.view(torch.int16).clone(), ws
    return run, nv.moe_workspace_layout(T, H, F, E, k)


def _same(a, b, lay, field, what):
    lo = lay[field]
    hi = min(v for v in lay.values() if v > lo) if any(v > lo for v in lay.values()) else lay["total"]
    d = (a[lo:hi] != b[lo:hi]).nonzero()
    assert d.numel() == 0, f"{what}: {field} differs at {d.numel()} bytes, first at {int(d[0])}"


def _check(run, lay, **kw):
    out_s, ws_s = run(fc2_requant="separate", **kw)
    out_c, ws_c = run(fc2_requant="in_fc2", requant_copy=True, **kw)
    assert int(ws_c[lay["err"]:lay["err"] + 4].view(torch.int32)[0]) == 0
    assert torch.equal(out_s, out_c), "output differs from the separate requantization"
    # every intermediate, the requantized copies included
    lo, hi = lay["err"], lay["total"]
    diff = (ws_s[lo:hi] != ws_c[lo:hi]).nonzero()
    assert diff.numel() == 0, f"workspace differs at {diff.numel()} bytes, first offset {int(diff[0]) + lo}"
    # as shipped: no copies, the same output and Y2
    out_p, ws_p = run(fc2_requant="in_fc2", **kw)
    assert torch.equal(out_s, out_p), "output differs without the copies"
    _same(ws_s, ws_p, lay, "y2", "no copies")
    return ws_p


@pytest.mark.parametrize("name", ["moe_8k", "moe_32k"])
def test_in_fc2_matches_the_separate_launch_bit_for_bit(name):
    d = getattr(workloads, name)()
    run, lay = _layer(d, 128, 8, 768)
    ws_p = _check(run, lay)
    # without the copies, nothing is written to the requantized slots (the workspace starts zeroed)
    a2 = ws_p[lay["a2_codes"]:lay["a2_codes"] + 4096]
    assert int(a2.count_nonzero()) == 0


@pytest.mark.parametrize("T,E,k,H,F,seed", [
    (700, 64, 8, 512, 256, 1),    # one K-stage, two n-tiles, ragged groups
    (333, 32, 4, 1024, 512, 2),   # two K-stages, groups with an odd number of m-tiles
    (1500, 64, 6, 768, 768, 3),   # three K-stages, three n-tiles
])
def test_in_fc2_ragged_layers(T, E, k, H, F, seed):
    """Reduced layers: groups that end mid-tile, odd m-tile counts (the pair's
    second CTA stages its partner's rows and stores nothing), empty experts,
    a zero token and an outlier token."""
    rng = np.random.default_rng(seed)
    x = workloads.gaussian_bf16(rng, (T, H))
    x[5] = 0                                     # a zero row: amax 0 through FC1 and FC2
    x[9, 3] = np.float32(3.0e4).view(np.uint32) >> 16
    logits = rng.standard_normal((T, E), dtype=np.float32)
    bias = np.zeros(E, np.float32)
    bias[: E // 8] = -1e4                        # experts that no token picks
    d = {"x": x, "logits": logits, "bias": bias,
         "w1": workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02),
         "w2": workloads.gaussian_bf16(rng, (E, H, F), std=0.02)}
    run, lay = _layer(d, E, k, F)
    _check(run, lay)


def test_in_fc2_with_the_router_weight_at_fc1():
    """The pages' weighted-SwiGLU placement (moe_options.weight_at_fc1): D
    carries the router weight before its amax and requantization, which FC2
    then performs; same bits as the separate launch."""
    rng = np.random.default_rng(5)
    T, E, k, H, F = 900, 64, 8, 512, 512
    d = {"x": workloads.gaussian_bf16(rng, (T, H)), "logits": rng.standard_normal((T, E), dtype=np.float32),
         "bias": rng.standard_normal(E, dtype=np.float32),
         "w1": workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02),
         "w2": workloads.gaussian_bf16(rng, (E, H, F), std=0.02)}
    run, lay = _layer(d, E, k, F)
    _check(run, lay, weight_at_fc1=True)


def test_in_fc2_falls_back_where_it_does_not_apply():
    """Four-over-six activations and F = 640 (not a multiple of 256) take the
    separate launch under MOE_REQUANT_IN_FC2: same bits, requantized slots
    written without the copy flag."""
    rng = np.random.default_rng(4)
    T, E, k, H = 400, 32, 4, 512
    for F, fos in ((256, "mse"), (640, None)):
        d = {"x": workloads.gaussian_bf16(rng, (T, H)), "logits": rng.standard_normal((T, E), dtype=np.float32),
             "bias": np.zeros(E, np.float32),
             "w1": workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02),
             "w2": workloads.gaussian_bf16(rng, (E, H, F), std=0.02)}
        run, lay = _layer(d, E, k, F)
        out_s, ws_s = run(fc2_requant="separate", four_over_six=fos)
        out_c, ws_c = run(fc2_requant="in_fc2", four_over_six=fos)
        assert torch.equal(out_s, out_c)
        lo, hi = lay["err"], lay["total"]
        assert int((ws_s[lo:hi] != ws_c[lo:hi]).sum()) == 0
