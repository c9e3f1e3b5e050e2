"""The router-weighted combine inside FC2's epilogue (moe_options.fc2_combine):
each 64-column block of a token's output is summed by the unit that writes
the last of the token's k rows of that block, from Y2, in slot order ("miniTE
Technical Report" 5.6: the consumer's work moved into the producing GEMM).

The sum is the combine kernel's own (the same fp32 fused multiply-adds in the
same order), so the layer must give the same bits as with the separate
combine launch, whose output the other MoE tests check against the oracle;
which unit arrives last must not matter (run-to-run identity)."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import workloads
from tests.helpers import to_dev_bf16

pytestmark = pytest.mark.gpu


def _layer(d, E, k, F):
    w1q = nv.quantize_grouped_weights(to_dev_bf16(d["w1"]))
    w2q = nv.quantize_grouped_weights(to_dev_bf16(d["w2"]))
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


def _check(run, lay, **kw):
    out_s, ws_s = run(**kw)
    out_c, ws_c = run(fc2_combine=True, **kw)
    assert int(ws_c[lay["err"]:lay["err"] + 4].view(torch.int32)[0]) == 0
    assert torch.equal(out_s, out_c), "output differs from the separate combine"
    y = slice(lay["y2"], lay["comb_cnt"])
    assert torch.equal(ws_s[y], ws_c[y]), "Y2 differs"
    out_c2, _ = run(fc2_combine=True, **kw)
    assert torch.equal(out_c, out_c2), "run-to-run difference"


@pytest.mark.parametrize("name", ["moe_8k", "moe_32k"])
def test_combine_in_fc2_matches_the_separate_combine(name):
    d = getattr(workloads, name)()
    run, lay = _layer(d, 128, 8, 768)
    _check(run, lay)


@pytest.mark.parametrize("T,E,k,H,F,seed", [
    (700, 64, 8, 512, 256, 1),
    (333, 32, 4, 1024, 512, 2),
    (1500, 64, 6, 768, 768, 3),
    (257, 32, 1, 512, 384, 4),    # top-1, F not a multiple of 256
])
def test_combine_in_fc2_ragged_layers(T, E, k, H, F, seed):
    """Reduced layers: groups that end mid-tile (rows stored directly), odd
    m-tile counts, empty experts, a zero token, k = 1, 4, 6, 8."""
    rng = np.random.default_rng(seed)
    x = workloads.gaussian_bf16(rng, (T, H))
    x[5] = 0
    bias = np.zeros(E, np.float32)
    bias[: E // 8] = -1e4
    d = {"x": x, "logits": rng.standard_normal((T, E), dtype=np.float32), "bias": bias,
         "w1": workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02),
         "w2": workloads.gaussian_bf16(rng, (E, H, F), std=0.02)}
    run, lay = _layer(d, E, k, F)
    _check(run, lay)


def test_combine_in_fc2_with_the_router_weight_at_fc1():
    """With the weight applied at FC1 the combine sums unweighted rows."""
    rng = np.random.default_rng(6)
    T, E, k, H, F = 900, 64, 8, 512, 512
    d = {"x": workloads.gaussian_bf16(rng, (T, H)), "logits": rng.standard_normal((T, E), dtype=np.float32),
         "bias": rng.standard_normal(E, dtype=np.float32),
         "w1": workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02),
         "w2": workloads.gaussian_bf16(rng, (E, H, F), std=0.02)}
    run, lay = _layer(d, E, k, F)
    _check(run, lay, weight_at_fc1=True)


def test_combine_in_fc2_yields_to_the_requant_in_fc2():
    """With the requantization inside FC2 as well, the combine stays its own
    launch: the same bits as the requantization inside FC2 alone."""
    rng = np.random.default_rng(7)
    T, E, k, H, F = 600, 32, 8, 512, 256
    d = {"x": workloads.gaussian_bf16(rng, (T, H)), "logits": rng.standard_normal((T, E), dtype=np.float32),
         "bias": np.zeros(E, np.float32),
         "w1": workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02),
         "w2": workloads.gaussian_bf16(rng, (E, H, F), std=0.02)}
    run, lay = _layer(d, E, k, F)
    out_a, _ = run(fc2_requant="in_fc2")
    out_b, _ = run(fc2_requant="in_fc2", fc2_combine=True)
    assert torch.equal(out_a, out_b)
