"""The expert layer exactly as it ships: the call without any debug output,
as bench.py times it, on the 8192- and 32768-token Qwen3-shaped layers.

1. Bit-identity with the debug run.  The stage-wise parity checks read the
   fp32 FC1 output that only a debug call writes (an extra store in FC1's
   epilogue); here the same inputs go through the plain call and through the
   debug call, and the output and every intermediate of the workspace must
   be the same bits, so those stage-wise checks speak for the plain call.
2. The independent end-to-end check: the oracle's own chain from the same
   inputs (route, quantize, permute, FC1, SwiGLU, requant, FC2, combine, no
   device intermediate fed in) on a seeded sample of tokens.  Rounding in
   FC1 (fp32 accumulation and the fast exp / reciprocal against fp64) can
   flip a rare FC2-input code, so the check is statistical: rel-L2 <= 1e-3
   over the sample, at least 99.9% of the elements within the GEMM
   tolerance carried through the combine, and the q2 code mismatch rate
   reported."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import oracle
import workloads
from tests.helpers import bf16_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

E, K_TOP, F = 128, 8, 768


def _weights(d):
    return nv.quantize_grouped_weights(to_dev_bf16(d["w1"])), nv.quantize_grouped_weights(to_dev_bf16(d["w2"]))


def _call(d, w1q, w2q, fc1_debug=None):
    T, H = d["x"].shape
    ws = torch.zeros(int(nv.lib().moe_expert_workspace(T, H, F, E, K_TOP)), dtype=torch.uint8, device="cuda")
    out, ws = nv.moe_expert_forward(to_dev_bf16(d["x"]), torch.from_numpy(d["logits"]).cuda(),
                                    torch.from_numpy(d["bias"]).cuda(), w1q, w2q, F, K_TOP, ws=ws,
                                    fc1_debug=fc1_debug)
    torch.cuda.synchronize()
    return out, ws


@pytest.mark.parametrize("name", ["moe_8k", "moe_32k"])
def test_plain_call_is_bit_identical_to_the_debug_call(name):
    d = getattr(workloads, name)()
    T, H = d["x"].shape
    w1q, w2q = _weights(d)
    out_a, ws_a = _call(d, w1q, w2q)
    fc1 = torch.empty((T * K_TOP, 2 * F), dtype=torch.float32, device="cuda")
    out_b, ws_b = _call(d, w1q, w2q, fc1_debug=fc1)
    lay = nv.moe_workspace_layout(T, H, F, E, K_TOP)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16)), "outputs differ"
    lo, hi = lay["err"], lay["total"]
    diff = (ws_a[lo:hi] != ws_b[lo:hi]).nonzero()
    assert diff.numel() == 0, f"workspace differs at {diff.numel()} bytes, first offset {int(diff[0]) + lo}"


@pytest.mark.parametrize("name,n_tok", [("moe_8k", 768), ("moe_32k", 512)])
def test_end_to_end_against_the_oracle_chain(name, n_tok):
    d = getattr(workloads, name)()
    T, H = d["x"].shape
    w1q, w2q = _weights(d)
    out, ws = _call(d, w1q, w2q)
    lay = nv.moe_workspace_layout(T, H, F, E, K_TOP)
    assert int(ws[lay["err"]:lay["err"] + 4].view(torch.int32)[0]) == 0
    toks = np.sort(np.random.default_rng(7).choice(T, n_tok, replace=False))
    w1o = [oracle.quantize(d["w1"][e], per_tensor=True) for e in range(E)]
    w2o = [oracle.quantize(d["w2"][e], per_tensor=True) for e in range(E)]
    ref = oracle.moe_forward(d["x"], d["logits"], d["bias"], w1o, w2o, K_TOP, rows=toks, with_abs=True)
    g = oracle.bf16_to_f64(bf16_bits(out)[toks])
    r = oracle.bf16_to_f64(ref["out"])
    rel = np.linalg.norm(g - r) / np.linalg.norm(r)
    # the GEMM tolerance of each slot's Y2 element (1 bf16 ulp + 1e-5 sum_k |a_k b_k|),
    # weighted by the router weight and summed over the slots, plus 1 bf16 ulp of the combine
    at = np.full(T * K_TOP, -1, np.int64)
    at[ref["rows_computed"]] = np.arange(len(ref["rows_computed"]))
    slot_rows = at[ref["meta"]["inv"].reshape(T, K_TOP)[toks]]
    wts = ref["w"][toks]
    y2, y2a = ref["y2"][slot_rows], ref["y2_abs"][slot_rows]  # [n_tok, k, H]
    tol = oracle.bf16_ulp(np.maximum(np.abs(g), np.abs(r))) + np.einsum(
        "tk,tkh->th", np.abs(wts), oracle.bf16_ulp(y2) + 1e-5 * y2a)
    within = float(np.mean(np.abs(g - r) <= tol))
    rows = ref["rows_computed"]
    n = R = T * K_TOP
    q2_dev = ws[lay["a2_codes"]:lay["a2_codes"] + R * F // 2].view(R, F // 2)[torch.from_numpy(rows).cuda()]
    qd = q2_dev.cpu().numpy()
    qo = ref["q2_codes"]
    mism = float(np.mean(np.concatenate([(qd & 15) != (qo & 15), (qd >> 4) != (qo >> 4)])))
    rows_flipped = float(np.mean((qd != qo).any(axis=1)))
    print(f"\n{name}: {n_tok} tokens, rel-L2 {rel:.3e}, within tolerance {within:.5%}, "
          f"q2 code mismatch rate {mism:.3e} ({rows_flipped:.3%} of {len(rows)} rows with a flip)")
    assert rel <= 1e-3, rel
    assert within >= 0.999, within


def test_graph_replay_is_bit_identical_to_the_eager_call():
    """The layer captured once into a CUDA graph and replayed (how bench.py
    times the step, and how a serving loop of fixed shape would run it): same
    bits as the eager call, on two replays with different inputs copied into
    the captured buffers in between."""
    rng = np.random.default_rng(21)
    T, E_, k, H, F_ = 700, 64, 8, 512, 256
    w1q = nv.quantize_grouped_weights(to_dev_bf16(workloads.gaussian_bf16(rng, (E_, 2 * F_, H), std=0.02)))
    w2q = nv.quantize_grouped_weights(to_dev_bf16(workloads.gaussian_bf16(rng, (E_, H, F_), std=0.02)))
    x = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    lg = torch.empty((T, E_), dtype=torch.float32, device="cuda")
    bs = torch.empty((E_,), dtype=torch.float32, device="cuda")
    ws = torch.zeros(int(nv.lib().moe_expert_workspace(T, H, F_, E_, k)), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")

    def fill(seed):
        r = np.random.default_rng(seed)
        x.copy_(to_dev_bf16(workloads.gaussian_bf16(r, (T, H))))
        lg.copy_(torch.from_numpy(r.standard_normal((T, E_), dtype=np.float32)))
        bs.copy_(torch.from_numpy(r.standard_normal(E_, dtype=np.float32)))

    fill(1)
    nv.moe_expert_forward(x, lg, bs, w1q, w2q, F_, k, out=out, ws=ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        nv.moe_expert_forward(x, lg, bs, w1q, w2q, F_, k, out=out, ws=ws)
    torch.cuda.current_stream().wait_stream(side)
    for seed in (2, 3):
        fill(seed)
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        ref, _ = nv.moe_expert_forward(x, lg, bs, w1q, w2q, F_, k)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"replay with inputs {seed}"
