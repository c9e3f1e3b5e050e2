"""Failure detection on the GPU without a fault.  moe_debug.stall_fc1 makes
FC1's MMA-issuing thread wait on a barrier that nothing arrives at, so its
bounded wait runs out.  The kernel must then record NVFP4_DEVERR_TIMEOUT in
the workspace's error word and return: every other role of both CTAs of each
pair sees the abort flag, the producers wait (bounded) for their copies in
flight, the pair meets at its cluster barrier and frees its tensor memory.
Nothing traps and nothing hangs, and the context stays usable: the next call
on the same workspace gives the same bits as a call made before the stall."""
import time

import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import workloads
from tests.helpers import bf16_bits, to_dev_bf16

pytestmark = pytest.mark.gpu

T, E, K, H, F = 256, 128, 8, 2048, 768


def test_fc1_wait_time_out_is_reported_and_the_context_survives():
    rng = np.random.default_rng(29)
    x = to_dev_bf16(workloads.gaussian_bf16(rng, (T, H)))
    logits = torch.from_numpy(rng.standard_normal((T, E), dtype=np.float32)).cuda()
    bias = torch.from_numpy(rng.standard_normal(E, dtype=np.float32)).cuda()
    w1q = nv.quantize_grouped_weights(to_dev_bf16(workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02)))
    w2q = nv.quantize_grouped_weights(to_dev_bf16(workloads.gaussian_bf16(rng, (E, H, F), std=0.02)))
    lay = nv.moe_workspace_layout(T, H, F, E, K)
    ws = torch.zeros(lay["total"], dtype=torch.uint8, device="cuda")
    err = ws[lay["err"]:lay["err"] + 4]

    def err_word():
        torch.cuda.synchronize()
        return int(err.cpu().numpy().view(np.uint32)[0])

    ref, _ = nv.moe_expert_forward(x, logits, bias, w1q, w2q, F, K, ws=ws)
    ref_bits = bf16_bits(ref)
    assert err_word() == 0

    t0 = time.monotonic()
    nv.moe_expert_forward(x, logits, bias, w1q, w2q, F, K, ws=ws, debug_stall_fc1=True)
    word = err_word()
    took = time.monotonic() - t0
    assert word & nv.DEVERR_TIMEOUT, f"error word {word:#x}: the time-out was not reported"
    assert not word & nv.DEVERR_BADEXPERT
    assert took < 60, f"the stalled layer took {took:.1f} s to return"

    # the context is intact: same workspace, same inputs, same bits as before the stall
    err.zero_()
    again, _ = nv.moe_expert_forward(x, logits, bias, w1q, w2q, F, K, ws=ws)
    assert err_word() == 0
    assert np.array_equal(bf16_bits(again), ref_bits)
