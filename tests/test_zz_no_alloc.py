"""moe_expert_forward_noalloc: the expert layer for callers that must not
allocate device memory (a plugin given only its input and output buffers,
or a step where cudaMalloc would synchronize the device).  Its workspace is
a fixed array inside the library, so the checks here are that it gives the
same output as moe_expert_forward with a caller workspace, twice in a row on
different inputs (the array keeps the previous call's contents), and that it
refuses layers too large for the array.  Named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import nvfp4_quantized_moe_token_gb300 as nv
import oracle
import workloads
from tests.helpers import bf16_bits, to_dev_bf16

T, E, K, H, F = 200, 128, 8, 2048, 768  # about 14 MiB of workspace, inside the 32 MiB array


def _lib():
    L = nv.lib()
    f = L.moe_expert_forward_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int, ctypes.POINTER(nv._Tensor), ctypes.POINTER(nv._Tensor),
                  ctypes.c_int64, ctypes.POINTER(nv._Options), ctypes.c_void_p, ctypes.c_void_p]
    return L


def _noalloc(L, x, logits, bias, w1q, w2q, out):
    a, b = w1q.c(), w2q.c()
    opt = nv._Options(0)
    rc = L.moe_expert_forward_noalloc(x.data_ptr(), T, H, logits.data_ptr(), bias.data_ptr(), E, K,
                                      ctypes.byref(a), ctypes.byref(b), F, ctypes.byref(opt), out.data_ptr(),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, L.nvfp4_last_error().decode()


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_on_two_calls_in_a_row():
    L = _lib()
    rng = np.random.default_rng(17)
    w1 = workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02)
    w2 = workloads.gaussian_bf16(rng, (E, H, F), std=0.02)
    w1q = nv.quantize_grouped_weights(to_dev_bf16(w1))
    w2q = nv.quantize_grouped_weights(to_dev_bf16(w2))
    for call in range(2):  # different inputs each call: nothing stale may leak through the shared array
        x = to_dev_bf16(workloads.gaussian_bf16(rng, (T, H)))
        logits = torch.from_numpy(rng.standard_normal((T, E), dtype=np.float32)).cuda()
        bias = torch.from_numpy(rng.standard_normal(E, dtype=np.float32) * np.float32(2.0)).cuda()
        ref, _ = nv.moe_expert_forward(x, logits, bias, w1q, w2q, F, K)
        out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        _noalloc(L, x, logits, bias, w1q, w2q, out)
        torch.cuda.synchronize()
        g = oracle.bf16_to_f64(bf16_bits(out))
        r = oracle.bf16_to_f64(bf16_bits(ref))
        assert np.all(np.isfinite(g)), f"call {call}: output not written"
        # the tolerance of the combine parity tests: one bf16 ulp (same kernels, so in fact bitwise)
        assert np.all(np.abs(g - r) <= oracle.bf16_ulp(np.maximum(np.abs(g), np.abs(r)))), f"call {call}"


def test_noalloc_rejects_layers_beyond_the_array():
    """Refused on the host before any CUDA call (runs without a GPU)."""
    L = _lib()
    w1 = nv._Tensor(4096, 4096, 4096, E * 2 * F, H)
    w2 = nv._Tensor(4096, 4096, 4096, E * H, F)
    opt = nv._Options(0)
    rc = L.moe_expert_forward_noalloc(4096, 32768, H, 4096, None, E, K, ctypes.byref(w1), ctypes.byref(w2), F,
                                      ctypes.byref(opt), 4096, None)
    assert rc == -4
    assert "scratch" in L.nvfp4_last_error().decode()


def test_noalloc_boundary_is_516_tokens_at_the_qwen3_shape():
    """The documented limit, pinned: 516 tokens fit the 32 MiB array at hidden
    2048, FFN 768, 128 experts, top-8, and 517 are refused on the host."""
    L = _lib()
    limit = 32 << 20
    assert L.moe_expert_workspace(516, H, F, E, K) <= limit < L.moe_expert_workspace(517, H, F, E, K)
    w1 = nv._Tensor(4096, 4096, 4096, E * 2 * F, H)
    w2 = nv._Tensor(4096, 4096, 4096, E * H, F)
    opt = nv._Options(0)
    rc = L.moe_expert_forward_noalloc(4096, 517, H, 4096, None, E, K, ctypes.byref(w1), ctypes.byref(w2), F,
                                      ctypes.byref(opt), 4096, None)
    assert rc == -4
    assert "scratch" in L.nvfp4_last_error().decode()


class _DevWord:
    """A uint32 at a raw device address, for torch.as_tensor (CUDA array interface)."""

    def __init__(self, ptr):
        self.__cuda_array_interface__ = {"shape": (1,), "typestr": "<u4", "data": (ptr, False), "version": 3}


@pytest.mark.gpu
def test_noalloc_error_word_is_the_calls_own_and_clear_after_a_good_call():
    """moe_noalloc_error_word gives the device address of the word the
    no-alloc call clears and its kernels set: poisoned before a good call,
    it reads zero after it."""
    L = _lib()
    f = L.moe_noalloc_error_word
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
    assert f(None) == -1  # NVFP4_EINVAL for a null out
    ptr = ctypes.c_void_p()
    assert f(ctypes.byref(ptr)) == 0 and ptr.value
    word = torch.as_tensor(_DevWord(ptr.value), device="cuda")
    word.fill_(0x7FFFFFFF)
    torch.cuda.synchronize()
    rng = np.random.default_rng(23)
    w1q = nv.quantize_grouped_weights(to_dev_bf16(workloads.gaussian_bf16(rng, (E, 2 * F, H), std=0.02)))
    w2q = nv.quantize_grouped_weights(to_dev_bf16(workloads.gaussian_bf16(rng, (E, H, F), std=0.02)))
    x = to_dev_bf16(workloads.gaussian_bf16(rng, (T, H)))
    logits = torch.from_numpy(rng.standard_normal((T, E), dtype=np.float32)).cuda()
    bias = torch.zeros(E, dtype=torch.float32, device="cuda")
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    _noalloc(L, x, logits, bias, w1q, w2q, out)
    torch.cuda.synchronize()
    assert int(word.item()) == 0
    ptr2 = ctypes.c_void_p()
    assert f(ctypes.byref(ptr2)) == 0 and ptr2.value == ptr.value  # one address for the process
