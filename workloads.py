"""Seeded synthetic inputs shared by the tests, bench.py and the oracle.

This module only draws random numbers and rounds them to bf16 (through
torch's CPU cast, round to nearest even); it holds none of the quantization,
routing or GEMM arithmetic.  bf16 tensors are returned as uint16 bit
patterns (numpy), the form both the oracle and the CUDA binding accept.

The shapes follow the pages' Qwen3-30B-A3B workload (hidden 2048, 128
experts, top-8, expert FFN width 768, 32 query + 4 KV heads of dim 128):
there are no real activations, weights or DAPO text here, so Gaussian draws
stand in for them.  Each tensor has its own child stream of the config's
seed (numpy SeedSequence.spawn), so adding a tensor never shifts another.
"""
import concurrent.futures as cf
import os

import numpy as np
import torch

HIDDEN = 2048
EXPERTS = 128
TOPK = 8
FFN = 768


def to_bf16_bits(a):
    """float32 numpy array -> bf16 bit patterns (uint16), RNE via torch."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _streams(seed, n):
    """n independent child seed sequences of `seed` (one per tensor)."""
    return list(np.random.SeedSequence(seed).spawn(n))


def _draw(rng, shape, std, outlier_frac, outlier_mult, zero_row_frac):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if outlier_frac > 0:
        x[rng.random(shape) < outlier_frac] *= np.float32(outlier_mult)
    if zero_row_frac > 0:
        rows = x.reshape(-1, shape[-1])
        rows[rng.random(rows.shape[0]) < zero_row_frac] = 0.0
    return to_bf16_bits(x)


def gaussian_bf16(src, shape, std=1.0, outlier_frac=0.0, outlier_mult=50.0, zero_row_frac=0.0):
    """bf16 bit patterns of N(0, std^2) draws; a fraction of entries scaled by
    outlier_mult and a fraction of rows (last axis) set to zero.

    src is a numpy Generator (drawn in one piece) or a SeedSequence: then the
    leading axis is cut into chunks of about 4M elements, each drawn from its
    own child sequence in a thread pool (numpy releases the GIL while
    filling), so the values do not depend on the thread count."""
    if isinstance(src, np.random.Generator):
        return _draw(src, shape, std, outlier_frac, outlier_mult, zero_row_frac)
    shape = tuple(shape)
    per_lead = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    step = max(1, (1 << 22) // per_lead)
    starts = list(range(0, shape[0], step))
    seqs = src.spawn(len(starts))
    out = np.empty(shape, np.uint16)

    def one(i):
        lo = starts[i]
        hi = min(shape[0], lo + step)
        out[lo:hi] = _draw(np.random.default_rng(seqs[i]), (hi - lo,) + shape[1:], std,
                           outlier_frac, outlier_mult, zero_row_frac)

    with cf.ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(one, range(len(starts))))
    return out


def linear_small(seed=0):
    """Single W4A4 linear: X [64 x 256] ~N(0,1), W stored [K=256 x N=512]
    ~N(0, 0.02^2) and handed to the GEMM K-major as [512 x 256]."""
    rx, rw = _streams(seed, 2)
    x = gaussian_bf16(rx, (64, 256))
    w_kn = np.random.default_rng(rw).standard_normal((256, 512), dtype=np.float32) * np.float32(0.02)
    w = to_bf16_bits(np.ascontiguousarray(w_kn.T))
    return dict(x=x, w=w)


def quant_rows(seed=1, rows=16384, cols=2048):
    """Per-token quantization workload: ~N(0,1), 1% of entries x50, 2% of rows zero."""
    (r,) = _streams(seed, 1)
    return dict(x=gaussian_bf16(r, (rows, cols), outlier_frac=0.01, zero_row_frac=0.02))


def moe_layer(seed, tokens, bias_std, hidden=HIDDEN, experts=EXPERTS, ffn=FFN,
              with_weights=True):
    """MoE expert layer inputs: X [T x H] ~N(0,1), router logits [T x E]
    ~N(0,1) fp32, per-expert bias ~N(0, bias_std^2) fp32, W1 [E x 2F x H]
    (gate rows then up rows) and W2 [E x H x F] ~N(0, 0.02^2)."""
    rx, rl, rb, r1, r2 = _streams(seed, 5)
    out = dict(
        x=gaussian_bf16(rx, (tokens, hidden)),
        logits=np.random.default_rng(rl).standard_normal((tokens, experts), dtype=np.float32),
        bias=(np.random.default_rng(rb).standard_normal(experts, dtype=np.float32) * np.float32(bias_std)),
    )
    if with_weights:
        out["w1"] = gaussian_bf16(r1, (experts, 2 * ffn, hidden), std=0.02)
        out["w2"] = gaussian_bf16(r2, (experts, hidden, ffn), std=0.02)
    return out


def moe_8k(seed=2, **kw):
    return moe_layer(seed, 8192, 1.0, **kw)


def moe_32k(seed=3, **kw):
    return moe_layer(seed, 32768, 2.0, **kw)


def attn_proj(seed=4, tokens=32768):
    """Dense attention projections: X [T x 2048] and O [T x 4096] ~N(0,1) with
    1% x50 outliers; Wqkv [5120 x 2048], Wo [2048 x 4096] ~N(0, 0.02^2)."""
    rx, ro, rq, rw = _streams(seed, 4)
    return dict(
        x=gaussian_bf16(rx, (tokens, 2048), outlier_frac=0.01),
        o=gaussian_bf16(ro, (tokens, 4096), outlier_frac=0.01),
        wqkv=gaussian_bf16(rq, (5120, 2048), std=0.02),
        wo=gaussian_bf16(rw, (2048, 4096), std=0.02),
    )
