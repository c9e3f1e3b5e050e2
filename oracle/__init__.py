"""CPU oracle for the per-token NVFP4 W4A4 forward path (test infrastructure).

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and the
cpu_baseline / reference leg of bench.py are the only callers.  It shares no
code with the CUDA library and never calls it.

The bit-level steps (E2M1/E4M3 encoding, per-token and per-tensor
quantization, scale-factor layout, routing, metadata, SwiGLU, combine) are the
plain C in nvfp4_oracle.c; this module marshals numpy arrays into it and
does the fp64 contractions with numpy's matmul (a library primitive: the sum
of products of the dequantized operands, nothing fused or reordered beyond
what a dot product is).

Sources, by page title and section:
  "miniTE Technical Report" 2.2 (decode x^ = q s_b s_g), 2.3 (per-token
  scaling domain, rel-L2 / SNR / MAE), 5.1 (per-row outer scale), 5.2
  (contiguous buffers, expert offsets), 5.3 (amax reuse, weighted SwiGLU +
  row amax), 5.4 (GEMM epilogue: ACC x alpha_a[m] x alpha_b, C = gate | up,
  D = act(gate, up)), 5.6 (gs = gamax / 2688, zero rows).
  "The 4-bitter Lesson": baseline recipe (per-token activations, per-tensor
  weights), Four-Over-Six (E2M1 grid).
"""
import ctypes
import numpy as np

from . import build as _build

_LIB = None

i64 = ctypes.c_int64
i32 = ctypes.c_int
u8p = ctypes.POINTER(ctypes.c_uint8)
u16p = ctypes.POINTER(ctypes.c_uint16)
i32p = ctypes.POINTER(ctypes.c_int32)
i64p = ctypes.POINTER(ctypes.c_int64)
f32p = ctypes.POINTER(ctypes.c_float)
f64p = ctypes.POINTER(ctypes.c_double)


def lib():
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(_build.build())
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_float]
        L.orc_bf16_from_f64.restype = ctypes.c_uint16
        L.orc_bf16_from_f64.argtypes = [ctypes.c_double]
        L.orc_bf16_from_f64_array.argtypes = [f64p, i64, u16p]
        L.orc_quantize.argtypes = [u16p, i64, i64, i64, i32, f32p, u8p, u8p, f32p]
        L.orc_quantize_46.argtypes = [u16p, i64, i64, i64, i32, f32p, i32, u8p, u8p, f32p, u8p]
        L.orc_dequantize.argtypes = [u8p, u8p, f32p, i64, i64, i32, f64p]
        L.orc_sf_offset.restype = i64
        L.orc_sf_offset.argtypes = [i64, i64, i64]
        L.orc_sf_bytes.restype = i64
        L.orc_sf_bytes.argtypes = [i64, i64]
        L.orc_sf_swizzle.argtypes = [u8p, i64, i64, i64p, i64, u8p]
        L.orc_sf_unswizzle.argtypes = [u8p, i64, i64, i64p, u8p]
        L.orc_route.argtypes = [f32p, f32p, i64, i32, i32, i32p, f64p, f32p]
        L.orc_route_metadata.argtypes = [i32p, i64, i32, i32, i32p, i32p, i32p, i32p, i32p]
        L.orc_swiglu.argtypes = [f64p, i64, i64, f64p, u16p, f32p]
        L.orc_combine.argtypes = [f64p, i64, i32p, f64p, i64, i32, u16p]
        _LIB = L
    return _LIB


def _p(a, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats

def e2m1_decode(code):
    return lib().orc_e2m1_decode(int(code))


def e4m3_decode(byte):
    return lib().orc_e4m3_decode(int(byte))


def e4m3_encode(u):
    return int(lib().orc_e4m3_encode(float(u)))


def e2m1_encode(v):
    return int(lib().orc_e2m1_encode(float(v)))


def bf16_round(x):
    """fp64 array -> bf16 bit patterns (uint16), round to nearest even."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_from_f64_array(_p(x, f64p), x.size, _p(out, u16p))
    return out


def bf16_to_f64(h):
    """bf16 bit patterns (uint16) -> fp64 values (exact)."""
    h = np.asarray(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(y):
    """Spacing of bf16 numbers at |y|: the gap from the bf16 binade holding |y|
    to its next value, 2^(floor(log2|y|) - 7), and the subnormal spacing 2^-133
    below 2^-126 (zero included).  floor(log2|y|) is read exactly off frexp."""
    a = np.abs(np.asarray(y, np.float64))
    _, ex = np.frexp(a)  # a = m 2^ex, 0.5 <= m < 1, so floor(log2 a) = ex - 1 (a > 0)
    e = np.where(a > 0, ex.astype(np.float64) - 1.0, -126.0)
    e = np.maximum(e, -126.0)
    return np.exp2(e - 7.0)


# ---------------------------------------------------------------- quantization

def quantize(x_bf16, per_tensor=False, amax_in=None):
    """x_bf16: uint16 [rows, cols] bf16 bit patterns.

    Returns (codes uint8 [rows, cols/2], sf_lin uint8 [rows, cols/16],
    scale float32 [rows] or [1])."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    assert cols % 16 == 0
    codes = np.empty((rows, cols // 2), np.uint8)
    sf = np.empty((rows, cols // 16), np.uint8)
    scale = np.empty(1 if per_tensor else rows, np.float32)
    am = None
    if amax_in is not None:
        am = _c(amax_in, np.float32).reshape(-1)
    lib().orc_quantize(_p(x, u16p), rows, cols, cols, int(per_tensor),
                       _p(am, f32p) if am is not None else None,
                       _p(codes, u8p), _p(sf, u8p), _p(scale, f32p))
    return codes, sf, scale


def quantize_46(x_bf16, err="mse", per_tensor=False, amax_in=None, with_choice=False):
    """Four-over-six quantization (see orc_quantize_46): err 'mse' or 'mae'.

    Returns (codes, sf_lin, scale) like quantize, plus the per-block choice
    uint8 [rows, cols/16] (4 or 6) when with_choice."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    assert cols % 16 == 0
    kind = {"mse": 1, "mae": 2}[err]
    codes = np.empty((rows, cols // 2), np.uint8)
    sf = np.empty((rows, cols // 16), np.uint8)
    scale = np.empty(1 if per_tensor else rows, np.float32)
    choice = np.empty((rows, cols // 16), np.uint8)
    am = None
    if amax_in is not None:
        am = _c(amax_in, np.float32).reshape(-1)
    lib().orc_quantize_46(_p(x, u16p), rows, cols, cols, int(per_tensor),
                          _p(am, f32p) if am is not None else None, kind,
                          _p(codes, u8p), _p(sf, u8p), _p(scale, f32p), _p(choice, u8p))
    if with_choice:
        return codes, sf, scale, choice
    return codes, sf, scale


def dequantize(codes, sf_lin, scale, per_tensor=False):
    codes = _c(codes, np.uint8)
    sf = _c(sf_lin, np.uint8)
    scale = _c(scale, np.float32).reshape(-1)
    rows, half = codes.shape
    out = np.empty((rows, half * 2), np.float64)
    lib().orc_dequantize(_p(codes, u8p), _p(sf, u8p), _p(scale, f32p), rows, half * 2,
                         int(per_tensor), _p(out, f64p))
    return out


def dequantize_bf16(codes, sf_lin, scale, per_tensor=False):
    """DQ(Q(x)): the BF16-dequantized value of the exact quantized tensor, the
    operand of the dequantized backward ("Per-token NVFP4 and Dequantized
    Backward", Improving Gradient Stability).  The exact value q s_b s_g
    (decode of "miniTE Technical Report" 2.2; at most 30 significant bits, so
    exact in fp64) rounded once to bf16, nearest even.  Returns uint16 bits."""
    return bf16_round(dequantize(codes, sf_lin, scale, per_tensor))


def sf_offset(r, c, sf_cols):
    return int(lib().orc_sf_offset(int(r), int(c), int(sf_cols)))


def sf_bytes(rows, sf_cols):
    return int(lib().orc_sf_bytes(int(rows), int(sf_cols)))


def sf_swizzle(sf_lin, row_map=None, dst_rows=None):
    sf = _c(sf_lin, np.uint8)
    rows, sc = sf.shape
    if dst_rows is None:
        dst_rows = rows
    rm = None if row_map is None else _c(row_map, np.int64)
    out = np.empty(sf_bytes(dst_rows, sc), np.uint8)
    lib().orc_sf_swizzle(_p(sf, u8p), rows, sc, _p(rm, i64p) if rm is not None else None,
                         dst_rows, _p(out, u8p))
    return out


def sf_unswizzle(sw, rows, sf_cols, row_map=None):
    sw = _c(sw, np.uint8).reshape(-1)
    rm = None if row_map is None else _c(row_map, np.int64)
    out = np.empty((rows, sf_cols), np.uint8)
    lib().orc_sf_unswizzle(_p(sw, u8p), rows, sf_cols, _p(rm, i64p) if rm is not None else None,
                           _p(out, u8p))
    return out


# ---------------------------------------------------------------- GEMM

def gemm_f64(a_deq, b_deq):
    """Y = A . B^T in fp64 on dequantized operands (A [M,K], B [N,K])."""
    return np.asarray(a_deq, np.float64) @ np.asarray(b_deq, np.float64).T


def linear(xq, wq):
    """Dense W4A4 linear: Y = bf16( deq(X) . deq(W)^T ), X per-token, W per-tensor.

    xq = (codes, sf_lin, scale[rows]); wq = (codes, sf_lin, scale[1])."""
    a = dequantize(*xq, per_tensor=False)
    b = dequantize(*wq, per_tensor=True)
    return bf16_round(gemm_f64(a, b))


def abs_product_sum(a_deq, b_deq):
    """sum_k |a_k b_k| for every output element (the tolerance term)."""
    return np.abs(np.asarray(a_deq, np.float64)) @ np.abs(np.asarray(b_deq, np.float64)).T


# ---------------------------------------------------------------- routing

def route(logits, bias, k):
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().orc_route(_p(logits, f32p), _p(bias, f32p), T, E, k, _p(ids, i32p), _p(w, f64p), None)
    return ids, w


def route_metadata(ids, E):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    cnt = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    poff = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    lib().orc_route_metadata(_p(ids, i32p), T, E, k, _p(cnt, i32p), _p(off, i32p),
                             _p(poff, i32p), _p(perm, i32p), _p(inv, i32p))
    return dict(cnt=cnt, off=off, poff=poff, perm=perm, inv=inv)


def expert_of_rows(off):
    """Expert index of each permuted row, from the offsets."""
    off = np.asarray(off, np.int64)
    return np.repeat(np.arange(len(off) - 1), np.diff(off))


def padded_rows(meta):
    """Destination scale-factor row of each permuted row: poff[e] + (r - off[e])."""
    off = meta["off"].astype(np.int64)
    poff = meta["poff"].astype(np.int64)
    e = expert_of_rows(off)
    r = np.arange(off[-1], dtype=np.int64)
    return poff[e] + (r - off[e])


def permute(xq, meta, k):
    """Gather the per-token quantized rows into expert order.

    Returns (codes [R, K/2], sf_lin [R, K/16], scale [R]); the swizzled
    per-expert-padded scale buffer is sf_swizzle(sf_lin, padded_rows(meta),
    meta['poff'][-1])."""
    codes, sf, scale = xq
    tok = meta["perm"].astype(np.int64) // k
    return codes[tok], sf[tok], scale[tok]


# ---------------------------------------------------------------- MoE pieces

def swiglu(c, prob=None):
    """c: fp64 [rows, 2F] = gate | up.  Returns (D bf16 [rows, F], amax fp32 [rows])."""
    c = _c(c, np.float64)
    rows, two_f = c.shape
    F = two_f // 2
    d = np.empty((rows, F), np.uint16)
    amax = np.empty(rows, np.float32)
    pr = None if prob is None else _c(prob, np.float64)
    lib().orc_swiglu(_p(c, f64p), rows, F, _p(pr, f64p) if pr is not None else None,
                     _p(d, u16p), _p(amax, f32p))
    return d, amax


def combine(y, inv, w):
    """y: fp64 [R, H]; inv int32 [T*k]; w fp64 [T, k] -> bf16 [T, H]."""
    y = _c(y, np.float64)
    w = _c(w, np.float64)
    inv = _c(inv, np.int32)
    T, k = w.shape
    H = y.shape[1]
    out = np.empty((T, H), np.uint16)
    lib().orc_combine(_p(y, f64p), H, _p(inv, i32p), _p(w, f64p), T, k, _p(out, u16p))
    return out


def moe_forward(x_bf16, logits, bias, w1q, w2q, k, rows=None, w_deq=None, with_abs=False):
    """Whole expert layer on the CPU, each stage from the previous oracle stage.

    w1q / w2q: lists over experts of (codes, sf_lin, scale[1]) per-tensor
    quantized weights, W1_e [2F, H] = gate | up, W2_e [H, F].
    rows (nullable): restrict the output to these token indices (the router,
    metadata and every expert GEMM row needed by them are still computed).
    w_deq (nullable): (list of dequantize(w1q[e]), list of dequantize(w2q[e]))
    computed once for static weights.
    with_abs: also return sum_k |a_k b_k| of FC2 for every computed element
    (the term of the GEMM tolerance).
    Returns a dict of every intermediate; the per-row ones (D, amax2,
    q2_codes, y2, y2_abs) hold the computed expert-ordered rows `rows_computed`
    (all R rows when rows is None), in that order."""
    E = len(w1q)
    ids, w = route(logits, bias, k)
    meta = route_metadata(ids, E)
    xq = quantize(x_bf16)
    a1 = permute(xq, meta, k)
    off = meta["off"]
    R = int(off[-1])
    F = w2q[0][0].shape[1] * 2
    H = w1q[0][0].shape[1] * 2
    inv_tk = meta["inv"].reshape(-1, k)
    if rows is None:
        need = np.arange(R, dtype=np.int64)
    else:
        need = np.unique(inv_tk[np.asarray(rows)].reshape(-1)).astype(np.int64)
    at = np.full(R, -1, np.int64)  # position of an expert-ordered row among the computed ones
    at[need] = np.arange(len(need))
    n = len(need)
    y2 = np.zeros((n, H), np.float64)
    y2_abs = np.zeros((n, H), np.float64) if with_abs else None
    d_all = np.zeros((n, F), np.uint16)
    amax2 = np.zeros(n, np.float32)
    q2_codes = np.zeros((n, F // 2), np.uint8)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        sel = need[(need >= lo) & (need < hi)]
        if len(sel) == 0:
            continue
        idx = at[sel]
        b1 = w_deq[0][e] if w_deq is not None else dequantize(*w1q[e], per_tensor=True)
        b2 = w_deq[1][e] if w_deq is not None else dequantize(*w2q[e], per_tensor=True)
        a = dequantize(a1[0][sel], a1[1][sel], a1[2][sel])
        c = gemm_f64(a, b1)
        d, am = swiglu(c)
        d_all[idx] = d
        amax2[idx] = am
        q2 = quantize(d, amax_in=am)
        q2_codes[idx] = q2[0]
        a2 = dequantize(*q2)
        y2[idx] = bf16_to_f64(bf16_round(gemm_f64(a2, b2)))
        if with_abs:
            y2_abs[idx] = abs_product_sum(a2, b2)
    if rows is None:
        out = combine(y2, meta["inv"], w)
    else:
        rows = np.asarray(rows)
        out = combine(y2, at[inv_tk[rows].reshape(-1)].astype(np.int32), w[rows])
    return dict(ids=ids, w=w, meta=meta, xq=xq, a1=a1, rows_computed=need, D=d_all, amax2=amax2,
                q2_codes=q2_codes, y2=y2, y2_abs=y2_abs, out=out)


# ---------------------------------------------------------------- dequantized backward GEMMs

def _groups(rows, poff):
    if poff is None:
        return [(0, rows)]
    poff = np.asarray(poff, np.int64)
    return [(int(poff[g]), int(poff[g + 1])) for g in range(len(poff) - 1)]


def grouped_dgrad(dy_bf16, w_bf16, poff=None):
    """dgrad of the dequantized backward ("Per-token NVFP4 and Dequantized
    Backward", Improving Gradient Stability: BF16 backward on DQ(Q(w))): for
    each row group g, dx[rows of g] = dy[rows of g] . w_g, in fp64 on the bf16
    operands (each product exact).  dy bf16 bits [rows, nf], w bf16 bits
    [G, nf, kf]; poff [G + 1] row offsets (None: one group).  Returns (dx fp64
    [rows, kf], sum_n |dy w| per element)."""
    dy = bf16_to_f64(dy_bf16)
    w = bf16_to_f64(w_bf16)
    dx = np.zeros((dy.shape[0], w.shape[2]))
    ab = np.zeros_like(dx)
    for g, (lo, hi) in enumerate(_groups(dy.shape[0], poff)):
        dx[lo:hi] = dy[lo:hi] @ w[g]
        ab[lo:hi] = np.abs(dy[lo:hi]) @ np.abs(w[g])
    return dx, ab


def grouped_wgrad(dy_bf16, x_bf16, poff=None, groups=None):
    """wgrad of the dequantized backward: for each row group g, dw_g =
    dy[rows of g]^T . x[rows of g] in fp64 on the bf16 operands (x = DQ(Q(x))).
    dy bf16 bits [rows, nf], x bf16 bits [rows, kf].  Returns (dw fp64
    [G, nf, kf], sum_r |dy x| per element); a group with no rows gives zero."""
    dy = bf16_to_f64(dy_bf16)
    x = bf16_to_f64(x_bf16)
    gr = _groups(dy.shape[0], poff)
    dw = np.zeros((len(gr), dy.shape[1], x.shape[1]))
    ab = np.zeros_like(dw)
    for g, (lo, hi) in enumerate(gr):
        dw[g] = dy[lo:hi].T @ x[lo:hi]
        ab[g] = np.abs(dy[lo:hi]).T @ np.abs(x[lo:hi])
    return dw, ab


# ---------------------------------------------------------------- single-pass FC2 (a research direction)

def fc2_single_pass(d_bf16, w2q_e, k_tile=128):
    """FC2 of one expert with online amax compensation ("miniTE Technical
    Report" 5.6, Exploring Single-Pass Fusion), in the pages' order: for each
    K-tile i of D (the FC1 slice that completes first), the running row amax
    gamax = max(gamax, max |P_i|); rows with gamax = 0 contribute nothing
    yet; gs = gamax / 2688; the tile's E4M3 block scales and E2M1 codes are
    generated with gs (the plain per-token rule with amax = gamax); dO_i is
    the block-scaled product (block scales included, gs and the weight's
    outer scale excluded); O = O * (gs_prev / gs) + dO_i; gs_prev = gs.  At
    the end Y = O * gs_prev * gs_W2 (all-zero rows give zero).

    d_bf16: uint16 [rows, F] (bf16 bits of SwiGLU's output); w2q_e: (codes,
    sf_lin, scale[1]) of W2_e [H, F].  Returns dict(y (bf16 bits [rows, H]),
    y_f64 (before rounding), codes, sf (the tiles' codes and block scales side
    by side, [rows, F/2] and [rows, F/16]), gs_tiles [rows, F/k_tile])."""
    d = _c(d_bf16, np.uint16)
    rows, F = d.shape
    assert F % k_tile == 0 and k_tile % 16 == 0
    codes_w, sf_w, gs_w = w2q_e
    b_bs = dequantize(codes_w, sf_w, np.ones(1, np.float32), per_tensor=True)  # q_w s_bw, gs_W2 excluded
    H = b_bs.shape[0]
    n_t = F // k_tile
    gamax = np.zeros(rows, np.float32)
    gs_prev = np.zeros(rows, np.float64)
    o = np.zeros((rows, H), np.float64)
    codes = np.zeros((rows, F // 2), np.uint8)
    sf = np.zeros((rows, F // 16), np.uint8)
    gs_tiles = np.zeros((rows, n_t), np.float32)
    for i in range(n_t):
        cols = slice(i * k_tile, (i + 1) * k_tile)
        p = np.ascontiguousarray(d[:, cols])
        rowmax = np.abs(bf16_to_f64(p)).max(axis=1).astype(np.float32)
        gamax = np.maximum(gamax, rowmax)
        live = gamax > 0
        q_c, q_sf, gs = quantize(p, amax_in=gamax)  # gs = gamax / 2688 in fp32, as the per-token rule
        codes[:, i * k_tile // 2:(i + 1) * k_tile // 2] = q_c
        sf[:, i * k_tile // 16:(i + 1) * k_tile // 16] = q_sf
        gs_tiles[:, i] = gs
        a_bs = dequantize(q_c, q_sf, np.ones(rows, np.float32))  # q s_b, gs excluded
        d_o = gemm_f64(a_bs, b_bs[:, cols])
        g = gs.astype(np.float64)
        ratio = np.where(live, gs_prev / np.where(live, g, 1.0), 0.0)
        o = np.where(live[:, None], o * ratio[:, None] + d_o, o)
        gs_prev = np.where(live, g, gs_prev)
    y = o * (gs_prev * np.float64(gs_w[0]))[:, None]
    return dict(y=bf16_round(y), y_f64=y, codes=codes, sf=sf, gs_tiles=gs_tiles)


# ---------------------------------------------------------------- metrics

def error_metrics(x, xhat):
    """Relative L2, SNR (dB) and MAE of a reconstruction ("miniTE Technical
    Report" 2.3)."""
    x = np.asarray(x, np.float64).reshape(-1)
    xhat = np.asarray(xhat, np.float64).reshape(-1)
    err = np.linalg.norm(xhat - x)
    nx = np.linalg.norm(x)
    return dict(rel_l2=err / nx, snr_db=20 * np.log10(nx / err) if err > 0 else np.inf,
                mae=np.mean(np.abs(xhat - x)))
