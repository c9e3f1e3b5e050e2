"""Python binding of libnvfp4moe.so (include/nvfp4moe.h): argument marshalling only.

Every step of the path runs in the library's sm_103a kernels; this module
only allocates device buffers with torch, passes raw pointers and the
current CUDA stream, and turns nonzero return codes into exceptions.  There
is no fallback: if the shared library is missing or a GPU is absent the
calls raise.
"""
import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

c_i64 = ctypes.c_int64
c_vp = ctypes.c_void_p


class _Tensor(ctypes.Structure):
    _fields_ = [("codes", c_vp), ("sf", c_vp), ("scale", c_vp), ("rows", c_i64), ("cols", c_i64)]


class _Options(ctypes.Structure):
    _fields_ = [("weight_at_fc1", ctypes.c_int), ("four_over_six", ctypes.c_int), ("fc2_requant", ctypes.c_int),
                ("fc2_combine", ctypes.c_int)]


class _Debug(ctypes.Structure):
    _fields_ = [("fc1_out", c_vp), ("stage_events", ctypes.POINTER(c_vp)), ("stall_fc1", ctypes.c_int),
                ("requant_copy", ctypes.c_int)]


STAGES = ["quantize", "route", "fc1", "requant", "fc2", "combine"]


LAYOUT_FIELDS = ["total", "err", "ids", "weights", "row_weights", "counts", "offsets", "padded_offsets",
                 "perm", "inv", "chunk_counts", "xq_codes", "xq_sf", "xq_scale", "a1_codes", "a1_sf",
                 "a1_scale", "d", "amax2", "a2_codes", "a2_sf", "a2_scale", "y2", "comb_cnt"]


class _Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in LAYOUT_FIELDS]


PER_ROW = 0
PER_TENSOR = 1
DQ_PADDED_ROWS = 8    # nvfp4_dequantize_rows: rows written at their padded positions
DEVERR_TIMEOUT = 1    # bits of the device error word
DEVERR_BADEXPERT = 2
DEVERR_BADGROUP = 4
FOUR_OVER_SIX = {None: 0, "mse": 2, "mae": 4}  # scale-mode flags of four-over-six block scaling
FC2_REQUANT = {None: 0, "separate": 1, "in_fc2": 2}  # moe_options.fc2_requant
SYMBOLS = ["nvfp4_sf_bytes", "nvfp4_quantize_workspace", "nvfp4_quantize_rows", "nvfp4_quantize_grouped",
           "nvfp4_dequantize_rows",
           "nvfp4_linear", "nvfp4_grouped_dgrad_bf16", "nvfp4_grouped_wgrad_bf16",
           "moe_expert_workspace_layout", "moe_expert_workspace", "moe_expert_forward",
           "moe_expert_forward_noalloc", "moe_noalloc_error_word", "nvfp4_last_error"]


class NVFP4Error(RuntimeError):
    pass


def library_path():
    return _build.LIB


def lib():
    """Load the shared library (built in-tree by build.build())."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise NVFP4Error(f"{path} is missing: run __graft_entry__.build() (or "
                             "nvfp4_quantized_moe_token_gb300.build.build()) first")
        L = ctypes.CDLL(path)
        L.nvfp4_sf_bytes.restype = ctypes.c_size_t
        L.nvfp4_sf_bytes.argtypes = [c_i64, c_i64]
        L.nvfp4_quantize_workspace.restype = ctypes.c_size_t
        L.nvfp4_quantize_workspace.argtypes = [c_i64, c_i64, ctypes.c_int]
        L.nvfp4_quantize_rows.restype = ctypes.c_int
        L.nvfp4_quantize_rows.argtypes = [c_vp, c_i64, c_i64, c_i64, ctypes.c_int, c_vp,
                                          ctypes.POINTER(_Tensor), c_vp, ctypes.c_size_t, c_vp]
        L.nvfp4_quantize_grouped.restype = ctypes.c_int
        L.nvfp4_quantize_grouped.argtypes = [c_vp, ctypes.c_int, c_i64, c_i64, ctypes.c_int, ctypes.POINTER(_Tensor),
                                             c_vp, ctypes.c_size_t, c_vp]
        L.nvfp4_dequantize_rows.restype = ctypes.c_int
        L.nvfp4_dequantize_rows.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_int, c_vp, c_vp, ctypes.c_int, c_vp,
                                            c_i64, c_vp]
        for fn in (L.nvfp4_grouped_dgrad_bf16, L.nvfp4_grouped_wgrad_bf16):
            fn.restype = ctypes.c_int
            fn.argtypes = [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, ctypes.c_int, c_vp, ctypes.c_size_t, c_vp]
        L.nvfp4_linear.restype = ctypes.c_int
        L.nvfp4_linear.argtypes = [ctypes.POINTER(_Tensor), ctypes.POINTER(_Tensor), c_vp, c_i64,
                                   c_vp, ctypes.c_size_t, c_vp]
        L.moe_expert_workspace_layout.restype = ctypes.c_int
        L.moe_expert_workspace_layout.argtypes = [c_i64, c_i64, c_i64, ctypes.c_int, ctypes.c_int,
                                                  ctypes.POINTER(_Layout)]
        L.moe_expert_workspace.restype = ctypes.c_size_t
        L.moe_expert_workspace.argtypes = [c_i64, c_i64, c_i64, ctypes.c_int, ctypes.c_int]
        L.moe_expert_forward.restype = ctypes.c_int
        L.moe_expert_forward.argtypes = [c_vp, c_i64, c_i64, c_vp, c_vp, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(_Tensor), ctypes.POINTER(_Tensor), c_i64,
                                         ctypes.POINTER(_Options), c_vp, ctypes.POINTER(_Debug),
                                         c_vp, ctypes.c_size_t, c_vp]
        L.nvfp4_last_error.restype = ctypes.c_char_p
        L.nvfp4_last_error.argtypes = []
        _LIB = L
    return _LIB


def _check(rc, what):
    if rc != 0:
        msg = lib().nvfp4_last_error().decode()
        raise NVFP4Error(f"{what} failed ({rc}): {msg}")


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class NVFP4Tensor:
    """An NVFP4 matrix on the device: packed E2M1 codes [rows, cols/2],
    swizzled E4M3 block scales (sf_bytes(rows, cols) bytes) and fp32 outer
    scales ([rows], [1] or one per stacked group)."""

    def __init__(self, codes, sf, scale, rows, cols):
        self.codes, self.sf, self.scale = codes, sf, scale
        self.rows, self.cols = int(rows), int(cols)

    @classmethod
    def empty(cls, rows, cols, n_scales, device="cuda"):
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
        sf = torch.empty(max(sf_bytes(rows, cols), 16), dtype=torch.uint8, device=device)
        scale = torch.empty(max(n_scales, 1), dtype=torch.float32, device=device)
        return cls(codes, sf, scale, rows, cols)

    def c(self):
        return _Tensor(self.codes.data_ptr(), self.sf.data_ptr(), self.scale.data_ptr(),
                       self.rows, self.cols)


def sf_bytes(rows, cols):
    return int(lib().nvfp4_sf_bytes(rows, cols))


def quantize_rows(x, per_tensor=False, amax_in=None, out=None, four_over_six=None, stream=None):
    """bf16 [rows, cols] (CUDA) -> NVFP4Tensor (per-row or per-tensor outer scale);
    four_over_six None, 'mse' or 'mae' selects four-over-six block scaling."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if out is None:
        out = NVFP4Tensor.empty(rows, cols, 1 if per_tensor else rows, x.device)
    mode = (PER_TENSOR if per_tensor else PER_ROW) | FOUR_OVER_SIX[four_over_six]
    ws_bytes = int(lib().nvfp4_quantize_workspace(rows, cols, mode))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device) if ws_bytes else None
    t = out.c()
    rc = lib().nvfp4_quantize_rows(_ptr(x), rows, cols, x.stride(0), mode, _ptr(amax_in), ctypes.byref(t),
                                   _ptr(ws), ws_bytes, _stream(stream))
    _check(rc, "nvfp4_quantize_rows")
    return out


def dequantize_rows(t, per_tensor=False, group_offsets=None, padded_offsets=None, out=None, padded_rows=False,
                    stream=None):
    """NVFP4Tensor -> bf16 [rows, cols] = bf16(q s_b s_g), the exact product rounded
    once (DQ(Q(x)), the BF16 backward operand).  group_offsets / padded_offsets
    (int32 CUDA tensors [G+1]): scale rows padded per group, as in the expert-ordered
    buffers of moe_expert_forward; per_tensor with offsets takes one scale per group.
    padded_rows: rows written at their padded positions, padding rows zeroed (out
    must then hold padded_offsets[G] rows)."""
    if out is None:
        assert not padded_rows, "padded_rows needs an out buffer of padded_offsets[G] rows"
        out = torch.empty((t.rows, t.cols), dtype=torch.bfloat16, device=t.codes.device)
    assert out.dtype == torch.bfloat16 and out.stride(1) == 1
    G = 0 if group_offsets is None else group_offsets.numel() - 1
    mode = (PER_TENSOR if per_tensor else PER_ROW) | (DQ_PADDED_ROWS if padded_rows else 0)
    rc = lib().nvfp4_dequantize_rows(ctypes.byref(t.c()), mode,
                                     _ptr(group_offsets), _ptr(padded_offsets), G, _ptr(out), out.stride(0),
                                     _stream(stream))
    _check(rc, "nvfp4_dequantize_rows")
    return out


def grouped_dgrad_bf16(dy, w, padded_offsets=None, out=None, err=None, stream=None):
    """dx = dy . w_g per row group: dy bf16 [rows, nf], w bf16 [G, nf, kf] (each
    group's DQ(Q(W)) in its forward layout), padded_offsets int32 [G+1] (ascending
    multiples of 128) or None for one dense group; returns dx bf16 [rows, kf]."""
    rows, nf = dy.shape
    G, nf2, kf = w.shape
    assert nf2 == nf and dy.is_contiguous() and w.is_contiguous()
    if out is None:
        out = torch.empty((rows, kf), dtype=torch.bfloat16, device=dy.device)
    rc = lib().nvfp4_grouped_dgrad_bf16(_ptr(dy), _ptr(w), _ptr(out), rows, nf, kf, _ptr(padded_offsets),
                                        G if padded_offsets is not None else 1, _ptr(err),
                                        0 if err is None else err.numel() * err.element_size(), _stream(stream))
    _check(rc, "nvfp4_grouped_dgrad_bf16")
    return out


def grouped_wgrad_bf16(dy, x, padded_offsets=None, groups=1, out=None, err=None, stream=None):
    """dw_g = dy[rows of g]^T . x[rows of g]: dy bf16 [rows, nf], x bf16 [rows, kf],
    padded_offsets int32 [G+1] or None (one group); returns dw bf16 [G, nf, kf]."""
    rows, nf = dy.shape
    rows2, kf = x.shape
    assert rows2 == rows and dy.is_contiguous() and x.is_contiguous()
    G = padded_offsets.numel() - 1 if padded_offsets is not None else 1
    if out is None:
        out = torch.empty((G, nf, kf), dtype=torch.bfloat16, device=dy.device)
    rc = lib().nvfp4_grouped_wgrad_bf16(_ptr(dy), _ptr(x), _ptr(out), rows, nf, kf, _ptr(padded_offsets), G,
                                        _ptr(err), 0 if err is None else err.numel() * err.element_size(),
                                        _stream(stream))
    _check(rc, "nvfp4_grouped_wgrad_bf16")
    return out


def quantize_grouped_weights(w, four_over_six=None, stream=None):
    """Per-expert weights bf16 [G, N, K] -> one stacked NVFP4Tensor [G*N, K]
    with one per-tensor scale per expert (scale has G entries).  Requires
    N % 128 == 0 so each expert's swizzled scales are a contiguous slice."""
    G, N, K = w.shape
    assert N % 128 == 0 and w.is_contiguous()
    out = NVFP4Tensor.empty(G * N, K, G, w.device)
    ws = torch.empty(16 + 4 * G, dtype=torch.uint8, device=w.device)
    rc = lib().nvfp4_quantize_grouped(_ptr(w), G, N, K, PER_TENSOR | FOUR_OVER_SIX[four_over_six], ctypes.byref(out.c()),
                                      _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "nvfp4_quantize_grouped")
    return out


def linear(xq, wq, out=None, err=None, stream=None):
    """y = bf16( deq(x) . deq(w)^T ): x per-row, w per-tensor (K-major [N, K])."""
    M, N = xq.rows, wq.rows
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.codes.device)
    a, b = xq.c(), wq.c()
    rc = lib().nvfp4_linear(ctypes.byref(a), ctypes.byref(b), _ptr(out), out.stride(0),
                            _ptr(err), 0 if err is None else err.numel() * err.element_size(),
                            _stream(stream))
    _check(rc, "nvfp4_linear")
    return out


def moe_workspace_layout(T, H, F, E, topk):
    L = _Layout()
    _check(lib().moe_expert_workspace_layout(T, H, F, E, topk, ctypes.byref(L)), "moe_expert_workspace_layout")
    return {n: int(getattr(L, n)) for n in LAYOUT_FIELDS}


def moe_expert_forward(x, logits, bias, w1q, w2q, F, topk, weight_at_fc1=False, out=None,
                       ws=None, fc1_debug=None, stage_events=None, four_over_six=None, stream=None,
                       debug_stall_fc1=False, fc2_requant=None, requant_copy=False, fc2_combine=False):
    """One W4A4 MoE expert layer on the device.  Returns (out bf16 [T, H], ws).
    four_over_six (None, 'mse', 'mae'): four-over-six scaling of the activations.
    fc2_requant (None: the library's choice, 'separate', 'in_fc2'): where D is
    requantized (moe_options.fc2_requant); requant_copy: with 'in_fc2', also
    write the encoded D to the workspace's a2 slots (moe_debug.requant_copy).
    fc2_combine: the router-weighted combine inside FC2's epilogue
    (moe_options.fc2_combine).
    debug_stall_fc1: test of the time-out path (moe_debug.stall_fc1): FC1's
    bounded wait runs out, DEVERR_TIMEOUT is set in the workspace's error
    word, the outputs are undefined.

    stage_events (optional): len(STAGES) + 1 torch.cuda.Event objects (or None
    for an event to skip) recorded on the stream before the first stage and
    after each stage."""
    T, H = x.shape
    E = logits.shape[1]
    need = int(lib().moe_expert_workspace(T, H, F, E, topk))
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    a, b = w1q.c(), w2q.c()
    opt = _Options(1 if weight_at_fc1 else 0, FOUR_OVER_SIX[four_over_six], FC2_REQUANT[fc2_requant],
                   1 if fc2_combine else 0)
    evs = None
    if stage_events is not None:
        assert len(stage_events) == len(STAGES) + 1
        st = stream if stream is not None else torch.cuda.current_stream()
        for e in stage_events:
            if e is not None and e.cuda_event == 0:  # torch creates the CUDA event on its first record
                e.record(st)
        evs = (c_vp * len(stage_events))(*[None if e is None else e.cuda_event for e in stage_events])
    dbg = _Debug(None if fc1_debug is None else fc1_debug.data_ptr(), evs, 1 if debug_stall_fc1 else 0,
                 1 if requant_copy else 0)
    rc = lib().moe_expert_forward(_ptr(x), T, H, _ptr(logits), _ptr(bias), E, topk, ctypes.byref(a),
                                  ctypes.byref(b), F, ctypes.byref(opt), _ptr(out), ctypes.byref(dbg),
                                  _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "moe_expert_forward")
    return out, ws


def ws_view(ws, layout, field, dtype, shape):
    """A typed view of one intermediate inside the MoE workspace."""
    off = layout[field]
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.empty(0, dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).view(*shape)
