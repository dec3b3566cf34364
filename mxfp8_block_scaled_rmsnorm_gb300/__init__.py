"""Fused RMSNorm + MXFP8 block quantization on GB300 (sm_103a).

Python binding of the C ABI declared in ``include/mxfp8norm.h`` (library
``libmxfp8norm.so`` next to this file). The calls have the C names:

``rmsnorm_quant_mxfp8(xs, gammas, eps, weight_offset, rowwise, columnwise)``
    RMSNorm of each bf16 matrix (float32 math), written as bf16 ``normed``,
    plus the MXFP8 planes of that same bf16.
``quant_mxfp8(ws, rowwise, columnwise)``
    MXFP8 planes of each bf16 matrix (weight storage; no norm).

MXFP8 planes of an [R, C] matrix: ``q_row`` [R, C] E4M3 codes with ``s_row``
[R, C/32] E8M0 scale bytes (blocks of 32 columns), and ``q_col`` [R, C] in the
same row-major layout with ``s_col`` [R/32, C] (blocks of 32 rows). Codes and
scales are returned as ``torch.uint8`` tensors; view them as
``torch.float8_e4m3fn`` / ``torch.float8_e8m0fnu`` where needed.

This module only marshals arguments: every step runs in the CUDA kernels of the
library, on the caller's current CUDA stream. PyTorch is used for device
memory and streams. There is no CPU fallback: if the library is not built the
calls raise.
"""
from __future__ import annotations

import collections
import ctypes
import os
from typing import Sequence

import torch

__all__ = ["rmsnorm_quant_mxfp8", "quant_mxfp8", "add_rmsnorm_quant_mxfp8", "update_planes",
           "mm_mxfp8", "quantize_weight_for_mm", "mm_mxfp8_workspace_size", "device_status",
           "NormQuantOut",
           "QuantOut",
           "MXFP8Error", "MXFP8Desc", "library", "make_outputs", "mma_scale_shape",
           "padded_scale_shape"]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmxfp8norm.so")

BLOCK = 32
MAX_TENSORS = 256
# scale layouts of the *_ex calls (include/mxfp8norm.h)
SCALE_LAYOUTS = {"compact": 0, "mma": 1, "padded": 2}
ERRORS = {-1: "MXFP8_ERR_POINTER", -2: "MXFP8_ERR_SHAPE", -3: "MXFP8_ERR_FLAGS",
          -4: "MXFP8_ERR_COUNT", -5: "MXFP8_ERR_CUDA"}

NormQuantOut = collections.namedtuple("NormQuantOut", "normed q_row s_row q_col s_col")
QuantOut = collections.namedtuple("QuantOut", "q_row s_row q_col s_col")


class MXFP8Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{ERRORS.get(code, code)}: {message}")
        self.code = code


class MXFP8Residual(ctypes.Structure):
    """``mxfp8_residual`` of include/mxfp8norm.h."""
    _fields_ = [("residual", ctypes.c_void_p), ("residual_out", ctypes.c_void_p)]


class MXFP8Planes(ctypes.Structure):
    """``mxfp8_planes`` of include/mxfp8norm.h."""
    _fields_ = [("q_row", ctypes.c_void_p), ("s_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("s_col", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class MXFP8Desc(ctypes.Structure):
    """``mxfp8_desc`` of include/mxfp8norm.h."""
    _fields_ = [("x", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
                ("normed", ctypes.c_void_p), ("q_row", ctypes.c_void_p),
                ("s_row", ctypes.c_void_p), ("q_col", ctypes.c_void_p),
                ("s_col", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("eps", ctypes.c_float),
                ("weight_offset", ctypes.c_float)]


_lib = None


def library() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first "
                "(python -m mxfp8_block_scaled_rmsnorm_gb300.build, or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        for name in ("rmsnorm_quant_mxfp8", "quant_mxfp8"):
            f = getattr(L, name)
            f.argtypes = [ctypes.POINTER(MXFP8Desc), ctypes.c_int, ctypes.c_int,
                          ctypes.c_int, ctypes.c_void_p]
            f.restype = ctypes.c_int
        for name in ("rmsnorm_quant_mxfp8_ex", "quant_mxfp8_ex"):
            f = getattr(L, name)
            f.argtypes = [ctypes.POINTER(MXFP8Desc), ctypes.c_int, ctypes.c_int,
                          ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
            f.restype = ctypes.c_int
        L.add_rmsnorm_quant_mxfp8.argtypes = [ctypes.POINTER(MXFP8Desc),
                                              ctypes.POINTER(MXFP8Residual), ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_void_p]
        L.add_rmsnorm_quant_mxfp8.restype = ctypes.c_int
        L.mxfp8_update_planes.argtypes = [ctypes.POINTER(MXFP8Planes),
                                          ctypes.POINTER(MXFP8Planes), ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_void_p]
        L.mxfp8_update_planes.restype = ctypes.c_int
        L.mm_mxfp8_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int64]
        L.mm_mxfp8_workspace_size.restype = ctypes.c_size_t
        L.mm_mxfp8.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.mm_mxfp8.restype = ctypes.c_int
        L.mm_mxfp8_static.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_void_p]
        L.mm_mxfp8_static.restype = ctypes.c_int
        L.mm_mxfp8_quantized.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        L.mm_mxfp8_quantized.restype = ctypes.c_int
        L.mxfp8_device_status.argtypes = [ctypes.c_int]
        L.mxfp8_device_status.restype = ctypes.c_int64
        L.mxfp8_set_test_hook.argtypes = [ctypes.c_int, ctypes.c_int]
        L.mxfp8_set_test_hook.restype = ctypes.c_int
        L.mxfp8_last_error.argtypes = []
        L.mxfp8_last_error.restype = ctypes.c_char_p
        L.mxfp8_abi_version.argtypes = []
        L.mxfp8_abi_version.restype = ctypes.c_int
        _lib = L
    return _lib


def _as_list(v, n, name):
    if isinstance(v, (list, tuple)):
        if len(v) != n:
            raise ValueError(f"{name}: {len(v)} values for {n} tensors")
        return list(v)
    return [v] * n


def _check_input(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D torch.bfloat16 tensor")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _scale_numel(rows: int, cols: int, columnwise: bool, scale_layout: str) -> int:
    """Bytes of one scale plane of a [rows, cols] matrix in ``scale_layout``."""
    if scale_layout == "mma":
        r, c = (mma_scale_shape(cols, rows // BLOCK) if columnwise
                else mma_scale_shape(rows, cols // BLOCK))
    elif scale_layout == "padded":
        r, c = padded_scale_shape(rows, cols, columnwise)
    else:
        r, c = (rows // BLOCK, cols) if columnwise else (rows, cols // BLOCK)
    return r * c


def _check_buffer(t, name: str, device, numel: int, shape=None, dtype=None,
                  at_least: bool = False):
    """A caller-supplied buffer: the kernels touch numel elements from its data
    pointer, so a smaller, strided or foreign-device buffer is rejected here
    (the C ABI sees raw pointers only). Outputs must match exactly; inputs that
    are only read (``at_least``) may be larger."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch tensor")
    if t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor on {device}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dtype is None and t.element_size() != 1:
        raise ValueError(f"{name} must have 1-byte elements (uint8 or an 8-bit float view)")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.numel() < numel or (t.numel() != numel and not at_least):
        raise ValueError(f"{name} must hold {'at least ' if at_least else ''}{numel} "
                         f"elements, got {t.numel()}")


def _check_planes(o, i: int, R: int, C: int, rowwise: bool, columnwise: bool,
                  scale_layout: str, device, what: str = "output"):
    """The code and scale planes of one entry, for the planes requested."""
    for on, q, sc, tag, colw in ((rowwise, o.q_row, o.s_row, "row", False),
                                 (columnwise, o.q_col, o.s_col, "col", True)):
        if not on:
            continue
        if q is None or sc is None:
            plane = "columnwise" if colw else "rowwise"
            raise ValueError(f"{what} {i}: the {plane} plane is requested but q_{tag} or "
                             f"s_{tag} is None")
        _check_buffer(q, f"{what} {i} q_{tag}", device, R * C, shape=(R, C))
        _check_buffer(sc, f"{what} {i} s_{tag}", device, _scale_numel(R, C, colw, scale_layout))


class _NoSwitch:
    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


_NO_SWITCH = _NoSwitch()


def _on_device(dev: torch.device):
    """The library launches on the current CUDA device: switch to ``dev`` only
    when it is not current already (the switch costs a few microseconds)."""
    if dev.index is None or dev.index == torch.cuda.current_device():
        return _NO_SWITCH
    return torch.cuda.device(dev)


# torch's current-stream lookup as a raw cudaStream_t: about 0.1 us, against
# about 3 us for torch.cuda.current_stream().cuda_stream, which builds a
# Stream object (a large share of a small call's host time)
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, dev) -> int:
    """cudaStream_t of ``stream`` (a torch stream or a raw handle), or of the
    current torch stream on ``dev`` (which must be the current device)."""
    if stream is None:
        if _raw_current_stream is not None:
            return _raw_current_stream(torch.cuda.current_device() if dev.index is None
                                       else dev.index)
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def mma_scale_shape(m: int, kb: int):
    """Byte count of the tiled ("mma") scale layout of an operand with m rows
    and kb scale columns, as a (rows, cols) pair: (roundup(m, 128),
    roundup(kb, 4)). The bytes are tiled, not row-major."""
    return (-(-m // 128) * 128, -(-kb // 4) * 4)


def padded_scale_shape(rows: int, cols: int, columnwise: bool):
    """Row-major padded ("padded") scale shape: rowwise [roundup(rows, 128),
    roundup(cols/32, 4)]; columnwise [roundup(rows/32, 4), roundup(cols, 128)]."""
    r = lambda v, m: -(-v // m) * m
    if columnwise:
        return (r(rows // BLOCK, 4), r(cols, 128))
    return (r(rows, 128), r(cols // BLOCK, 4))


def make_outputs(x: torch.Tensor, fused: bool, rowwise: bool, columnwise: bool,
                 scale_layout: str = "compact"):
    """Allocate the output tensors of one list entry. Codes and normed use
    ``torch.empty``; tiled ("mma") scale buffers are zero-filled once, since
    the kernels leave their padding untouched."""
    R, C = x.shape
    u8 = dict(dtype=torch.uint8, device=x.device)
    q_row = torch.empty((R, C), **u8) if rowwise else None
    q_col = torch.empty((R, C), **u8) if columnwise else None
    if scale_layout == "mma":
        s_row = torch.zeros(mma_scale_shape(R, C // BLOCK), **u8) if rowwise else None
        s_col = torch.zeros(mma_scale_shape(C, R // BLOCK), **u8) if columnwise else None
    elif scale_layout == "padded":
        s_row = torch.zeros(padded_scale_shape(R, C, False), **u8) if rowwise else None
        s_col = torch.zeros(padded_scale_shape(R, C, True), **u8) if columnwise else None
    else:
        s_row = torch.empty((R, C // BLOCK), **u8) if rowwise else None
        s_col = torch.empty((R // BLOCK, C), **u8) if columnwise else None
    if fused:
        return NormQuantOut(torch.empty_like(x), q_row, s_row, q_col, s_col)
    return QuantOut(q_row, s_row, q_col, s_col)


def _call(fused, xs, gammas, eps, offsets, rowwise, columnwise, out, stream,
          scale_layout="compact", residual=None):
    if scale_layout not in SCALE_LAYOUTS:
        raise ValueError(f"scale_layout must be one of {sorted(SCALE_LAYOUTS)}")
    single = isinstance(xs, torch.Tensor)
    xs = [xs] if single else list(xs)
    n = len(xs)
    if fused:
        gammas = [gammas] if isinstance(gammas, torch.Tensor) else list(gammas)
        if len(gammas) != n:
            raise ValueError(f"{len(gammas)} gammas for {n} inputs")
    for i, x in enumerate(xs):
        _check_input(x, f"input {i}")
    if out is None:
        out = [make_outputs(x, fused, rowwise, columnwise, scale_layout) for x in xs]
    else:
        out = [out] if isinstance(out, tuple) and hasattr(out, "_fields") else list(out)
        if len(out) != n:
            raise ValueError(f"{len(out)} output sets for {n} inputs")
        for i, (x, o) in enumerate(zip(xs, out)):
            R, C = x.shape
            if fused:
                _check_buffer(o.normed, f"output {i} normed", x.device, R * C, shape=(R, C),
                              dtype=torch.bfloat16)
            if (columnwise and R % BLOCK) or C % BLOCK:
                continue  # the C ABI reports the shape error
            _check_planes(o, i, R, C, rowwise, columnwise, scale_layout, x.device)
    descs = (MXFP8Desc * max(n, 1))()
    eps_l = _as_list(eps, n, "eps")
    off_l = _as_list(offsets, n, "weight_offset")
    for i, x in enumerate(xs):
        d = descs[i]
        o = out[i]
        d.x = x.data_ptr()
        d.rows, d.cols = x.shape
        if fused:
            g = gammas[i]
            if (not isinstance(g, torch.Tensor) or g.dtype != torch.bfloat16
                    or g.dim() != 1 or not g.is_contiguous() or g.device != x.device):
                raise ValueError(f"gamma {i} must be a contiguous 1-D bf16 tensor on {x.device}")
            d.gamma = g.data_ptr()
            d.normed = _ptr(o.normed)
            d.eps = float(eps_l[i])
            d.weight_offset = float(off_l[i])
        d.q_row, d.s_row = _ptr(o.q_row), _ptr(o.s_row)
        d.q_col, d.s_col = _ptr(o.q_col), _ptr(o.s_col)
    L = library()
    dev = xs[0].device
    layout = SCALE_LAYOUTS[scale_layout]
    rw, cw = int(bool(rowwise)), int(bool(columnwise))
    with _on_device(dev):
        handle = _stream_handle(stream, dev)
        if residual is not None:
            rc = L.add_rmsnorm_quant_mxfp8(descs, residual, n, rw, cw, layout, handle)
        else:
            fn = L.rmsnorm_quant_mxfp8_ex if fused else L.quant_mxfp8_ex
            rc = fn(descs, n, rw, cw, layout, handle)
    if rc != 0:
        raise MXFP8Error(rc, L.mxfp8_last_error().decode())
    return out[0] if single else out


def rmsnorm_quant_mxfp8(xs, gammas, eps: float | Sequence[float] = 1e-6,
                        weight_offset: float | Sequence[float] = 0.0,
                        rowwise: bool = True, columnwise: bool = True,
                        out=None, stream=None, scale_layout: str = "compact"):
    """Fused RMSNorm + MXFP8 of one bf16 [R, C] tensor or a list of them (one launch).

    ``gammas``: bf16 [C] per input; ``eps`` and ``weight_offset``: float32
    scalars, one for all inputs or one per input. Returns a ``NormQuantOut``
    (or a list of them); disabled planes are ``None``. ``out`` takes
    preallocated outputs (e.g. from :func:`make_outputs`) to be overwritten in
    place, which keeps CUDA-graph captures valid. ``scale_layout="mma"``
    writes the scales in the tiled layout of a block-scaled GEMM operand
    (s_row as an operand with M = R rows, s_col with M = C rows; see
    include/mxfp8norm.h) instead of the compact [R, C/32] / [R/32, C] arrays;
    ``"padded"`` writes row-major arrays with TE's padded allocation shape.
    """
    return _call(True, xs, gammas, eps, weight_offset, rowwise, columnwise, out, stream,
                 scale_layout)


def quant_mxfp8(ws, rowwise: bool = True, columnwise: bool = True, out=None, stream=None,
                scale_layout: str = "compact"):
    """MXFP8 planes of one bf16 [R, C] tensor or a list of them (one launch).

    Returns a ``QuantOut`` (or a list of them); disabled planes are ``None``.
    ``scale_layout`` as for :func:`rmsnorm_quant_mxfp8`.
    """
    return _call(False, ws, None, 0.0, 0.0, rowwise, columnwise, out, stream, scale_layout)


def add_rmsnorm_quant_mxfp8(xs, residuals, gammas, eps: float | Sequence[float] = 1e-6,
                            weight_offset: float | Sequence[float] = 0.0,
                            rowwise: bool = True, columnwise: bool = True, out=None,
                            residual_out=True, stream=None, scale_layout: str = "compact"):
    """Residual add + RMSNorm + MXFP8 in one launch: h = bf16(x + residual)
    (one rounding of the exact sum), then the planes of RMSNorm(h).

    ``residuals``: a bf16 tensor per input (or ``None`` entries: nothing
    added). ``residual_out``: ``True`` to allocate h, ``False``/``None`` not to
    write it, or tensors to write it into. Returns ``(h, NormQuantOut)`` (or a
    list of them); h is ``None`` when not written.
    """
    single = isinstance(xs, torch.Tensor)
    xl = [xs] if single else list(xs)
    rl = [residuals] if (single or residuals is None or isinstance(residuals, torch.Tensor)) \
        else list(residuals)
    if len(rl) != len(xl):
        rl = rl * len(xl) if len(rl) == 1 else rl
    if len(rl) != len(xl):
        raise ValueError(f"{len(rl)} residuals for {len(xl)} inputs")
    if residual_out is True:
        houts = [torch.empty_like(x) for x in xl]
    elif residual_out is None or residual_out is False:
        houts = [None] * len(xl)
    else:
        houts = [residual_out] if isinstance(residual_out, torch.Tensor) else list(residual_out)
    res = (MXFP8Residual * max(1, len(xl)))()
    for i, (x, r, h) in enumerate(zip(xl, rl, houts)):
        for t, name in ((r, "residual"), (h, "residual_out")):
            if t is not None and (t.shape != x.shape or t.dtype != torch.bfloat16
                                  or not t.is_contiguous() or t.device != x.device):
                raise ValueError(f"{name} {i} must be a contiguous bf16 tensor shaped like x")
        res[i].residual = _ptr(r)
        res[i].residual_out = _ptr(h)
    outs = _call(True, xl, gammas, eps, weight_offset, rowwise, columnwise, out, stream,
                 scale_layout, residual=res)
    pairs = list(zip(houts, outs))
    return pairs[0] if single else pairs


def update_planes(src, dst, rowwise: bool = True, columnwise: bool = True,
                  scale_layout: str = "padded", stream=None) -> None:
    """In-place plane update (update_mxfp8_tensor): for each pair, copy the
    selected planes of ``src`` (compact scales) into ``dst`` (scales in
    ``scale_layout``, padding untouched); a selected plane that ``src`` lacks
    (its tensors are ``None``) is cleared in ``dst``. ``src``/``dst``: objects
    with ``q_row, s_row, q_col, s_col`` (e.g. ``QuantOut``) or lists of them."""
    if scale_layout not in SCALE_LAYOUTS:
        raise ValueError(f"scale_layout must be one of {sorted(SCALE_LAYOUTS)}")
    single = hasattr(src, "q_row")
    sl = [src] if single else list(src)
    dl = [dst] if single else list(dst)
    if len(sl) != len(dl) or not sl:
        raise ValueError("src and dst must be non-empty and of equal length")
    arr_s = (MXFP8Planes * len(sl))()
    arr_d = (MXFP8Planes * len(dl))()
    dev = None
    for i, (a, b) in enumerate(zip(sl, dl)):
        ref = b.q_row if b.q_row is not None else b.q_col
        if ref is None or ref.dim() != 2:
            raise ValueError(f"dst {i} needs a 2-D code plane")
        dev = ref.device
        R, C = ref.shape
        if C % BLOCK == 0 and not (columnwise and R % BLOCK):
            _check_planes(b, i, R, C, rowwise, columnwise, scale_layout, dev, "dst")
            for on, q, sc, tag, colw in ((rowwise, a.q_row, a.s_row, "row", False),
                                         (columnwise, a.q_col, a.s_col, "col", True)):
                if on and q is not None and sc is not None:
                    _check_buffer(q, f"src {i} q_{tag}", dev, R * C, shape=(R, C),
                                  at_least=True)
                    _check_buffer(sc, f"src {i} s_{tag}", dev,
                                  _scale_numel(R, C, colw, "compact"), at_least=True)
        for arr, o in ((arr_s, a), (arr_d, b)):
            arr[i].q_row, arr[i].s_row = _ptr(o.q_row), _ptr(o.s_row)
            arr[i].q_col, arr[i].s_col = _ptr(o.q_col), _ptr(o.s_col)
            arr[i].rows, arr[i].cols = R, C
    L = library()
    with _on_device(dev):
        rc = L.mxfp8_update_planes(arr_s, arr_d, len(sl), int(bool(rowwise)),
                                   int(bool(columnwise)), SCALE_LAYOUTS[scale_layout],
                                   _stream_handle(stream, dev))
    if rc != 0:
        raise MXFP8Error(rc, L.mxfp8_last_error().decode())


def quantize_weight_for_mm(w: torch.Tensor, stream=None) -> QuantOut:
    """The rowwise plane of a bf16 weight [N, K] with its scales in the tiled
    GEMM-operand layout: the form mm_mxfp8 takes (quantize once, reuse)."""
    return quant_mxfp8(w, True, False, stream=stream, scale_layout="mma")


def mm_mxfp8(x: torch.Tensor, w_q: torch.Tensor, w_s: torch.Tensor, out=None,
             workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[M, N] = x[M, K] w^T in MXFP8: x (bf16) is quantized on the fly, the
    weight comes as ``quantize_weight_for_mm(w)``'s ``q_row``/``s_row``.
    ``workspace``: a uint8 CUDA buffer of at least
    ``mm_mxfp8_workspace_size(M, K)`` bytes (allocated here if omitted)."""
    _check_input(x, "x")
    M, K = x.shape
    N = w_q.shape[0]
    if w_q.shape != (N, K) or w_q.dtype != torch.uint8 or w_s.dtype != torch.uint8:
        raise ValueError("w_q must be uint8 [N, K] codes and w_s uint8 tiled scales")
    _check_buffer(w_q, "w_q", x.device, N * K, shape=(N, K))
    if K % BLOCK == 0:
        _check_buffer(w_s, "w_s", x.device, _scale_numel(N, K, False, "mma"), at_least=True)
    L = library()
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    else:
        _check_buffer(out, "out", x.device, M * N, shape=(M, N), dtype=torch.bfloat16)
    if workspace is None:
        workspace = torch.empty(int(L.mm_mxfp8_workspace_size(M, K)), dtype=torch.uint8,
                                device=x.device)
    else:
        _check_buffer(workspace, "workspace", x.device, workspace.numel(), dtype=torch.uint8)
    with _on_device(x.device):
        rc = L.mm_mxfp8(x.data_ptr(), M, K, w_q.data_ptr(), w_s.data_ptr(), N, out.data_ptr(),
                        workspace.data_ptr(), workspace.numel(), _stream_handle(stream, x.device))
    if rc != 0:
        raise MXFP8Error(rc, L.mxfp8_last_error().decode())
    return out


def mm_mxfp8_quantized(x_q: torch.Tensor, x_s: torch.Tensor, w_q: torch.Tensor,
                       w_s: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """The GEMM of mm_mxfp8 alone: out[M, N] = deq(x_q, x_s) deq(w_q, w_s)^T for
    an activation quantized beforehand (e.g. ``rmsnorm_quant_mxfp8(...,
    scale_layout="mma")``'s ``q_row``/``s_row``); one launch, no workspace."""
    if x_q.dim() != 2 or x_q.dtype != torch.uint8 or w_q.dim() != 2 or w_q.dtype != torch.uint8:
        raise ValueError("x_q and w_q must be uint8 [M, K] and [N, K] codes")
    M, K = x_q.shape
    N = w_q.shape[0]
    if w_q.shape[1] != K or x_s.dtype != torch.uint8 or w_s.dtype != torch.uint8:
        raise ValueError("x_q [M, K] and w_q [N, K] must share K; scales must be uint8")
    dev = x_q.device
    _check_buffer(x_q, "x_q", dev, M * K, shape=(M, K))
    _check_buffer(w_q, "w_q", dev, N * K, shape=(N, K))
    if K % BLOCK == 0:
        _check_buffer(x_s, "x_s", dev, _scale_numel(M, K, False, "mma"), at_least=True)
        _check_buffer(w_s, "w_s", dev, _scale_numel(N, K, False, "mma"), at_least=True)
    L = library()
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    else:
        _check_buffer(out, "out", dev, M * N, shape=(M, N), dtype=torch.bfloat16)
    with _on_device(dev):
        rc = L.mm_mxfp8_quantized(x_q.data_ptr(), x_s.data_ptr(), M, K, w_q.data_ptr(),
                                  w_s.data_ptr(), N, out.data_ptr(), _stream_handle(stream, dev))
    if rc != 0:
        raise MXFP8Error(rc, L.mxfp8_last_error().decode())
    return out


def mm_mxfp8_workspace_size(M: int, K: int) -> int:
    """Bytes of scratch mm_mxfp8 needs for an [M, K] activation (its
    quantized codes and tiled scales)."""
    return int(library().mm_mxfp8_workspace_size(M, K))


def device_status(clear: bool = True) -> int:
    """The library's device-side status on the current device (synchronizes):
    0 when no kernel wait has given up since the last clear, else the code
    described in include/mxfp8norm.h (mxfp8_device_status)."""
    L = library()
    st = int(L.mxfp8_device_status(int(bool(clear))))
    if st < 0:
        raise MXFP8Error(st, L.mxfp8_last_error().decode())
    return st
