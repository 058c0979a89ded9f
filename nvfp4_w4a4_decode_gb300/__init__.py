"""Python binding of the GB300 small-M NVFP4 W4A4 decode linear.

A thin ctypes layer over the C ABI in ``include/nvfp4.h`` (library
``libnvfp4_gb300.so``): it checks tensor devices/dtypes/shapes, allocates
outputs with torch, passes raw device pointers and the current CUDA stream,
and raises on a non-zero status.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback -- if the library
is missing or fails to load, every call raises.

Entry points keep the C names (``nvfp4_quantize_act`` ...) and have short
aliases (``quantize_act`` ...).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "Nvfp4Error", "library", "nvfp4_global_scale", "nvfp4_pack_weight",
    "nvfp4_quantize_act", "nvfp4_gemm_smallm", "global_scale", "pack_weight",
    "quantize_act", "gemm_smallm", "nvfp4_linear", "linear", "MAX_M",
    "nvfp4_gemm_workspace_size", "nvfp4_workspace", "gemm_workspace_size", "workspace",
    "nvfp4_gemm_smallm_static", "gemm_smallm_static", "nvfp4_read_probe", "read_probe",
    "ChainLinear", "Chain", "CHAIN_MAX_LINEARS", "nvfp4_chain_supported", "chain_supported",
    "TiledWeight", "nvfp4_tile_weight", "tile_weight",
]

MAX_M = 8
STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_UNSUPPORTED", 3: "NVFP4_ERR_CUDA"}

_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64

SIGNATURES = {
    "nvfp4_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "nvfp4_version": ([], ctypes.c_char_p),
    "nvfp4_global_scale": ([_p, _i64, _p, _p], ctypes.c_int),
    "nvfp4_pack_weight": ([_p, _i64, _i64, _p, _p, _p, _p], ctypes.c_int),
    "nvfp4_quantize_act": ([_p, _i64, _i64, _p, _p, _p, _p], ctypes.c_int),
    "nvfp4_gemm_smallm": ([_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p], ctypes.c_int),
    "nvfp4_quantize_act_ex": ([_p, _i64, _i64, _p, _p, _p, ctypes.c_uint32, _p], ctypes.c_int),
    "nvfp4_gemm_smallm_ex": ([_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, ctypes.c_uint32, _p],
                             ctypes.c_int),
    "nvfp4_gemm_select": ([_i64, _i64, _i64, ctypes.c_uint32], ctypes.c_int),
    "nvfp4_device_status": ([_p, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int], ctypes.c_int),
    "nvfp4_linear": ([_p, _i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p, ctypes.c_uint32, _p],
                     ctypes.c_int),
    "nvfp4_quantize_act_dynamic": ([_p, _i64, _i64, _p, _p, _p, _p], ctypes.c_int),
    "nvfp4_gemm_workspace_size": ([_i64, _i64, _i64, ctypes.c_uint32], _i64),
    "nvfp4_gemm_select_ws": ([_i64, _i64, _i64, ctypes.c_uint32, ctypes.c_size_t], ctypes.c_int),
    "nvfp4_gemm_smallm_static": ([_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, ctypes.c_uint32,
                                  _p], ctypes.c_int),
    "nvfp4_gemm_static_scratch_bytes": ([], _i64),
    "nvfp4_gemm_smallm_ws": ([_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, ctypes.c_uint32, _p,
                              ctypes.c_size_t, _p], ctypes.c_int),
    "nvfp4_linear_ws": ([_p, _i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p, ctypes.c_uint32, _p,
                         ctypes.c_size_t, _p], ctypes.c_int),
    "nvfp4_read_probe": ([_p, _i64, _p, _p], ctypes.c_int),
    "nvfp4_linear_chain": ([_p, _i64, _i64, ctypes.c_uint32, _p], ctypes.c_int),
    "nvfp4_gemm_chain": ([_p, _i64, _i64, ctypes.c_uint32, _p], ctypes.c_int),
    "nvfp4_chain_supported": ([_i64, _i64, _i64], ctypes.c_int),
    "nvfp4_linear_chain_ws": ([_p, _i64, _i64, ctypes.c_uint32, _p, ctypes.c_size_t, _p],
                              ctypes.c_int),
    "nvfp4_gemm_chain_ws": ([_p, _i64, _i64, ctypes.c_uint32, _p, ctypes.c_size_t, _p],
                            ctypes.c_int),
    "nvfp4_chain_workspace_size": ([_i64, ctypes.c_uint32], _i64),
    "nvfp4_tiled_weight_bytes": ([_i64, _i64, ctypes.POINTER(_i64)], _i64),
    "nvfp4_tile_weight": ([_p, _p, _i64, _i64, _p, _p, _p], ctypes.c_int),
}

KERNEL_AUTO, KERNEL_GENERIC, KERNEL_GEMV, KERNEL_MMA, KERNEL_TMA, KERNEL_SPLITK = 0, 1, 2, 3, 4, 5
KERNEL_TC = 6
KERNEL_NAMES = {KERNEL_GENERIC: "generic", KERNEL_GEMV: "gemv", KERNEL_MMA: "mma",
                KERNEL_TMA: "tma", KERNEL_SPLITK: "splitk", KERNEL_TC: "tc"}
FLAG_PDL = 0x100
FLAG_FUSED_QUANTIZE = 0x200
FLAG_X_BF16 = 0x400
FLAG_Y_BF16 = 0x800
FLAG_W_TILED = 0x1000
FLAG_TEST_WAIT_TIMEOUT = 0x10000
DEVICE_WAIT_TIMEOUT = 1


class Nvfp4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


def library(path: str | None = None) -> ctypes.CDLL:
    """Load ``libnvfp4_gb300.so`` (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            raise ImportError(f"{path} is not built; run nvfp4_w4a4_decode_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(name: str, status: int):
    if status != 0:
        raise Nvfp4Error(name, status)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _dev(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def nvfp4_global_scale(t: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Tensor scale amax(|t|)/2688 as a 1-element float32 device tensor."""
    _dev(t, torch.float32, "t")
    g = out if out is not None else torch.empty(1, dtype=torch.float32, device=t.device)
    _check("nvfp4_global_scale",
           library().nvfp4_global_scale(t.data_ptr(), t.numel(), g.data_ptr(), _stream(t)))
    return g


def nvfp4_pack_weight(w: torch.Tensor):
    """Quantise W[n, k] (float32) -> (w_q uint8 [n, k/2], w_s uint8 [n, k/16], w_g float32 [1])."""
    _dev(w, torch.float32, "w")
    n, k = w.shape
    wq = torch.empty((n, k // 2), dtype=torch.uint8, device=w.device)
    ws = torch.empty((n, k // 16), dtype=torch.uint8, device=w.device)
    wg = torch.empty(1, dtype=torch.float32, device=w.device)
    _check("nvfp4_pack_weight", library().nvfp4_pack_weight(
        w.data_ptr(), n, k, wq.data_ptr(), ws.data_ptr(), wg.data_ptr(), _stream(w)))
    return wq, ws, wg


def _x_flag(x: torch.Tensor) -> int:
    """The dtype flag of an activation tensor (FP32 or BF16)."""
    if x.dtype == torch.bfloat16:
        _dev(x, torch.bfloat16, "x")
        return FLAG_X_BF16
    _dev(x, torch.float32, "x")
    return 0


def _y_out(out, m: int, n: int, dtype, device):
    """The output tensor and its dtype flag (FP32 or BF16)."""
    if out is None:
        out = torch.empty((m, n), dtype=dtype, device=device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"output must be float32 or bfloat16, got {out.dtype}")
    _dev(out, out.dtype, "out")
    return out, (FLAG_Y_BF16 if out.dtype == torch.bfloat16 else 0)


def nvfp4_quantize_act(x: torch.Tensor, xg: torch.Tensor, out=None, pdl: bool = False):
    """Quantise X[m, k] (float32 or bfloat16) with tensor scale xg ->
    (x_q [m, k/2], x_s [m, k/16])."""
    xflag = _x_flag(x)
    _dev(xg, torch.float32, "xg")
    m, k = x.shape
    if out is None:
        xq = torch.empty((m, k // 2), dtype=torch.uint8, device=x.device)
        xs = torch.empty((m, k // 16), dtype=torch.uint8, device=x.device)
    else:
        xq, xs = out
    _check("nvfp4_quantize_act", library().nvfp4_quantize_act_ex(
        x.data_ptr(), m, k, xg.data_ptr(), xq.data_ptr(), xs.data_ptr(),
        (FLAG_PDL if pdl else 0) | xflag, _stream(x)))
    return xq, xs


def nvfp4_quantize_act_dynamic(x: torch.Tensor, out=None):
    """Quantise X[m, k] with its own tensor scale amax(|X|)/2688 ->
    (x_q [m, k/2], x_s [m, k/16], x_g [1])."""
    _dev(x, torch.float32, "x")
    m, k = x.shape
    if out is None:
        xq = torch.empty((m, k // 2), dtype=torch.uint8, device=x.device)
        xs = torch.empty((m, k // 16), dtype=torch.uint8, device=x.device)
        xg = torch.empty(1, dtype=torch.float32, device=x.device)
    else:
        xq, xs, xg = out
    _check("nvfp4_quantize_act_dynamic", library().nvfp4_quantize_act_dynamic(
        x.data_ptr(), m, k, xg.data_ptr(), xq.data_ptr(), xs.data_ptr(), _stream(x)))
    return xq, xs, xg


def nvfp4_gemm_workspace_size(m: int, n: int, k: int, kernel: int = KERNEL_AUTO) -> int:
    """Bytes of workspace the GEMM of this shape uses (0: none)."""
    v = int(library().nvfp4_gemm_workspace_size(m, n, k, int(kernel) & 0xFF))
    if v < 0:
        raise Nvfp4Error("nvfp4_gemm_workspace_size", -v)
    return v


def nvfp4_workspace(m: int, n: int, k: int, kernel: int = KERNEL_AUTO,
                    device=None) -> torch.Tensor | None:
    """A zeroed workspace for GEMMs of this shape (None when none is needed).
    It can be reused by any number of calls that do not overlap in time."""
    size = nvfp4_gemm_workspace_size(m, n, k, kernel)
    if size == 0:
        return None
    return torch.zeros(size, dtype=torch.uint8,
                       device=device if device is not None else torch.cuda.current_device())


def _ws_args(workspace, m, n, k, kernel, device):
    """(pointer, bytes, keep-alive) of the workspace for one call; a zeroed
    one is made for this call when none is given and the GEMM wants one;
    ``False`` offers none (as the plain boundary call does)."""
    if workspace is False:
        return None, 0, None
    if workspace is None:
        workspace = nvfp4_workspace(m, n, k, kernel, device) if m and n and k else None
    if workspace is None:
        return None, 0, None
    _dev(workspace, torch.uint8, "workspace")
    return workspace.data_ptr(), workspace.numel(), workspace


def nvfp4_gemm_smallm(xq, xs, xg, wq, ws, wg, out: torch.Tensor | None = None,
                      kernel: int = KERNEL_AUTO, pdl: bool = False,
                      test_wait_timeout: bool = False,
                      workspace: torch.Tensor | None = None,
                      out_dtype=torch.float32) -> torch.Tensor:
    """Y[m, n] = dequant(X) . dequant(W)^T for m <= 8, float32.

    ``kernel`` forces one kernel (KERNEL_GENERIC, KERNEL_GEMV, KERNEL_MMA,
    KERNEL_TMA, KERNEL_SPLITK); ``pdl`` lets the launch overlap the previous
    kernel (weights must not be written by it); ``workspace`` (from
    ``nvfp4_workspace``) is made per call when the kernel needs one and none
    is given (``False``: none is offered, so the split-K kernel takes one
    chunk or its cluster form).  The output is float32, or bfloat16
    (``out_dtype`` or the dtype
    of ``out``): the float32 result rounded to nearest even."""
    tiled = isinstance(wq, TiledWeight)
    if tiled:                        # gemm_smallm(xq, xs, xg, TiledWeight, ...)
        tw = wq
        if ws is not None or wg is not None:
            raise ValueError("pass a TiledWeight in place of (wq, ws, wg), with ws = wg = None")
        wq, ws, wg = tw.t_q, tw.t_s, tw.w_g
    for t, name in ((xq, "xq"), (xs, "xs"), (wq, "wq"), (ws, "ws")):
        _dev(t, torch.uint8, name)
    _dev(xg, torch.float32, "xg")
    _dev(wg, torch.float32, "wg")
    m, kh = xq.shape
    k = kh * 2
    if tiled:
        n = tw.n
        if tw.k != k or xs.shape != (m, k // 16):
            raise ValueError("operand shapes disagree")
        kernel = KERNEL_TC
    else:
        n = wq.shape[0]
        if wq.shape[1] != kh or xs.shape != (m, k // 16) or ws.shape != (n, k // 16):
            raise ValueError("operand shapes disagree")
    y, yflag = _y_out(out, m, n, out_dtype, xq.device)
    opts = int(kernel) | (FLAG_PDL if pdl else 0) | (FLAG_TEST_WAIT_TIMEOUT if test_wait_timeout else 0)
    opts |= yflag | (FLAG_W_TILED if tiled else 0)
    wp, wn, _keep = _ws_args(workspace, m, n, k, kernel, xq.device)
    _check("nvfp4_gemm_smallm", library().nvfp4_gemm_smallm_ws(
        xq.data_ptr(), xs.data_ptr(), xg.data_ptr(), wq.data_ptr(), ws.data_ptr(),
        wg.data_ptr(), y.data_ptr(), m, n, k, opts, wp, wn, _stream(xq)))
    return y


def nvfp4_gemm_smallm_static(xq, xs, xg, wq, ws, wg, out: torch.Tensor | None = None,
                             pdl: bool = False, out_dtype=torch.float32) -> torch.Tensor:
    """The split-K GEMM on the library's static scratch array (no workspace,
    no allocation in the library): same result bits as ``nvfp4_gemm_smallm``
    with KERNEL_SPLITK and a full workspace.  Calls that may overlap in time
    share the one array and race."""
    for t, name in ((xq, "xq"), (xs, "xs"), (wq, "wq"), (ws, "ws")):
        _dev(t, torch.uint8, name)
    _dev(xg, torch.float32, "xg")
    _dev(wg, torch.float32, "wg")
    m, kh = xq.shape
    n = wq.shape[0]
    k = kh * 2
    if wq.shape[1] != kh or xs.shape != (m, k // 16) or ws.shape != (n, k // 16):
        raise ValueError("operand shapes disagree")
    y, yflag = _y_out(out, m, n, out_dtype, xq.device)
    _check("nvfp4_gemm_smallm_static", library().nvfp4_gemm_smallm_static(
        xq.data_ptr(), xs.data_ptr(), xg.data_ptr(), wq.data_ptr(), ws.data_ptr(),
        wg.data_ptr(), y.data_ptr(), m, n, k, KERNEL_SPLITK | (FLAG_PDL if pdl else 0) | yflag,
        _stream(xq)))
    return y


def nvfp4_gemm_select(m: int, n: int, k: int, kernel: int = KERNEL_AUTO,
                      workspace_bytes: int = 0) -> int:
    """Kernel id the library runs for this shape when offered
    ``workspace_bytes`` of workspace (negative status if none)."""
    return library().nvfp4_gemm_select_ws(m, n, k, kernel, workspace_bytes)


def nvfp4_read_probe(buf: torch.Tensor, sink: torch.Tensor | None = None) -> torch.Tensor:
    """Read-only streaming probe over a contiguous CUDA tensor (16-byte
    aligned, size a multiple of 16 bytes): returns a uint64 device scalar
    (as int64 storage) holding the XOR of all 8-byte words of ``buf``.  A
    measurement aid; time it with CUDA events on the current stream."""
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    if sink is None:
        sink = torch.empty(1, dtype=torch.int64, device=buf.device)
    _check("nvfp4_read_probe", library().nvfp4_read_probe(
        buf.data_ptr(), buf.numel() * buf.element_size(), sink.data_ptr(), _stream(buf)))
    return sink


def nvfp4_device_status(clear: bool = True, stream=None) -> int:
    """Device status bits recorded by the kernels (synchronises the stream)."""
    v = ctypes.c_uint32(0)
    st = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _check("nvfp4_device_status", library().nvfp4_device_status(st, ctypes.byref(v), int(clear)))
    return int(v.value)


def nvfp4_linear(x: torch.Tensor, xg: torch.Tensor, wq, ws, wg, out=None, x_out=None,
                 kernel: int = KERNEL_AUTO, pdl: bool = False,
                 fused: bool = False, workspace: torch.Tensor | None = None,
                 out_dtype=torch.float32) -> torch.Tensor:
    """One W4A4 decode linear: quantise X[m, k] on the fly and multiply by the
    packed W[n, k].  ``fused`` asks for one kernel (where the CUDA-core stream
    takes the shape); ``x_out`` = (x_q, x_s) receive the quantised activations;
    ``workspace`` as in ``nvfp4_gemm_smallm``.  X may be float32 or bfloat16;
    the output is float32 or bfloat16 (``out_dtype`` or the dtype of ``out``)."""
    xflag = _x_flag(x)
    for t, name in ((wq, "wq"), (ws, "ws")):
        _dev(t, torch.uint8, name)
    _dev(xg, torch.float32, "xg")
    _dev(wg, torch.float32, "wg")
    m, k = x.shape
    n = wq.shape[0]
    if wq.shape[1] * 2 != k or ws.shape != (n, k // 16):
        raise ValueError("operand shapes disagree")
    if x_out is None:
        xq = torch.empty((m, k // 2), dtype=torch.uint8, device=x.device)
        xs = torch.empty((m, k // 16), dtype=torch.uint8, device=x.device)
    else:
        xq, xs = x_out
    y, yflag = _y_out(out, m, n, out_dtype, x.device)
    opts = int(kernel) | (FLAG_PDL if pdl else 0) | (FLAG_FUSED_QUANTIZE if fused else 0)
    opts |= xflag | yflag
    wp, wn, _keep = _ws_args(workspace, m, n, k, kernel, x.device)
    _check("nvfp4_linear", library().nvfp4_linear_ws(
        x.data_ptr(), m, n, k, xg.data_ptr(), wq.data_ptr(), ws.data_ptr(), wg.data_ptr(),
        y.data_ptr(), xq.data_ptr(), xs.data_ptr(), opts, wp, wn, _stream(x)))
    return y


linear = nvfp4_linear


# ---- tile-major weights of the tensor-core kernel ------------------------------

class TiledWeight:
    """Packed weights in the tensor-core kernel's tile-major layout
    (``nvfp4_tile_weight``): ``t_q`` / ``t_s`` flat uint8 device tensors, the
    tensor scale ``w_g`` and the logical shape (n, k).  Accepted wherever a
    ``(w_q, w_s, w_g)`` triple is, on the tensor-core kernel."""

    def __init__(self, t_q, t_s, w_g, n: int, k: int):
        self.t_q, self.t_s, self.w_g, self.n, self.k = t_q, t_s, w_g, int(n), int(k)


def nvfp4_tile_weight(wq: torch.Tensor, ws: torch.Tensor, wg: torch.Tensor) -> TiledWeight:
    """Repack row-major packed weights (w_q [n, k/2], w_s [n, k/16]) into the
    tile-major layout; k a multiple of 256."""
    _dev(wq, torch.uint8, "wq")
    _dev(ws, torch.uint8, "ws")
    _dev(wg, torch.float32, "wg")
    n, kh = wq.shape
    k = kh * 2
    if ws.shape != (n, k // 16):
        raise ValueError("operand shapes disagree")
    sb = _i64(0)
    qb = int(library().nvfp4_tiled_weight_bytes(n, k, ctypes.byref(sb)))
    if qb < 0:
        raise Nvfp4Error("nvfp4_tiled_weight_bytes", -qb)
    tq = torch.empty(max(qb, 16), dtype=torch.uint8, device=wq.device)
    ts = torch.empty(max(sb.value, 16), dtype=torch.uint8, device=wq.device)
    _check("nvfp4_tile_weight", library().nvfp4_tile_weight(
        wq.data_ptr(), ws.data_ptr(), n, k, tq.data_ptr(), ts.data_ptr(), _stream(wq)))
    return TiledWeight(tq, ts, wg, n, k)


tile_weight = nvfp4_tile_weight


# ---- many independent linears in one persistent launch ----------------------

CHAIN_MAX_LINEARS = 256
TC_MAX_LINEARS = 150


class ChainLinear(ctypes.Structure):
    """``nvfp4_chain_linear`` of include/nvfp4.h (device pointers, sizes)."""
    _fields_ = [("x", _p), ("x_g", _p), ("x_q", _p), ("x_s", _p), ("w_q", _p), ("w_s", _p),
                ("w_g", _p), ("y", _p), ("n", _i64), ("k", _i64)]


def nvfp4_chain_supported(m: int, n: int, k: int) -> bool:
    """Whether a linear of this shape can be part of a chain."""
    return bool(library().nvfp4_chain_supported(m, n, k))


class Chain:
    """A fixed list of independent linears run as one multi-linear call
    (``nvfp4_linear_chain_ws`` / ``nvfp4_gemm_chain_ws``).

    ``linears`` is a sequence of ``(x, xg, (xq, xs), (wq, ws, wg), y)``: x
    [m, k] float32 or bfloat16 (the same dtype for every linear), xg [1]
    float32, xq [m, k/2] / xs [m, k/16] uint8 (written by ``run``, read by
    ``gemm_only``), the packed weights, and y [m, n] float32 or bfloat16 (the
    same dtype for every linear).  The descriptions are built once; the
    tensors must stay alive and in place while the chain is used.  With
    ``workspace`` (default) the tensor-core kernel gets a zeroed workspace of
    its own, so calls of one Chain must not overlap in time."""

    def __init__(self, linears, kernel: int = KERNEL_AUTO, workspace: bool = True):
        if not linears:
            raise ValueError("a chain needs at least one linear")
        descs = []
        self._keep = []
        xdt = ydt = None
        m = None
        tiled = None
        for x, xg, (xq, xs), wts, y in linears:
            is_tiled = isinstance(wts, TiledWeight)
            if tiled is None:
                tiled = is_tiled
            elif tiled != is_tiled:
                raise ValueError("every linear of a chain has the same weight layout")
            if is_tiled:
                wq, ws, wg = wts.t_q, wts.t_s, wts.w_g
            else:
                wq, ws, wg = wts
            if x.dtype not in (torch.float32, torch.bfloat16):
                raise ValueError(f"x must be float32 or bfloat16, got {x.dtype}")
            _dev(x, x.dtype, "x")
            _dev(xg, torch.float32, "xg")
            for t, name in ((xq, "xq"), (xs, "xs"), (wq, "wq"), (ws, "ws")):
                _dev(t, torch.uint8, name)
            _dev(wg, torch.float32, "wg")
            if y.dtype not in (torch.float32, torch.bfloat16):
                raise ValueError(f"y must be float32 or bfloat16, got {y.dtype}")
            _dev(y, y.dtype, "y")
            mm, k = x.shape
            n = wts.n if is_tiled else wq.shape[0]
            if is_tiled:
                wshape_ok = wts.k == k
            else:
                wshape_ok = wq.shape == (n, k // 2) and ws.shape == (n, k // 16)
            if (xq.shape != (mm, k // 2) or xs.shape != (mm, k // 16) or not wshape_ok
                    or y.shape != (mm, n)):
                raise ValueError("operand shapes disagree")
            if m is None:
                m, xdt, ydt = mm, x.dtype, y.dtype
            elif mm != m or x.dtype != xdt or y.dtype != ydt:
                raise ValueError("every linear of a chain has the same m and dtypes")
            descs.append(ChainLinear(x.data_ptr(), xg.data_ptr(), xq.data_ptr(), xs.data_ptr(),
                                     wq.data_ptr(), ws.data_ptr(), wg.data_ptr(), y.data_ptr(),
                                     n, k))
            self._keep.append((x, xg, xq, xs, wq, ws, wg, y))
        self.m = m
        self.count = len(descs)
        self._arr = (ChainLinear * self.count)(*descs)
        self.tiled = bool(tiled)
        self._flags = (FLAG_X_BF16 if xdt == torch.bfloat16 else 0) | \
                      (FLAG_Y_BF16 if ydt == torch.bfloat16 else 0) | \
                      (FLAG_W_TILED if self.tiled else 0)
        self.device = linears[0][0].device
        self.kernel = int(kernel)
        if self.kernel == KERNEL_AUTO:
            self.engine = KERNEL_TC          # the library's choice at every m
        else:
            self.engine = self.kernel
        # the tensor-core kernel balances its CTAs through a zeroed workspace
        self.workspace = None
        if workspace:
            size = int(library().nvfp4_chain_workspace_size(m, self.kernel))
            if size < 0:
                raise Nvfp4Error("nvfp4_chain_workspace_size", -size)
            if size:
                self.workspace = torch.zeros(size, dtype=torch.uint8, device=self.device)

    def _ws(self):
        if self.workspace is None:
            return None, 0
        return self.workspace.data_ptr(), self.workspace.numel()

    def run(self, pdl: bool = False):
        """Quantise every linear's X and compute every Y (two launches per
        CHAIN_MAX_LINEARS linears) on the current stream."""
        wp, wn = self._ws()
        _check("nvfp4_linear_chain", library().nvfp4_linear_chain_ws(
            ctypes.cast(self._arr, ctypes.c_void_p), self.count, self.m,
            self.kernel | self._flags | (FLAG_PDL if pdl else 0), wp, wn,
            torch.cuda.current_stream(self.device).cuda_stream))

    def launches(self, quantize: bool = True) -> int:
        """Kernel launches of one call."""
        per = TC_MAX_LINEARS if self.engine == KERNEL_TC else CHAIN_MAX_LINEARS
        return -(-self.count // per) * (2 if quantize else 1)

    def gemm_only(self, pdl: bool = False):
        """Every Y from the codes already in each xq / xs (one launch per
        CHAIN_MAX_LINEARS, or TC_MAX_LINEARS, linears)."""
        wp, wn = self._ws()
        _check("nvfp4_gemm_chain", library().nvfp4_gemm_chain_ws(
            ctypes.cast(self._arr, ctypes.c_void_p), self.count, self.m,
            self.kernel | (self._flags & (FLAG_Y_BF16 | FLAG_W_TILED)) | (FLAG_PDL if pdl else 0),
            wp, wn,
            torch.cuda.current_stream(self.device).cuda_stream))


chain_supported = nvfp4_chain_supported


global_scale = nvfp4_global_scale
pack_weight = nvfp4_pack_weight
quantize_act = nvfp4_quantize_act
quantize_act_dynamic = nvfp4_quantize_act_dynamic
gemm_smallm = nvfp4_gemm_smallm
gemm_select = nvfp4_gemm_select
gemm_workspace_size = nvfp4_gemm_workspace_size
gemm_smallm_static = nvfp4_gemm_smallm_static
workspace = nvfp4_workspace
device_status = nvfp4_device_status
read_probe = nvfp4_read_probe
