"""Thin ctypes binding of the C ABI in include/qmm.h.

Argument marshalling only: every step of the computation runs in the CUDA
library (``_build/libqmm_gb300.so``).  There is no CPU fallback; if the
library has not been built, every call raises.

The ``qmm_*`` functions mirror the C entry points one to one (same names,
same argument order; tensors stand in for device pointers, ``stream`` defaults
to torch's current stream) and return the integer ``qmm_status``.  The short
names (``gemv``, ``gemm``, ``matmul``, ``dequant``) allocate the output and
raise ``QmmError`` on any non-OK status.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

Q8_0, Q4_0, Q4_K, Q6_K, Q5_K = 0, 1, 2, 3, 4
X_F32, X_BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
GEMV_MAX_N, GEMM_MAX_N = 16, 512
MATMUL_GEMV_MAX_N = 8    # qmm_matmul's default GEMV/GEMM crossover (QMM_MATMUL_GEMV_MAX_N)
BLOCK = {Q8_0: (32, 34), Q4_0: (32, 18), Q4_K: (256, 144), Q6_K: (256, 210), Q5_K: (256, 176)}
EXPORTS = ("qmm_gemv", "qmm_gemv_argmax", "qmm_gemv_multi", "qmm_gemm", "qmm_gemm_workspace_bytes", "qmm_matmul", "qmm_matmul_host",
           "qmm_dequant", "qmm_block_info", "qmm_last_device_error", "qmm_status_str",
           "qmm_set_wait_limit", "qmm_set_static_weights", "qmm_set_gemv_i8", "qmm_set_gemv_tc", "qmm_quantize_q8_0",
           "qmm_gemv_preq", "qmm_q8act_workspace_bytes", "qmm_gemv_q8act", "qmm_gemv_swiglu",
           "qmm_gemm_q8act_workspace_bytes", "qmm_gemm_q8act", "qmm_gemm_swiglu_workspace_bytes", "qmm_gemm_swiglu",
           "qmm_kernel_launches", "qmm_set_gemv_stream", "qmm_gemv_stream_plan")

_lock = threading.Lock()
_lib = None


class QmmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_name(status)}" if what else status_name(status))


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"CUDA library not built ({_build.LIB}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB)
        i64, sz, p, ci = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
        lib.qmm_gemv.argtypes = [ci, p, sz, i64, i64, p, ci, i64, p, p]
        lib.qmm_gemv_argmax.argtypes = [ci, p, sz, i64, i64, p, ci, i64, p, p, p, sz, p]
        lib.qmm_gemv_multi.argtypes = [ci, p, ci, i64, p, ci, i64, p]
        lib.qmm_gemm.argtypes = [ci, p, sz, i64, i64, p, ci, i64, p, p, sz, p]
        lib.qmm_matmul.argtypes = [ci, p, sz, i64, i64, p, ci, i64, p, p, sz, p]
        lib.qmm_matmul_host.argtypes = [ci, p, sz, i64, i64, p, ci, i64, p, p, p, p, sz, p]
        lib.qmm_dequant.argtypes = [ci, p, sz, i64, i64, p, p]
        lib.qmm_block_info.argtypes = [ci, p, p]
        lib.qmm_last_device_error.argtypes = [p]
        lib.qmm_gemm_workspace_bytes.argtypes = [i64, i64, ci]
        lib.qmm_gemm_workspace_bytes.restype = sz
        lib.qmm_status_str.argtypes = [ci]
        lib.qmm_status_str.restype = ctypes.c_char_p
        lib.qmm_set_wait_limit.argtypes = [ctypes.c_uint64]
        lib.qmm_set_wait_limit.restype = None
        lib.qmm_set_static_weights.argtypes = [ctypes.c_int]
        lib.qmm_set_static_weights.restype = None
        lib.qmm_set_gemv_i8.argtypes = [ctypes.c_int]
        lib.qmm_set_gemv_i8.restype = None
        lib.qmm_set_gemv_tc.argtypes = [ctypes.c_int]
        lib.qmm_set_gemv_tc.restype = None
        lib.qmm_set_gemv_stream.argtypes = [ci, ci, ci, ci, ci]
        lib.qmm_set_gemv_stream.restype = None
        lib.qmm_gemv_stream_plan.argtypes = [ci, i64, i64, p]
        lib.qmm_quantize_q8_0.argtypes = [p, ci, i64, i64, p, p, p]
        lib.qmm_gemv_preq.argtypes = [ci, p, sz, i64, i64, p, p, i64, p, p]
        lib.qmm_q8act_workspace_bytes.argtypes = [i64, i64]
        lib.qmm_q8act_workspace_bytes.restype = sz
        lib.qmm_gemv_q8act.argtypes = [ci, p, sz, i64, i64, p, ci, i64, p, p, sz, p]
        lib.qmm_gemv_swiglu.argtypes = [ci, p, sz, p, sz, i64, i64, p, ci, i64, p, p, sz, p]
        lib.qmm_gemm_q8act_workspace_bytes.argtypes = [i64, i64]
        lib.qmm_gemm_q8act_workspace_bytes.restype = sz
        lib.qmm_gemm_q8act.argtypes = [ci, p, sz, i64, i64, p, ci, i64, p, p, sz, p]
        lib.qmm_gemm_swiglu_workspace_bytes.argtypes = [i64, i64, i64, ci]
        lib.qmm_gemm_swiglu_workspace_bytes.restype = sz
        lib.qmm_gemm_swiglu.argtypes = [ci, p, sz, p, sz, i64, i64, p, ci, i64, p, p, sz, p]
        lib.qmm_kernel_launches.argtypes = []
        lib.qmm_kernel_launches.restype = ctypes.c_uint64
        for f in ("qmm_gemv", "qmm_gemv_argmax", "qmm_gemv_multi", "qmm_gemm", "qmm_matmul", "qmm_matmul_host", "qmm_dequant", "qmm_block_info",
                  "qmm_last_device_error", "qmm_quantize_q8_0", "qmm_gemv_preq", "qmm_gemv_q8act", "qmm_gemv_swiglu",
                  "qmm_gemm_q8act", "qmm_gemm_swiglu"):
            getattr(lib, f).restype = ci
        _lib = lib
        return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


def _xtype(X) -> int:
    if X.dtype == torch.float32:
        return X_F32
    if X.dtype == torch.bfloat16:
        return X_BF16
    raise TypeError("X must be float32 or bfloat16")


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def status_name(s: int) -> str:
    return load().qmm_status_str(s).decode()


# --------------------------------------------------------------------------
# one-to-one mirrors of the C entry points (return qmm_status)
# --------------------------------------------------------------------------
def qmm_gemv(wt, W, M, K, X, N, Y, stream=None, w_bytes=None, xt=None) -> int:
    return load().qmm_gemv(wt, _ptr(W), _nbytes(W) if w_bytes is None else w_bytes, M, K, _ptr(X),
                           _xtype(X) if xt is None else xt, N, _ptr(Y), _stream(stream))


def qmm_gemv_argmax(wt, W, M, K, X, N, idx, val, workspace, stream=None, w_bytes=None, xt=None) -> int:
    return load().qmm_gemv_argmax(wt, _ptr(W), _nbytes(W) if w_bytes is None else w_bytes, M, K, _ptr(X),
                                  _xtype(X) if xt is None else xt, N, _ptr(idx), _ptr(val), _ptr(workspace),
                                  _nbytes(workspace), _stream(stream))


class QmmMatrix(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("w_bytes", ctypes.c_size_t), ("M", ctypes.c_int64), ("Y", ctypes.c_void_p)]


def qmm_gemv_multi(wt, mats, K, X, N, stream=None, xt=None) -> int:
    """mats: list of (W, M, Y) sharing X; one launch."""
    arr = (QmmMatrix * len(mats))(*[QmmMatrix(_ptr(W), _nbytes(W), M, _ptr(Y)) for (W, M, Y) in mats])
    return load().qmm_gemv_multi(wt, ctypes.cast(arr, ctypes.c_void_p), len(mats), K, _ptr(X),
                                 _xtype(X) if xt is None else xt, N, _stream(stream))


def gemv_multi(wt, Ws_and_Ms, K, X, stream=None):
    """[Y_i [N, M_i]] for [(W_i, M_i)] sharing X, in one launch."""
    N = _shape(X, K)
    Ys = [torch.empty(N, M, dtype=torch.float32, device=X.device) for (_, M) in Ws_and_Ms]
    _check(qmm_gemv_multi(wt, [(W, M, Y) for (W, M), Y in zip(Ws_and_Ms, Ys)], K, X, N, stream), "qmm_gemv_multi")
    return Ys


def gemv_argmax(wt, W, M, K, X, stream=None):
    """(idx int32 [N], val float32 [N]): per token, the row of the largest
    GEMV output and that output, without materializing the outputs."""
    N = _shape(X, K)
    idx = torch.empty(N, dtype=torch.int32, device=X.device)
    val = torch.empty(N, dtype=torch.float32, device=X.device)
    ws = torch.empty(N + 1, dtype=torch.int64, device=X.device)
    _check(qmm_gemv_argmax(wt, W, M, K, X, N, idx, val, ws, stream), "qmm_gemv_argmax")
    return idx, val


def qmm_gemm(wt, W, M, K, X, N, Y, workspace=None, ws_bytes=None, stream=None, w_bytes=None, xt=None) -> int:
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else _nbytes(workspace)
    return load().qmm_gemm(wt, _ptr(W), _nbytes(W) if w_bytes is None else w_bytes, M, K, _ptr(X),
                           _xtype(X) if xt is None else xt, N, _ptr(Y), _ptr(workspace), ws_bytes,
                           _stream(stream))


def qmm_matmul(wt, W, M, K, X, N, Y, workspace=None, ws_bytes=None, stream=None, w_bytes=None, xt=None) -> int:
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else _nbytes(workspace)
    return load().qmm_matmul(wt, _ptr(W), _nbytes(W) if w_bytes is None else w_bytes, M, K, _ptr(X),
                             _xtype(X) if xt is None else xt, N, _ptr(Y), _ptr(workspace), ws_bytes,
                             _stream(stream))


def qmm_matmul_host(wt, W, M, K, X_host, N, Y_host, x_dev, y_dev, workspace=None, ws_bytes=None,
                    stream=None) -> int:
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else _nbytes(workspace)
    return load().qmm_matmul_host(wt, _ptr(W), _nbytes(W), M, K, _ptr(X_host), _xtype(X_host), N, _ptr(Y_host),
                                  _ptr(x_dev), _ptr(y_dev), _ptr(workspace), ws_bytes, _stream(stream))


def qmm_dequant(wt, W, M, K, out, stream=None, w_bytes=None) -> int:
    return load().qmm_dequant(wt, _ptr(W), _nbytes(W) if w_bytes is None else w_bytes, M, K, _ptr(out),
                              _stream(stream))


def qmm_block_info(wt):
    e, b = ctypes.c_int(), ctypes.c_int()
    s = load().qmm_block_info(wt, ctypes.byref(e), ctypes.byref(b))
    return s, e.value, b.value


def qmm_gemm_workspace_bytes(N, K, xt) -> int:
    return load().qmm_gemm_workspace_bytes(N, K, xt)


def qmm_kernel_launches() -> int:
    return int(load().qmm_kernel_launches())


def qmm_last_device_error(stream=None) -> int:
    return load().qmm_last_device_error(_stream(stream))


def qmm_status_str(s: int) -> str:
    return status_name(s)


def qmm_set_wait_limit(cycles: int) -> None:
    load().qmm_set_wait_limit(cycles)


# --------------------------------------------------------------------------
# convenience wrappers (allocate the output, raise on error)
# --------------------------------------------------------------------------
def qmm_set_static_weights(on: bool) -> None:
    """Static-weights mode (see include/qmm.h): weights stream before the
    preceding kernel on the stream ends; W must not be written meanwhile."""
    load().qmm_set_static_weights(1 if on else 0)


def qmm_set_gemv_i8(on: int) -> None:
    """GEMV kernel for N <= 2 (see include/qmm.h): 1 integer kernel, 0 bf16
    kernel, -1 the environment's choice (QMM_GEMV_I8, default off)."""
    load().qmm_set_gemv_i8(int(on))


def qmm_set_gemv_tc(on: int) -> None:
    """GEMV kernel for 2 <= N <= 4 (see include/qmm.h): 1 the 16-row-tile
    tensor-core kernel, 0 the ring kernel, -1 the environment's choice
    (QMM_GEMV_TC, default off)."""
    load().qmm_set_gemv_tc(int(on))


def qmm_set_gemv_stream(rows_per_task: int, warps: int = 0, slots: int = 0, ctas_per_sm: int = 0,
                        direct: int = -1) -> None:
    """Plan parameters of the N = 1 streaming GEMV (see include/qmm.h):
    0 = the planner's choice, -1 = the environment's."""
    load().qmm_set_gemv_stream(int(rows_per_task), int(warps), int(slots), int(ctas_per_sm), int(direct))


def qmm_gemv_stream_plan(wt: int, M: int, K: int):
    """(status, {grid, warps, slots, rows_per_task, smem, direct}) of the streaming
    GEMV for an M x K matrix under the present settings."""
    out = (ctypes.c_int32 * 6)()
    st = load().qmm_gemv_stream_plan(int(wt), int(M), int(K), out)
    keys = ("grid", "warps", "slots", "rows_per_task", "smem", "direct")
    return st, (dict(zip(keys, (int(v) for v in out))) if st == OK else None)


def qmm_quantize_q8_0(X, N, K, scales, quants, stream=None, xt=None) -> int:
    return load().qmm_quantize_q8_0(_ptr(X), _xtype(X) if xt is None else xt, N, K, _ptr(scales), _ptr(quants),
                                    _stream(stream))


def qmm_gemv_preq(wt, W, M, K, scales, quants, N, Y, stream=None, w_bytes=None) -> int:
    return load().qmm_gemv_preq(wt, _ptr(W), _nbytes(W) if w_bytes is None else w_bytes, M, K, _ptr(scales),
                                _ptr(quants), N, _ptr(Y), _stream(stream))


def qmm_q8act_workspace_bytes(N, K) -> int:
    return load().qmm_q8act_workspace_bytes(N, K)


def qmm_gemv_q8act(wt, W, M, K, X, N, Y, workspace, ws_bytes=None, stream=None, w_bytes=None, xt=None) -> int:
    return load().qmm_gemv_q8act(wt, _ptr(W), _nbytes(W) if w_bytes is None else w_bytes, M, K, _ptr(X),
                                 _xtype(X) if xt is None else xt, N, _ptr(Y), _ptr(workspace),
                                 _nbytes(workspace) if ws_bytes is None else ws_bytes, _stream(stream))


def qmm_gemv_swiglu(wt, Wg, Wu, M, K, X, N, Y, workspace, stream=None, xt=None) -> int:
    return load().qmm_gemv_swiglu(wt, _ptr(Wg), _nbytes(Wg), _ptr(Wu), _nbytes(Wu), M, K, _ptr(X),
                                  _xtype(X) if xt is None else xt, N, _ptr(Y), _ptr(workspace), _nbytes(workspace),
                                  _stream(stream))


def gemv_swiglu(wt, Wg, Wu, M, K, X, Y=None, workspace=None, stream=None):
    """silu(X Wg^T) * (X Wu^T), [N, M]; the workspace keeps both projections."""
    N = _shape(X, K)
    Y = torch.empty((N, M), dtype=torch.float32, device=X.device) if Y is None else Y
    if workspace is None:
        workspace = torch.empty(2 * N * M, dtype=torch.float32, device=X.device)
    _check(qmm_gemv_swiglu(wt, Wg, Wu, M, K, X, N, Y, workspace, stream), "qmm_gemv_swiglu")
    return Y


def qmm_gemm_q8act(wt, W, M, K, X, N, Y, workspace, stream=None, w_bytes=None, xt=None) -> int:
    return load().qmm_gemm_q8act(wt, _ptr(W), _nbytes(W) if w_bytes is None else w_bytes, M, K, _ptr(X),
                                 _xtype(X) if xt is None else xt, N, _ptr(Y), _ptr(workspace), _nbytes(workspace),
                                 _stream(stream))


def gemm_q8act(wt, W, M, K, X, Y=None, workspace=None, stream=None):
    """Y [N, M]: the tensor-core GEMM on the Q8_0-quantized activations of X."""
    N = _shape(X, K)
    Y = torch.empty((N, M), dtype=torch.float32, device=X.device) if Y is None else Y
    if workspace is None:
        workspace = torch.empty(load().qmm_gemm_q8act_workspace_bytes(N, K), dtype=torch.uint8, device=X.device)
    _check(qmm_gemm_q8act(wt, W, M, K, X, N, Y, workspace, stream=stream), "qmm_gemm_q8act")
    return Y


def qmm_gemm_swiglu(wt, Wg, Wu, M, K, X, N, Y, workspace, stream=None, xt=None) -> int:
    return load().qmm_gemm_swiglu(wt, _ptr(Wg), _nbytes(Wg), _ptr(Wu), _nbytes(Wu), M, K, _ptr(X),
                                  _xtype(X) if xt is None else xt, N, _ptr(Y), _ptr(workspace), _nbytes(workspace),
                                  _stream(stream))


def gemm_swiglu(wt, Wg, Wu, M, K, X, Y=None, workspace=None, stream=None):
    """silu(X Wg^T) * (X Wu^T), [N, M], on the tensor-core GEMM (one launch
    for both projections)."""
    N = _shape(X, K)
    Y = torch.empty((N, M), dtype=torch.float32, device=X.device) if Y is None else Y
    if workspace is None:
        n = load().qmm_gemm_swiglu_workspace_bytes(N, M, K, _xtype(X))
        workspace = torch.empty(n, dtype=torch.uint8, device=X.device)
    _check(qmm_gemm_swiglu(wt, Wg, Wu, M, K, X, N, Y, workspace, stream), "qmm_gemm_swiglu")
    return Y


def quantize_q8_0(X, stream=None):
    """(scales f32 [N, K/32], quants int8 [N, K]) of X [N, K] (f32 or bf16)."""
    N, K = X.shape
    scales = torch.empty((N, K // 32), dtype=torch.float32, device=X.device)
    quants = torch.empty((N, K), dtype=torch.int8, device=X.device)
    _check(qmm_quantize_q8_0(X, N, K, scales, quants, stream), "qmm_quantize_q8_0")
    return scales, quants


def gemv_q8act(wt, W, M, K, X, Y=None, workspace=None, stream=None):
    """Y [N, M] of the Q8_0-activation GEMV of X [N, K] (1 <= N <= 16)."""
    N = _shape(X, K)
    Y = torch.empty((N, M), dtype=torch.float32, device=X.device) if Y is None else Y
    if workspace is None:
        workspace = torch.empty(qmm_q8act_workspace_bytes(N, K), dtype=torch.uint8, device=X.device)
    _check(qmm_gemv_q8act(wt, W, M, K, X, N, Y, workspace, stream=stream), "qmm_gemv_q8act")
    return Y


def _check(s: int, what: str):
    if s != OK:
        raise QmmError(s, what)


def _shape(X, K):
    if X.dim() != 2 or X.shape[1] != K:
        raise ValueError(f"X must be [N, {K}]")
    return X.shape[0]


def gemv(wt, W, M, K, X, Y=None, stream=None):
    N = _shape(X, K)
    Y = torch.empty((N, M), dtype=torch.float32, device=X.device) if Y is None else Y
    _check(qmm_gemv(wt, W, M, K, X, N, Y, stream), "qmm_gemv")
    return Y


def workspace_for(N, K, X):
    n = qmm_gemm_workspace_bytes(N, K, _xtype(X))
    return torch.empty(max(n, 16), dtype=torch.uint8, device=X.device) if n else None


def gemm(wt, W, M, K, X, Y=None, workspace=None, stream=None):
    N = _shape(X, K)
    Y = torch.empty((N, M), dtype=torch.float32, device=X.device) if Y is None else Y
    workspace = workspace_for(N, K, X) if workspace is None else workspace
    _check(qmm_gemm(wt, W, M, K, X, N, Y, workspace, stream=stream), "qmm_gemm")
    return Y


def matmul(wt, W, M, K, X, Y=None, workspace=None, stream=None):
    N = _shape(X, K)
    Y = torch.empty((N, M), dtype=torch.float32, device=X.device) if Y is None else Y
    workspace = workspace_for(N, K, X) if workspace is None else workspace
    _check(qmm_matmul(wt, W, M, K, X, N, Y, workspace, stream=stream), "qmm_matmul")
    return Y


def dequant(wt, W, M, K, out=None, stream=None):
    out = torch.empty((M, K), dtype=torch.float32, device=W.device) if out is None else out
    _check(qmm_dequant(wt, W, M, K, out, stream), "qmm_dequant")
    return out
