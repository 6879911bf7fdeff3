"""Oracle for the block-quantized projection matmul -- TEST INFRASTRUCTURE ONLY.

A plain C implementation (``qmm_oracle.c``) in IEEE double precision, loaded
through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the CUDA library never
touches it and shares no code with it.

What it computes (cera, "cera 0.5.2 src/backend/cpu.rs", matmul_q4_0_f32 /
matmul_q8_0_f32 / matmul_q4km_f32 and the scalar GEMV row loops): for weights
W[M,K] stored as consecutive quant blocks per row,

    Y[n, m] = sum_k w(m, k) * x(n, k)      S[n, m] = sum_k |w(m, k) * x(n, k)|

with w(m,k) the exact dequantized value and x exactly what the GPU received
(f32, or bf16).  S scales the tolerance |y - Y| <= rel * S + abs.

Parity pins live in ``tests/test_oracle_pins.py``.  The Q4_K 6-bit scale
packing and the Q6_K bit map follow the GGUF reading and are pinned only to
that reading: parity unpinned against real GGUF files for those two layouts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libqmm_oracle.so")
_SRC = os.path.join(_HERE, "qmm_oracle.c")

Q8_0, Q4_0, Q4_K, Q6_K, Q5_K = 0, 1, 2, 3, 4
X_F32, X_BF16 = 0, 1
BLOCK = {Q8_0: (32, 34), Q4_0: (32, 18), Q4_K: (256, 144), Q6_K: (256, 210), Q5_K: (256, 176)}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE semantics: no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.join(_HERE, "qmm_oracle.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.orc_block_info.argtypes = [ctypes.c_int, p, p]
            lib.orc_block_info.restype = ctypes.c_int
            lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f64.restype = ctypes.c_double
            lib.orc_dequant_block.argtypes = [ctypes.c_int, p, p]
            lib.orc_dequant.argtypes = [ctypes.c_int, p, i64, i64, p]
            lib.orc_dequant_f32.argtypes = [ctypes.c_int, p, i64, i64, p]
            lib.orc_matmul_rows.argtypes = [ctypes.c_int, p, i64, i64, p, ctypes.c_int, i64,
                                            p, i64, p, p, ctypes.c_int]
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_quantize_q8_0.argtypes = [p, i64, p, p]
            lib.orc_quantize_q8_0.restype = ctypes.c_int
            for f in (lib.orc_dequant_block, lib.orc_dequant, lib.orc_dequant_f32, lib.orc_matmul_rows):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def block_info(wtype: int):
    """(elements, bytes) per block as the C oracle defines them."""
    e, b = ctypes.c_int(), ctypes.c_int()
    if _load().orc_block_info(wtype, ctypes.byref(e), ctypes.byref(b)):
        raise ValueError(f"unknown weight type {wtype}")
    return e.value, b.value


def f16_to_f64(h: int) -> float:
    return _load().orc_f16_to_f64(h)


def dequant_block(wtype: int, blk: bytes | np.ndarray) -> np.ndarray:
    E, B = BLOCK[wtype]
    b = np.frombuffer(bytes(blk), dtype=np.uint8) if not isinstance(blk, np.ndarray) else blk
    b = np.ascontiguousarray(b, dtype=np.uint8)
    assert b.size == B
    out = np.empty(E, dtype=np.float64)
    if _load().orc_dequant_block(wtype, _ptr(b), _ptr(out)):
        raise ValueError("orc_dequant_block failed")
    return out


def dequant(wtype: int, w: np.ndarray, M: int, K: int) -> np.ndarray:
    """Exact dequantized weights, float64 [M, K]."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    out = np.empty((M, K), dtype=np.float64)
    if _load().orc_dequant(wtype, _ptr(w), M, K, _ptr(out)):
        raise ValueError("orc_dequant: bad arguments")
    return out


def dequant_f32(wtype: int, w: np.ndarray, M: int, K: int) -> np.ndarray:
    """Dequantized weights rounded once (RN-even) to float32 [M, K]."""
    w = np.ascontiguousarray(w, dtype=np.uint8)
    out = np.empty((M, K), dtype=np.float32)
    if _load().orc_dequant_f32(wtype, _ptr(w), M, K, _ptr(out)):
        raise ValueError("orc_dequant_f32: bad arguments")
    return out


def matmul(wtype: int, w: np.ndarray, M: int, K: int, x: np.ndarray, rows=None,
           nthreads: int = 0):
    """Return (Y, S), float64 [N, len(rows)] (rows=None: all M rows).

    x is float32 [N, K] or a bf16 bit-pattern array (uint16 [N, K]).
    """
    w = np.ascontiguousarray(w, dtype=np.uint8)
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        xt = X_F32
    elif x.dtype == np.uint16:
        xt = X_BF16
    else:
        raise TypeError("x must be float32 or uint16 (bf16 bits)")
    N = x.shape[0] if x.ndim == 2 else 1
    assert x.size == N * K
    if rows is None:
        nrows, rp = M, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rp = rows.size, _ptr(rows)
    Y = np.empty((N, nrows), dtype=np.float64)
    S = np.empty((N, nrows), dtype=np.float64)
    if _load().orc_matmul_rows(wtype, _ptr(w), M, K, _ptr(x), xt, N, rp, nrows,
                               _ptr(Y), _ptr(S), nthreads):
        raise ValueError("orc_matmul_rows: bad arguments")
    return Y, S


def f32_to_f16(f: float) -> int:
    """binary16 bit pattern of float32 f, round to nearest even."""
    return int(_load().orc_f32_to_f16(float(np.float32(f))))


def quantize_q8_0(x: np.ndarray):
    """Q8_0 activations of float32 x [..., K] (K % 32 == 0): (scales float32
    [..., K/32], quants int8 [..., K]), per "cera 0.5.2 src/backend/cpu.rs",
    quantize_f32_to_q8_0_scalar."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    K = x.shape[-1]
    scales = np.empty(x.shape[:-1] + (K // 32,), dtype=np.float32)
    quants = np.empty(x.shape, dtype=np.int8)
    if _load().orc_quantize_q8_0(_ptr(x), x.size, _ptr(scales), _ptr(quants)):
        raise ValueError("orc_quantize_q8_0: bad arguments")
    return scales, quants


def dequant_q8_0_act(scales: np.ndarray, quants: np.ndarray) -> np.ndarray:
    """The activation values the Q8_0 codes stand for, scales[b] * quants[e]
    (exact in float32: an 11-bit scale times an 8-bit code)."""
    K = quants.shape[-1]
    s = np.repeat(scales.astype(np.float64), 32, axis=-1).reshape(quants.shape)
    return (s * quants.astype(np.float64)).astype(np.float32)


def matmul_q8act(wtype: int, w: np.ndarray, M: int, K: int, x: np.ndarray, rows=None, nthreads: int = 0):
    """(Y, S) of the Q8_0-activation product: X is first quantized to Q8_0
    blocks, then Y[n, m] = sum_k w(m, k) * xq(n, k) with xq the dequantized
    activations (the pages' int8 decode and prefill arithmetic)."""
    scales, quants = quantize_q8_0(np.asarray(x, dtype=np.float32).reshape(-1, K))
    return matmul(wtype, w, M, K, dequant_q8_0_act(scales, quants), rows=rows, nthreads=nthreads)


def swiglu(Yg: np.ndarray, Sg: np.ndarray, Yu: np.ndarray, Su: np.ndarray, rel: float, abs_: float):
    """Fused gate/up activation ("cera 0.5.2 src/backend/cpu.rs",
    gemv_q4_0_gate_up_swiglu_with_q8: out = silu(gate . x) * (up . x), and
    silu_mul_inplace: silu(v) = v * sigmoid(v) = v / (1 + exp(-v))), in
    double on the exact projections.  Returns (out, bound): bound carries
    a per-projection error rel * S + abs through the activation to first
    order, |silu'(g) u| e_g + |silu(g)| e_u, plus 1e-6 of |out| for the f32
    evaluation of the activation itself."""
    g = np.asarray(Yg, dtype=np.float64)
    u = np.asarray(Yu, dtype=np.float64)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    out = silu * u
    dsilu = sig * (1.0 + g * (1.0 - sig))
    eg = rel * np.asarray(Sg) + abs_
    eu = rel * np.asarray(Su) + abs_
    bound = np.abs(dsilu * u) * eg + np.abs(silu) * eu + eg * eu + 1e-6 * np.abs(out) + 1e-7
    return out, bound


def within(y: np.ndarray, Y: np.ndarray, S: np.ndarray, rel: float, abs_: float):
    """Element-wise tolerance test |y - Y| <= rel*S + abs; returns (ok, worst ratio)."""
    err = np.abs(y.astype(np.float64) - Y)
    bound = rel * S + abs_
    ratio = float(np.max(err / bound)) if err.size else 0.0
    return bool(np.all(err <= bound)), ratio
