"""Seeded synthetic inputs: raw GGUF/ggml quant blocks and activations.

This module only draws random numbers and places them into the block byte
layouts; it performs none of the matmul or dequantization arithmetic, so both
the CUDA path and the oracle can consume what it produces.

Distributions (the workloads of the projection-matmul benchmarks):
  Q8_0 : d ~ U[1e-3, 1e-2] stored as f16, 32 int8 q ~ U{-127..127}
  Q4_0 : d ~ U[1e-3, 1e-2] as f16, 16 bytes of uniform nibbles
  Q4_K : d ~ U[1e-3, 1e-2], dmin ~ U[0, 1e-2] as f16, 12 uniform scale bytes,
         128 uniform nibble bytes
  Q6_K : 128 uniform ql bytes, 64 uniform qh bytes, 16 int8 scales
         ~ U{-64..63}, d ~ U[1e-4, 1e-3] as f16
  Q5_K : as Q4_K, with 32 uniform qh bytes between the scales and qs
  X    : N(0, 1) drawn in double and rounded to f32; bf16 X is the
         round-to-nearest-even bf16 of those same f32 values.
Block byte layouts (field offsets) are the ones documented in include/qmm.h.

Every tensor has its own seed derived from a base seed and its name, so a
tensor can be regenerated alone (e.g. one layer of the decoder sweep).
"""
from __future__ import annotations

import hashlib

import numpy as np

BASE_SEED = 20261202

Q8_0, Q4_0, Q4_K, Q6_K, Q5_K = 0, 1, 2, 3, 4
NAMES = {Q8_0: "Q8_0", Q4_0: "Q4_0", Q4_K: "Q4_K", Q6_K: "Q6_K", Q5_K: "Q5_K"}
BLOCK = {Q8_0: (32, 34), Q4_0: (32, 18), Q4_K: (256, 144), Q6_K: (256, 210), Q5_K: (256, 176)}


def seed_for(name: str, base: int = BASE_SEED) -> int:
    h = hashlib.sha256(f"{base}:{name}".encode()).digest()
    return int.from_bytes(h[:8], "little")


def rng_for(name: str, base: int = BASE_SEED) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_for(name, base)))


def row_bytes(wtype: int, K: int) -> int:
    E, B = BLOCK[wtype]
    assert K % E == 0, f"K={K} is not a multiple of {E}"
    return K // E * B


def weight_bytes(wtype: int, M: int, K: int) -> int:
    return M * row_bytes(wtype, K)


def _f16_bytes(v: np.ndarray) -> np.ndarray:
    """float values -> little-endian binary16 bytes, shape v.shape + (2,)."""
    h = v.astype(np.float16).astype("<f2")
    return h.view(np.uint8).reshape(v.shape + (2,))


def gen_weights(wtype: int, M: int, K: int, name: str, base: int = BASE_SEED,
                out: np.ndarray | None = None) -> np.ndarray:
    """Raw blocks for W[M, K] as a flat uint8 array of M*row_bytes bytes."""
    E, B = BLOCK[wtype]
    nb = K // E
    rng = rng_for(f"W:{NAMES[wtype]}:{M}x{K}:{name}", base)
    n = M * nb * B
    if out is None:
        out = np.empty(n, dtype=np.uint8)
    assert out.size == n and out.dtype == np.uint8
    out[:] = np.frombuffer(rng.bytes(n), dtype=np.uint8)
    blk = out.reshape(M, nb, B)
    if wtype == Q8_0:
        blk[:, :, 0:2] = _f16_bytes(rng.uniform(1e-3, 1e-2, size=(M, nb)))
        blk[:, :, 2:34] = rng.integers(-127, 128, size=(M, nb, 32), dtype=np.int8).view(np.uint8)
    elif wtype == Q4_0:
        blk[:, :, 0:2] = _f16_bytes(rng.uniform(1e-3, 1e-2, size=(M, nb)))
    elif wtype in (Q4_K, Q5_K):
        blk[:, :, 0:2] = _f16_bytes(rng.uniform(1e-3, 1e-2, size=(M, nb)))
        blk[:, :, 2:4] = _f16_bytes(rng.uniform(0.0, 1e-2, size=(M, nb)))
    elif wtype == Q6_K:
        blk[:, :, 192:208] = rng.integers(-64, 64, size=(M, nb, 16), dtype=np.int8).view(np.uint8)
        blk[:, :, 208:210] = _f16_bytes(rng.uniform(1e-4, 1e-3, size=(M, nb)))
    else:
        raise ValueError(f"unknown weight type {wtype}")
    return out


def gen_x(N: int, K: int, name: str, base: int = BASE_SEED) -> np.ndarray:
    """Activations X[N, K], float32 ~ N(0, 1)."""
    rng = rng_for(f"X:{N}x{K}:{name}", base)
    return rng.standard_normal(size=(N, K)).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16, returned as uint16 bit patterns.

    Input preparation only (finite inputs); used to hand the same activations
    to both sides in bf16 form.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Named workloads (shapes only).  Sizes are those of the projection-matmul
# benchmarks: a small Q8_0 case, Llama-3-8B projection shapes in Q4_0, a Q4_K
# prefill GEMM, a 128256-row Q6_K LM head and a 32-layer Q4_K_M-style decoder.
# ----------------------------------------------------------------------------

SMALL_Q8_0 = dict(wtype=Q8_0, shapes=[(256, 512)], Ns=[1])
DECODE_Q4_0 = dict(wtype=Q4_0, shapes=[(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)], Ns=[1])
PREFILL_Q4_K = dict(wtype=Q4_K, shapes=[(4096, 4096), (14336, 4096)], Ns=[64, 256, 512])
LMHEAD_Q6_K = dict(wtype=Q6_K, shapes=[(128256, 4096)], Ns=[1, 4, 8])
# One decoder layer: (name, wtype, M, K).  32 layers, N sweep below.
DECODER_LAYER = [
    ("attn_q", Q4_K, 4096, 4096),
    ("attn_k", Q4_K, 1024, 4096),
    ("attn_v", Q6_K, 1024, 4096),
    ("attn_output", Q4_K, 4096, 4096),
    ("ffn_gate", Q4_K, 14336, 4096),
    ("ffn_up", Q4_K, 14336, 4096),
    ("ffn_down", Q6_K, 4096, 14336),
]
DECODER_LAYERS = 32
DECODER_NS = [1, 2, 4, 8, 16, 32, 64, 128, 256, 512]
