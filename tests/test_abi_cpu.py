"""CPU-side checks of the C ABI: the library builds, loads without a GPU and
exports every entry point that include/qmm.h declares; host-only entry points
(block geometry, status names, workspace size) answer correctly."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import oracle
from block_quantized_gemv_gguf_gb300 import build, qmm, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qmm.load()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"QMM_API\s+[\w\s\*]*?\b(qmm_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared()
    for n in qmm.EXPORTS:
        assert n in names, f"{n} not declared in include/"


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} missing from {qmm.library_path()}"
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_block_info(lib):
    assert qmm.qmm_block_info(qmm.Q8_0) == (0, 32, 34)
    assert qmm.qmm_block_info(qmm.Q4_0) == (0, 32, 18)
    assert qmm.qmm_block_info(qmm.Q4_K) == (0, 256, 144)
    assert qmm.qmm_block_info(qmm.Q6_K) == (0, 256, 210)
    assert qmm.qmm_block_info(qmm.Q5_K) == (0, 256, 176)
    assert qmm.qmm_block_info(9)[0] == qmm.ERR_INVALID_ARG
    # the library, the oracle and the input generators agree on every format
    for wt, (e, b) in synth.BLOCK.items():
        assert qmm.qmm_block_info(wt) == (0, e, b) and oracle.block_info(wt) == (e, b)


def test_status_strings(lib):
    assert qmm.status_name(qmm.OK) == "QMM_OK"
    assert qmm.status_name(qmm.ERR_TIMEOUT) == "QMM_ERR_TIMEOUT"
    assert qmm.status_name(77) == "QMM_UNKNOWN_STATUS"


def test_workspace_bytes(lib):
    assert qmm.qmm_gemm_workspace_bytes(512, 4096, qmm.X_F32) == 512 * 4096 * 2
    assert qmm.qmm_gemm_workspace_bytes(512, 4096, qmm.X_BF16) == 0
    assert qmm.qmm_gemm_workspace_bytes(0, 4096, qmm.X_F32) == 0


def test_no_runtime_dependency_on_driver(lib):
    # The CUDA runtime is linked statically; the library must load on a
    # machine without libcuda (this container) -- the fixture proves it.
    assert os.path.exists(qmm.library_path())


def test_invalid_arguments_rejected_before_any_device_work(lib):
    # Null pointers / bad formats / bad shapes return without touching a GPU.
    L = lib
    assert L.qmm_gemv(7, 1, 1 << 20, 1, 32, 1, 0, 1, 1, None) == qmm.ERR_INVALID_ARG      # unknown format
    assert L.qmm_gemv(qmm.Q4_0, None, 18, 1, 32, 16, 0, 1, 64, None) == qmm.ERR_INVALID_ARG  # null W
    assert L.qmm_gemv(qmm.Q4_0, 16, 18, 1, 31, 64, 0, 1, 256, None) == qmm.ERR_INVALID_ARG   # K % 32
    assert L.qmm_gemv(qmm.Q4_0, 16, 17, 1, 32, 64, 0, 1, 256, None) == qmm.ERR_INVALID_ARG   # short W
    assert L.qmm_gemv(qmm.Q4_0, 16, 18, 1, 32, 64, 0, 17, 256, None) == qmm.ERR_INVALID_ARG  # N > 16
    assert L.qmm_gemv(qmm.Q4_0, 16, 18, 1, 32, 64, 0, 0, 256, None) == qmm.ERR_INVALID_ARG   # N < 1
    assert L.qmm_gemv(qmm.Q4_0, 16, 18, 1, 32, 64, 5, 1, 256, None) == qmm.ERR_INVALID_ARG   # bad xtype
    assert L.qmm_gemv(qmm.Q4_0, 1024, 18, 1, 32, 4096, 0, 1, 1024, None) == qmm.ERR_INVALID_ARG  # Y overlaps W
    assert L.qmm_gemm(qmm.Q4_K, 4096, 1 << 20, 16, 256, 1 << 24, 0, 513, 1 << 28, None, 0, None) == \
        qmm.ERR_INVALID_ARG                                                                    # N > 512
    # f32 X needs a workspace on the GEMM path
    assert L.qmm_gemm(qmm.Q4_K, 4096, 1 << 20, 16, 256, 1 << 24, 0, 64, 1 << 28, None, 0, None) == \
        qmm.ERR_INVALID_ARG
    assert L.qmm_dequant(qmm.Q6_K, 4096, 210, 1, 256, None, None) == qmm.ERR_INVALID_ARG


def test_q8_activation_entry_points_validate_exact_sizes(lib):
    # Codes are N*K bytes: an output right after them is not an overlap, so
    # validation passes and the call only fails for want of a device.
    L = lib
    wt, M, K, N = qmm.Q4_0, 64, 512, 2
    base = 1 << 32                                   # fake, never dereferenced
    W, S, Q = base, base + (1 << 20), base + (2 << 20)
    Y = Q + N * K                                    # adjacent to the codes
    assert L.qmm_gemv_preq(wt, W, M * 16 * 18, M, K, S, Q, N, Y, None) == qmm.ERR_CUDA
    assert L.qmm_gemv_preq(wt, W, M * 16 * 18, M, K, S, Q, N, Q + N * K - 4, None) == qmm.ERR_INVALID_ARG
    assert L.qmm_gemv_preq(wt, W, M * 16 * 18, M, K, S, Q, 17, Y, None) == qmm.ERR_INVALID_ARG
    assert L.qmm_gemv_preq(wt, W, M * 16 * 18, M, K, None, Q, N, Y, None) == qmm.ERR_INVALID_ARG
    assert L.qmm_quantize_q8_0(base, qmm.X_F32, N, 500, S, Q, None) == qmm.ERR_INVALID_ARG     # K % 32
    assert L.qmm_quantize_q8_0(base, qmm.X_F32, N, K, base + 64, Q, None) == qmm.ERR_INVALID_ARG  # scales on X
    assert L.qmm_q8act_workspace_bytes(N, K) == N * K + N * (K // 32) * 4
    ws = base + (3 << 20)
    assert L.qmm_gemv_q8act(wt, W, M * 16 * 18, M, K, base + (4 << 20), qmm.X_F32, N, base + (5 << 20), ws, 16,
                            None) == qmm.ERR_INVALID_ARG                                         # small workspace
