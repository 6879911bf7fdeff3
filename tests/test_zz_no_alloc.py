"""qmm_gemm_noalloc: the GEMM entry point for callers that may not allocate.

Some callers cannot hand the library a workspace or call cudaMalloc (a host
framework that owns all device memory, a fixed memory budget, a path that must
not stall on allocator synchronization).  qmm_gemm_noalloc keeps the bf16 copy
of an f32 X in a fixed library-owned device array instead.  This file checks,
through the C ABI, that two calls in a row match qmm_gemm with a
caller-provided workspace bit for bit (same kernels, same inputs) and the
oracle within the GEMM tolerance, with f32 and bf16 X, and that sizes beyond
the array are refused.  It is named to be collected last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20
TOL = (2e-3, 1e-5)


def _fn():
    f = qmm.load().qmm_gemm_noalloc
    f.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _noalloc(wt, W, M, K, X, N, Y):
    f = _fn()
    xt = qmm.X_F32 if X.dtype == torch.float32 else qmm.X_BF16
    return f(wt, W.data_ptr(), W.numel(), M, K, X.data_ptr(), xt, N, Y.data_ptr(),
             torch.cuda.current_stream().cuda_stream)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()


@pytest.mark.parametrize("xbf16", [False, True], ids=["f32x", "bf16x"])
def test_two_calls_match_workspace_entry_point_and_oracle(xbf16):
    wt, M, K = synth.Q4_K, 640, 4096
    w = synth.gen_weights(wt, M, K, "noalloc")
    W = torch.from_numpy(w).cuda()
    for call, N in enumerate((300, 512)):       # two calls in a row, different inputs
        x = synth.gen_x(N, K, f"noalloc-{call}")
        xo = synth.f32_to_bf16_bits(x) if xbf16 else x
        X = torch.from_numpy(xo).cuda()
        if xbf16:
            X = X.view(torch.bfloat16)
        Y_ref = torch.empty(N, M, device="cuda")
        ws = qmm.workspace_for(N, K, X)
        assert qmm.qmm_gemm(wt, W, M, K, X, N, Y_ref, ws) == qmm.OK
        Y = torch.full((N, M), float("nan"), device="cuda")
        assert _noalloc(wt, W, M, K, X, N, Y) == qmm.OK
        torch.cuda.synchronize()
        # the same kernels on the same inputs: identical bits
        assert torch.equal(Y.view(torch.int32), Y_ref.view(torch.int32)), f"call {call}: differs from qmm_gemm"
        # and the method's result: the oracle's exact sum, GEMM tolerance
        Yr, S = oracle.matmul(wt, w, M, K, xo)
        ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, *TOL)
        assert ok, f"call {call}: worst |err|/tol = {ratio:.3g}"
    assert qmm.qmm_last_device_error() == qmm.OK


def test_bad_argument_reported_before_the_size_limit():
    wt, M = synth.Q4_K, 128
    K = 2 * SCRATCH_BYTES // (2 * 512)          # too big for the array at N = 512
    X = torch.zeros(512, K, device="cuda")
    Y = torch.full((512, M), 7.0, device="cuda")
    f = _fn()
    # null W: an invalid argument, not an unsupported size
    st = f(wt, None, 0, M, K, X.data_ptr(), qmm.X_F32, 512, Y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == qmm.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)


def test_size_beyond_scratch_is_refused():
    wt, M = synth.Q4_K, 128
    K = 2 * SCRATCH_BYTES // (2 * 512)          # N*K*2 = 2 x the array at N = 512
    W = torch.zeros(M * synth.row_bytes(wt, K), dtype=torch.uint8, device="cuda")
    X = torch.zeros(512, K, device="cuda")
    Y = torch.full((512, M), 7.0, device="cuda")
    assert _noalloc(wt, W, M, K, X, 512, Y) == qmm.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)
