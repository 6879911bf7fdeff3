"""qmm_matmul_host: X from pinned host memory, Y back to it, through the C ABI.

Checks the result against the oracle (GEMV bar where qmm_matmul takes the GEMV, GEMM bar above)
and that an invalid argument returns before anything is copied: the device
staging buffers and the host output keep their poison.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()


@pytest.mark.parametrize("N", [1, 4, 64])
def test_host_buffers_match_oracle(N):
    wt, M, K = synth.Q4_K, 777, 2048
    w = synth.gen_weights(wt, M, K, "host-io")
    x = synth.gen_x(N, K, "host-io")
    W = torch.from_numpy(w).cuda()
    Xh = torch.from_numpy(x).pin_memory()
    Yh = torch.full((N, M), float("nan")).pin_memory()
    xd = torch.empty(N, K, device="cuda")
    yd = torch.empty(N, M, device="cuda")
    ws = qmm.workspace_for(N, K, xd)
    s = qmm.qmm_matmul_host(wt, W, M, K, Xh, N, Yh, xd, yd, ws)
    assert s == qmm.OK, qmm.status_name(s)
    torch.cuda.synchronize()
    Yr, S = oracle.matmul(wt, w, M, K, x)
    tol = (1e-5, 1e-6) if N <= qmm.MATMUL_GEMV_MAX_N else (2e-3, 1e-5)
    ok, ratio = oracle.within(Yh.numpy(), Yr, S, *tol)
    assert ok, f"worst |err|/tol = {ratio:.3g}"


@pytest.mark.parametrize("N", [2, 100])
def test_bad_argument_copies_nothing(N):
    wt, M, K = synth.Q4_0, 64, 512
    W = torch.from_numpy(synth.gen_weights(wt, M, K, "host-bad")).cuda()
    Xh = torch.from_numpy(synth.gen_x(N, K, "host-bad")).pin_memory()
    Yh = torch.full((N, M), 5.0).pin_memory()
    xd = torch.full((N, K), 3.0, device="cuda")
    yd = torch.full((N, M), 4.0, device="cuda")
    ws = qmm.workspace_for(N, K, xd)
    # K not a multiple of the block: rejected before the host-to-device copy
    s = load_host(wt, W, M, K + 1, Xh, N, Yh, xd, yd, ws)
    assert s == qmm.ERR_INVALID_ARG
    # y_dev overlapping W: rejected too
    s = load_host(wt, W, M, K, Xh, N, Yh, xd, W, ws)
    assert s == qmm.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(xd == 3.0) and torch.all(yd == 4.0) and torch.all(Yh == 5.0)


def load_host(wt, W, M, K, Xh, N, Yh, xd, yd, ws):
    ws_bytes = 0 if ws is None else ws.numel()
    return qmm.load().qmm_matmul_host(wt, W.data_ptr(), W.numel(), M, K, Xh.data_ptr(), qmm.X_F32, N,
                                      Yh.data_ptr(), xd.data_ptr(), yd.data_ptr(),
                                      None if ws is None else ws.data_ptr(), ws_bytes,
                                      torch.cuda.current_stream().cuda_stream)
