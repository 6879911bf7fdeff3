"""Static-weights mode (programmatic dependent launch) on chains of calls
where each call's X is the previous call's Y, issued back to back on one
stream with no host synchronization in between.  Every stage is checked
against the oracle on the intermediate values the GPU produced, so a call
that read its X before the preceding kernel had written it would fail."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _mode():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    qmm.qmm_set_static_weights(True)
    yield
    qmm.qmm_set_static_weights(False)
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def _chain(specs, x0, tol):
    """specs: list of (wt, M); K of each stage = M of the previous one (all
    row pitches 16-byte aligned, so every stage takes the tensor-core path)."""
    K = x0.shape[1]
    N = x0.shape[0]
    ws, Ws, Ys = [], [], []
    for i, (wt, M) in enumerate(specs):
        w = synth.gen_weights(wt, M, K, f"chain-{i}")
        ws.append((wt, w, M, K))
        Ws.append(torch.from_numpy(w).cuda())
        Ys.append(torch.full((N, M), float("nan"), device="cuda"))
        K = M
    X0 = torch.from_numpy(x0).cuda()
    wss = [qmm.workspace_for(N, k, X0) for (_, _, _, k) in ws]
    for rep in range(3):
        x = X0
        for (wt, w, M, K), W, Y, wsp in zip(ws, Ws, Ys, wss):
            assert qmm.qmm_matmul(wt, W, M, K, x, N, Y, wsp) == qmm.OK
            x = Y
        torch.cuda.synchronize()
        xin = x0
        for (wt, w, M, K), Y in zip(ws, Ys):
            y = Y.cpu().numpy()
            Yr, S = oracle.matmul(wt, w, M, K, xin)
            ok, ratio = oracle.within(y, Yr, S, *tol)
            assert ok, f"rep {rep} stage {wt}: {ratio}"
            xin = np.ascontiguousarray(y)
        for Y in Ys:
            Y.fill_(float("nan"))


def test_gemv_chain_n1():
    x0 = synth.gen_x(1, 4096, "chain")
    _chain([(synth.Q4_0, 2048), (synth.Q6_K, 1024), (synth.Q4_K, 512), (synth.Q8_0, 768)], x0, (1e-5, 1e-6))


def test_gemv_chain_n4():
    x0 = synth.gen_x(4, 2048, "chain4")
    _chain([(synth.Q4_K, 4096), (synth.Q6_K, 1024), (synth.Q4_0, 2560)], x0, (1e-5, 1e-6))


def test_gemm_chain_n64():
    x0 = synth.gen_x(64, 2048, "chain64")
    _chain([(synth.Q4_K, 2048), (synth.Q6_K, 1024), (synth.Q8_0, 512)], x0, (2e-3, 1e-5))
