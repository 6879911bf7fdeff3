"""Argmax-fused GEMV (greedy decode through the LM head).

qmm_gemv_argmax computes every output exactly as qmm_gemv does but keeps only
each token's largest output and its row.  Checks:
  * bit-exact agreement with the argmax of qmm_gemv's Y (lowest row on ties);
  * validity against the oracle: the chosen row's exact output is within the
    GEMV tolerance of the exact maximum;
  * ties between identical rows resolve to the lower row;
  * the K-split (cluster) path, the ring path (N > 2) and the LM-head shape;
  * argument errors and the unsupported (unaligned) case.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu
TOL = (1e-5, 1e-6)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    yield
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def _argmax_lowest(y: np.ndarray) -> np.ndarray:
    return np.argmax(y, axis=1)          # numpy returns the first maximum


def _check(wt, w, M, K, x, xbf16=False, rows_for_oracle=None):
    N = x.shape[0]
    W = torch.from_numpy(w).cuda()
    xo = synth.f32_to_bf16_bits(x) if xbf16 else x
    X = torch.from_numpy(xo).cuda()
    if xbf16:
        X = X.view(torch.bfloat16)
    idx, val = qmm.gemv_argmax(wt, W, M, K, X)
    y = qmm.gemv(wt, W, M, K, X)
    torch.cuda.synchronize()
    idx, val, y = idx.cpu().numpy(), val.cpu().numpy(), y.cpu().numpy()
    ref_idx = _argmax_lowest(y)
    assert np.array_equal(idx, ref_idx), (idx, ref_idx)
    assert np.array_equal(val.view(np.uint32), y[np.arange(N), ref_idx].view(np.uint32))
    # valid against exact arithmetic
    Y, S = oracle.matmul(wt, w, M, K, xo)
    tol = TOL[0] * S + TOL[1]
    best = Y.max(axis=1)
    for n in range(N):
        i = int(idx[n])
        j = int(np.argmax(Y[n]))
        assert Y[n, i] >= best[n] - (tol[n, i] + tol[n, j]), (n, i, j)
        assert abs(float(val[n]) - Y[n, i]) <= tol[n, i]
    return idx


@pytest.mark.parametrize("wt", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K],
                         ids=["Q8_0", "Q4_0", "Q4_K", "Q6_K", "Q5_K"])
@pytest.mark.parametrize("M,K,N", [(300, 4096, 1), (1024, 2048, 2), (4000, 4096, 5), (777, 2048, 8), (20000, 2048, 16)])
def test_argmax_matches_gemv_and_oracle(wt, M, K, N):
    w = synth.gen_weights(wt, M, K, "amax")
    x = synth.gen_x(N, K, "amax")
    _check(wt, w, M, K, x)


@pytest.mark.parametrize("N", [1, 3])
def test_argmax_bf16_x(N):
    wt, M, K = synth.Q4_K, 2000, 4096
    _check(wt, synth.gen_weights(wt, M, K, "amax-bf"), M, K, synth.gen_x(N, K, "amax-bf"), xbf16=True)


@pytest.mark.parametrize("N", [1, 4, 8])
def test_argmax_lm_head(N):
    """Q6_K LM head, 128256 x 4096."""
    wt, M, K = synth.Q6_K, 128256, 4096
    _check(wt, synth.gen_weights(wt, M, K, "amax-head"), M, K, synth.gen_x(N, K, "amax-head"))


def test_ties_go_to_the_lower_row():
    wt, M, K, N = synth.Q4_0, 1000, 2048, 2
    w = synth.gen_weights(wt, M, K, "amax-tie")
    x = synth.gen_x(N, K, "amax-tie")
    Y, _ = oracle.matmul(wt, w, M, K, x)
    rb = synth.row_bytes(wt, K)
    wr = w.reshape(M, rb)
    top = int(np.argmax(Y[0]))
    low = 3 if top != 3 else 4
    wr[low] = wr[top]                      # identical bytes: identical outputs on the GPU
    idx = _check(wt, wr.reshape(-1), M, K, x)
    assert idx[0] == min(low, top)


def test_argmax_errors():
    wt, M, K, N = synth.Q4_0, 64, 512, 2
    W = torch.from_numpy(synth.gen_weights(wt, M, K, "amax-err")).cuda()
    X = torch.from_numpy(synth.gen_x(N, K, "amax-err")).cuda()
    idx = torch.empty(N, dtype=torch.int32, device="cuda")
    val = torch.empty(N, device="cuda")
    ws = torch.empty(N + 1, dtype=torch.int64, device="cuda")
    assert qmm.qmm_gemv_argmax(wt, W, M, K, X, N, idx, val, ws[:N]) == qmm.ERR_INVALID_ARG   # workspace too small
    assert qmm.qmm_gemv_argmax(wt, W, M, K, X, 17, idx, val, ws) == qmm.ERR_INVALID_ARG      # N > 16
    base = torch.zeros(W.numel() + 16, dtype=torch.uint8, device="cuda")
    base[1:1 + W.numel()] = W
    assert qmm.qmm_gemv_argmax(wt, base[1:1 + W.numel()], M, K, X, N, idx, val, ws) == qmm.ERR_UNSUPPORTED
    torch.cuda.synchronize()


def test_argmax_small_outputs_next_to_inputs():
    """idx/val/workspace are N-entry buffers: placing them right after X (in
    one allocation) is not an overlap."""
    wt, M, K, N = synth.Q6_K, 4096, 2048, 4
    w = synth.gen_weights(wt, M, K, "amax-adj")
    x = synth.gen_x(N, K, "amax-adj")
    W = torch.from_numpy(w).cuda()
    buf = torch.empty(N * K + 64, dtype=torch.float32, device="cuda")   # X, then val, idx, workspace
    X = buf[:N * K].view(N, K)
    X.copy_(torch.from_numpy(x).cuda())
    val = buf[N * K:N * K + N]
    idx = buf[N * K + 16:N * K + 16 + N].view(torch.int32)
    ws = buf[N * K + 32:N * K + 32 + 2 * (N + 1)].view(torch.int64)
    assert qmm.qmm_gemv_argmax(wt, W, M, K, X, N, idx, val, ws) == qmm.OK
    y = qmm.gemv(wt, W, M, K, X)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), np.argmax(y.cpu().numpy(), axis=1))
