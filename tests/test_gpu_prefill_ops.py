"""The pages' prefill variants on the tensor-core GEMM, through the C ABI:

  qmm_gemm_q8act   X quantized to Q8_0 blocks, the GEMM on the dequantized
                   activations; reference: the oracle's exact product on the
                   oracle's own Q8_0 quantization of X (oracle.matmul_q8act);
  qmm_gemm_swiglu  gate and up projections in one GEMM launch, then
                   silu(g) * u; reference: oracle.swiglu on the exact
                   projections, and g, u (left in the workspace) each
                   within the GEMM bar of its exact projection.

Bar: the GEMM tolerance 2e-3 * S + 1e-5 (carried through the activation for
SwiGLU).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

GEMM_TOL = (2e-3, 1e-5)
ALL = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K]
IDS = [synth.NAMES[f] for f in ALL]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    yield
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def _x(N, K, name, xbf16):
    x = synth.gen_x(N, K, name)
    if not xbf16:
        return x, torch.from_numpy(x).cuda()
    xb = synth.f32_to_bf16_bits(x)
    return synth.bf16_bits_to_f32(xb), torch.from_numpy(xb).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("M,K,N", [(300, 2048, 100), (129, 2048, 33), (512, 4096, 512)])
@pytest.mark.parametrize("xbf16", [False, True], ids=["f32x", "bf16x"])
def test_gemm_q8act_matches_oracle(wt, M, K, N, xbf16):
    w = synth.gen_weights(wt, M, K, "gemm-q8act")
    x, X = _x(N, K, "gemm-q8act", xbf16)
    Y = qmm.gemm_q8act(wt, torch.from_numpy(w).cuda(), M, K, X)
    torch.cuda.synchronize()
    Yr, S = oracle.matmul_q8act(wt, w, M, K, x)
    ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, *GEMM_TOL)
    assert ok, f"worst |err|/tol = {ratio:.3g}"


def test_gemm_q8act_differs_from_the_plain_product_where_quantization_matters():
    """The activations really are quantized: with a block holding one large
    and many small values, the Q8_0 result follows the oracle's quantized
    product, not the exact one."""
    wt, M, K, N = synth.Q4_K, 256, 2048, 32
    w = synth.gen_weights(wt, M, K, "q8act-range")
    x = synth.gen_x(N, K, "q8act-range")
    x[:, 0::32] *= 200.0                     # small entries fall to a few codes
    X = torch.from_numpy(x).cuda()
    Y = qmm.gemm_q8act(wt, torch.from_numpy(w).cuda(), M, K, X).cpu().numpy()
    Yq, Sq = oracle.matmul_q8act(wt, w, M, K, x)
    Yx, Sx = oracle.matmul(wt, w, M, K, x)
    assert oracle.within(Y, Yq, Sq, *GEMM_TOL)[0]
    assert not oracle.within(Y, Yx, Sx, *GEMM_TOL)[0]


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("M,K,N", [(384, 2048, 96), (1000, 4096, 300)])
@pytest.mark.parametrize("xbf16", [False, True], ids=["f32x", "bf16x"])
def test_gemm_swiglu_matches_oracle(wt, M, K, N, xbf16):
    wg = synth.gen_weights(wt, M, K, "gemm-gate")
    wu = synth.gen_weights(wt, M, K, "gemm-up")
    x, X = _x(N, K, "gemm-swiglu", xbf16)
    Wg, Wu = torch.from_numpy(wg).cuda(), torch.from_numpy(wu).cuda()
    n = qmm.load().qmm_gemm_swiglu_workspace_bytes(N, M, K, qmm.X_BF16 if xbf16 else qmm.X_F32)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    Y = qmm.gemm_swiglu(wt, Wg, Wu, M, K, X, workspace=ws)
    torch.cuda.synchronize()
    Yg, Sg = oracle.matmul(wt, wg, M, K, x)
    Yu, Su = oracle.matmul(wt, wu, M, K, x)
    out, bound = oracle.swiglu(Yg, Sg, Yu, Su, *GEMM_TOL)
    err = np.abs(Y.cpu().numpy().astype(np.float64) - out)
    assert np.all(err <= bound), f"worst err/bound {np.max(err / bound):.3g}"
    # g and u left in the workspace: each projection within the GEMM bar
    xws = (qmm.qmm_gemm_workspace_bytes(N, K, qmm.X_BF16 if xbf16 else qmm.X_F32) + 15) // 16 * 16
    g = ws[xws:xws + N * M * 4].view(torch.float32).view(N, M).cpu().numpy()
    u = ws[xws + N * M * 4:xws + 2 * N * M * 4].view(torch.float32).view(N, M).cpu().numpy()
    assert oracle.within(g, Yg, Sg, *GEMM_TOL)[0]
    assert oracle.within(u, Yu, Su, *GEMM_TOL)[0]


@pytest.mark.parametrize("wt", [synth.Q4_K, synth.Q8_0], ids=["Q4_K", "Q8_0"])
def test_gemm_swiglu_two_launch_plan(wt):
    """More 128-row tiles (both matrices) than one wave holds: whole waves run
    unsplit and the last tiles (the second matrix's) run as a second,
    K-split launch; every row checked against the oracle."""
    M, K, N = 5000, 2048, 300
    wg = synth.gen_weights(wt, M, K, "gemm-gate-big")
    wu = synth.gen_weights(wt, M, K, "gemm-up-big")
    x, X = _x(N, K, "gemm-swiglu-big", True)
    n = qmm.load().qmm_gemm_swiglu_workspace_bytes(N, M, K, qmm.X_BF16)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    Y = qmm.gemm_swiglu(wt, torch.from_numpy(wg).cuda(), torch.from_numpy(wu).cuda(), M, K, X, workspace=ws)
    torch.cuda.synchronize()
    Yg, Sg = oracle.matmul(wt, wg, M, K, x)
    Yu, Su = oracle.matmul(wt, wu, M, K, x)
    out, bound = oracle.swiglu(Yg, Sg, Yu, Su, *GEMM_TOL)
    err = np.abs(Y.cpu().numpy().astype(np.float64) - out)
    assert np.all(err <= bound), f"worst err/bound {np.max(err / bound):.3g}"


@pytest.mark.parametrize("xbf16", [False, True], ids=["f32x", "bf16x"])
def test_gemm_swiglu_full_size(xbf16):
    """Gate/up at 14336 x 4096, N = 300: 448 tiles of both matrices in one
    paired plan (whole waves, then the rest).  Sampled rows (the last tile
    in full) against the oracle, and g, u left in the workspace."""
    wt, M, K, N = synth.Q4_K, 14336, 4096, 300
    wg = synth.gen_weights(wt, M, K, "gemm-gate-sep")
    wu = synth.gen_weights(wt, M, K, "gemm-up-sep")
    x, X = _x(N, K, "gemm-swiglu-sep", xbf16)
    xt = qmm.X_BF16 if xbf16 else qmm.X_F32
    ws = torch.empty(qmm.load().qmm_gemm_swiglu_workspace_bytes(N, M, K, xt), dtype=torch.uint8, device="cuda")
    Y = qmm.gemm_swiglu(wt, torch.from_numpy(wg).cuda(), torch.from_numpy(wu).cuda(), M, K, X, workspace=ws)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    rows = np.sort(np.concatenate([rng.choice(M - 128, 192, replace=False), np.arange(M - 128, M)]))
    Yg, Sg = oracle.matmul(wt, wg, M, K, x, rows=rows)
    Yu, Su = oracle.matmul(wt, wu, M, K, x, rows=rows)
    out, bound = oracle.swiglu(Yg, Sg, Yu, Su, *GEMM_TOL)
    err = np.abs(Y.cpu().numpy()[:, rows].astype(np.float64) - out)
    assert np.all(err <= bound), f"worst err/bound {np.max(err / bound):.3g}"
    xws = (qmm.qmm_gemm_workspace_bytes(N, K, xt) + 15) // 16 * 16
    g = ws[xws:xws + N * M * 4].view(torch.float32).view(N, M).cpu().numpy()[:, rows]
    u = ws[xws + N * M * 4:xws + 2 * N * M * 4].view(torch.float32).view(N, M).cpu().numpy()[:, rows]
    assert oracle.within(g, Yg, Sg, *GEMM_TOL)[0]
    assert oracle.within(u, Yu, Su, *GEMM_TOL)[0]


@pytest.mark.parametrize("wt", [synth.Q4_K, synth.Q8_0, synth.Q6_K], ids=["Q4_K", "Q8_0", "Q6_K"])
def test_gemm_two_launch_plan_ragged_rows(wt):
    """155 row tiles (the last one partial) at N = 100: a wave of 152 tiles,
    then 3 tiles split over clusters; sampled rows, the last tiles in full."""
    M, K, N = 152 * 128 + 300, 2048, 100
    w = synth.gen_weights(wt, M, K, "gemm-two-launch")
    x, X = _x(N, K, "gemm-two-launch", False)
    Y = torch.full((N, M), float("nan"), device="cuda")
    assert qmm.qmm_gemm(wt, torch.from_numpy(w).cuda(), M, K, X, N, Y, qmm.workspace_for(N, K, X)) == qmm.OK
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    rows = np.sort(np.concatenate([rng.choice(152 * 128, 256, replace=False), np.arange(152 * 128, M)]))
    Yr, S = oracle.matmul(wt, w, M, K, x, rows=rows)
    ok, ratio = oracle.within(Y.cpu().numpy()[:, rows], Yr, S, *GEMM_TOL)
    assert ok, f"worst |err|/tol = {ratio:.3g}"
    assert torch.all(torch.isfinite(Y))


def test_invalid_arguments_write_nothing():
    wt, M, K, N = synth.Q4_K, 256, 2048, 64
    W = torch.from_numpy(synth.gen_weights(wt, M, K, "bad")).cuda()
    X = torch.from_numpy(synth.gen_x(N, K, "bad")).cuda()
    Y = torch.full((N, M), 9.0, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert qmm.qmm_gemm_q8act(wt, W, M, K, X, N, Y, small) == qmm.ERR_INVALID_ARG
    assert qmm.qmm_gemm_swiglu(wt, W, W, M, K, X, N, Y, small) == qmm.ERR_INVALID_ARG
    ws = torch.empty(qmm.load().qmm_gemm_q8act_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    assert qmm.qmm_gemm_q8act(wt, W, M, K + 1, X, N, Y, ws) == qmm.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(Y == 9.0)
