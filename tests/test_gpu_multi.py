"""Fused projections: qmm_gemv_multi runs several weight matrices that share X
in one launch.  Each output is checked against the oracle (GEMV bound) and
against a separate qmm_gemv call of its matrix (same bound, twice)."""
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


def _run(wt, Ms, K, N, tag, unaligned=None, xbf16=False):
    ws = [synth.gen_weights(wt, M, K, f"multi-{tag}-{i}") for i, M in enumerate(Ms)]
    x = synth.gen_x(N, K, f"multi-{tag}")
    xo = synth.f32_to_bf16_bits(x) if xbf16 else x
    X = torch.from_numpy(xo).cuda()
    if xbf16:
        X = X.view(torch.bfloat16)
    Ws = []
    for i, w in enumerate(ws):
        if unaligned == i:
            base = torch.zeros(w.size + 16, dtype=torch.uint8, device="cuda")
            base[2:2 + w.size] = torch.from_numpy(w).cuda()
            Ws.append(base[2:2 + w.size])
        else:
            Ws.append(torch.from_numpy(w).cuda())
    Ys = qmm.gemv_multi(wt, list(zip(Ws, Ms)), K, X)
    singles = [qmm.gemv(wt, W, M, K, X) for W, M in zip(Ws, Ms)]
    torch.cuda.synchronize()
    for w, M, Y, Y1 in zip(ws, Ms, Ys, singles):
        Yr, S = oracle.matmul(wt, w, M, K, xo)
        y = Y.cpu().numpy()
        ok, ratio = oracle.within(y, Yr, S, *TOL)
        assert ok, ratio
        assert np.all(np.abs(y - Y1.cpu().numpy()) <= 2 * (TOL[0] * S + TOL[1]))


@pytest.mark.parametrize("wt", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K], ids=["Q8_0", "Q4_0", "Q4_K", "Q6_K", "Q5_K"])
@pytest.mark.parametrize("N", [1, 2, 5, 16])
def test_qkv_like(wt, N):
    _run(wt, [512, 128, 128], 2048, N, f"qkv-{wt}-{N}")


@pytest.mark.parametrize("wt", [synth.Q4_K, synth.Q4_0])
def test_gate_up_like_and_four(wt):
    _run(wt, [1408, 1408], 4096, 1, f"gu-{wt}")
    _run(wt, [300, 64, 1000, 17], 2048, 3, f"four-{wt}")


def test_bf16_x():
    _run(synth.Q6_K, [640, 256], 4096, 4, "bf16", xbf16=True)


def test_one_unaligned_matrix_takes_the_byte_path():
    _run(synth.Q4_0, [256, 96], 1024, 2, "unal", unaligned=1)


def test_multi_errors():
    wt, K, N = synth.Q4_0, 512, 2
    W = torch.from_numpy(synth.gen_weights(wt, 64, K, "multi-err")).cuda()
    X = torch.from_numpy(synth.gen_x(N, K, "multi-err")).cuda()
    Y = torch.empty(N, 64, device="cuda")
    assert qmm.qmm_gemv_multi(wt, [], K, X, N) == qmm.ERR_INVALID_ARG
    assert qmm.qmm_gemv_multi(wt, [(W, 64, Y)] * 5, K, X, N) == qmm.ERR_INVALID_ARG
    # an output overlapping another output
    assert qmm.qmm_gemv_multi(wt, [(W, 64, Y), (W, 64, Y)], K, X, N) == qmm.ERR_INVALID_ARG
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# gate/up with the SwiGLU product (qmm_gemv_swiglu)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wt", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K],
                         ids=["Q8_0", "Q4_0", "Q4_K", "Q6_K", "Q5_K"])
@pytest.mark.parametrize("N", [1, 4, 16])
def test_swiglu_parity(wt, N):
    M, K = 1408, 4096
    wg = synth.gen_weights(wt, M, K, "swiglu-gate")
    wu = synth.gen_weights(wt, M, K, "swiglu-up")
    x = synth.gen_x(N, K, f"swiglu-{N}") * np.float32(3.0)    # gate values across silu's curve
    X = torch.from_numpy(x).cuda()
    ws = torch.full((2 * N * M,), float("nan"), device="cuda")
    Y = qmm.gemv_swiglu(wt, torch.from_numpy(wg).cuda(), torch.from_numpy(wu).cuda(), M, K, X, workspace=ws)
    torch.cuda.synchronize()
    Yg, Sg = oracle.matmul(wt, wg, M, K, x)
    Yu, Su = oracle.matmul(wt, wu, M, K, x)
    out, bound = oracle.swiglu(Yg, Sg, Yu, Su, *TOL)
    y = Y.cpu().numpy()
    err = np.abs(y - out)
    assert np.all(err <= bound), float(np.max(err / bound))
    # the projections stay in the workspace and meet the GEMV bar
    g = ws[: N * M].view(N, M).cpu().numpy()
    u = ws[N * M:].view(N, M).cpu().numpy()
    assert oracle.within(g, Yg, Sg, *TOL)[0] and oracle.within(u, Yu, Su, *TOL)[0]


def test_swiglu_errors():
    wt, M, K, N = synth.Q4_0, 64, 512, 2
    Wg = torch.from_numpy(synth.gen_weights(wt, M, K, "sw-err-g")).cuda()
    Wu = torch.from_numpy(synth.gen_weights(wt, M, K, "sw-err-u")).cuda()
    X = torch.from_numpy(synth.gen_x(N, K, "sw-err")).cuda()
    Y = torch.empty(N, M, device="cuda")
    ws = torch.empty(2 * N * M, device="cuda")
    assert qmm.qmm_gemv_swiglu(wt, Wg, Wu, M, K, X, N, Y, ws[: N * M]) == qmm.ERR_INVALID_ARG   # too small
    assert qmm.qmm_gemv_swiglu(wt, Wg, Wu, M, K, X, N, ws[:N * M].view(N, M), ws) == qmm.ERR_INVALID_ARG  # Y in ws
    assert qmm.qmm_gemv_swiglu(wt, Wg, Wu, M, K, X, 17, Y, ws) == qmm.ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.parametrize("wt", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K],
                         ids=["Q8_0", "Q4_0", "Q4_K", "Q6_K", "Q5_K"])
@pytest.mark.parametrize("plan", [(-1, -1, -1, -1, -1), (1, 0, 0, 1, 2), (2, 0, 0, 2, 2), (1, 0, 0, 0, 1)],
                         ids=["auto", "r1-c1", "r2-c2", "direct"])
def test_one_token_multi_streaming(wt, plan):
    """N = 1 over several matrices runs the streaming kernel in one launch,
    its CTAs split over the matrices by rows: four ragged matrices (1, 17,
    300 and 4100 rows) and the Q/K/V shape, each plan."""
    qmm.qmm_set_gemv_stream(*plan)
    try:
        _run(wt, [17, 4100, 1, 300], 2048, 1, f"ms-four-{wt}-{plan[0]}")
        _run(wt, [4096, 1024, 1024], 4096, 1, f"ms-qkv-{wt}-{plan[0]}", xbf16=plan[0] == 2)
    finally:
        qmm.qmm_set_gemv_stream(-1, -1, -1, -1, -1)


def test_one_token_multi_is_one_streaming_launch():
    wt, K = synth.Q4_K, 4096
    Ms = [4096, 1024, 1024]
    Ws = [torch.from_numpy(synth.gen_weights(wt, M, K, f"ms1-{i}")).cuda() for i, M in enumerate(Ms)]
    X = torch.from_numpy(synth.gen_x(1, K, "ms1")).cuda()
    Ys = [torch.empty(1, M, device="cuda") for M in Ms]
    torch.cuda.synchronize()
    n0 = qmm.qmm_kernel_launches()
    assert qmm.qmm_gemv_multi(wt, list(zip(Ws, Ms, Ys)), K, X, 1) == qmm.OK
    torch.cuda.synchronize()
    assert qmm.qmm_kernel_launches() - n0 == 1
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        assert qmm.qmm_gemv_multi(wt, list(zip(Ws, Ms, Ys)), K, X, 1) == qmm.OK
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    if names:
        assert any("gemv_stream_kernel" in n for n in names), names
