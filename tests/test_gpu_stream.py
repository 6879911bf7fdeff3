"""GPU parity of the streaming one-token GEMV (the N = 1 decode kernel).

It owns whole rows per CTA and streams 32-unit stages (a unit = 256 weights
of one row) per warp, so the shapes below cover: fewer rows than SMs, rows
shorter than a stage (1, 2, 4, 8 units), rows that cross stages (56 units),
partial last stages, very long rows (128 units), and every warp count the
planner may choose.  Bar: |y - Y| <= 1e-5 * S + 1e-6 against the oracle.
"""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GEMV_TOL = (1e-5, 1e-6)
ALL = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K]
IDS = [synth.NAMES[f] for f in ALL]
GUARD = 256
POISON = 0x7FC0DEAD


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    yield
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def row_aligned(wt, K):
    E, B = synth.BLOCK[wt]
    return (K // E * B) % 16 == 0


SHAPES = [(1, 256), (7, 512), (33, 1024), (151, 2048), (153, 2048), (300, 4096), (1000, 14336), (5, 32768)]


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("xbf16", [False, True], ids=["f32x", "bf16x"])
def test_stream_parity(wt, M, K, xbf16):
    if not row_aligned(wt, K):
        pytest.skip("rows not 16-byte multiples: another kernel serves this shape")
    w = synth.gen_weights(wt, M, K, "stream")
    x = synth.gen_x(1, K, "stream")
    xo = synth.f32_to_bf16_bits(x) if xbf16 else x
    X = torch.from_numpy(xo).cuda()
    if xbf16:
        X = X.view(torch.bfloat16)
    W = torch.from_numpy(w).cuda()
    buf = torch.full((M + 2 * GUARD,), POISON, dtype=torch.int32, device="cuda")
    Y = buf[GUARD:GUARD + M].view(torch.float32).view(1, M)
    assert qmm.qmm_gemv(wt, W, M, K, X, 1, Y) == qmm.OK
    torch.cuda.synchronize()
    b = buf.cpu()
    assert torch.all(b[:GUARD] == POISON) and torch.all(b[GUARD + M:] == POISON), "write outside Y"
    Yr, S = oracle.matmul(wt, w, M, K, xo)
    ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, *GEMV_TOL)
    assert ok, f"worst |err|/tol = {ratio:.3g}"
    # deterministic: a second call gives the same bits
    Y2 = torch.empty_like(Y)
    assert qmm.qmm_gemv(wt, W, M, K, X, 1, Y2) == qmm.OK
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int32), Y2.view(torch.int32))


def test_stream_kernel_is_the_one_that_runs():
    """N = 1 on an aligned shape launches the streaming kernel (profiler
    kernel names), not another GEMV."""
    wt, M, K = synth.Q4_0, 4096, 4096
    W = torch.from_numpy(synth.gen_weights(wt, M, K, "which")).cuda()
    X = torch.from_numpy(synth.gen_x(1, K, "which")).cuda()
    Y = torch.empty(1, M, device="cuda")
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        assert qmm.qmm_gemv(wt, W, M, K, X, 1, Y) == qmm.OK
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    if not names:
        pytest.skip("the profiler recorded no device activity on this machine")
    assert any("gemv_stream_kernel" in n for n in names), names


CHILD = r'''
import numpy as np, torch, oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth
qmm.load()
bad = []
for wt in (synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K):
    for (M, K) in ((300, 4096), (77, 2048), (40, 14336)):
        w = synth.gen_weights(wt, M, K, "stream-tune")
        W = torch.from_numpy(w).cuda()
        x = synth.gen_x(1, K, "stream-tune")
        X = torch.from_numpy(x).cuda()
        Y = torch.full((1, M), float("nan"), device="cuda")
        s = qmm.qmm_gemv(wt, W, M, K, X, 1, Y)
        torch.cuda.synchronize()
        if s != qmm.OK:
            bad.append((wt, M, K, qmm.status_name(s)))
            continue
        Yr, S = oracle.matmul(wt, w, M, K, x)
        ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, 1e-5, 1e-6)
        if not ok:
            bad.append((wt, M, K, ratio))
assert qmm.qmm_last_device_error() == qmm.OK
print("BAD" if bad else "OK", bad)
'''


@pytest.mark.parametrize("env", [{"QMM_STREAM_WARPS": "4"}, {"QMM_STREAM_WARPS": "8"},
                                 {"QMM_STREAM_WARPS": "12"}, {"QMM_STREAM_WARPS": "16"},
                                 {"QMM_STREAM_SLOTS": "2"}, {"QMM_STREAM_SLOTS": "3"},
                                 {"QMM_STREAM_SLOTS": "2", "QMM_STREAM_STAGGER": "0"},
                                 {"QMM_STREAM_SLOTS": "3", "QMM_STREAM_STAGGER": "0"},
                                 {"QMM_GEMV_STREAM": "0"}, {"QMM_STATIC_WEIGHTS": "1"}],
                         ids=lambda e: "-".join(f"{k[4:].lower()}{v}" for k, v in e.items()))
def test_stream_forced_shapes(env):
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env={**os.environ, **env, "PYTHONPATH": ROOT},
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().startswith("OK"), r.stdout[-3000:]


def _hard_x(N, K, name):
    """Blocks with a 1e6 range between their largest and smallest entries,
    whole blocks 1e-20 or 1e20 times the rest, a zero block, a lone spike."""
    x = synth.gen_x(N, K, name).astype(np.float64)
    rng = np.random.default_rng(7)
    nb = K // 32
    for n in range(N):
        for b in rng.choice(nb, size=max(1, nb // 8), replace=False):
            x[n, 32 * b:32 * b + 32] *= 10.0 ** rng.uniform(-6, 0, 32)
        x[n, 0:32] = 0.0
        x[n, 32:64] *= 1e-20
        x[n, 64:96] *= 1e20
        x[n, 100] = 3e4
    return x.astype(np.float32)


@pytest.mark.parametrize("wt", [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K],
                         ids=["Q8_0", "Q4_0", "Q4_K", "Q6_K", "Q5_K"])
@pytest.mark.parametrize("N", [1, 2, 4])
def test_hard_values(wt, N):
    """Hard activations through the default dispatch (this kernel serves
    N = 1), against the oracle at the GEMV bar."""
    M, K = 512, 2048
    w = synth.gen_weights(wt, M, K, "hard")
    x = _hard_x(N, K, f"hard-{N}")
    W = torch.from_numpy(w).cuda()
    X = torch.from_numpy(x).cuda()
    Y = torch.empty(N, M, device="cuda")
    assert qmm.qmm_gemv(wt, W, M, K, X, N, Y) == qmm.OK
    torch.cuda.synchronize()
    Yr, S = oracle.matmul(wt, w, M, K, x)
    ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, *GEMV_TOL)
    assert ok, f"worst |err|/tol = {ratio:.3g}"
