"""GPU parity of the 16-row-tile tensor-core GEMV (opt-in, 2 <= N <= 8;
Q8_0, Q4_0, Q4_K, Q5_K with 16-byte aligned 256-weight units).

Its CTAs own whole 16-row groups; with fewer groups per CTA than warps the
warps split K and add partial sums in shared memory.  The shapes below cover
both modes, partial last row groups (M % 16 != 0), fewer rows than SMs, one-
and two-n-tile token counts (N <= 4 and 5 <= N <= 8), f32 and bf16 X, and
activations spread over many binades (the per-token binary16 scaling).
Bar: |y - Y| <= 1e-5 * S + 1e-6 against the oracle.
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
TC = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q5_K]
IDS = [synth.NAMES[f] for f in TC]
GUARD = 256
POISON = 0x7FC0DEAD


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    qmm.qmm_set_gemv_tc(1)      # the kernel is opt-in
    yield
    qmm.qmm_set_gemv_tc(-1)
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def run_check(wt, M, K, x, xbf16=False):
    """N = 1 takes the streaming kernel; 2 <= N <= 4 this one when it is
    switched on (the forced-setting children below also route 5 <= N <= 8
    here)."""
    N = x.shape[0]
    w = synth.gen_weights(wt, M, K, "tc")
    xo = synth.f32_to_bf16_bits(x) if xbf16 else x
    X = torch.from_numpy(xo).cuda()
    if xbf16:
        X = X.view(torch.bfloat16)
    W = torch.from_numpy(w).cuda()
    buf = torch.full((N * M + 2 * GUARD,), POISON, dtype=torch.int32, device="cuda")
    Y = buf[GUARD:GUARD + N * M].view(torch.float32).view(N, M)
    assert qmm.qmm_gemv(wt, W, M, K, X, N, Y) == qmm.OK
    torch.cuda.synchronize()
    b = buf.cpu()
    assert torch.all(b[:GUARD] == POISON) and torch.all(b[GUARD + N * M:] == POISON), "write outside Y"
    Yr, S = oracle.matmul(wt, w, M, K, xo)
    ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, *GEMV_TOL)
    assert ok, f"worst |err|/tol = {ratio:.3g}"
    Y2 = torch.empty_like(Y)
    assert qmm.qmm_gemv(wt, W, M, K, X, N, Y2) == qmm.OK
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int32), Y2.view(torch.int32)), "not deterministic"


# (M, K): fewer groups than SMs, partial groups, K split and owner modes
SHAPES = [(1, 256), (7, 512), (33, 1024), (300, 4096), (2449, 2048), (20000, 1024), (40, 14336), (9, 32768)]


@pytest.mark.parametrize("wt", TC, ids=IDS)
@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("N", [1, 3, 4, 6, 8])
def test_tc_parity(wt, M, K, N):
    if M * K * N > 40000 * 4096 * 2:
        pytest.skip("size")
    run_check(wt, M, K, synth.gen_x(N, K, "tc"))


@pytest.mark.parametrize("wt", TC, ids=IDS)
@pytest.mark.parametrize("N", [1, 5])
def test_tc_bf16_x(wt, N):
    run_check(wt, 333, 2048, synth.gen_x(N, 2048, "tc-bf16"), xbf16=True)


@pytest.mark.parametrize("wt", TC, ids=IDS)
def test_tc_wide_dynamic_range(wt):
    """Activations spanning ~60 binades per token (the binary16 pieces use a
    per-token power-of-two scale), plus an all-zero token."""
    K = 2048
    rng = np.random.default_rng(7)
    x = synth.gen_x(3, K, "tc-range")
    x[0] *= np.exp2(rng.integers(-30, 30, size=K)).astype(np.float32)
    x[1] = 0.0
    x[2] *= np.float32(1e-30)
    run_check(wt, 257, K, x)


CHILD = r'''
import numpy as np, torch, oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth
qmm.load()
bad = []
for wt in (synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q5_K):
    for (M, K) in ((300, 4096), (2449, 2048), (40, 14336)):
        w = synth.gen_weights(wt, M, K, "tc-tune")
        W = torch.from_numpy(w).cuda()
        for N in (1, 2, 7):
            x = synth.gen_x(N, K, "tc-tune")
            X = torch.from_numpy(x).cuda()
            Y = torch.full((N, M), float("nan"), device="cuda")
            s = qmm.qmm_gemv(wt, W, M, K, X, N, Y)
            torch.cuda.synchronize()
            if s != qmm.OK:
                bad.append((wt, M, K, N, qmm.status_name(s)))
                continue
            Yr, S = oracle.matmul(wt, w, M, K, x)
            ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, 1e-5, 1e-6)
            if not ok:
                bad.append((wt, M, K, N, ratio))
assert qmm.qmm_last_device_error() == qmm.OK
print("BAD" if bad else "OK", bad)
'''


@pytest.mark.parametrize("env", [{"QMM_GEMV_TC": "1", "QMM_TC_WARPS": "4", "QMM_TC_MAX_N": "8"},
                                 {"QMM_GEMV_TC": "1", "QMM_TC_WARPS": "8", "QMM_TC_MAX_N": "8"},
                                 {"QMM_GEMV_TC": "1", "QMM_TC_WARPS": "16", "QMM_TC_MAX_N": "8"},
                                 {"QMM_GEMV_TC": "0"},
                                 {"QMM_GEMV_TC": "1", "QMM_STATIC_WEIGHTS": "1", "QMM_TC_MAX_N": "8"}],
                         ids=lambda e: "-".join(f"{k[4:].lower()}{v}" for k, v in e.items()))
def test_tc_forced(env):
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env={**os.environ, **env, "PYTHONPATH": ROOT},
                       capture_output=True, text=True, timeout=900)
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
    """Hard activations (1e+-20 blocks, 1e6 ranges, spikes, zero blocks)
    through the dispatch with this kernel switched on, against the oracle at
    the GEMV bar.  The per-token binary16 range is a documented limit of
    this kernel (an entry 2^40 below the token's largest is lost), so the
    spike that sits 2^40 below the 1e20 block is checked by the default
    kernels (test_gpu_stream.py) and here the huge block is 1e8, not 1e20."""
    M, K = 512, 2048
    w = synth.gen_weights(wt, M, K, "hard")
    x = _hard_x(N, K, f"hard-{N}")
    x[:, 64:96] *= np.float32(1e-12)   # 1e20 -> 1e8: inside the per-token range of this kernel
    W = torch.from_numpy(w).cuda()
    X = torch.from_numpy(x).cuda()
    Y = torch.empty(N, M, device="cuda")
    assert qmm.qmm_gemv(wt, W, M, K, X, N, Y) == qmm.OK
    torch.cuda.synchronize()
    Yr, S = oracle.matmul(wt, w, M, K, x)
    ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, *GEMV_TOL)
    assert ok, f"worst |err|/tol = {ratio:.3g}"
