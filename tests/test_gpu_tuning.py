"""GPU parity of every GEMV launch shape, forced through the library's tuning
overrides (rows per tile, K split, resident-X on or off).

The overrides are read once per process, so each combination runs in a child
process that checks a few shapes against the oracle and prints one line.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import numpy as np, torch, oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth
qmm.load()
bad = []
for wt in (synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K):
    for (M, K) in ((300, 4096), (77, 2048)):
        w = synth.gen_weights(wt, M, K, "tune")
        W = torch.from_numpy(w).cuda()
        for N in (1, 2, 3, 5, 8, 16):
            for bf in (False, True):
                x = synth.gen_x(N, K, "tune")
                xo = synth.f32_to_bf16_bits(x) if bf else x
                X = torch.from_numpy(xo).cuda()
                if bf:
                    X = X.view(torch.bfloat16)
                Y = torch.full((N, M), float("nan"), device="cuda")
                s = qmm.qmm_gemv(wt, W, M, K, X, N, Y)
                torch.cuda.synchronize()
                if s != qmm.OK:
                    bad.append((wt, M, K, N, bf, qmm.status_name(s)))
                    continue
                Yr, S = oracle.matmul(wt, w, M, K, xo)
                ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, 1e-5, 1e-6)
                if not ok:
                    bad.append((wt, M, K, N, bf, ratio))
assert qmm.qmm_last_device_error() == qmm.OK
print("BAD" if bad else "OK", bad)
'''

COMBOS = [
    {"QMM_GEMV_ROWS": "64", "QMM_GEMV_KS": "1", "QMM_GEMV_RESIDENT": "1"},
    {"QMM_GEMV_ROWS": "64", "QMM_GEMV_KS": "8", "QMM_GEMV_RESIDENT": "1"},
    {"QMM_GEMV_ROWS": "128", "QMM_GEMV_RG": "2", "QMM_GEMV_KS": "2", "QMM_GEMV_RESIDENT": "1"},
    {"QMM_GEMV_ROWS": "128", "QMM_GEMV_RG": "1", "QMM_GEMV_KS": "4", "QMM_GEMV_RESIDENT": "1"},
    {"QMM_GEMV_ROWS": "256", "QMM_GEMV_KS": "1", "QMM_GEMV_RESIDENT": "1"},
    {"QMM_GEMV_ROWS": "128", "QMM_GEMV_KS": "1", "QMM_GEMV_RESIDENT": "0"},
    {"QMM_GEMV_ROWS": "64", "QMM_GEMV_KS": "4", "QMM_GEMV_RESIDENT": "0"},
    # the integer kernel (exact int8 digits) for N <= 2
    {"QMM_GEMV_ROWS": "64", "QMM_GEMV_KS": "2", "QMM_GEMV_I8": "1"},
    {"QMM_GEMV_ROWS": "128", "QMM_GEMV_RG": "2", "QMM_GEMV_KS": "1", "QMM_GEMV_I8": "1"},
]


@pytest.mark.parametrize("env", COMBOS, ids=lambda e: "-".join(f"{k[9:].lower()}{v}" for k, v in e.items()))
def test_forced_launch_shapes(env):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env={**os.environ, **env, "PYTHONPATH": ROOT},
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().startswith("OK"), r.stdout[-3000:]


GEMM_CHILD = r'''
import numpy as np, torch, oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth
qmm.load()
bad = []
for wt in (synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q8_0, synth.Q5_K):
    for (M, K, N) in ((300, 2048, 100), (128, 2048, 17), (520, 4096, 512), (200, 2304, 40), (130, 256, 20)):
        E, B = synth.BLOCK[wt]
        if (K // E * B) % 16:
            continue   # rows not 16-byte multiples: the GEMM does not take them
        w = synth.gen_weights(wt, M, K, "tune-gemm")
        W = torch.from_numpy(w).cuda()
        x = synth.gen_x(N, K, "tune-gemm")
        X = torch.from_numpy(x).cuda()
        Y = torch.full((N, M), float("nan"), device="cuda")
        s = qmm.qmm_gemm(wt, W, M, K, X, N, Y, qmm.workspace_for(N, K, X))
        torch.cuda.synchronize()
        if s != qmm.OK:
            bad.append((wt, M, K, N, qmm.status_name(s)))
            continue
        Yr, S = oracle.matmul(wt, w, M, K, x)
        ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, 2e-3, 1e-5)
        if not ok:
            bad.append((wt, M, K, N, ratio))
assert qmm.qmm_last_device_error() == qmm.OK
print("BAD" if bad else "OK", bad)
'''

GEMM_COMBOS = [
    {"QMM_GEMM_BN": "64"},
    {"QMM_GEMM_BN": "128"},
    {"QMM_GEMM_BN": "256"},
    {"QMM_GEMM_KS": "1"},
    {"QMM_GEMM_KS": "2", "QMM_GEMM_BN": "256"},
    {"QMM_GEMM_KS": "4", "QMM_GEMM_BN": "64"},
    {"QMM_GEMM_KS": "4", "QMM_GEMM_BN": "128"},
]


@pytest.mark.parametrize("env", GEMM_COMBOS, ids=lambda e: "-".join(f"{k[9:].lower()}{v}" for k, v in e.items()))
def test_forced_gemm_shapes(env):
    """The tensor-core GEMM with every token tile (M not a multiple of the
    128-row tile: the partial tiles must stay inside Y) and every K split
    (K = 2304 splits its 9 chunks 4/5 and 2/2/2/3; K = 256 cannot split)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    r = subprocess.run([sys.executable, "-c", GEMM_CHILD], cwd=ROOT, env={**os.environ, **env, "PYTHONPATH": ROOT},
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().startswith("OK"), r.stdout[-3000:]
