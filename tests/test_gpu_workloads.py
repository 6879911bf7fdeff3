"""Parity at the full benchmark sizes, through the same C-ABI calls bench.py
times (qmm_matmul, default dispatch).  Small matrices are checked in full;
large ones on a seeded sample of output rows that the oracle computes one by
one (every token column of those rows).

Workloads:
  Q8_0 256x512, N=1
  Q4_0 decode shapes (4096,4096) (1024,4096) (14336,4096) (4096,14336), N=1
  Q4_K prefill (4096,4096) (14336,4096), N in {64, 256, 512}, f32 and bf16 X
  Q6_K LM head 128256x4096, N in {1, 4, 8}
  32-layer Q4_K_M-style decoder, all 7 projections of every layer, N in
  {1, 2, 4, 8, 16, 32, 64, 128, 256, 512}: layers 0 and 31 on every row,
  layers 1..30 on a seeded 1/16 of the rows
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

GEMV_TOL = (1e-5, 1e-6)
GEMM_TOL = (2e-3, 1e-5)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()


def tol_for(N):
    return GEMV_TOL if N <= qmm.MATMUL_GEMV_MAX_N else GEMM_TOL


def run_and_check(wt, w_np, W, M, K, N, name, rows=None, xbf16=False):
    x = synth.gen_x(N, K, name)
    X = torch.from_numpy(x).cuda()
    xo = x
    if xbf16:
        xo = synth.f32_to_bf16_bits(x)
        X = torch.from_numpy(xo).cuda().view(torch.bfloat16)
    Y = qmm.matmul(wt, W, M, K, X)
    torch.cuda.synchronize()
    y = Y.cpu().numpy()
    Yr, S = oracle.matmul(wt, w_np, M, K, xo, rows=rows)
    yy = y if rows is None else y[:, rows]
    ok, ratio = oracle.within(yy, Yr, S, *tol_for(N))
    assert ok, f"{synth.NAMES[wt]} M={M} K={K} N={N}: worst |err|/tol = {ratio:.3g}"
    assert np.all(np.isfinite(y))


def sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    r = rng.choice(M, size=min(n, M), replace=False)
    return np.sort(np.concatenate([r, [0, M - 1]]))


def test_q8_0_small():
    wt, M, K = synth.Q8_0, 256, 512
    w = synth.gen_weights(wt, M, K, "wl-q8")
    run_and_check(wt, w, torch.from_numpy(w).cuda(), M, K, 1, "wl-q8")


@pytest.mark.parametrize("M,K", [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)])
def test_q4_0_decode_shapes(M, K):
    wt = synth.Q4_0
    w = synth.gen_weights(wt, M, K, f"bench-decode-{M}x{K}")
    run_and_check(wt, w, torch.from_numpy(w).cuda(), M, K, 1, f"wl-decode-{K}")


@pytest.mark.parametrize("M,K", [(4096, 4096), (14336, 4096)])
@pytest.mark.parametrize("N", [64, 256, 512])
@pytest.mark.parametrize("xbf16", [False, True], ids=["f32x", "bf16x"])
def test_q4_k_prefill(M, K, N, xbf16):
    wt = synth.Q4_K
    w = synth.gen_weights(wt, M, K, f"wl-prefill-{M}x{K}")
    rows = sample_rows(M, 192, M + N)
    run_and_check(wt, w, torch.from_numpy(w).cuda(), M, K, N, f"wl-prefill-{N}", rows=rows, xbf16=xbf16)


@pytest.fixture(scope="module")
def lmhead():
    M, K = 128256, 4096
    w = synth.gen_weights(synth.Q6_K, M, K, "bench-lmhead")
    return w, torch.from_numpy(w).cuda()


@pytest.mark.parametrize("N", [1, 4, 8])
def test_q6_k_lm_head(lmhead, N):
    w, W = lmhead
    M, K = 128256, 4096
    run_and_check(synth.Q6_K, w, W, M, K, N, f"wl-lmhead-{N}", rows=sample_rows(M, 1024, N))


@pytest.mark.parametrize("layer", range(synth.DECODER_LAYERS))
def test_decoder_sweep_layers(layer):
    full = layer in (0, synth.DECODER_LAYERS - 1)
    for name, wt, M, K in synth.DECODER_LAYER:
        w = synth.gen_weights(wt, M, K, f"layer{layer}.{name}")
        W = torch.from_numpy(w).cuda()
        for N in synth.DECODER_NS:
            rows = None if full else np.sort(np.random.default_rng(layer * 1000 + N).choice(M, M // 16, replace=False))
            run_and_check(wt, w, W, M, K, N, f"layer{layer}.{name}.x{N}", rows=rows)
        del W
