"""The integer tensor-core GEMV (N <= 2; Q6_K N == 1) on exact int8 digits of
X, through the C ABI, against the oracle at the GEMV bar
|y - Y| <= 1e-5 * S + 1e-6, plus the cases its digit split has to get
right: wide dynamic range inside a block, zero and tiny blocks, non-finite
blocks, K splits over clusters, ragged M, bf16 X, fused matrices."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth
from test_gpu_parity import ALL, IDS, GEMV_TOL, dev, guarded, guards_intact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    qmm.qmm_set_gemv_i8(1)
    yield
    qmm.qmm_set_gemv_i8(-1)
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def run_gemv(wt, w, M, K, x, xbf16=False):
    N = x.shape[0]
    X = dev(synth.f32_to_bf16_bits(x)).view(torch.bfloat16) if xbf16 else dev(x)
    buf, Y = guarded(N * M)
    Y = Y.view(N, M)
    s = qmm.qmm_gemv(wt, dev(w), M, K, X, N, Y)
    assert s == qmm.OK, qmm.status_name(s)
    torch.cuda.synchronize()
    assert guards_intact(buf, N * M), "write outside Y"
    return Y.cpu().numpy()


def check(y, wt, w, M, K, x, xbf16=False):
    xo = synth.f32_to_bf16_bits(x) if xbf16 else x
    Yr, S = oracle.matmul(wt, w, M, K, xo)
    ok, ratio = oracle.within(y, Yr, S, *GEMV_TOL)
    assert ok, f"max err/tol {ratio:.3g}"
    return ratio


def max_n(wt):
    return 1 if wt == synth.Q6_K else 2


# (M, K): one tile, ragged tails, 128-row tiles, K splits (2, 4, 8 slices)
SHAPES = [(64, 256), (200, 1024), (1000, 2048), (4096, 4096), (777, 14336), (40000, 512)]


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("MK", SHAPES, ids=[f"{m}x{k}" for m, k in SHAPES])
def test_parity_f32(wt, MK):
    M, K = MK
    if wt in (synth.Q4_K, synth.Q6_K, synth.Q5_K) and K % 256:
        pytest.skip("K-quants need K % 256 == 0")
    w = synth.gen_weights(wt, M, K, f"i8-{M}x{K}")
    for N in range(1, max_n(wt) + 1):
        x = synth.gen_x(N, K, f"i8-x-{M}x{K}-{N}")
        check(run_gemv(wt, w, M, K, x), wt, w, M, K, x)


@pytest.mark.parametrize("wt", ALL, ids=IDS)
def test_parity_bf16(wt):
    M, K = 1000, 4096
    w = synth.gen_weights(wt, M, K, "i8-bf16")
    for N in range(1, max_n(wt) + 1):
        x = synth.gen_x(N, K, f"i8-bf16-{N}")
        check(run_gemv(wt, w, M, K, x, xbf16=True), wt, w, M, K, x, xbf16=True)


def hard_x(N, K, name):
    """Blocks with a 1e6 range between their largest and smallest entries,
    whole blocks 1e-20 or 1e20 times the rest, zero blocks, lone spikes."""
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


@pytest.mark.parametrize("wt", ALL, ids=IDS)
def test_parity_hard_values(wt):
    M, K = 512, 2048
    w = synth.gen_weights(wt, M, K, "i8-hard")
    for N in range(1, max_n(wt) + 1):
        x = hard_x(N, K, f"i8-hard-{N}")
        check(run_gemv(wt, w, M, K, x), wt, w, M, K, x)


def test_subnormal_scale_blocks_count_as_zero():
    # a block whose largest |x| is below 2^-98 contributes nothing; every
    # other block exactly as usual (1e-6 absolute slack covers the rest)
    wt, M, K = synth.Q4_0, 256, 1024
    w = synth.gen_weights(wt, M, K, "i8-tiny")
    x = synth.gen_x(1, K, "i8-tiny")
    x[0, 256:288] = np.float32(1e-31)
    y = run_gemv(wt, w, M, K, x)
    check(y, wt, w, M, K, x)
    x2 = x.copy()
    x2[0, 256:288] = 0
    Y2, _ = oracle.matmul(wt, w, M, K, x2)
    assert np.all(np.abs(y[0] - Y2[0]) <= 1e-5 * np.abs(Y2[0]) + 1e-6)


def test_nonfinite_block_gives_nan():
    wt, M, K = synth.Q4_0, 128, 512
    w = synth.gen_weights(wt, M, K, "i8-nan")
    for v in (np.nan, np.inf):
        x = synth.gen_x(1, K, "i8-nan")
        x[0, 40] = v
        y = run_gemv(wt, w, M, K, x)
        assert np.all(np.isnan(y))


@pytest.mark.parametrize("wt", ALL, ids=IDS)
def test_i8_and_bf16_kernels_agree(wt):
    M, K = 3000, 4096
    w = synth.gen_weights(wt, M, K, "i8-vs-bf16")
    x = synth.gen_x(1, K, "i8-vs-bf16")
    y_i8 = run_gemv(wt, w, M, K, x)
    qmm.qmm_set_gemv_i8(0)
    try:
        y_bf = run_gemv(wt, w, M, K, x)
    finally:
        qmm.qmm_set_gemv_i8(1)
    r1 = check(y_i8, wt, w, M, K, x)
    r2 = check(y_bf, wt, w, M, K, x)
    # the digit split is closer to exact than hi/lo bf16 pieces
    assert r1 <= max(r2, 0.05)


def test_fused_matrices_and_argmax_through_i8():
    wt, K = synth.Q4_K, 4096
    Ms = [1024, 256, 256]
    ws = [synth.gen_weights(wt, M, K, f"i8-multi-{i}") for i, M in enumerate(Ms)]
    x = synth.gen_x(1, K, "i8-multi")
    Ys = qmm.gemv_multi(wt, [(dev(w), M) for w, M in zip(ws, Ms)], K, dev(x))
    torch.cuda.synchronize()
    for w, M, Y in zip(ws, Ms, Ys):
        check(Y.cpu().numpy(), wt, w, M, K, x)
    idx, val = qmm.gemv_argmax(wt, dev(ws[0]), Ms[0], K, dev(x))
    torch.cuda.synchronize()
    Yr, S = oracle.matmul(wt, ws[0], Ms[0], K, x)
    i = int(idx.cpu()[0])
    tol = 1e-5 * S[0] + 1e-6
    assert Yr[0, i] >= Yr[0].max() - 2 * tol.max()
    assert abs(float(val.cpu()[0]) - Yr[0, i]) <= tol[i]
