"""GPU parity: the CUDA path through the C ABI against the oracle.

Bars (the method's tolerances):
  dequant            bit-exact against the oracle's once-rounded f32 values
  GEMV (N <= 16)     |y - Y| <= 1e-5 * S + 1e-6      S = sum_k |w x|
  GEMM (tensor core) |y - Y| <= 2e-3 * S + 1e-5
Outputs are written into buffers with poisoned guard bands that must survive.
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
ALL = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K]
IDS = [synth.NAMES[f] for f in ALL]
GUARD = 256  # floats of poison on each side of every output
POISON = 0x7FC0DEAD


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    yield
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded(n: int):
    buf = torch.full((n + 2 * GUARD,), 0, dtype=torch.int32, device="cuda")
    buf.fill_(POISON)
    return buf, buf[GUARD:GUARD + n].view(torch.float32)


def guards_intact(buf: torch.Tensor, n: int) -> bool:
    b = buf.cpu()
    return bool(torch.all(b[:GUARD] == POISON)) and bool(torch.all(b[GUARD + n:] == POISON))


def run(path, wt, w, M, K, x, xbf16=False):
    """Run one call with guarded output; returns y (numpy, [N, M])."""
    N = x.shape[0]
    W = dev(w)
    if xbf16:
        X = dev(synth.f32_to_bf16_bits(x)).view(torch.bfloat16)
    else:
        X = dev(x)
    buf, Y = guarded(N * M)
    Y = Y.view(N, M)
    if path == "gemv":
        s = qmm.qmm_gemv(wt, W, M, K, X, N, Y)
    elif path == "gemm":
        ws = qmm.workspace_for(N, K, X)
        s = qmm.qmm_gemm(wt, W, M, K, X, N, Y, ws)
    else:
        ws = qmm.workspace_for(N, K, X)
        s = qmm.qmm_matmul(wt, W, M, K, X, N, Y, ws)
    assert s == qmm.OK, qmm.status_name(s)
    torch.cuda.synchronize()
    assert guards_intact(buf, N * M), "write outside Y"
    return Y.cpu().numpy()


def check(y, w, wt, M, K, x, tol, xbf16=False, rows=None):
    xo = synth.f32_to_bf16_bits(x) if xbf16 else x
    Yr, S = oracle.matmul(wt, w, M, K, xo, rows=rows)
    yy = y if rows is None else y[:, rows]
    ok, ratio = oracle.within(yy, Yr, S, *tol)
    assert ok, f"worst |err|/tol = {ratio:.3g}"
    return ratio


# --------------------------------------------------------------------------
# dequant: bit exact
# --------------------------------------------------------------------------
def _edge_blocks(wt, M, K):
    """Random blocks with edge values planted in the scale fields."""
    w = synth.gen_weights(wt, M, K, "edge").reshape(M, -1, synth.BLOCK[wt][1])
    specials = np.array([0x0000, 0x8000, 0x0001, 0x83ff, 0x3c00, 0xbc00, 0x7bff, 0x0400], np.uint16)
    sp = specials.view(np.uint8).reshape(-1, 2)
    nb = w.shape[1]
    for i in range(min(nb * M, 64)):
        r, b = divmod(i, nb)
        k = i % len(specials)
        if wt in (synth.Q8_0, synth.Q4_0):
            w[r, b, 0:2] = sp[k]
        elif wt in (synth.Q4_K, synth.Q5_K):
            w[r, b, 0:2] = sp[k]
            w[r, b, 2:4] = sp[(k + 3) % len(specials)]
        else:
            w[r, b, 208:210] = sp[k]
            w[r, b, 192:208] = np.array([-64, 63, -1, 0] * 4, np.int8).view(np.uint8)
    if wt == synth.Q8_0:
        w[0, 0, 2:34] = np.array([-128, 127] * 16, np.int8).view(np.uint8)
    return w.reshape(-1)


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("kind", ["random", "edge"])
def test_dequant_bit_exact(wt, kind):
    M, K = 37, 2048
    w = synth.gen_weights(wt, M, K, "deq") if kind == "random" else _edge_blocks(wt, M, K)
    out = qmm.dequant(wt, dev(w), M, K)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = oracle.dequant_f32(wt, w, M, K)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------------------------
# GEMV (N <= 16)
# --------------------------------------------------------------------------
GEMV_SHAPES = [(1, 256), (7, 512), (128, 2048), (300, 4096)]


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("M,K", GEMV_SHAPES)
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 13, 16])
def test_gemv_parity(wt, M, K, N):
    w = synth.gen_weights(wt, M, K, "gemv")
    x = synth.gen_x(N, K, "gemv")
    y = run("gemv", wt, w, M, K, x)
    check(y, w, wt, M, K, x, GEMV_TOL)


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("N", [1, 8, 16])
@pytest.mark.parametrize("M", [16000, 40000])
def test_gemv_many_rows_no_k_split(wt, N, M):
    """Enough row tiles that the GEMV runs without a K split (one CTA per
    tile); 40000 rows selects the 128-row tile variant on a 152-SM GPU."""
    K = 2048
    w = synth.gen_weights(wt, M, K, "gemv-big")
    x = synth.gen_x(N, K, "gemv-big")
    y = run("gemv", wt, w, M, K, x)
    rows = np.sort(np.random.default_rng(N).choice(M, 512, replace=False))
    check(y, w, wt, M, K, x, GEMV_TOL, rows=rows)


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("N", [1, 4, 9, 16])
def test_gemv_bf16_x(wt, N):
    M, K = 257, 2048
    w = synth.gen_weights(wt, M, K, "gemv-bf16")
    x = synth.gen_x(N, K, "gemv-bf16")
    y = run("gemv", wt, w, M, K, x, xbf16=True)
    check(y, w, wt, M, K, x, GEMV_TOL, xbf16=True)


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("offset", [1, 2, 6])
def test_gemv_unaligned_weights(wt, offset):
    """W not 16-byte aligned: the byte-addressed path must give the same result."""
    M, K, N = 33, 512, 3
    w = synth.gen_weights(wt, M, K, "unaligned")
    x = synth.gen_x(N, K, "unaligned")
    base = torch.zeros(w.size + 64, dtype=torch.uint8, device="cuda")
    base[offset:offset + w.size] = dev(w)
    W = base[offset:offset + w.size]
    X = dev(x)
    buf, Y = guarded(N * M)
    assert qmm.qmm_gemv(wt, W, M, K, X, N, Y.view(N, M)) == qmm.OK
    torch.cuda.synchronize()
    assert guards_intact(buf, N * M)
    check(Y.view(N, M).cpu().numpy(), w, wt, M, K, x, GEMV_TOL)


@pytest.mark.parametrize("wt", ALL, ids=IDS)
def test_gemv_batch_equals_single_token_calls(wt):
    """Decode/prefill identity in spirit: GEMV at N equals N GEMVs at N=1 (within tolerance)."""
    M, K, N = 200, 4096, 8
    w = synth.gen_weights(wt, M, K, "ident")
    x = synth.gen_x(N, K, "ident")
    yb = run("gemv", wt, w, M, K, x)
    ys = np.stack([run("gemv", wt, w, M, K, x[n:n + 1])[0] for n in range(N)])
    _, S = oracle.matmul(wt, w, M, K, x)
    assert np.all(np.abs(yb - ys) <= 2 * (1e-5 * S + 1e-6))


# --------------------------------------------------------------------------
# GEMM (tensor cores)
# --------------------------------------------------------------------------
GEMM_CASES = [
    # (M, K, N)
    (128, 256, 17),
    (128, 2048, 64),
    (300, 2048, 100),
    (256, 4096, 256),
    (129, 2048, 512),
    (512, 4096, 33),
]


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("M,K,N", GEMM_CASES)
def test_gemm_parity(wt, M, K, N):
    if wt == synth.Q6_K and K % 2048:
        pytest.skip("Q6_K tensor-core path needs K % 2048 == 0")
    w = synth.gen_weights(wt, M, K, "gemm")
    x = synth.gen_x(N, K, "gemm")
    y = run("gemm", wt, w, M, K, x)
    check(y, w, wt, M, K, x, GEMM_TOL)


@pytest.mark.parametrize("wt", ALL, ids=IDS)
def test_gemm_bf16_x(wt):
    M, K, N = 384, 2048, 96
    w = synth.gen_weights(wt, M, K, "gemm-bf16")
    x = synth.gen_x(N, K, "gemm-bf16")
    y = run("gemm", wt, w, M, K, x, xbf16=True)
    check(y, w, wt, M, K, x, GEMM_TOL, xbf16=True)


@pytest.mark.parametrize("N", [1, 16])
def test_gemm_small_n(N):
    wt, M, K = synth.Q4_K, 256, 1024
    w = synth.gen_weights(wt, M, K, "gemm-small")
    x = synth.gen_x(N, K, "gemm-small")
    y = run("gemm", wt, w, M, K, x)
    check(y, w, wt, M, K, x, GEMM_TOL)


def test_gemm_unsupported_shape_is_an_error_not_a_fallback():
    wt, M, K, N = synth.Q6_K, 64, 256, 32      # Q6_K rows of 210 B are not 16-byte multiples
    W = dev(synth.gen_weights(wt, M, K, "unsup"))
    X = dev(synth.gen_x(N, K, "unsup"))
    Y = torch.zeros(N, M, device="cuda")
    ws = qmm.workspace_for(N, K, X)
    assert qmm.qmm_gemm(wt, W, M, K, X, N, Y, ws) == qmm.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(Y == 0)


# --------------------------------------------------------------------------
# dispatcher
# --------------------------------------------------------------------------
@pytest.mark.parametrize("N", [1, 16, 17, 512])
def test_dispatcher(N):
    wt, M, K = synth.Q4_K, 256, 2048
    w = synth.gen_weights(wt, M, K, "disp")
    x = synth.gen_x(N, K, "disp")
    y = run("matmul", wt, w, M, K, x)
    # N <= QMM_MATMUL_GEMV_MAX_N takes the f32 GEMV and must meet the tighter bar
    check(y, w, wt, M, K, x, GEMV_TOL if N <= qmm.MATMUL_GEMV_MAX_N else GEMM_TOL)


# --------------------------------------------------------------------------
# error paths on the device
# --------------------------------------------------------------------------
def test_validation_leaves_output_untouched():
    wt, M, K, N = synth.Q4_0, 64, 256, 2
    W = dev(synth.gen_weights(wt, M, K, "val"))
    X = dev(synth.gen_x(N, K, "val"))
    buf, Y = guarded(N * M)
    Y.fill_(3.0)
    assert qmm.qmm_gemv(wt, W, M, K + 1, X, N, Y.view(N, M)) == qmm.ERR_INVALID_ARG
    assert qmm.qmm_gemv(wt, W, M, K, X, N, Y.view(N, M), w_bytes=W.numel() - 1) == qmm.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(Y == 3.0) and guards_intact(buf, N * M)


def test_bounded_wait_reports_timeout_and_context_survives():
    """A tiny wait limit makes the GEMM's waits give up: the kernel must exit
    cleanly with QMM_ERR_TIMEOUT in the status word, and the next call works."""
    wt, M, K, N = synth.Q4_K, 1024, 4096, 256
    w = synth.gen_weights(wt, M, K, "timeout")
    x = synth.gen_x(N, K, "timeout")
    W, X = dev(w), dev(x)
    Y = torch.empty(N, M, device="cuda")
    ws = qmm.workspace_for(N, K, X)
    assert qmm.qmm_last_device_error() == qmm.OK
    qmm.qmm_set_wait_limit(1)
    try:
        assert qmm.qmm_gemm(wt, W, M, K, X, N, Y, ws) == qmm.OK
        assert qmm.qmm_last_device_error() == qmm.ERR_TIMEOUT
    finally:
        qmm.qmm_set_wait_limit(1 << 31)
    assert qmm.qmm_last_device_error() == qmm.OK
    assert qmm.qmm_gemm(wt, W, M, K, X, N, Y, ws) == qmm.OK
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK
    check(Y.cpu().numpy(), w, wt, M, K, x, GEMM_TOL)
