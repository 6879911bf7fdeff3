"""Q8_0 activations ("cera 0.5.2 src/backend/cpu.rs",
quantize_f32_to_q8_0_scalar) and the integer GEMV on them, through the C ABI:
  * qmm_quantize_q8_0 equals the oracle's quantizer bit for bit (codes and
    binary16-rounded scales), special blocks included;
  * qmm_gemv_preq / qmm_gemv_q8act equal the oracle's product of dequant(W)
    with the dequantized activations within 1e-5 * S + 1e-6;
  * a token's outputs do not depend on the other tokens of the batch.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth
from test_gpu_parity import ALL, IDS, GEMV_TOL, dev, guarded, guards_intact
import test_oracle_pins as pins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    yield
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def special_x(N, K):
    x = synth.gen_x(N, K, "q8act-special")
    cases = [pins.q8act_case_arrays(c)[0] for c in pins.Q8ACT_CASES]
    for i, c in enumerate(cases):
        n, b = i % N, (3 * i + 1) % (K // 32)
        x[n, 32 * b:32 * b + 32] = c
    x[0, 32 * 5:32 * 6] *= np.float32(1e-3)
    return x


@pytest.mark.parametrize("xbf16", [False, True], ids=["f32", "bf16"])
def test_quantizer_bit_exact(xbf16):
    N, K = 5, 4096
    x = special_x(N, K)
    if xbf16:
        bits = synth.f32_to_bf16_bits(x)
        xin = dev(bits).view(torch.bfloat16)
        xref = (bits.astype(np.uint32) << 16).view(np.float32)
    else:
        xin, xref = dev(x), x
    s, q = qmm.quantize_q8_0(xin)
    torch.cuda.synchronize()
    s_ref, q_ref = oracle.quantize_q8_0(xref)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    s_got = s.cpu().numpy()
    assert np.array_equal(s_got.view(np.uint32), s_ref.view(np.uint32))


def run_preq(wt, w, M, K, x):
    N = x.shape[0]
    s_ref, q_ref = oracle.quantize_q8_0(x)
    buf, Y = guarded(N * M)
    Y = Y.view(N, M)
    st = qmm.qmm_gemv_preq(wt, dev(w), M, K, dev(s_ref), dev(q_ref), N, Y)
    assert st == qmm.OK, qmm.status_name(st)
    torch.cuda.synchronize()
    assert guards_intact(buf, N * M)
    return Y.cpu().numpy()


SHAPES = [(64, 256), (300, 2048), (4096, 4096), (1000, 14336)]


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("MK", SHAPES, ids=[f"{m}x{k}" for m, k in SHAPES])
def test_preq_parity(wt, MK):
    M, K = MK
    w = synth.gen_weights(wt, M, K, f"q8act-{M}x{K}")
    if synth.row_bytes(wt, K) % 16:
        # no tensor-core geometry (16-byte row pitch) and no other variant
        s_ref, q_ref = oracle.quantize_q8_0(synth.gen_x(1, K, "q8act-unsup"))
        Y = torch.empty(1, M, device="cuda")
        assert qmm.qmm_gemv_preq(wt, dev(w), M, K, dev(s_ref), dev(q_ref), 1, Y) == qmm.ERR_UNSUPPORTED
        return
    for N in (1, 3, 8, 13, 16):
        x = synth.gen_x(N, K, f"q8act-x-{M}-{N}")
        y = run_preq(wt, w, M, K, x)
        Yr, S = oracle.matmul_q8act(wt, w, M, K, x)
        ok, ratio = oracle.within(y, Yr, S, *GEMV_TOL)
        assert ok, f"N={N}: max err/tol {ratio:.3g}"


@pytest.mark.parametrize("wt", ALL, ids=IDS)
def test_q8act_end_to_end_and_token_independence(wt):
    M, K, N = 2000, 4096, 8
    w = synth.gen_weights(wt, M, K, "q8act-e2e")
    x = special_x(N, K)
    # finite outputs to compare: no non-finite entries, no binary16 scale overflow
    x = np.clip(np.nan_to_num(x, nan=0.0, posinf=0.0, neginf=0.0), -1e4, 1e4).astype(np.float32)
    W, X = dev(w), dev(x)
    Y = qmm.gemv_q8act(wt, W, M, K, X)
    torch.cuda.synchronize()
    Yr, S = oracle.matmul_q8act(wt, w, M, K, x)
    y = Y.cpu().numpy()
    ok, ratio = oracle.within(y, Yr, S, *GEMV_TOL)
    assert ok, ratio
    # token 3 alone gives the same outputs within the bar (decode = prefill)
    y3 = qmm.gemv_q8act(wt, W, M, K, X[3:4].contiguous()).cpu().numpy()
    assert np.all(np.abs(y3[0] - y[3]) <= 2 * (GEMV_TOL[0] * S[3] + GEMV_TOL[1]))


def test_q8act_errors():
    wt, M, K, N = synth.Q4_0, 64, 512, 2
    W = dev(synth.gen_weights(wt, M, K, "q8act-err"))
    x = synth.gen_x(N, K, "q8act-err")
    s, q = oracle.quantize_q8_0(x)
    S, Q = dev(s), dev(q)
    Y = torch.empty(N, M, device="cuda")
    assert qmm.qmm_gemv_preq(wt, W, M, K, S, Q, 17, Y) == qmm.ERR_INVALID_ARG
    assert qmm.qmm_gemv_preq(wt, W, M, K, None, Q, N, Y) == qmm.ERR_INVALID_ARG
    # misaligned scales: no tensor-core geometry, and no other variant
    S2 = torch.zeros(S.numel() + 4, device="cuda")[1:1 + S.numel()]
    S2.copy_(S.view(-1))
    assert qmm.qmm_gemv_preq(wt, W, M, K, S2, Q, N, Y) == qmm.ERR_UNSUPPORTED
    # workspace too small
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    assert qmm.qmm_gemv_q8act(wt, W, M, K, dev(x), N, Y, ws) == qmm.ERR_INVALID_ARG
    # quantizer: K not a multiple of 32
    assert qmm.qmm_quantize_q8_0(dev(x), N, 500, S, Q) == qmm.ERR_INVALID_ARG
    torch.cuda.synchronize()
