"""GPU parity of the streaming one-token GEMV under every plan it can take.

A task of that kernel is R consecutive rows (R = 1, 2, 4) at one 256-weight
column, computed by one lane against one read of the column's x values;
a warp stage is 32 consecutive tasks.  A stage is one contiguous copy of W
when R = 1 or the unit count U of a row divides 32, and one copy per
(row, run of columns) piece otherwise.  The shapes below cover: U = 1, 3, 8,
12, 16, 32, 56, 112 (contiguous and piecewise stages, row groups inside one
stage and groups spanning up to four stages), fewer rows than R and than
SMs, a short last row group, and the forced plans one warp / one slot / one
or two CTAs per SM.  Each plan is checked with qmm_gemv_stream_plan before
it runs, so the kernel under test is the one that was asked for.  Bar:
|y - Y| <= 1e-5 * S + 1e-6 against the oracle, bit-identical on repeat.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu

GEMV_TOL = (1e-5, 1e-6)
ALL = [synth.Q8_0, synth.Q4_0, synth.Q4_K, synth.Q6_K, synth.Q5_K]
IDS = [synth.NAMES[f] for f in ALL]
SHAPES = [(1, 256), (5, 256), (7, 768), (33, 2048), (151, 3072), (300, 4096), (130, 8192), (61, 14336),
          (9, 28672), (3001, 4096)]
# (rows per task, warps, slots, CTAs per SM); 0 = the planner's choice
PLANS = [(1, 0, 0, 0), (2, 0, 0, 0), (4, 0, 0, 0), (4, 1, 1, 1), (4, 2, 2, 1), (2, 5, 1, 2), (4, 0, 1, 2),
         (2, 3, 1, 0)]
GUARD = 256
POISON = 0x7FC0DEAD


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()
    yield
    qmm.qmm_set_gemv_stream(-1, -1, -1, -1, -1)
    torch.cuda.synchronize()
    assert qmm.qmm_last_device_error() == qmm.OK


def _aligned(wt, K):
    E, B = synth.BLOCK[wt]
    return (K // E * B) % 16 == 0


def _run_plan(wt, plan, direct=2):
    """Returns the number of shapes the forced plan served (direct: 2 the
    staged kernel, 1 the direct-load variant)."""
    r, nw, s, cps = plan
    qmm.qmm_set_gemv_stream(r, nw, s, cps, direct)
    served = 0
    try:
        for M, K in SHAPES:
            if not _aligned(wt, K):
                continue
            st, p = qmm.qmm_gemv_stream_plan(wt, M, K)
            if st != qmm.OK:
                # shared memory too small for the forced plan, or a piecewise
                # stage of 210-byte (Q6_K) units: another kernel would run
                assert st == qmm.ERR_UNSUPPORTED
                continue
            if direct == 1 and wt in (synth.Q4_0, synth.Q4_K):
                assert p["direct"] == 1 and p["rows_per_task"] == 1 and p["slots"] == 0, p
            else:
                assert p["direct"] == 0, p
                assert (r == 0 or p["rows_per_task"] == r) and (s == 0 or p["slots"] == s), p
            assert nw == 0 or p["warps"] == nw, p
            w = synth.gen_weights(wt, M, K, f"rows-{M}-{K}")
            x = synth.gen_x(1, K, f"rows-{M}-{K}")
            W = torch.from_numpy(w).cuda()
            X = torch.from_numpy(x).cuda()
            buf = torch.full((M + 2 * GUARD,), POISON, dtype=torch.int32, device="cuda")
            Y = buf[GUARD:GUARD + M].view(torch.float32).view(1, M)
            assert qmm.qmm_gemv(wt, W, M, K, X, 1, Y) == qmm.OK
            torch.cuda.synchronize()
            b = buf.cpu()
            assert torch.all(b[:GUARD] == POISON) and torch.all(b[GUARD + M:] == POISON), (M, K, "write outside Y")
            Yr, S = oracle.matmul(wt, w, M, K, x)
            ok, ratio = oracle.within(Y.cpu().numpy(), Yr, S, *GEMV_TOL)
            assert ok, (M, K, p, f"worst |err|/tol = {ratio:.3g}")
            Y2 = torch.empty_like(Y)
            assert qmm.qmm_gemv(wt, W, M, K, X, 1, Y2) == qmm.OK
            torch.cuda.synchronize()
            assert torch.equal(Y.view(torch.int32), Y2.view(torch.int32)), (M, K, "not deterministic")
            served += 1
    finally:
        qmm.qmm_set_gemv_stream(-1, -1, -1, -1, -1)
    return served


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("plan", PLANS, ids=lambda p: "r{}-w{}-s{}-c{}".format(*p))
def test_forced_plan_parity(wt, plan):
    served = _run_plan(wt, plan)
    if plan[1:] == (0, 0, 0) and not (wt == synth.Q6_K and plan[0] > 1):
        assert served >= 6
    else:
        assert served >= 1   # forced warps and slots fit only the smaller X / narrower units


DIRECT_PLANS = [(0, 0, 0, 0), (0, 0, 0, 1), (0, 0, 0, 2), (0, 5, 0, 1), (0, 3, 0, 2)]


@pytest.mark.parametrize("wt", ALL, ids=IDS)
@pytest.mark.parametrize("plan", DIRECT_PLANS, ids=lambda p: "w{}-c{}".format(p[1], p[3]))
def test_direct_variant_parity(wt, plan):
    """The direct-load variant (Q4_0, Q4_K; other formats keep the staged
    kernel when it is requested) on every shape and CTA shape."""
    assert _run_plan(wt, plan, direct=1) >= 5   # two CTAs per SM cannot hold X of K = 28672


@pytest.mark.parametrize("wt", [synth.Q4_0, synth.Q4_K], ids=["Q4_0", "Q4_K"])
def test_direct_variant_argmax(wt):
    M, K = 2999, 4096
    w = synth.gen_weights(wt, M, K, "rows-amax")
    x = synth.gen_x(1, K, "rows-amax")
    W = torch.from_numpy(w).cuda()
    X = torch.from_numpy(x).cuda()
    qmm.qmm_set_gemv_stream(0, 0, 0, 0, 1)
    try:
        st, p = qmm.qmm_gemv_stream_plan(wt, M, K)
        assert st == qmm.OK and p["direct"] == 1
        idx, val = qmm.gemv_argmax(wt, W, M, K, X)
        y = qmm.gemv(wt, W, M, K, X)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_gemv_stream(-1, -1, -1, -1, -1)
    y = y.cpu().numpy()
    j = int(np.argmax(y[0]))
    assert int(idx.cpu()[0]) == j
    assert val.cpu().numpy().view(np.uint32)[0] == y[0, j].view(np.uint32)


@pytest.mark.parametrize("wt", [synth.Q4_0, synth.Q4_K, synth.Q6_K], ids=["Q4_0", "Q4_K", "Q6_K"])
@pytest.mark.parametrize("r", [2, 4])
def test_forced_plan_argmax(wt, r):
    """Argmax mode of the same kernel: the row of qmm_gemv's largest output
    (lowest row on ties) and its bits."""
    M, K = 2999, 4096
    w = synth.gen_weights(wt, M, K, "rows-amax")
    x = synth.gen_x(1, K, "rows-amax")
    W = torch.from_numpy(w).cuda()
    X = torch.from_numpy(x).cuda()
    qmm.qmm_set_gemv_stream(r, 0, 0, 0, 2)
    try:
        st, p = qmm.qmm_gemv_stream_plan(wt, M, K)
        assert st == qmm.OK and p["rows_per_task"] == r
        idx, val = qmm.gemv_argmax(wt, W, M, K, X)
        y = qmm.gemv(wt, W, M, K, X)
        torch.cuda.synchronize()
    finally:
        qmm.qmm_set_gemv_stream(-1, -1, -1, -1, -1)
    y = y.cpu().numpy()
    j = int(np.argmax(y[0]))
    assert int(idx.cpu()[0]) == j
    assert val.cpu().numpy().view(np.uint32)[0] == y[0, j].view(np.uint32)


def test_default_plans_of_the_decode_shapes():
    """The planner's choice on the Llama-3-8B decode shapes: two rows per
    task where every SM gets several stages and a stage is one contiguous
    copy (K = 4096), or for the offset-free K-quants also when it is copied
    in pieces (K = 14336); one row per task for small M; one slot per warp;
    two CTAs per SM for rows of 4096 up to 64 MB (at least 8 rows per CTA),
    each holding more than a third of the SM's shared memory, else one CTA
    per SM holding more than half."""
    sm_smem = 233472
    half = sm_smem // 2
    for wt, slots in ((synth.Q4_0, 1), (synth.Q4_K, 1), (synth.Q8_0, 1), (synth.Q5_K, 1)):
        st, p = qmm.qmm_gemv_stream_plan(wt, 14336, 4096)
        assert st == qmm.OK and p["rows_per_task"] == 2 and p["slots"] == slots and p["smem"] <= half, (wt, p)
        # no SM can hold a third CTA of the launch
        assert 3 * p["smem"] > sm_smem, p
    for wt, r in ((synth.Q4_0, 1), (synth.Q8_0, 1), (synth.Q4_K, 2), (synth.Q6_K, 1)):
        st, p = qmm.qmm_gemv_stream_plan(wt, 4096, 14336)
        assert st == qmm.OK and p["rows_per_task"] == r, (wt, p)
    st, p = qmm.qmm_gemv_stream_plan(synth.Q4_0, 1024, 4096)
    # few rows per SM: one CTA per SM, alone on it
    assert st == qmm.OK and p["rows_per_task"] == 1 and p["grid"] <= 1024 and 2 * p["smem"] > sm_smem, p
    st, p = qmm.qmm_gemv_stream_plan(synth.Q6_K, 128256, 4096)
    assert st == qmm.OK and p["rows_per_task"] == 2, p
