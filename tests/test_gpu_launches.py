"""The library's launch counter (qmm_kernel_launches), which bench.py uses
for its gpu_launches figure: one count per kernel the library launches or
records into a graph, none for a rejected call or a graph replay."""
from __future__ import annotations

import pytest
import torch

from block_quantized_gemv_gguf_gb300 import qmm, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    qmm.load()


def _weights(wt, M, K):
    return torch.from_numpy(synth.gen_weights(wt, M, K, "launches")).cuda()


def _delta(f):
    torch.cuda.synchronize()
    n0 = qmm.qmm_kernel_launches()
    f()
    torch.cuda.synchronize()
    return qmm.qmm_kernel_launches() - n0


def test_gemv_is_one_launch():
    M, K = 4096, 4096
    W = _weights(synth.Q4_0, M, K)
    X = torch.from_numpy(synth.gen_x(1, K, "launches")).cuda()
    Y = torch.empty(1, M, device="cuda")
    assert _delta(lambda: qmm.qmm_gemv(synth.Q4_0, W, M, K, X, 1, Y)) == 1


def test_gemm_launches_and_the_f32_conversion():
    M, K, N = 14336, 4096, 512
    W = _weights(synth.Q4_K, M, K)
    x = synth.gen_x(N, K, "launches")
    X = torch.from_numpy(x).cuda()
    XB = torch.from_numpy(synth.f32_to_bf16_bits(x)).cuda().view(torch.bfloat16)
    Y = torch.empty(N, M, device="cuda")
    ws = qmm.workspace_for(N, K, X)
    nb = _delta(lambda: qmm.qmm_gemm(synth.Q4_K, W, M, K, XB, N, Y))
    nf = _delta(lambda: qmm.qmm_gemm(synth.Q4_K, W, M, K, X, N, Y, ws))
    assert nb in (1, 2)          # whole waves, and possibly the split last wave
    assert nf == nb + 1          # plus the f32 -> bf16 conversion


def test_rejected_call_launches_nothing():
    M, K = 256, 512
    W = _weights(synth.Q8_0, M, K)
    X = torch.zeros(1, K + 32, device="cuda")
    Y = torch.empty(1, M, device="cuda")
    # K not a multiple of the block size: rejected on the host
    assert _delta(lambda: qmm.qmm_gemv(synth.Q8_0, W, M, K + 1, X, 1, Y)) == 0


def test_graph_recording_counts_and_replay_does_not():
    M, K = 1024, 4096
    W = _weights(synth.Q4_0, M, K)
    X = torch.from_numpy(synth.gen_x(1, K, "launches")).cuda()
    Y = torch.empty(1, M, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert qmm.qmm_gemv(synth.Q4_0, W, M, K, X, 1, Y, stream=s) == qmm.OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = qmm.qmm_kernel_launches()
    with torch.cuda.graph(g, stream=s):
        assert qmm.qmm_gemv(synth.Q4_0, W, M, K, X, 1, Y, stream=s) == qmm.OK
    assert qmm.qmm_kernel_launches() - n0 == 1
    n1 = qmm.qmm_kernel_launches()
    g.replay()
    torch.cuda.synchronize()
    assert qmm.qmm_kernel_launches() == n1
