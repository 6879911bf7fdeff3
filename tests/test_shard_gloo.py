"""Row sharding over ranks (host logic), on CPU with the gloo backend.

Two ranks each compute the rows they own of a Q4_K matrix (the oracle
stands in for the per-rank GEMV: the split itself is what is tested), gather
the slices with shard.gather_rows, and must reproduce the single-rank result
exactly; row_partition's slices must tile the rows.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

from block_quantized_gemv_gguf_gb300.shard import row_partition


@pytest.mark.parametrize("M", [1, 15, 16, 17, 300, 4096, 128256])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_row_partition_tiles_the_rows(M, world):
    b = [row_partition(M, world, g) for g in range(world)]
    assert b[0][0] == 0 and b[-1][1] == M
    assert all(b[g][1] == b[g + 1][0] for g in range(world - 1))
    assert all(r0 % 16 == 0 and r0 <= r1 for r0, r1 in b)
    sizes = [r1 - r0 for r0, r1 in b]
    assert max(sizes) - min(sizes) <= 16


def test_row_partition_rejects_bad_ranks():
    with pytest.raises(ValueError):
        row_partition(100, 2, 2)
    with pytest.raises(ValueError):
        row_partition(100, 0, 0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist

    import oracle
    from block_quantized_gemv_gguf_gb300 import synth
    from block_quantized_gemv_gguf_gb300.shard import gather_rows
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wt, M, K, N = synth.Q4_K, 200, 512, 3
        w = synth.gen_weights(wt, M, K, "shard")
        x = synth.gen_x(N, K, "shard")
        r0, r1 = row_partition(M, world, rank)
        rb = synth.row_bytes(wt, K)
        y_local, _ = oracle.matmul(wt, w[r0 * rb:r1 * rb], r1 - r0, K, x)
        Y = gather_rows(torch.from_numpy(np.ascontiguousarray(y_local)), M, world).numpy()
        Yfull, _ = oracle.matmul(wt, w, M, K, x)
        q.put((rank, bool(np.array_equal(Y, Yfull)), Y.shape))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gather_equals_single_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for p in procs:
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] for r in res), res
    assert all(r[2] == (3, 200) for r in res)
