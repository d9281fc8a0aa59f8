"""Output-channel (column-parallel) split on CPU ranks: the shards cover the
output channels exactly once, and gathering each rank's shard, computed by the
oracle from that rank's weight rows, reproduces the unsplit layer bit for bit
(output channels are independent: no reduction across ranks)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402
import w4a8_quantized_gemm_int8_b300 as cider  # noqa: E402


@pytest.mark.parametrize("N", [1, 127, 128, 300, 1000, 10240])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_column_shards_partition_the_channels(N, world):
    spans = [cider.column_shard(N, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == N
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0 and a0 <= a1
    widths = [n1 - n0 for n0, n1 in spans]
    assert all(n0 % 128 == 0 for n0, _ in spans if n0 < N)  # shards start on tile boundaries
    units = [(w + 127) // 128 for w in widths]
    assert max(units) - min(units) <= 1                      # balanced in 128-channel tiles


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, gs, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    M, N, K = 5, 300, 256
    li = synth.linear_inputs(M, N, K, n_out=2, seed=3)
    x, w = li.x.numpy(), li.w.numpy()
    wq, s = oracle.quantize_weight_int8(w, gs)
    n0, n1 = cider.column_shard(N, world, rank)
    y_shard = oracle.w8a8_linear(x, wq[n0:n1], s[n0:n1], gs)  # this rank's weight rows only
    # gloo has no 16-bit collectives: carry the fp16 values as fp32 (exact)
    y = cider.gather_columns(torch.from_numpy(y_shard.astype(np.float32)), N, world)
    out[rank] = y.numpy().astype(np.float16).tobytes()
    dist.destroy_process_group()


@pytest.mark.parametrize("gs", [0, 64])
def test_gathered_shards_equal_the_unsplit_layer(gs):
    world = 3
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), gs, out), nprocs=world, join=True)
        res = dict(out)
    M, N, K = 5, 300, 256
    li = synth.linear_inputs(M, N, K, n_out=2, seed=3)
    x, w = li.x.numpy(), li.w.numpy()
    wq, s = oracle.quantize_weight_int8(w, gs)
    ref = oracle.w8a8_linear(x, wq, s, gs)
    for r in range(world):
        y = np.frombuffer(res[r], dtype=np.float16).reshape(M, N)
        assert np.array_equal(y.view(np.uint16), ref.view(np.uint16))
