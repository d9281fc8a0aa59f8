"""Parity at the full workload sizes, through the same C-ABI calls (and so the
same launch configurations) that bench.py times.

The whole layer runs on the GPU at full size and the oracle recomputes the
whole layer: EVERY output is compared, so each tile that a persistent cluster
takes after its first (the next tile's scale prefetch, the TMA ring and the
accumulator phases carried across tiles, the ragged last tile) is checked.
Bars: bit-identical fp16 (the kernels perform the oracle's operations in its
order; 1 ulp is the outer tolerance), bit-exact int32. Workloads:
  - W8A8 per-channel, N10240 K2560, M in {1, 128, 1024, 4096, 8192};
  - W8A8 per-group gs 64 / 128, N2560 K10240, same M sweep;
  - W4A8 gs 128, N10240 K2560 and N2560 K10240, M in {1, 1024, 8192};
  - the seven linears of an 8B-class decoder layer at M = 2048;
  - raw int32 products with more tiles than the grid has clusters (SM
    pairs) or SMs (single-SM engine), per channel and per group.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a8_quantized_gemm_int8_b300 as cider
from gpu_helpers import assert_f16_within_1ulp, host

pytestmark = pytest.mark.gpu

M_SWEEP = [1, 128, 1024, 4096, 8192]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cider.load_library()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    st, site = cider.device_status()
    assert st == cider.CIDER_OK, f"device status {st} at site {site:#x}"


# Weight preparation goes through the oracle (its codes are what the GEMM
# consumes); a module-level cache keeps one prepared weight per shape.
_weights: dict = {}


def _prepared(N, K, bits, gs, seed):
    key = (N, K, bits, gs, seed)
    if key not in _weights:
        _weights.clear()
        w = synth.weights(N, K, synth.generator(seed)).numpy()
        if bits == 8:
            wq, s = oracle.quantize_weight_int8(w, gs)
        else:
            wq, s = oracle.pack_weight_int4(w, gs)
        _weights[key] = (wq, s, torch.from_numpy(wq).cuda(), torch.from_numpy(s).cuda())
    return _weights[key]


def _acts(M, K, seed):
    return synth.activations(M, K, 4, synth.generator(seed))


@pytest.mark.parametrize("M", M_SWEEP)
def test_w8a8_pc_full_size(M):
    N, K = 10240, 2560
    wq, s, wqd, sd = _prepared(N, K, 8, 0, 100)
    x = _acts(M, K, 1000 + M)
    y = cider.w8a8_linear(x.cuda(), wqd, sd, 0)
    assert_f16_within_1ulp(host(y), oracle.w8a8_linear(x.numpy(), wq, s, 0), f"pc M={M}")


@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("M", M_SWEEP)
def test_w8a8_pg_full_size(M, gs):
    N, K = 2560, 10240
    wq, s, wqd, sd = _prepared(N, K, 8, gs, 200 + gs)
    x = _acts(M, K, 2000 + M + gs)
    y = cider.w8a8_linear(x.cuda(), wqd, sd, gs)
    assert_f16_within_1ulp(host(y), oracle.w8a8_linear(x.numpy(), wq, s, gs),
                           f"pg{gs} M={M}")


@pytest.mark.parametrize("N,K", [(10240, 2560), (2560, 10240)])
@pytest.mark.parametrize("M", [1, 128, 1024, 8192])
def test_w4a8_full_size(M, N, K):
    wp, s, wpd, sd = _prepared(N, K, 4, 128, 300 + N)
    x = _acts(M, K, 3000 + M + N)
    y = cider.w4a8_linear(x.cuda(), wpd, sd, 128)
    assert_f16_within_1ulp(host(y), oracle.w4a8_linear(x.numpy(), wp, s, 128),
                           f"w4 N={N} K={K} M={M}")


def test_decoder_layer_linears():
    """q, k, v, o, gate, up, down of an 8B-class layer at 2048 tokens, each
    with its own inputs (1 % outlier channels), weights prepared on the GPU
    (bit-exact with the oracle's prep), every output against the oracle."""
    for name, li in synth.decoder_layer_inputs(2048, seed=0):
        wq_d, s_d = cider.quantize_weight_int8(li.w.cuda(), 0)
        wq, s = oracle.quantize_weight_int8(li.w.numpy(), 0)
        assert np.array_equal(host(wq_d), wq) and np.array_equal(host(s_d), s), name
        y = cider.w8a8_linear(li.x.cuda(), wq_d, s_d, 0)
        assert_f16_within_1ulp(host(y), oracle.w8a8_linear(li.x.numpy(), wq, s, 0), name)


def _codes(shape, seed):
    g = np.random.default_rng(seed)
    return g.integers(-127, 128, size=shape, dtype=np.int16).astype(np.int8)


@pytest.mark.parametrize("M,N,K,gs", [
    (2048, 5120, 2560, 0),   # 8 x 20 = 160 pair tiles on at most 74 clusters
    (2304, 2560, 512, 64),   # 9 x 10 = 90 per-group pair tiles
    (128, 20480, 1024, 0),   # 160 single-SM 128 x 128 tiles on 148 SMs
    (96, 10240, 512, 64),    # 160 single-SM 128 x 64 per-group tiles
])
def test_raw_int32_more_tiles_than_clusters(M, N, K, gs):
    """Raw int32 products (totals, or per-group partials) where every
    cluster of the persistent grid walks several tiles; bit-exact against the
    oracle's int32 products."""
    q = _codes((M, K), M + K)
    w = _codes((N, K), N + K)
    out = cider.raw_gemm_s32(torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(), K, 8, gs)
    ref = oracle.gemm_s32(q, w, gs)
    got = host(out)
    assert got.shape == ref.shape
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} int32 outputs differ"
