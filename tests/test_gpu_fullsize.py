"""Parity at the full workload sizes, through the same C-ABI calls (and so the
same launch configurations) that bench.py times.

The whole layer runs on the GPU at full size; the oracle recomputes a sample
of token rows (every output of each sampled row, all N) and those rows must
agree within 1 fp16 ulp. Sampled rows: first, second, middle, last and a few
seeded random ones, so every M-tile position class (first tile, interior,
ragged last tile) is visited. Workloads:
  - W8A8 per-channel, N10240 K2560, M in {1, 128, 1024, 4096, 8192};
  - W8A8 per-group gs 64 / 128, N2560 K10240, same M sweep;
  - W4A8 gs 128, N10240 K2560 and N2560 K10240, M in {1, 1024, 8192};
  - the seven linears of an 8B-class decoder layer at M = 2048.
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


def _sample_rows(M: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = {0, min(1, M - 1), M // 2, M - 1}
    rows.update(int(r) for r in rng.integers(0, M, 4))
    return np.array(sorted(rows))


def _check_rows(y_gpu: torch.Tensor, x: np.ndarray, ref_fn, what: str, seed: int):
    M = x.shape[0]
    rows = _sample_rows(M, seed)
    ref = ref_fn(x[rows])
    assert_f16_within_1ulp(host(y_gpu[rows]), ref, what)


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
    _check_rows(y, x.numpy(), lambda xr: oracle.w8a8_linear(xr, wq, s, 0), f"pc M={M}", M)


@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("M", M_SWEEP)
def test_w8a8_pg_full_size(M, gs):
    N, K = 2560, 10240
    wq, s, wqd, sd = _prepared(N, K, 8, gs, 200 + gs)
    x = _acts(M, K, 2000 + M + gs)
    y = cider.w8a8_linear(x.cuda(), wqd, sd, gs)
    _check_rows(y, x.numpy(), lambda xr: oracle.w8a8_linear(xr, wq, s, gs), f"pg{gs} M={M}",
                M + gs)


@pytest.mark.parametrize("N,K", [(10240, 2560), (2560, 10240)])
@pytest.mark.parametrize("M", [1, 1024, 8192])
def test_w4a8_full_size(M, N, K):
    wp, s, wpd, sd = _prepared(N, K, 4, 128, 300 + N)
    x = _acts(M, K, 3000 + M + N)
    y = cider.w4a8_linear(x.cuda(), wpd, sd, 128)
    _check_rows(y, x.numpy(), lambda xr: oracle.w4a8_linear(xr, wp, s, 128),
                f"w4 N={N} K={K} M={M}", M + N)


def test_decoder_layer_linears():
    """q, k, v, o, gate, up, down of an 8B-class layer at 2048 tokens, each
    with its own inputs (1 % outlier channels), weights prepared on the GPU
    (bit-exact with the oracle's prep), sampled rows against the oracle."""
    for i, (name, li) in enumerate(synth.decoder_layer_inputs(2048, seed=0)):
        wq_d, s_d = cider.quantize_weight_int8(li.w.cuda(), 0)
        wq, s = oracle.quantize_weight_int8(li.w.numpy(), 0)
        assert np.array_equal(host(wq_d), wq) and np.array_equal(host(s_d), s), name
        y = cider.w8a8_linear(li.x.cuda(), wq_d, s_d, 0)
        _check_rows(y, li.x.numpy(), lambda xr: oracle.w8a8_linear(xr, wq, s, 0), name, 50 + i)
