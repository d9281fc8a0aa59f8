"""bfloat16 activations and outputs (README roadmap: float16/bfloat16
dtypes), CUDA path against the CPU oracle through the C ABI. bf16 values are
handed to the oracle as uint16 bit patterns. Bars as for fp16: codes, scales
and int32 exact; outputs bit-identical (both sides round the same fp32 value
to nearest even)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a8_quantized_gemm_int8_b300 as cider
from gpu_helpers import cuda, every_pair_rows, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cider.load_library()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    st, site = cider.device_status()
    assert st == cider.CIDER_OK, f"device status {st} at site {site:#x}"


def _bf16_bits(x32: np.ndarray) -> np.ndarray:
    return oracle.float_to_bf16(np.ascontiguousarray(x32, dtype=np.float32))


def _to_gpu_bf16(bits: np.ndarray) -> torch.Tensor:
    return cuda(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))


def _bits_of(y: torch.Tensor) -> np.ndarray:
    return host(y.view(torch.int16)).view(np.uint16)


def _acts(M, K, seed, n_out=4):
    x = synth.activations(M, K, n_out if K >= 64 else 0, synth.generator(seed)).float().numpy()
    return _bf16_bits(x * 1.7)


@pytest.mark.parametrize("M,K", [(1, 16), (3, 40), (128, 512), (257, 2560), (64, 12288)])
def test_quantize_act_bf16_bitexact(M, K):
    xb = _acts(M, K, M + K)
    q, s = cider.quantize_act_any(_to_gpu_bf16(xb))
    qo, so = oracle.quantize_act_bf16(xb)
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32))
    assert np.array_equal(host(q), qo)


def test_quantize_bf16_exhaustive_rows_up_to_16k():
    """For a sweep of absmax values a (both ends of the range included), rows
    of 16384 elements that hold a and a window of every bf16 value |x| <= a,
    both signs: codes and scales bit for bit."""
    pos = np.arange(1, 0x7F80, dtype=np.int32)  # positive finite bf16 bit patterns
    chosen = np.unique(np.concatenate([pos[::487], pos[-6:], pos[:6],
                                       np.array([0x3F80, 0x42FE, 0x4300, 0x7F7F])]))
    width, win = 16384, 8191
    rows = []
    for a in chosen:
        for lo in range(0, a + 1, win):
            xs = np.arange(lo, min(lo + win, a + 1), dtype=np.uint16)
            r = np.zeros(width, np.uint16)
            r[0] = a
            r[1:1 + len(xs)] = xs
            r[1 + win:1 + win + len(xs)] = xs | 0x8000
            rows.append(r)
    xb = np.stack(rows)
    q, s = cider.quantize_act_any(_to_gpu_bf16(xb))
    qo, so = oracle.quantize_act_bf16(xb)
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32))
    assert np.array_equal(host(q), qo)


def test_quantize_act_bf16_every_pair():
    """Every finite bf16 x against every positive finite bf16 absmax a with
    |x| <= a, both signs of x (about 10^9 pairs, one row per a): codes and
    scales bit for bit."""
    for rows in every_pair_rows(0x7F7F):
        q, s = cider.quantize_act_any(_to_gpu_bf16(rows))
        qo, so = oracle.quantize_act_bf16(rows)
        assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32)), rows.shape
        assert np.array_equal(host(q), qo), rows.shape
        del q, s


def _weights(N, K, seed):
    return synth.weights(N, K, synth.generator(seed)).numpy()


@pytest.mark.parametrize("out", ["bf16", "f16"])
@pytest.mark.parametrize("gs", [0, 64])
@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (5, 260, 1152), (130, 264, 2560),
                                   (300, 520, 1024)])
def test_w8a8_layer_bf16(M, N, K, gs, out):
    xb = _acts(M, K, 5 * M + N)
    wq, s = oracle.quantize_weight_int8(_weights(N, K, N + K), gs)
    y = cider.linear(_to_gpu_bf16(xb), cuda(torch.from_numpy(wq)), cuda(torch.from_numpy(s)),
                     8, gs, out_dtype=torch.bfloat16 if out == "bf16" else torch.float16)
    ref = oracle.w8a8_linear(xb, wq, s, gs, x_dtype="bf16", y_dtype=out)
    assert np.array_equal(_bits_of(y), ref.view(np.uint16))


@pytest.mark.parametrize("gs", [0, 128])
@pytest.mark.parametrize("M,N,K", [(1, 300, 1024), (3, 264, 2560), (200, 264, 1024)])
def test_w4a8_layer_bf16(M, N, K, gs):
    xb = _acts(M, K, 3 * M + K)
    wp, s = oracle.pack_weight_int4(_weights(N, K, N * 3 + K), gs)
    y = cider.linear(_to_gpu_bf16(xb), cuda(torch.from_numpy(wp)), cuda(torch.from_numpy(s)),
                     4, gs)
    ref = oracle.w4a8_linear(xb, wp, s, gs, x_dtype="bf16")
    assert np.array_equal(_bits_of(y), ref.view(np.uint16))


def test_fp16_input_bf16_output():
    M, N, K = 130, 264, 512
    x = synth.activations(M, K, 4, synth.generator(11)).numpy()
    wq, s = oracle.quantize_weight_int8(_weights(N, K, 12), 0)
    y = cider.linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                     cuda(torch.from_numpy(s)), 8, 0, out_dtype=torch.bfloat16)
    ref = oracle.w8a8_linear(x, wq, s, 0, x_dtype="f16", y_dtype="bf16")
    assert np.array_equal(_bits_of(y), ref.view(np.uint16))


def test_bf16_gemv_equals_gemm_row():
    """Routing on M never changes a result: the M = 1 GEMV equals the first
    row of the GEMM on the same bf16 token."""
    M, N, K = 140, 520, 2560
    xb = _acts(M, K, 77)
    wq, s = oracle.quantize_weight_int8(_weights(N, K, 78), 64)
    wd, sd = cuda(torch.from_numpy(wq)), cuda(torch.from_numpy(s))
    y = cider.linear(_to_gpu_bf16(xb), wd, sd, 8, 64)
    y1 = cider.linear(_to_gpu_bf16(xb[:1]), wd, sd, 8, 64)
    assert torch.equal(y1.view(torch.int16), y[:1].view(torch.int16))
