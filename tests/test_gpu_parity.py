"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bars: INT8 codes, scales and INT32 accumulators bit-exact; fp16 outputs
within 1 ulp of the oracle (the tests also count the outputs that are not
bit-identical; the kernels follow the oracle's operation order, so the
expected count is 0).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a8_quantized_gemm_int8_b300 as cider
from gpu_helpers import assert_f16_within_1ulp, cuda, every_pair_rows, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cider.load_library()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    st, site = cider.device_status()
    assert st == cider.CIDER_OK, f"device status {st} at site {site:#x}"


# ---------------------------------------------------------------------------
# failure detection: a bounded device wait gives up and reports
# ---------------------------------------------------------------------------

def test_bounded_wait_reports_timeout():
    cider.device_status()  # clear
    cider.wait_timeout_probe(20_000_000)  # 20 ms
    st, site = cider.device_status()
    assert st == cider.CIDER_ERR_TIMEOUT and site == 0x901
    st, _ = cider.device_status()
    assert st == cider.CIDER_OK
    # the context is still usable
    x = torch.ones(4, 16, dtype=torch.float16, device="cuda")
    q, s = cider.quantize_act(x)
    assert int(q[0, 0]) == 127


# ---------------------------------------------------------------------------
# activation quantization
# ---------------------------------------------------------------------------

def _special_rows(K):
    rows = [np.zeros(K), np.zeros(K)]
    rows[1][K // 2] = -3.0
    r = (np.arange(K) % 9 - 4) * 0.5
    r[0] = 4.0 * 127 / 127  # absmax 4 -> scale 4/127
    rows.append(r)
    t = np.full(K, 0.5)
    t[1] = 127.0  # scale 1: 0.5 ties to 0
    rows.append(t)
    return np.array(rows, dtype=np.float16)


@pytest.mark.parametrize("M,K", [(1, 16), (3, 40), (5, 13), (128, 512), (257, 2560),
                                 (64, 12288), (2, 1 << 16)])
def test_quantize_act_bitexact(M, K):
    x = synth.activations(M, K, 4 if K >= 64 else 0, synth.generator(M * 7 + K)).numpy()
    x = np.concatenate([x, _special_rows(K)])
    q, s = cider.quantize_act(cuda(torch.from_numpy(x)))
    qo, so = oracle.quantize_act(x)
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32))
    assert np.array_equal(host(q), qo)


def test_quantize_exhaustive_over_x_for_many_scales():
    """For each chosen absmax a, one row holds a and every fp16 x with
    |x| <= a (zero padded): all codes must match the oracle bit for bit."""
    pos = np.arange(1, 0x7C00, dtype=np.int32)      # positive finite fp16 bit patterns
    chosen = np.unique(np.concatenate([pos[::97], pos[-40:], pos[:40],
                                       np.array([0x3C00, 0x57F0, 0x5BF0, 0x7BFF])]))
    width = 2 * 0x7C00
    width += (-width) % 16
    rows = np.zeros((len(chosen), width), np.uint16)
    for i, a in enumerate(chosen):
        xs = np.arange(0, a + 1, dtype=np.uint16)
        rows[i, :a + 1] = xs
        rows[i, a + 1:2 * a + 2] = xs | 0x8000
    x = rows.view(np.float16)
    q, s = cider.quantize_act(cuda(torch.from_numpy(x)))
    qo, so = oracle.quantize_act(x)
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32))
    assert np.array_equal(host(q), qo)


def test_quantize_exhaustive_rows_up_to_16k():
    """The same exhaustive coverage on rows of 16384 elements (the width the
    one-pass register kernels take): for each chosen absmax a, a set of rows
    that each hold a and a window of the fp16 values |x| <= a, both signs."""
    pos = np.arange(1, 0x7C00, dtype=np.int32)
    chosen = np.unique(np.concatenate([pos[::211], pos[-12:], pos[:12],
                                       np.array([0x3C00, 0x57F0, 0x5BF0, 0x7BFF])]))
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
    x = np.stack(rows).view(np.float16)
    q, s = cider.quantize_act(cuda(torch.from_numpy(x)))
    qo, so = oracle.quantize_act(x)
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32))
    assert np.array_equal(host(q), qo)
    img, s2 = cider.act_image(cuda(torch.from_numpy(x)))
    assert np.array_equal(host(s2).view(np.uint32), so.view(np.uint32))
    assert np.array_equal(host(img).astype(np.int32), qo.astype(np.int32))


def test_quantize_act_every_fp16_pair():
    """Every finite fp16 x against every positive finite fp16 absmax a with
    |x| <= a, both signs of x (about 10^9 pairs, one row per a, rows 11584
    to 63488 elements wide): codes, scales and the fp16 operand image bit for
    bit."""
    for rows in every_pair_rows(0x7BFF):
        x = rows.view(np.float16)
        xd = cuda(torch.from_numpy(x))
        q, s = cider.quantize_act(xd)
        qo, so = oracle.quantize_act(x)
        assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32)), rows.shape
        assert np.array_equal(host(q), qo), rows.shape
        img, s2 = cider.act_image(xd)
        assert np.array_equal(host(s2).view(np.uint32), so.view(np.uint32)), rows.shape
        assert np.array_equal(host(img).astype(np.int32), qo.astype(np.int32)), rows.shape
        del xd, q, s, img, s2


# ---------------------------------------------------------------------------
# weight preparation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gs", [0, 64, 128])
def test_quantize_weight_int8_bitexact(gs):
    w = synth.weights(300, 512, synth.generator(gs + 1)).numpy()
    w[3] = 0
    wq, s = cider.quantize_weight_int8(cuda(torch.from_numpy(w)), gs)
    wqo, so = oracle.quantize_weight_int8(w, gs)
    assert np.array_equal(host(wq), wqo)
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("gs", [0, 64, 128])
def test_pack_weight_int4_bitexact(gs):
    w = synth.weights(130, 768, synth.generator(gs + 2)).numpy()
    w[5, :128] = 0
    wp, s = cider.pack_weight_int4(cuda(torch.from_numpy(w)), gs)
    wpo, so = oracle.pack_weight_int4(w, gs)
    assert np.array_equal(host(wp), wpo)
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32))


# ---------------------------------------------------------------------------
# INT32 accumulators of the tensor-core engine (raw, bit-exact)
# ---------------------------------------------------------------------------

def _codes(shape, seed, lo=-127, hi=127):
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, shape, dtype=np.int8)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (1, 16, 64), (7, 300, 192), (130, 257, 1088),
                                   (300, 520, 2560), (129, 256, 12288),
                                   # K not a multiple of the 64-deep k-block (zero-filled tail)
                                   (5, 33, 96), (64, 130, 224), (150, 40, 224)])
def test_gemm_s32_bitexact(M, N, K):
    q = _codes((M, K), M + N)
    w = _codes((N, K), K)
    acc = cider.raw_gemm_s32(cuda(torch.from_numpy(q)), cuda(torch.from_numpy(w)), K)
    assert np.array_equal(host(acc), oracle.gemm_s32(q, w, 0))


def test_gemm_s32_worst_case_magnitudes():
    """All codes +-127: each 1024-deep segment reaches 127^2 * 1024 (just
    under 2^24) and the total reaches 127^2 * K; signs alternate by row so
    large partial sums cancel and rebuild."""
    M, N, K = 256, 256, 12288
    q = np.full((M, K), 127, np.int8)
    q[1::2] = -127
    q[2::4, ::3] = -127
    w = np.full((N, K), 127, np.int8)
    w[::3, ::2] = -127
    w[5] = 127
    acc = cider.raw_gemm_s32(cuda(torch.from_numpy(q)), cuda(torch.from_numpy(w)), K)
    assert np.array_equal(host(acc), oracle.gemm_s32(q, w, 0))


def test_gemm_s32_worst_case_small_m():
    """The worst-case magnitudes on the few-token engine, whose weights are
    widened on chip from raw INT8 codes."""
    M, N, K = 96, 200, 12288
    q = np.full((M, K), -127, np.int8)
    q[::2] = 127
    q[1::4, ::5] = 127
    w = np.full((N, K), 127, np.int8)
    w[::2, ::3] = -127
    acc = cider.raw_gemm_s32(cuda(torch.from_numpy(q)), cuda(torch.from_numpy(w)), K)
    assert np.array_equal(host(acc), oracle.gemm_s32(q, w, 0))


@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("M,K", [(140, 1024), (40, 1152), (3, 1152)])
def test_gemm_s32_group_partials(gs, M, K):
    """Per-group partials; K = 1152 gives a group count that is not a
    multiple of the four groups the few-token engine folds per round."""
    N = 270
    q = _codes((M, K), 11)
    w = _codes((N, K), 12)
    part = cider.raw_gemm_s32(cuda(torch.from_numpy(q)), cuda(torch.from_numpy(w)), K,
                               group_size=gs)
    assert np.array_equal(host(part), oracle.gemm_s32(q, w, gs))


@pytest.mark.parametrize("gs,M,K", [(64, 40, 192), (64, 3, 320), (192, 40, 576),
                                    (192, 7, 1344), (192, 140, 576)])
def test_gemm_s32_group_partials_odd_blocks(gs, M, K):
    """Per-group partials where K is an odd number of 64-k blocks (the
    few-token engine stages two blocks at a time: the last stage holds one
    block past K) and where a 192-k group ends inside a stage."""
    N = 200
    q = _codes((M, K), 13)
    w = _codes((N, K), 14)
    part = cider.raw_gemm_s32(cuda(torch.from_numpy(q)), cuda(torch.from_numpy(w)), K,
                               group_size=gs)
    assert np.array_equal(host(part), oracle.gemm_s32(q, w, gs))


@pytest.mark.parametrize("M,N,K", [(130, 300, 512), (40, 300, 96), (1, 77, 224)])
def test_gemm_s32_int4_weights(M, N, K):
    q = _codes((M, K), 21)
    wp = np.random.default_rng(22).integers(0, 256, (N, K // 2), dtype=np.uint8)
    acc = cider.raw_gemm_s32(cuda(torch.from_numpy(q)), cuda(torch.from_numpy(wp)), K, bits=4)
    assert np.array_equal(host(acc), oracle.gemm_s32(q, oracle.unpack_int4(wp, K), 0))


# ---------------------------------------------------------------------------
# whole linear layers
# ---------------------------------------------------------------------------

def _layer_inputs(M, N, K, seed):
    li = synth.linear_inputs(M, N, K, n_out=4, seed=seed)
    return li.x.numpy(), li.w.numpy()


LAYER_SHAPES = [(128, 256, 512), (2, 16, 64), (3, 300, 192), (130, 257, 1088), (200, 8, 2560),
                (129, 384, 4096), (4, 40, 80), (150, 72, 208)]


@pytest.mark.parametrize("M,N,K", LAYER_SHAPES)
def test_w8a8_pc_layer(M, N, K):
    x, w = _layer_inputs(M, N, K, seed=M + N + K)
    wq, s = oracle.quantize_weight_int8(w, 0)
    y = cider.w8a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                          cuda(torch.from_numpy(s)), 0)
    ref = oracle.w8a8_linear(x, wq, s, 0)
    assert_f16_within_1ulp(host(y), ref, "pc")


# Per-channel layers of at most 128 tokens share the k-blocks of all tiles
# evenly among the SMs (stream-K): these shapes give CTAs whose runs cross a
# tile boundary, tiles summed from two or three CTAs' int32 partials, and
# runs from 1 to about 20 k-blocks, so segments of 15 and 16 k-blocks too.
SK_SHAPES = [(32, 5120, 4096), (77, 2560, 8192), (128, 1280, 2560), (9, 10240, 1024)]


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("M,N,K", SK_SHAPES)
def test_pc_layer_stream_k(M, N, K, bits):
    x, w = _layer_inputs(M, N, K, seed=M + K + bits)
    if bits == 8:
        wq, s = oracle.quantize_weight_int8(w, 0)
        y = cider.w8a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                              cuda(torch.from_numpy(s)), 0)
        ref = oracle.w8a8_linear(x, wq, s, 0)
    else:
        wq, s = oracle.pack_weight_int4(w, 0)
        y = cider.w4a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                              cuda(torch.from_numpy(s)), 0)
        ref = oracle.w4a8_linear(x, wq, s, 0)
    assert_f16_within_1ulp(host(y), ref, f"stream-K w{bits}")


# Per-group layers of at most 128 tokens whose SM-pair tiles fill as many
# SMs as single-SM tiles would (wide layers) run on SM pairs with 128-token
# tiles, the weights widened into tensor memory.
@pytest.mark.parametrize("bits,gs", [(8, 64), (8, 128), (4, 128), (4, 64)])
@pytest.mark.parametrize("M", [128, 37])
def test_pg_few_token_layer_on_pairs(M, bits, gs):
    N, K = 10240, 1024
    x, w = _layer_inputs(M, N, K, seed=M + gs + bits)
    if bits == 8:
        wq, s = oracle.quantize_weight_int8(w, gs)
        y = cider.w8a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                              cuda(torch.from_numpy(s)), gs)
        ref = oracle.w8a8_linear(x, wq, s, gs)
    else:
        wq, s = oracle.pack_weight_int4(w, gs)
        y = cider.w4a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                              cuda(torch.from_numpy(s)), gs)
        ref = oracle.w4a8_linear(x, wq, s, gs)
    assert_f16_within_1ulp(host(y), ref, f"few-token pg{gs} w{bits} on pairs")


@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (3, 300, 1024), (130, 264, 2560),
                                   (5, 260, 1152)])
def test_w8a8_pg_layer(M, N, K, gs):
    x, w = _layer_inputs(M, N, K, seed=gs + M)
    wq, s = oracle.quantize_weight_int8(w, gs)
    y = cider.w8a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                          cuda(torch.from_numpy(s)), gs)
    ref = oracle.w8a8_linear(x, wq, s, gs)
    assert_f16_within_1ulp(host(y), ref, f"pg{gs}")


@pytest.mark.parametrize("bits,gs,M,N,K", [(8, 64, 40, 300, 192), (8, 64, 100, 300, 320),
                                            (8, 192, 7, 300, 576), (8, 192, 77, 520, 1344),
                                            (8, 192, 130, 264, 576), (4, 64, 40, 300, 192),
                                            (4, 192, 77, 520, 1344)])
def test_pg_layer_odd_k_blocks(bits, gs, M, N, K):
    """Per-group layers whose K is an odd number of 64-k blocks, and 192-k
    groups that end inside one of the few-token engine's two-block stages."""
    x, w = _layer_inputs(M, N, K, seed=gs + M + bits)
    if bits == 8:
        wq, s = oracle.quantize_weight_int8(w, gs)
        y = cider.w8a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                              cuda(torch.from_numpy(s)), gs)
        ref = oracle.w8a8_linear(x, wq, s, gs)
    else:
        wq, s = oracle.pack_weight_int4(w, gs)
        y = cider.w4a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                              cuda(torch.from_numpy(s)), gs)
        ref = oracle.w4a8_linear(x, wq, s, gs)
    assert_f16_within_1ulp(host(y), ref, f"pg{gs} w{bits} K{K}")


@pytest.mark.parametrize("gs", [0, 128, 64])
@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (2, 300, 1024), (131, 264, 2560)])
def test_w4a8_layer(M, N, K, gs):
    x, w = _layer_inputs(M, N, K, seed=gs + 3 * M)
    wp, s = oracle.pack_weight_int4(w, gs)
    y = cider.w4a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wp)),
                          cuda(torch.from_numpy(s)), gs)
    ref = oracle.w4a8_linear(x, wp, s, gs)
    assert_f16_within_1ulp(host(y), ref, f"w4 gs{gs}")


@pytest.mark.parametrize("cls,gs", [("W8A8Linear", 0), ("W8A8Linear", 64), ("W4A8Linear", 0),
                                    ("W4A8Linear", 128)])
def test_layer_classes_match_oracle(cls, gs):
    """The layer-level names: from_weights prepares the weights on the GPU and
    a call flattens leading dimensions into tokens (2 x 65 here, the pair
    engine) or runs the GEMV for one token; outputs match the oracle's on the
    same weights."""
    M, N, K = 130, 300, 1024
    x, w = _layer_inputs(M, N, K, seed=7 + gs)
    layer = getattr(cider, cls).from_weights(cuda(torch.from_numpy(w)), gs)
    if cls == "W8A8Linear":
        wq, s = oracle.quantize_weight_int8(w, gs)
        ref = oracle.w8a8_linear(x, wq, s, gs)
    else:
        wq, s = oracle.pack_weight_int4(w, gs)
        ref = oracle.w4a8_linear(x, wq, s, gs)
    y = layer(cuda(torch.from_numpy(x)).reshape(2, 65, K))
    assert tuple(y.shape) == (2, 65, N)
    assert_f16_within_1ulp(host(y).reshape(M, N), ref, cls)
    y1 = layer(cuda(torch.from_numpy(x[:1])))
    assert_f16_within_1ulp(host(y1), ref[:1], cls + " one token")


def test_empty_inputs_give_empty_outputs():
    """No tokens (M = 0) or no output channels (N = 0): every call returns an
    empty result of the right shape and type and launches nothing."""
    M, N, K = 4, 64, 256
    x, w = _layer_inputs(M, N, K, seed=3)
    xd = cuda(torch.from_numpy(x))
    wq, s = oracle.quantize_weight_int8(w, 0)
    wqd, sd = cuda(torch.from_numpy(wq)), cuda(torch.from_numpy(s))
    wg, sg = oracle.quantize_weight_int8(w, 64)
    wp, s4 = oracle.pack_weight_int4(w, 0)
    cases = {
        "pc": (cider.w8a8_linear(xd[:0], wqd, sd), (0, N), torch.float16),
        "pg": (cider.w8a8_linear(xd[:0], cuda(torch.from_numpy(wg)), cuda(torch.from_numpy(sg)),
                                 64), (0, N), torch.float16),
        "w4": (cider.w4a8_linear(xd[:0], cuda(torch.from_numpy(wp)), cuda(torch.from_numpy(s4))),
               (0, N), torch.float16),
        "bf16": (cider.linear(xd[:0].bfloat16(), wqd, sd), (0, N), torch.bfloat16),
        "no channels": (cider.w8a8_linear(xd, wqd[:0], sd[:0]), (M, 0), torch.float16),
        "gemv": (cider.int8_gemv(xd[0], wqd[:0], sd[:0]), (0,), torch.float16),
        "a16": (cider.a16_gemv(xd[0], wqd[:0], sd[:0]), (0,), torch.float16),
        "quant": (cider.quantize_act(xd[:0])[0], (0, K), torch.int8),
        "quant bf16": (cider.quantize_act_any(xd[:0].bfloat16())[1], (0,), torch.float32),
        "weights": (cider.quantize_weight_int8(cuda(torch.from_numpy(w[:0])), 64)[1], (0, K // 64),
                    torch.float32),
        "int4": (cider.pack_weight_int4(cuda(torch.from_numpy(w[:0])))[0], (0, K // 2),
                 torch.uint8),
    }
    for name, (y, shape, dtype) in cases.items():
        assert tuple(y.shape) == shape and y.dtype == dtype, name


def test_layer_edge_rows():
    """All-zero tokens, a single non-zero, exact-scale rows, overflow to inf."""
    M, N, K = 6, 64, 128
    x = np.zeros((M, K), np.float16)
    x[1, 5] = -2.0
    x[2] = 127.0
    x[3, ::2] = 127.0
    x[3, 1::2] = -127.0
    x[4] = np.linspace(-60, 60, K).astype(np.float16)
    x[5] = 65504.0
    w = synth.weights(N, K, synth.generator(5)).numpy()
    w[0] = 127.0
    w[1] = 0.0
    for gs in (0, 64):
        wq, s = oracle.quantize_weight_int8(w, gs)
        y = cider.w8a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                              cuda(torch.from_numpy(s)), gs)
        ref = oracle.w8a8_linear(x, wq, s, gs)
        assert np.array_equal(host(y).view(np.uint16), ref.view(np.uint16))


def test_group_size_limit_of_tensor_core_paths():
    """A group partial over more than 1024 products could leave the range
    where the tensor core's fp32 accumulator is exact (127^2 * 1024 < 2^24):
    the tensor-core paths take groups of up to 1024 and refuse larger ones
    instead of rounding."""
    M, N, K = 4, 32, 4096
    x, w = _layer_inputs(M, N, K, seed=77)
    wq, s = oracle.quantize_weight_int8(w, 1024)
    y = cider.w8a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                          cuda(torch.from_numpy(s)), 1024)
    assert_f16_within_1ulp(host(y), oracle.w8a8_linear(x, wq, s, 1024), "gs1024")
    wq, s = oracle.quantize_weight_int8(w, 2048)
    with pytest.raises(cider.CiderError) as e:
        cider.w8a8_linear(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                          cuda(torch.from_numpy(s)), 2048)
    assert e.value.status == cider.CIDER_ERR_UNSUPPORTED


@pytest.mark.parametrize("gs", [0, 64])
def test_column_shards_reproduce_the_full_layer(gs):
    """The output-channel split, each shard run on the GPU from its own weight
    rows (as each rank of a column-parallel run does), concatenates to the
    unsplit layer bit for bit."""
    M, N, K, world = 130, 700, 1024, 3
    x, w = _layer_inputs(M, N, K, seed=91)
    wq, s = oracle.quantize_weight_int8(w, gs)
    xd, wd, sd = cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)), cuda(torch.from_numpy(s))
    full = cider.w8a8_linear(xd, wd, sd, gs)
    parts = []
    for r in range(world):
        n0, n1 = cider.column_shard(N, world, r)
        parts.append(cider.w8a8_linear(xd, wd[n0:n1], sd[n0:n1], gs))
    y = torch.cat(parts, dim=1)
    assert torch.equal(y.view(torch.int16), full.view(torch.int16))


@pytest.mark.parametrize("gs", [0, 64])
@pytest.mark.parametrize("M", [1, 40, 300])
def test_concatenated_linears_equal_separate_calls(M, gs):
    """q|k|v-style fusion: one call on the weights stacked along N gives, in
    each linear's columns, exactly that linear's own output."""
    K = 1024
    x, _ = _layer_inputs(M, 8, K, seed=M + 500)
    xd = cuda(torch.from_numpy(x))
    lins = []
    for i, N in enumerate((384, 128, 136)):
        w = synth.weights(N, K, synth.generator(600 + i)).numpy()
        wq, s = oracle.quantize_weight_int8(w, gs)
        lins.append((cuda(torch.from_numpy(wq)), cuda(torch.from_numpy(s))))
    wcat, scat, sizes = cider.concat_linears(lins)
    parts = cider.split_columns(cider.w8a8_linear(xd, wcat, scat, gs), sizes)
    for (wq, s), y in zip(lins, parts):
        ref = cider.w8a8_linear(xd, wq, s, gs)
        assert torch.equal(y.contiguous().view(torch.int16), ref.view(torch.int16))


# ---------------------------------------------------------------------------
# M = 1 GEMV
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits,gs", [(8, 0), (8, 64), (8, 128), (4, 0), (4, 128), (4, 64)])
@pytest.mark.parametrize("N,K", [(10240, 2560), (2560, 10240), (37, 512), (1, 12288)])
def test_gemv_matches_oracle(bits, gs, N, K):
    x, w = _layer_inputs(1, N, K, seed=N + bits + gs)
    if bits == 8:
        wq, s = oracle.quantize_weight_int8(w, gs)
        ref = oracle.w8a8_linear(x, wq, s, gs)
    else:
        wq, s = oracle.pack_weight_int4(w, gs)
        ref = oracle.w4a8_linear(x, wq, s, gs)
    y = cider.int8_gemv(cuda(torch.from_numpy(x)), cuda(torch.from_numpy(wq)),
                        cuda(torch.from_numpy(s)), bits=bits, group_size=gs)
    assert np.array_equal(host(y).view(np.uint16), ref[0].view(np.uint16))


@pytest.mark.parametrize("gs", [0, 64])
def test_gemv_equals_gemm_row(gs):
    """Routing on M never changes a result: GEMV(x[m]) is bit-identical to
    row m of the tensor-core GEMM over the whole batch."""
    M, N, K = 130, 1000, 2560
    x, w = _layer_inputs(M, N, K, seed=77 + gs)
    wq, s = oracle.quantize_weight_int8(w, gs)
    xd, wd, sd = (cuda(torch.from_numpy(a)) for a in (x, wq, s))
    y = host(cider.w8a8_linear(xd, wd, sd, gs))
    for m in (0, 1, 64, 129):
        ym = host(cider.int8_gemv(xd[m], wd, sd, bits=8, group_size=gs))
        assert np.array_equal(ym.view(np.uint16), y[m].view(np.uint16))
    # the public GEMM entry point at M == 1 takes the GEMV
    y1 = host(cider.w8a8_linear(xd[5:6].contiguous(), wd, sd, gs))
    assert np.array_equal(y1.view(np.uint16), y[5:6].view(np.uint16))


@pytest.mark.parametrize("prep,bits,gs", [("int8", 8, 0), ("int8", 8, 64), ("int4", 4, 128),
                                          ("clipped", 8, 0), ("clipped", 4, 128)])
def test_gpu_weight_prep_then_decode_without_sync(prep, bits, gs):
    """A weight-preparation call followed at once, on the same stream and with
    no synchronization, by an M = 1 call that reads those weights: the
    decode kernel may start early (programmatic dependent launch) but must
    read the weights and scales only after the preparation has finished. The
    weight buffers first hold other codes, so an early read would show."""
    lib = cider.load_library()
    N, K = 10240, 2560
    x, w = _layer_inputs(1, N, K, seed=900 + bits + gs)
    if prep == "clipped":
        wq_ref, s_ref = oracle.quantize_weight_clipped(w, gs, 99.9, bits)
    elif bits == 8:
        wq_ref, s_ref = oracle.quantize_weight_int8(w, gs)
    else:
        wq_ref, s_ref = oracle.pack_weight_int4(w, gs)
    ref = (oracle.w8a8_linear(x, wq_ref, s_ref, gs) if bits == 8
           else oracle.w4a8_linear(x, wq_ref, s_ref, gs))
    xd, wd = cuda(torch.from_numpy(x)), cuda(torch.from_numpy(w))
    G = 1 if gs == 0 else K // gs
    wq = torch.full((N, K if bits == 8 else K // 2), 0x11, dtype=torch.int8 if bits == 8
                    else torch.uint8, device="cuda")
    s = torch.full((N,) if gs == 0 else (N, G), 1e-3, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for route in ("gemv", "layer"):
        wq.fill_(0x11)
        s.fill_(1e-3)
        if prep == "clipped":
            st = lib.cider_quantize_weight_clipped(wd.data_ptr(), 0, N, K, gs, bits, 99.9,
                                                   wq.data_ptr(), s.data_ptr(), stream)
        elif bits == 8:
            st = lib.cider_quantize_weight_int8(wd.data_ptr(), N, K, gs, wq.data_ptr(),
                                                s.data_ptr(), stream)
        else:
            st = lib.cider_pack_weight_int4(wd.data_ptr(), N, K, gs, wq.data_ptr(),
                                            s.data_ptr(), stream)
        assert st == cider.CIDER_OK
        if route == "gemv":
            y = cider.int8_gemv(xd, wq, s, bits=bits, group_size=gs)
        else:
            y = cider.linear(xd, wq, s, bits=bits, group_size=gs)
        got = host(y).reshape(-1)
        assert np.array_equal(got.view(np.uint16), ref.reshape(-1).view(np.uint16)), route
        assert np.array_equal(host(wq), wq_ref) and np.array_equal(host(s), s_ref)
