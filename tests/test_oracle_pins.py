"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test pins one part of the oracle to a hand-worked example (the golden
fixtures), to a closed form or invariant of the definition, to a special case
that reduces to an independent library routine (numpy's binary16 conversion,
numpy's rint, numpy's int64 matmul), or to brute force on tiny inputs.
The definition pinned is the Cider README's "Quantization" table (symmetric
per-token INT8 activations, symmetric INT8 / INT4 weights, INT32
accumulation, C_fp16 = C_int32 * s_act * s_weight).
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(json.loads(line))
    return rows


# --------------------------------------------------------------------------
# binary16 conversions (pinned to numpy's independent implementation)
# --------------------------------------------------------------------------

def test_half_to_float_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_float(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_matches_numpy():
    rng = np.random.default_rng(0)
    finite = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    finite = finite[np.isfinite(finite)].astype(np.float32)
    # midpoints between consecutive binary16 values exercise ties-to-even
    pos = np.sort(finite[finite >= 0])
    mids = ((pos[1:].astype(np.float64) + pos[:-1]) / 2).astype(np.float32)
    cases = [
        finite, mids, -mids,
        np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0)),
        (rng.standard_normal(200000) * 10.0 ** rng.uniform(-9, 5, 200000)).astype(np.float32),
        np.array([65504, 65519.996, 65520, 65536, 1e9, 2 ** -25, 3 * 2 ** -26,
                  2 ** -24, 2 ** -14, 2 ** -14 - 2 ** -25, 0.0, -0.0], np.float32),
    ]
    for c in cases:
        ours = oracle.float_to_half(c)
        ref = c.astype(np.float16).view(np.uint16)
        assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------
# quantization
# --------------------------------------------------------------------------

def test_quant_hand_examples():
    for ex in _golden("quant_hand_examples.txt"):
        v = np.array([ex["values"]], np.float16)
        if ex["kind"] == "int8":
            q, s = oracle.quantize_act(v)
            assert q[0].tolist() == ex["codes"]
            assert float(s[0]) == ex["scale"]
            wq, sw = oracle.quantize_weight_int8(v, 0)
            assert wq[0].tolist() == ex["codes"] and float(sw[0]) == ex["scale"]
        else:
            wp, sw = oracle.pack_weight_int4(v, 0)
            assert wp[0].tolist() == ex["bytes"]
            assert float(sw[0]) == ex["scale"]
            assert oracle.unpack_int4(wp, v.shape[1])[0].tolist() == ex["codes"]
            nib = [(b >> (4 * (i % 2))) & 0xF for i, b in
                   enumerate(np.repeat(wp[0], 2).tolist())]
            assert nib == ex["nibbles"]


def test_quant_unit_scale_is_rint():
    """absmax 127 gives scale exactly 1, where the code must be the textbook
    round-half-even of x (numpy.rint)."""
    rng = np.random.default_rng(1)
    x = (rng.uniform(-127, 127, (64, 300)) * 4).round() / 4  # quarter steps: many ties
    x[:, 7] = 127.0
    x[::2, 7] = -127.0
    x = x.astype(np.float16)
    q, s = oracle.quantize_act(x)
    assert np.all(s == 1.0)
    assert np.array_equal(q, np.rint(x.astype(np.float64)).astype(np.int8))


def test_quant_power_of_two_scales():
    """absmax 127 * 2^j gives scale 2^j exactly, so code = rint(x / 2^j) with
    an exact division; also pins the group indexing of weight quantization."""
    rng = np.random.default_rng(2)
    N, K, gs = 6, 256, 64
    G = K // gs
    j = rng.integers(-6, 4, (N, G))
    base = (rng.uniform(-127, 127, (N, K)) * 2).round() / 2
    w = np.empty((N, K))
    for n in range(N):
        for g in range(G):
            blk = base[n, g * gs:(g + 1) * gs].copy()
            blk[(n + g) % gs] = 127.0 if (n + g) % 2 else -127.0
            w[n, g * gs:(g + 1) * gs] = blk * 2.0 ** j[n, g]
    w16 = w.astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w)  # all exact in fp16
    wq, s = oracle.quantize_weight_int8(w16, gs)
    assert np.array_equal(s, (2.0 ** j).astype(np.float32))
    expect = np.rint(w / np.repeat(2.0 ** j, gs, axis=1)).astype(np.int8)
    assert np.array_equal(wq, expect)
    # per-channel on the same rows: one scale per row = max of its groups
    wq_pc, s_pc = oracle.quantize_weight_int8(w16, 0)
    assert np.array_equal(s_pc, (2.0 ** j.max(axis=1)).astype(np.float32))


def test_quant_invariants_random():
    """Odd symmetry, the absmax element maps to +-127, the range is
    [-127, 127], and |x - q*s| <= s * (1/2 + 127 * 2^-24) (rounding of the
    quotient plus the final round to an integer)."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((50, 777)) * 10.0 ** rng.uniform(-4, 4, (50, 1))).astype(np.float16)
    x[3] = 0
    q, s = oracle.quantize_act(x)
    qn, sn = oracle.quantize_act(-x)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    assert q.min() >= -127 and q.max() <= 127
    assert s[3] == 0 and not q[3].any()
    xf = x.astype(np.float64)
    amax = np.abs(xf).max(axis=1)
    nz = amax > 0
    arg = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(50), arg])[nz] == 127)
    assert np.array_equal(s[nz], (amax[nz].astype(np.float32) / np.float32(127)))
    err = np.abs(xf - q * s[:, None].astype(np.float64))
    bound = s[:, None].astype(np.float64) * (0.5 + 127 * 2.0 ** -24)
    assert np.all(err <= bound)


def test_int4_invariants():
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((9, 256)) * 0.02).astype(np.float16)
    for gs in (0, 128, 64):
        wp, s = oracle.pack_weight_int4(w, gs)
        codes = oracle.unpack_int4(wp, 256)
        assert codes.min() >= -7 and codes.max() <= 7
        lo, hi = wp & 0xF, wp >> 4
        assert lo.min() >= 1 and hi.min() >= 1 and lo.max() <= 15 and hi.max() <= 15
        s2 = s.reshape(9, -1)
        gsz = 256 if gs == 0 else gs
        err = np.abs(w.astype(np.float64) - codes * np.repeat(s2, gsz, axis=1))
        assert np.all(err <= np.repeat(s2, gsz, axis=1) * (0.5 + 7 * 2.0 ** -24))
    # nibble 0 (never written by the quantizer) decodes to -8
    assert oracle.unpack_int4(np.array([[0x80]], np.uint8), 2)[0].tolist() == [-8, 0]


# --------------------------------------------------------------------------
# INT32 products (brute force / numpy int64)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (3, 5, 64), (17, 33, 256), (33, 9, 128)])
def test_gemm_s32_brute_force(M, N, K):
    rng = np.random.default_rng(M * 1000 + N)
    q = rng.integers(-127, 128, (M, K), dtype=np.int8)
    w = rng.integers(-127, 128, (N, K), dtype=np.int8)
    acc = oracle.gemm_s32(q, w, 0)
    brute = np.zeros((M, N), np.int64)
    for m in range(M):
        for n in range(N):
            brute[m, n] = sum(int(q[m, k]) * int(w[n, k]) for k in range(K))
    assert np.array_equal(acc, brute)
    for gs in (16, 64):
        if K % gs:
            continue
        part = oracle.gemm_s32(q, w, gs)
        ref = np.einsum("mgk,ngk->mng", q.reshape(M, -1, gs).astype(np.int64),
                        w.reshape(N, -1, gs).astype(np.int64))
        assert np.array_equal(part, ref)
        assert np.array_equal(part.sum(axis=2), acc)


def test_gemm_s32_worst_case_no_overflow():
    K = 12288
    q = np.full((2, K), 127, np.int8)
    q[1] = -127
    w = np.full((2, K), 127, np.int8)
    acc = oracle.gemm_s32(q, w, 0)
    assert acc.tolist() == [[127 * 127 * K] * 2, [-127 * 127 * K] * 2]


def test_gemm_identity_weights():
    """wq = 127 * I (a slice): acc = 127 * q."""
    rng = np.random.default_rng(5)
    q = rng.integers(-127, 128, (7, 64), dtype=np.int8)
    w = np.zeros((32, 64), np.int8)
    w[np.arange(32), np.arange(32)] = 127
    assert np.array_equal(oracle.gemm_s32(q, w, 0), 127 * q[:, :32].astype(np.int32))


# --------------------------------------------------------------------------
# dequant epilogues and the whole layer
# --------------------------------------------------------------------------

def test_epilogue_hand_examples():
    for ex in _golden("epilogue_hand_examples.txt"):
        x = np.array([ex["x"]], np.float16)
        w = np.array([ex["w"]], np.float16)
        gs = ex["group_size"]
        q, _ = oracle.quantize_act(x)
        wq, sw = oracle.quantize_weight_int8(w, gs)
        part = oracle.gemm_s32(q, wq, gs)
        assert part.reshape(-1).tolist() == ex["partials"]
        y = oracle.w8a8_linear(x, wq, sw, gs)
        expect = np.float16(np.inf) if ex["y"] == "inf" else np.float16(ex["y"])
        assert y[0, 0] == expect


def test_epilogue_pc_unit_scales_is_fp16_of_acc():
    """s_act = s_w = 1: y = binary16 rounding of the integer accumulator,
    which numpy's float64 -> float16 conversion gives independently."""
    rng = np.random.default_rng(6)
    for acc in rng.integers(-(2 ** 31) + 1, 2 ** 31 - 1, 4000).tolist() + [0, 1, -1, 2049, 16129, 65519, 65520]:
        bits = oracle.epilogue_pc(acc, 1.0, 1.0)
        # (float)acc first rounds to binary32, then to binary16
        ref = np.float16(np.float32(acc)).view(np.uint16)
        assert bits == ref


def test_epilogue_pc_matches_float64_when_exact():
    """With power-of-two scales every fp32 step is exact for |acc| < 2^24, so
    y is the single binary16 rounding of acc * s_a * s_w."""
    rng = np.random.default_rng(7)
    for _ in range(3000):
        acc = int(rng.integers(-(2 ** 24) + 1, 2 ** 24))
        ea, ew = rng.integers(-20, 2, 2)
        sa, sw = 2.0 ** int(ea), 2.0 ** int(ew)
        ref = np.float16(acc * sa * sw).view(np.uint16)
        assert oracle.epilogue_pc(acc, sa, sw) == ref


def test_epilogue_pg_order_and_exact_case():
    rng = np.random.default_rng(8)
    # exact case: power-of-two scales, small partials -> the sum is exact
    for _ in range(500):
        G = int(rng.integers(1, 40))
        P = rng.integers(-(2 ** 14), 2 ** 14, G)
        sw = 2.0 ** rng.integers(-12, -4, G)
        sa = 2.0 ** int(rng.integers(-8, 0))
        ref = np.float16(float(np.sum(P * sw)) * sa).view(np.uint16)
        assert oracle.epilogue_pg(P, sw, sa) == ref
    # the rounded ascending-order sum is what the definition says: a group
    # that is tiny next to a large earlier one is absorbed
    P = np.array([1 << 24, 1, 1], np.int32)
    sw = np.ones(3, np.float32)
    assert oracle.epilogue_pg(P, sw, 2.0 ** -20) == np.float16(16.0).view(np.uint16)
    P2 = np.array([1, 1, 1 << 24], np.int32)
    assert oracle.epilogue_pg(P2, sw, 2.0 ** -20) == np.float16(np.float32(16777218.0) * 2.0 ** -20).view(np.uint16)


def test_epilogue_pg_rounds_each_product_then_each_sum():
    """Per-group reading (README "Quantization": each group's int32 partial
    rescaled by its weight scale, the rescaled partials summed): every
    product and every sum is its own binary32 rounding. Hand-worked case:
    P = [-3, 2531], s_w = [1, 13259 * 2^-23], s_a = 1.
      group 0: f = 0 + (-3 * 1) = -3 (exact)
      group 1: 2531 * 13259 = 33558529, so P*s = 33558529 * 2^-23
               = 4 + 2^-11 + 2^-23; binary32 in [4, 8) has spacing 2^-21,
               so fl(P*s) = 4 + 2^-11 (the 2^-23 is below half a spacing);
               f = fl(-3 + 4 + 2^-11) = 1 + 2^-11 (exact)
      y = fp16(1 + 2^-11): halfway between 1 and 1 + 2^-10, ties to even
          -> 1.0 (0x3C00).
    A fused multiply-add, or any wider accumulator, keeps the 2^-23 and
    rounds 1 + 2^-11 + 2^-23 up to 1 + 2^-10 (0x3C01) instead."""
    P = np.array([-3, 2531], np.int32)
    sw = np.array([1.0, 13259 * 2.0 ** -23], np.float32)
    assert 2531 * 13259 == 33558529 == (4 << 23) + (1 << 12) + 1
    assert oracle.epilogue_pg(P, sw, 1.0) == 0x3C00
    fused = np.float16(np.float32(-3.0 + 2531.0 * float(sw[1])))  # exact in float64
    assert fused.view(np.uint16) == 0x3C01


def test_epilogue_pc_multiplies_left_to_right():
    """README "Quantization", row "Output dequant: C_fp16 = C_int32 * s_act *
    s_weight", read left to right, each product rounded to binary32.
    Hand-worked: acc = 2275, s_act = 1 + 2^-12 = 4097/4096,
    s_weight = 1 + 35 * 2^-12 = 4131/4096.
      t = 2275 * 4097/4096 = 9320675/4096 (exact: binary32 spacing in
          [2048, 4096) is 2^-12)
      t * s_weight = 9400319.44 * 2^-12, rounded to 9400319 * 2^-12
          = 2294.99976; fp16 spacing there is 2, the midpoint 2295 is not
          reached -> 2294.0 (0x687B).
    The scales multiplied first: 4097 * 4131 = 16924707, an odd count of
    2^-24, halfway between binary32 neighbours; ties to even give
    16924708 * 2^-24; then 2275 times that rounds to exactly 2295, an fp16
    tie that rounds to even -> 2296.0 (0x687C)."""
    assert 4097 * 4131 == 16924707
    assert oracle.epilogue_pc(2275, 1 + 2.0 ** -12, 1 + 35 * 2.0 ** -12) == 0x687B


def test_epilogue_pg_sums_groups_in_ascending_order():
    """Groups summed in ascending order, each sum rounded. Hand-worked:
    P = [8392704, 1, 1] (8392704 = 2^23 + 2^12), s_w = [2, 1, 1],
    s_act = 2^-14.
      ascending: f = 2^24 + 2^13 (exact); adding 1 is a tie between
          binary32 neighbours 2 apart and rounds to the even one, so f stays
          2^24 + 2^13, twice; y = fp16((2^24 + 2^13) * 2^-14) = fp16(1024.5),
          an fp16 tie -> 1024.0 (0x6400).
    In descending order the two 1s add to 2 first and 2^24 + 2^13 + 2 is
    exact, so y = fp16(1024.5 + 2^-13) = 1025.0 (0x6401)."""
    P = np.array([8392704, 1, 1], np.int32)
    sw = np.array([2.0, 1.0, 1.0], np.float32)
    assert oracle.epilogue_pg(P, sw, 2.0 ** -14) == 0x6400


def test_epilogue_pg_applies_token_scale_once_at_the_end():
    """The token scale multiplies the finished group sum (README "Output
    dequant" row: C_int32 * s_act * s_weight, with the per-group sum in place
    of C_int32 * s_weight). Hand-worked: P = [986, 4093], s_w = [1, 1],
    s_act = 1 + 25 * 2^-12 = 4121/4096.
      f = 986 + 4093 = 5079 (exact); 5079 * 4121/4096 = 10465279.5 * 2^-11,
      a binary32 tie (spacing 2^-11 in [4096, 8192)) -> 10465280 * 2^-11 =
      5110, itself an fp16 tie between 5108 and 5112 -> 5112.0 (0x6CFE).
    Scaling each group before the sum gives 992.018066 + 4117.981445 =
    5109.99951, below the midpoint -> 5108.0 (0x6CFD)."""
    P = np.array([986, 4093], np.int32)
    sw = np.array([1.0, 1.0], np.float32)
    assert 5079 * 4121 == 2 * 10465279 + 1 and 10465280 * 2.0 ** -11 == 5110.0
    assert oracle.epilogue_pg(P, sw, 1 + 25 * 2.0 ** -12) == 0x6CFE


def test_pg_with_one_group_equals_pc_for_exact_scales():
    rng = np.random.default_rng(9)
    M, N, K = 5, 7, 128
    x = np.rint(rng.uniform(-127, 127, (M, K))).astype(np.float16)
    x[:, 0] = 127
    w = np.rint(rng.uniform(-127, 127, (N, K))).astype(np.float16)
    w[:, 1] = -127
    wq, s = oracle.quantize_weight_int8(w, 0)
    y_pc = oracle.w8a8_linear(x, wq, s, 0)
    y_pg = oracle.w8a8_linear(x, wq, s.reshape(N, 1), K)
    assert np.array_equal(y_pc.view(np.uint16), y_pg.view(np.uint16))


def test_layer_close_to_float64_product():
    """A dropped term, a wrong sign or index, or a transposed operand moves y
    far from x @ W^T; the quantized layer must stay within the error that
    the two quantizations allow."""
    rng = np.random.default_rng(10)
    M, N, K = 9, 40, 512
    x = rng.standard_normal((M, K))
    x[:, [3, 100]] *= 20
    x = x.astype(np.float16)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    xf, wf = x.astype(np.float64), w.astype(np.float64)
    exact = xf @ wf.T
    for gs in (0, 64, 128):
        wq, s = oracle.quantize_weight_int8(w, gs)
        y = oracle.w8a8_linear(x, wq, s, gs).astype(np.float64)
        sa = np.abs(xf).max(axis=1) / 127
        swf = np.abs(wf).max(axis=1) / 127 if gs == 0 else None
        # |x w - q s_a wq s_w| <= sum(|x| e_w + |w| e_a + e_a e_w) with e = s/2
        e_a = sa[:, None] / 2
        if gs == 0:
            e_w = np.repeat((swf / 2)[:, None], K, axis=1)
        else:
            e_w = np.repeat(s.astype(np.float64) / 2, gs, axis=1)
        bound = (np.abs(xf) @ e_w.T + e_a * np.abs(wf).sum(axis=1)[None, :]
                 + e_a * e_w.sum(axis=1)[None, :])
        bound = bound * 1.001 + np.abs(exact) * 2.0 ** -10 + 1e-6
        assert np.all(np.abs(y - exact) <= bound)


def test_w4a8_layer_equals_w8a8_on_unpacked_codes():
    rng = np.random.default_rng(11)
    M, N, K = 4, 12, 256
    x = rng.standard_normal((M, K)).astype(np.float16)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    for gs in (0, 128):
        wp, s = oracle.pack_weight_int4(w, gs)
        y4 = oracle.w4a8_linear(x, wp, s, gs)
        y8 = oracle.w8a8_linear(x, oracle.unpack_int4(wp, K), s, gs)
        assert np.array_equal(y4.view(np.uint16), y8.view(np.uint16))


def test_gemv_is_gemm_row():
    """The M=1 path is the same function as the GEMM: computing one row alone
    gives the bits of that row computed inside a batch."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((6, 192)).astype(np.float16)
    w = (rng.standard_normal((10, 192)) * 0.02).astype(np.float16)
    wq, s = oracle.quantize_weight_int8(w, 64)
    y = oracle.w8a8_linear(x, wq, s, 64)
    for m in range(6):
        assert np.array_equal(oracle.w8a8_linear(x[m:m + 1], wq, s, 64).view(np.uint16),
                              y[m:m + 1].view(np.uint16))


# ---------------------------------------------------------------------------
# bfloat16 activations and outputs (README roadmap: float16/bfloat16 dtypes)
# ---------------------------------------------------------------------------

def test_bf16_to_float_all_patterns():
    """Every bf16 bit pattern against torch's independent conversion (NaNs
    only need to stay NaN)."""
    import torch
    b = np.arange(65536, dtype=np.uint16)
    f = oracle.bf16_to_float(b)
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(f), nan)
    assert np.array_equal(f[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_bf16_hand_examples():
    """Worked roundings at 8 significant bits, ties to even, overflow."""
    cases = [
        (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
        (1.0 + 2.0 ** -8, 0x3F80),          # halfway between 1 and 1 + 2^-7: even (1)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),      # halfway between 1 + 2^-7 and 1 + 2^-6: even
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),  # just above the tie: up
        (3.3895313892515355e38, 0x7F7F),   # largest finite bf16
        (3.4028234663852886e38, 0x7F80),   # largest fp32 rounds past it to inf
        (2.0 ** -133, 0x0001),              # smallest bf16 subnormal
        (2.0 ** -134, 0x0000),              # halfway to it: even (0)
        (float("inf"), 0x7F80), (float("-inf"), 0xFF80),
    ]
    for v, want in cases:
        got = int(oracle.float_to_bf16(np.float32(v)))
        assert got == want, (v, hex(got), hex(want))


def test_float_to_bf16_matches_torch_random():
    import torch
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(200000).astype(np.float32)
         * np.float32(10.0) ** rng.integers(-40, 38, 200000).astype(np.float32))
    got = oracle.float_to_bf16(v)
    ref = torch.from_numpy(v).bfloat16().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_quant_equals_fp16_quant_on_shared_values():
    """Values exact in both formats (small integers and binary fractions)
    give the same codes and scales from bf16 and fp16 inputs."""
    rng = np.random.default_rng(8)
    x32 = (rng.integers(-256, 257, (5, 96)) / np.float32(8.0)).astype(np.float32)
    q16, s16 = oracle.quantize_act(x32.astype(np.float16))
    qbf, sbf = oracle.quantize_act_bf16(oracle.float_to_bf16(x32))
    assert np.array_equal(q16, qbf) and np.array_equal(s16, sbf)


def test_bf16_layer_epilogue_against_numpy_float32():
    """bf16 in / bf16 out layer: codes from the exact bf16 values, int32
    products from numpy int64, the fp32 epilogue restated in numpy float32
    (IEEE single) and rounded by torch's bf16 conversion."""
    import torch
    rng = np.random.default_rng(9)
    M, N, K = 4, 6, 64
    x_bits = oracle.float_to_bf16(rng.standard_normal((M, K)).astype(np.float32) * 3)
    wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s_w = (rng.random(N).astype(np.float32) * np.float32(0.01) + np.float32(1e-4))
    y = oracle.w8a8_linear(x_bits, wq, s_w, 0, x_dtype="bf16")
    q, s_a = oracle.quantize_act_bf16(x_bits)
    acc = (q.astype(np.int64) @ wq.astype(np.int64).T).astype(np.int32)
    t = (acc.astype(np.float32) * s_a[:, None]).astype(np.float32)
    t = (t * s_w[None, :]).astype(np.float32)
    ref = torch.from_numpy(t).bfloat16().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, ref)
    # fp16 output from the same bf16 input: the same fp32 values rounded to fp16.
    y16 = oracle.w8a8_linear(x_bits, wq, s_w, 0, x_dtype="bf16", y_dtype="f16")
    assert np.array_equal(y16.view(np.uint16), t.astype(np.float16).view(np.uint16))


def test_bf16_subnormal_scale_closed_form():
    """bf16 reaches values whose scale absmax / 127 is an fp32 subnormal: with
    u = 2^-149, absmax = 3 * 2^-133 = 196608 u gives s = rint(196608 / 127) u
    = 1548 u, and the codes are rint(x / s): 65536 / 1548 = 42.3 -> 42,
    196608 / 1548 = 127.0 -> 127."""
    u = 2.0 ** -149
    x = oracle.float_to_bf16(np.array([2.0 ** -133, -2.0 ** -133, 0.0, 3 * 2.0 ** -133],
                                      dtype=np.float32))
    q, s = oracle.quantize_act_bf16(x.reshape(1, 4))
    assert float(s[0]) == 1548 * u
    assert q.tolist() == [[42, -42, 0, 127]]


# ---------------------------------------------------------------------------
# A16 decode matrix-vector product (weight-only dequantization)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits,gs", [(8, 0), (8, 64), (4, 0), (4, 128)])
def test_a16_gemv_against_numpy_float64(bits, gs):
    """Independent restatement: dequantize the weights in numpy float64
    (code * scale) and take numpy's float64 matrix-vector product."""
    rng = np.random.default_rng(bits * 10 + gs)
    N, K = 37, 512
    x = (rng.standard_normal(K) * 3).astype(np.float16)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    if bits == 8:
        wq, s = oracle.quantize_weight_int8(w, gs)
        codes = wq.astype(np.float64)
        wdev = wq
    else:
        wdev, s = oracle.pack_weight_int4(w, gs)
        codes = oracle.unpack_int4(wdev, K).astype(np.float64)
    G = 1 if gs == 0 else K // gs
    scale = np.repeat(np.asarray(s, np.float64).reshape(N, G), K // G, axis=1)
    ref = (codes * scale) @ x.astype(np.float64)
    y = oracle.a16_gemv(x, wdev, s, bits, gs)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_a16_gemv_hand_examples():
    """One non-zero product per row: the value is exactly x * code * scale."""
    K = 64
    x = np.zeros(K, np.float16)
    x[5] = 1.5
    x[9] = -0.25
    wq = np.zeros((3, K), np.int8)
    wq[0, 5] = 100          # 1.5 * 100 * s0
    wq[1, 9] = -127         # -0.25 * -127 * s1
    wq[2, 5], wq[2, 9] = 2, 4  # 1.5 * 2 - 0.25 * 4 = 2
    s = np.array([0.5, 2.0, 0.125], np.float32)
    y = oracle.a16_gemv(x, wq, s, 8, 0)
    assert y.tolist() == [75.0, 63.5, 0.25]
    # bf16 input reads the same exact values
    xb = oracle.float_to_bf16(x.astype(np.float32))
    assert oracle.a16_gemv(xb, wq, s, 8, 0, x_dtype="bf16").tolist() == [75.0, 63.5, 0.25]


# ---------------------------------------------------------------------------
# percentile-clipped weight scales (clip_percentile)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gs", [0, 64])
@pytest.mark.parametrize("bits", [8, 4])
def test_clip_percentile_100_is_min_max(gs, bits):
    w = (np.random.default_rng(30 + gs + bits).standard_normal((9, 256)) * 0.02).astype(np.float16)
    got = oracle.quantize_weight_clipped(w, gs, 100.0, bits)
    ref = oracle.quantize_weight_int8(w, gs) if bits == 8 else oracle.pack_weight_int4(w, gs)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


@pytest.mark.parametrize("pct", [99.9, 99.0, 50.0, 1.0])
def test_clip_value_matches_numpy_percentile(pct):
    """The scale is numpy's linear-interpolation percentile of |w| (float64,
    rounded to float32) divided by qmax; codes saturate beyond the clip."""
    rng = np.random.default_rng(int(pct * 10))
    w = (rng.standard_normal((7, 1024)) * 0.05).astype(np.float16)
    wq, s = oracle.quantize_weight_clipped(w, 128, pct, 8)
    a = np.abs(w.astype(np.float64)).reshape(7, 8, 128)
    clip = np.percentile(a, pct, axis=2, method="linear").astype(np.float32)
    assert np.array_equal(s, clip / np.float32(127.0))
    x = w.astype(np.float32).reshape(7, 8, 128) / s[:, :, None]
    ref = np.clip(np.rint(x), -127, 127).astype(np.int8).reshape(7, 1024)
    assert np.array_equal(wq, ref)


def test_clip_percentile_hand_example():
    """|w| = 1..5 (one block of 8 with three zeros): the 50th percentile of
    [0, 0, 0, 1, 2, 3, 4, 5] sits at position 3.5 -> 1.5; scale 1.5 / 127."""
    w = np.array([[0, 1, -2, 3, 0, -4, 5, 0]], np.float16)
    wq, s = oracle.quantize_weight_clipped(w, 0, 50.0, 8)
    assert s[0] == np.float32(1.5) / np.float32(127.0)
    assert wq.tolist() == [[0, 85, -127, 127, 0, -127, 127, 0]]


def test_clip_zero_block_gives_zero_scale_and_zero_codes():
    """Reading (the pages are silent): when the p-th percentile of a block's
    |w| is 0 (more than p % of its entries are zero), the block's scale is 0
    and EVERY code is 0, non-zero weights included - the rule min-max applies
    to an all-zero block. The other plausible reading, saturating the
    non-zero weights to +-qmax (w / 0 = +-inf, clamped), fails here.
    Sorted |w| = [0, 0, 0, 0, 0, 0, 3, 5]: p = 50 sits at position 3.5 -> 0;
    p = 80 at 5.6 -> 0 + 0.6 * (3 - 0) = 1.8, a non-zero clip (contrast)."""
    w = np.array([[0, 0, 3, 0, 0, -5, 0, 0]], np.float16)
    wq, s = oracle.quantize_weight_clipped(w, 0, 50.0, 8)
    assert s.view(np.uint32)[0] == 0
    assert wq.tolist() == [[0, 0, 0, 0, 0, 0, 0, 0]]
    wp, s4 = oracle.quantize_weight_clipped(w, 0, 50.0, 4)
    assert s4[0] == 0.0 and wp.tolist() == [[0x88, 0x88, 0x88, 0x88]]  # nibble 8 = code 0
    wq, s = oracle.quantize_weight_clipped(w, 0, 80.0, 8)
    assert s[0] == np.float32(1.8) / np.float32(127.0)
    assert wq.tolist() == [[0, 0, 127, 0, 0, -127, 0, 0]]
