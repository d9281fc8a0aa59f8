"""Canary guard bands: no kernel writes outside the buffers it was given.

compute-sanitizer is closed on this machine, so out-of-bounds writes are caught
the plain way. Every output (y, the codes and scales of the quantization and
weight-preparation calls) and the workspace are carved out of one larger
device buffer filled with a sentinel byte pattern; after the call the bands
before and after each carved range must still hold the pattern, and the
outputs must still match the oracle. The shapes include ragged tails in M, N
and K, so that predicated tile edges are exercised on both engines and on
the GEMV.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a8_quantized_gemm_int8_b300 as cider
from gpu_helpers import assert_f16_within_1ulp, host

pytestmark = pytest.mark.gpu

BAND = 64 << 10  # bytes of sentinel before and after every carved range
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cider.load_library()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    st, site = cider.device_status()
    assert st == cider.CIDER_OK, f"device status {st} at site {site:#x}"


class Guarded:
    """Device ranges with sentinel bands around each (256-byte aligned)."""

    def __init__(self, sizes):
        self.offs = []
        off = BAND
        for n in sizes:
            self.offs.append((off, n))
            off += (n + 255) // 256 * 256 + BAND
        self.buf = torch.full((off,), PATTERN, dtype=torch.uint8, device="cuda:0")

    def view(self, i, dtype, shape):
        off, n = self.offs[i]
        t = self.buf[off:off + n].view(dtype)
        return t.view(shape) if shape else t

    def ptr(self, i):
        return self.buf.data_ptr() + self.offs[i][0]

    def check(self, what):
        torch.cuda.synchronize()
        b = host(self.buf)
        mask = np.ones(b.size, bool)
        for off, n in self.offs:
            mask[off:off + n] = False
        bad = np.flatnonzero(mask & (b != PATTERN))
        assert bad.size == 0, f"{what}: {bad.size} bytes written outside the buffers, first at " \
                              f"{self._where(int(bad[0]))}"

    def _where(self, pos):
        for i, (off, n) in enumerate(self.offs):
            if pos < off:
                return f"{off - pos} bytes before range {i}"
            if pos < off + n + BAND:
                return f"{pos - off - n} bytes after range {i}"
        return f"byte {pos}"


def _inputs(M, N, K, seed):
    li = synth.linear_inputs(M, N, K, n_out=4, seed=seed)
    return li.x.numpy(), li.w.numpy()


# The last two take stream-K on SM pairs for per-channel layers (their
# partial tiles live in the guarded workspace).
SHAPES = [(130, 257, 1088), (200, 8, 2560), (3, 300, 192), (4, 40, 80), (257, 136, 512),
          (1, 1000, 2560), (32, 1280, 8192), (77, 2500, 4096)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("bits,gs", [(8, 0), (8, 64), (4, 0), (4, 64)])
def test_layer_writes_only_y_and_workspace(M, N, K, bits, gs):
    if gs and K % gs:
        pytest.skip("group size does not divide K")
    if bits == 4 and K % 32:
        pytest.skip("INT4 needs K % 32 == 0")
    x, w = _inputs(M, N, K, seed=M + N + K + gs + bits)
    if bits == 8:
        wq, s = oracle.quantize_weight_int8(w, gs)
        ref = oracle.w8a8_linear(x, wq, s, gs)
    else:
        wq, s = oracle.pack_weight_int4(w, gs)
        ref = oracle.w4a8_linear(x, wq, s, gs)
    need = cider.workspace_bytes(M, N, K, group_size=gs, bits=bits)
    g = Guarded([2 * M * N, max(need, 16)])
    y = g.view(0, torch.float16, (M, N))
    ws = g.view(1, torch.uint8, None)[:need] if need else None
    cider.linear(torch.from_numpy(x).cuda(), torch.from_numpy(wq).cuda(),
                 torch.from_numpy(s).cuda(), bits=bits, group_size=gs, out=y, ws=ws)
    g.check(f"layer M={M} N={N} K={K} bits={bits} gs={gs}")
    assert_f16_within_1ulp(host(y), ref, "guarded layer")


@pytest.mark.parametrize("M,K", [(5, 13), (130, 1088), (3, 40)])
def test_act_quant_writes_only_its_outputs(M, K):
    lib = cider.load_library()
    x = synth.activations(M, K, 0, synth.generator(M + K)).numpy()
    g = Guarded([M * K, 4 * M])
    st = lib.cider_quantize_act(torch.from_numpy(x).cuda().data_ptr(), M, K, g.ptr(0), g.ptr(1),
                                torch.cuda.current_stream().cuda_stream)
    assert st == cider.CIDER_OK
    g.check(f"quantize_act M={M} K={K}")
    qo, so = oracle.quantize_act(x)
    assert np.array_equal(host(g.view(0, torch.int8, (M, K))), qo)
    assert np.array_equal(host(g.view(1, torch.float32, (M,))).view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("N,K,gs,bits", [(37, 192, 0, 8), (37, 192, 64, 8), (9, 96, 32, 4),
                                         (300, 1088, 0, 4)])
def test_weight_prep_writes_only_its_outputs(N, K, gs, bits):
    lib = cider.load_library()
    w = synth.weights(N, K, synth.generator(N + K)).numpy()
    G = 1 if gs == 0 else K // gs
    nbytes = N * K if bits == 8 else N * K // 2
    g = Guarded([nbytes, 4 * N * G])
    wd = torch.from_numpy(w).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    if bits == 8:
        st = lib.cider_quantize_weight_int8(wd.data_ptr(), N, K, gs, g.ptr(0), g.ptr(1), stream)
        qo, so = oracle.quantize_weight_int8(w, gs)
        got = host(g.view(0, torch.int8, (N, K)))
    else:
        st = lib.cider_pack_weight_int4(wd.data_ptr(), N, K, gs, g.ptr(0), g.ptr(1), stream)
        qo, so = oracle.pack_weight_int4(w, gs)
        got = host(g.view(0, torch.uint8, (N, K // 2)))
    assert st == cider.CIDER_OK
    g.check(f"weight prep N={N} K={K} gs={gs} bits={bits}")
    assert np.array_equal(got, qo)
    assert np.array_equal(host(g.view(1, torch.float32, (N * G,))).view(np.uint32),
                          np.asarray(so).reshape(-1).view(np.uint32))


def test_noalloc_layer_writes_only_y():
    lib = cider.load_library()
    M, N, K = 130, 257, 1088
    x, w = _inputs(M, N, K, seed=3)
    wq, s = oracle.quantize_weight_int8(w, 0)
    g = Guarded([2 * M * N])
    xd, wqd, sd = (torch.from_numpy(a).cuda() for a in (x, wq, s))
    st = lib.cider_w8a8_gemm_pc_noalloc(xd.data_ptr(), M, N, K, wqd.data_ptr(), sd.data_ptr(),
                                        g.ptr(0), torch.cuda.current_stream().cuda_stream)
    assert st == cider.CIDER_OK
    g.check("noalloc layer")
    assert_f16_within_1ulp(host(g.view(0, torch.float16, (M, N))),
                           oracle.w8a8_linear(x, wq, s, 0), "noalloc guarded")
