"""CPU oracle for the per-token INT8 quantize -> INT8 GEMM -> dequant layer.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the CUDA product path
never does. The arithmetic lives in ``cider_oracle.c`` (plain C, one IEEE
binary32 operation per written operation); this file only builds that C file
with gcc and marshals numpy arrays to it.

Every function cites the passage it follows in its docstring; the pages are
the Cider project's README mirror ("cider", Mininglamp-AI) and its two blog
posts. Where the pages are silent, the readings listed at the top of
``cider_oracle.c`` apply.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cider_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fexcess-precision=standard", "-fPIC", "-shared", "-fopenmp"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles cider_oracle.c into liboracle.so next to it (gcc)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_float.restype = ctypes.c_float
            lib.oracle_float_to_half.argtypes = [ctypes.c_float]
            lib.oracle_float_to_half.restype = ctypes.c_uint16
            lib.oracle_half_to_float_array.argtypes = [p, i64, p]
            lib.oracle_half_to_float_array.restype = None
            lib.oracle_float_to_half_array.argtypes = [p, i64, p]
            lib.oracle_float_to_half_array.restype = None
            lib.oracle_quantize_act.argtypes = [p, i64, i64, p, p]
            lib.oracle_quantize_act.restype = None
            lib.oracle_quantize_weight_int8.argtypes = [p, i64, i64, i32, p, p]
            lib.oracle_pack_weight_int4.argtypes = [p, i64, i64, i32, p, p]
            lib.oracle_unpack_int4.argtypes = [p, i64, i64, p]
            lib.oracle_unpack_int4.restype = None
            lib.oracle_gemm_s32.argtypes = [p, p, i64, i64, i64, i32, p]
            lib.oracle_epilogue_pc.argtypes = [ctypes.c_int32, ctypes.c_float, ctypes.c_float]
            lib.oracle_epilogue_pc.restype = ctypes.c_uint16
            lib.oracle_epilogue_pg.argtypes = [p, p, i64, ctypes.c_float]
            lib.oracle_epilogue_pg.restype = ctypes.c_uint16
            lib.oracle_w8a8_linear.argtypes = [p, i64, i64, i64, p, p, i32, p]
            lib.oracle_w4a8_linear.argtypes = [p, i64, i64, i64, p, p, i32, p]
            lib.oracle_bf16_to_float_array.argtypes = [p, i64, p]
            lib.oracle_bf16_to_float_array.restype = None
            lib.oracle_float_to_bf16_array.argtypes = [p, i64, p]
            lib.oracle_float_to_bf16_array.restype = None
            lib.oracle_quantize_act_ex.argtypes = [p, i32, i64, i64, p, p]
            lib.oracle_quantize_act_ex.restype = None
            lib.oracle_w8a8_linear_ex.argtypes = [p, i32, i64, i64, i64, p, p, i32, p, i32]
            lib.oracle_w4a8_linear_ex.argtypes = [p, i32, i64, i64, i64, p, p, i32, p, i32]
            lib.oracle_a16_gemv.argtypes = [p, i32, i64, i64, p, i32, p, i32, p]
            lib.oracle_quantize_weight_pct.argtypes = [p, i32, i64, i64, i32, ctypes.c_double,
                                                       ctypes.c_float, p, p]
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = None
            lib.oracle_get_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


_DTYPES = {"f16": 0, "bf16": 1}


def _bits(x, dtype: str) -> np.ndarray:
    """Activation bits: fp16 arrays (or uint16 bits) for "f16"; uint16 bit
    patterns for "bf16" (numpy has no bfloat16)."""
    if dtype == "f16":
        return _f16_bits(x)
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 values are passed as uint16 bit patterns, got {a.dtype}")
    return a


def _out(y_bits: np.ndarray, dtype: str) -> np.ndarray:
    return y_bits.view(np.float16) if dtype == "f16" else y_bits


def _f16_bits(x) -> np.ndarray:
    """fp16 array (or uint16 bit patterns) -> contiguous uint16 bit patterns."""
    a = np.ascontiguousarray(x)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected float16 or uint16 bits, got {a.dtype}")
    return a


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def half_to_float(bits) -> np.ndarray:
    """binary16 bit patterns -> exact float32 values (IEEE 754 binary16)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).ravel()
    out = np.empty(b.shape, np.float32)
    _load().oracle_half_to_float_array(_ptr(b), b.size, _ptr(out))
    return out.reshape(np.shape(bits))


def float_to_half(vals) -> np.ndarray:
    """float32 values -> binary16 bits, round to nearest, ties to even."""
    v = np.ascontiguousarray(np.asarray(vals, dtype=np.float32)).ravel()
    out = np.empty(v.shape, np.uint16)
    _load().oracle_float_to_half_array(_ptr(v), v.size, _ptr(out))
    return out.reshape(np.shape(vals))


def bf16_to_float(bits) -> np.ndarray:
    """bfloat16 bit patterns -> exact float32 values (the upper half of a
    binary32 encoding)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).ravel()
    out = np.empty(b.shape, np.float32)
    _load().oracle_bf16_to_float_array(_ptr(b), b.size, _ptr(out))
    return out.reshape(np.shape(bits))


def float_to_bf16(vals) -> np.ndarray:
    """float32 values -> bfloat16 bits, round to nearest, ties to even."""
    v = np.ascontiguousarray(np.asarray(vals, dtype=np.float32)).ravel()
    out = np.empty(v.shape, np.uint16)
    _load().oracle_float_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out.reshape(np.shape(vals))


def quantize_act_bf16(x_bits):
    """Per-token symmetric INT8 quantization of bf16 activations (uint16 bit
    patterns): the same formulas as quantize_act on the exact fp32 values
    (README "Quantization" table, row "Activations"; README roadmap,
    "automatic dtype handling (float16/bfloat16)")."""
    xb = _bits(x_bits, "bf16")
    M, K = xb.shape
    q = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    _load().oracle_quantize_act_ex(_ptr(xb), 1, M, K, _ptr(q), _ptr(s))
    return q, s


def quantize_act(x):
    """Per-token symmetric INT8 activation quantization.

    README "Quantization" table, row "Activations: Symmetric INT8, Per-token";
    README "Metal Kernel Pipeline", prefill step 1 (fp16 activations -> INT8
    plus per-token scales). Returns (q int8 [M,K], s float32 [M]).
    """
    xb = _f16_bits(x)
    M, K = xb.shape
    q = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    _load().oracle_quantize_act(_ptr(xb), M, K, _ptr(q), _ptr(s))
    return q, s


def quantize_weight_int8(w, group_size: int = 0):
    """Symmetric INT8 weight quantization, per output channel (group_size 0)
    or per group of ``group_size`` along K.

    README "Quantization" table, row "W8A8 weights"; README "W8A8 Quantization
    Granularity" table; README "Low-Level API" (quantize_weight_int8).
    Returns (wq int8 [N,K], s_w float32 [N] or [N, K/gs]).
    """
    wb = _f16_bits(w)
    N, K = wb.shape
    G = 1 if group_size == 0 else K // group_size
    wq = np.empty((N, K), np.int8)
    s = np.empty((N, G), np.float32)
    rc = _load().oracle_quantize_weight_int8(_ptr(wb), N, K, group_size, _ptr(wq), _ptr(s))
    if rc:
        raise ValueError(f"unsupported K={K} / group_size={group_size}")
    return wq, (s[:, 0].copy() if group_size == 0 else s)


def pack_weight_int4(w, group_size: int = 0):
    """Symmetric INT4 weight quantization (codes in [-7, 7], nibble = code + 8),
    two codes per byte, element 2j in the low nibble.

    README "Quantization" table, row "W4A8 weights: Symmetric INT4 (zp=8)";
    README "Low-Level API" (pack_weight_int4). Returns (wp uint8 [N, K/2],
    s_w float32 [N] or [N, K/gs]).
    """
    wb = _f16_bits(w)
    N, K = wb.shape
    G = 1 if group_size == 0 else K // group_size
    wp = np.empty((N, K // 2), np.uint8)
    s = np.empty((N, G), np.float32)
    rc = _load().oracle_pack_weight_int4(_ptr(wb), N, K, group_size, _ptr(wp), _ptr(s))
    if rc:
        raise ValueError(f"unsupported K={K} / group_size={group_size}")
    return wp, (s[:, 0].copy() if group_size == 0 else s)


def unpack_int4(wp, K: int) -> np.ndarray:
    """Packed INT4 [N, K/2] -> INT8 codes [N, K] (README "Modes" table, W4A8
    compute path "Unpack -> TensorOps")."""
    wp = np.ascontiguousarray(wp, dtype=np.uint8)
    N = wp.shape[0]
    wq = np.empty((N, K), np.int8)
    _load().oracle_unpack_int4(_ptr(wp), N, K, _ptr(wq))
    return wq


def gemm_s32(q, wq, group_size: int = 0) -> np.ndarray:
    """INT8 x INT8 -> INT32 products (README "Quantization" table, row
    "Accumulation: INT32"): [M,N] totals for group_size 0, else per-group
    partials [M, N, K/gs]."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    M, K = q.shape
    N = wq.shape[0]
    G = 1 if group_size == 0 else K // group_size
    out = np.empty((M, N, G), np.int32)
    rc = _load().oracle_gemm_s32(_ptr(q), _ptr(wq), M, N, K, group_size, _ptr(out))
    if rc:
        raise ValueError("unsupported group_size")
    return out[:, :, 0].copy() if group_size == 0 else out


def epilogue_pc(acc: int, s_act: float, s_w: float) -> int:
    """C_fp16 = C_int32 * s_act * s_weight (README "Quantization" table,
    row "Output dequant"); returns binary16 bits."""
    return int(_load().oracle_epilogue_pc(int(acc), float(s_act), float(s_w)))


def epilogue_pg(partials, s_w_row, s_act: float) -> int:
    """Per-group dequant: partials rescaled by their group scales, summed in
    ascending group order, times the token scale; returns binary16 bits."""
    p = np.ascontiguousarray(partials, dtype=np.int32)
    s = np.ascontiguousarray(s_w_row, dtype=np.float32)
    return int(_load().oracle_epilogue_pg(_ptr(p), _ptr(s), p.size, float(s_act)))


def w8a8_linear(x, wq, s_w, group_size: int = 0, x_dtype: str = "f16",
                y_dtype: str | None = None) -> np.ndarray:
    """W8A8 linear layer y = dequant(quant(x) . wq^T) (README "Metal Kernel
    Pipeline", prefill steps 1-2; "Quantization" table). x and y are fp16 by
    default; "bf16" takes / returns bfloat16 uint16 bit patterns (README
    roadmap, "automatic dtype handling (float16/bfloat16)"); y_dtype defaults
    to x_dtype."""
    y_dtype = y_dtype or x_dtype
    xb = _bits(x, x_dtype)
    M, K = xb.shape
    wq = np.ascontiguousarray(wq, dtype=np.int8)
    N = wq.shape[0]
    s = np.ascontiguousarray(s_w, dtype=np.float32)
    y = np.empty((M, N), np.uint16)
    rc = _load().oracle_w8a8_linear_ex(_ptr(xb), _DTYPES[x_dtype], M, N, K, _ptr(wq), _ptr(s),
                                       group_size, _ptr(y), _DTYPES[y_dtype])
    if rc:
        raise ValueError("unsupported shape / group_size")
    return _out(y, y_dtype)


def w4a8_linear(x, wp, s_w, group_size: int = 0, x_dtype: str = "f16",
                y_dtype: str | None = None) -> np.ndarray:
    """W4A8 linear layer: INT4 nibbles unpacked to INT8, then the W8A8 layer
    (README "Modes" table, W4A8 "Unpack -> TensorOps"; "Metal Kernel
    Pipeline", W4A8 note). Dtypes as in w8a8_linear."""
    y_dtype = y_dtype or x_dtype
    xb = _bits(x, x_dtype)
    M, K = xb.shape
    wp = np.ascontiguousarray(wp, dtype=np.uint8)
    N = wp.shape[0]
    s = np.ascontiguousarray(s_w, dtype=np.float32)
    y = np.empty((M, N), np.uint16)
    rc = _load().oracle_w4a8_linear_ex(_ptr(xb), _DTYPES[x_dtype], M, N, K, _ptr(wp), _ptr(s),
                                       group_size, _ptr(y), _DTYPES[y_dtype])
    if rc:
        raise ValueError("unsupported shape / group_size")
    return _out(y, y_dtype)


def a16_gemv(x, w, s_w, bits: int = 8, group_size: int = 0, x_dtype: str = "f16") -> np.ndarray:
    """A16 decode matrix-vector product with weight-only dequantization
    (README "Metal Kernel Pipeline", decode: "on-the-fly weight
    dequantization (no activation quantization needed)"): y[n] = sum over
    groups of s_w[n,g] * sum_k x[k] * code[n,k], accumulated in float64 and
    returned unrounded (float64 [N]). x: fp16 [K] or bf16 bits; w: int8
    [N,K] (bits 8) or packed uint8 [N,K/2] (bits 4)."""
    xb = _bits(np.asarray(x).reshape(-1), x_dtype)
    K = xb.size
    w = np.ascontiguousarray(w, dtype=np.int8 if bits == 8 else np.uint8)
    N = w.shape[0]
    s = np.ascontiguousarray(s_w, dtype=np.float32)
    y = np.empty((N,), np.float64)
    rc = _load().oracle_a16_gemv(_ptr(xb), _DTYPES[x_dtype], K, N, _ptr(w), bits, _ptr(s),
                                 group_size, _ptr(y))
    if rc:
        raise ValueError("unsupported bits / group_size")
    return y


def quantize_weight_clipped(w, group_size: int = 0, clip_percentile: float = 99.9,
                            bits: int = 8, w_dtype: str = "f16"):
    """Weight quantization with percentile-clipped scales (README "LLM
    Quantization" note: "the 99th percentile method (clip_percentile=99.9)"):
    per block (output channel, or group of ``group_size``), the clip value is
    the ``clip_percentile``-th percentile of |w| (linear interpolation between
    order statistics), scale = clip / qmax, codes = clamp(rint(w / scale)).
    bits 8: returns (wq int8 [N,K], s_w); bits 4: (packed uint8 [N,K/2],
    s_w), nibble = code + 8, element 2j in the low nibble."""
    wb = _bits(w, w_dtype)
    N, K = wb.shape
    G = 1 if group_size == 0 else K // group_size
    codes = np.empty((N, K), np.int8)
    s = np.empty((N, G), np.float32)
    qmax = 127.0 if bits == 8 else 7.0
    rc = _load().oracle_quantize_weight_pct(_ptr(wb), _DTYPES[w_dtype], N, K, group_size,
                                            float(clip_percentile), qmax, _ptr(codes), _ptr(s))
    if rc:
        raise ValueError("unsupported K / group_size / percentile")
    s = s[:, 0].copy() if group_size == 0 else s
    if bits == 8:
        return codes, s
    nib = (codes.astype(np.int16) + 8).astype(np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8), s
