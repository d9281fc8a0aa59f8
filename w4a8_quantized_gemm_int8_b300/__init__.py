"""B300 (sm_103a) quantized linear layers: online per-token INT8 activation
quantization, exact INT8 x INT8 -> INT32 products on the tensor cores, fused
dequant to fp16; W8A8 per-channel, W8A8 per-group, W4A8, and the M = 1 GEMV.

This module is a thin ctypes binding over ``libcider.so`` (the C ABI in
``include/cider.h``): it checks tensors, allocates outputs and workspace with
torch, and passes raw device pointers and the current CUDA stream. Every
arithmetic step runs in the library's CUDA kernels; there is no CPU path. If
the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcider.so")

# The C-ABI entry points (names as declared in include/cider.h).
ABI_FUNCTIONS = (
    "cider_status_string", "cider_abi_version", "cider_quantize_act",
    "cider_quantize_weight_int8", "cider_pack_weight_int4", "cider_workspace_bytes",
    "cider_w8a8_gemm_pc", "cider_w8a8_gemm_pg", "cider_w4a8_gemm", "cider_int8_gemv",
    "cider_linear", "cider_quantize_act_ex", "cider_a16_gemv", "cider_quantize_weight_clipped",
    "cider_w8a8_gemm_pc_noalloc",
    "cider_act_image", "cider_weight_image", "cider_gemm_images",
    "cider_test_gemm_s32", "cider_device_status", "cider_test_wait_timeout",
    "cider_test_int8_mma_loop", "cider_test_read_bytes",
)

CIDER_OK = 0
CIDER_DTYPE_F16 = 0
CIDER_DTYPE_BF16 = 1
_DTYPE_CODES = {torch.float16: CIDER_DTYPE_F16, torch.bfloat16: CIDER_DTYPE_BF16}
CIDER_ERR_INVALID_ARG = 1
CIDER_ERR_UNSUPPORTED = 2
CIDER_ERR_CUDA = 3
CIDER_ERR_TIMEOUT = 4

_lock = threading.Lock()
_lib = None


class CiderError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def load_library():
    """Loads libcider.so (built by ``build.py``); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m "
                "w4a8_quantized_gemm_int8_b300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "cider_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "cider_abi_version": ([], ctypes.c_int),
            "cider_quantize_act": ([p, i64, i64, p, p, p], ctypes.c_int),
            "cider_quantize_weight_int8": ([p, i64, i64, i32, p, p, p], ctypes.c_int),
            "cider_pack_weight_int4": ([p, i64, i64, i32, p, p, p], ctypes.c_int),
            "cider_workspace_bytes": ([i64, i64, i64, i32, i32], sz),
            "cider_w8a8_gemm_pc": ([p, i64, i64, i64, p, p, p, p, sz, p], ctypes.c_int),
            "cider_w8a8_gemm_pg": ([p, i64, i64, i64, p, p, i32, p, p, sz, p], ctypes.c_int),
            "cider_w4a8_gemm": ([p, i64, i64, i64, p, p, i32, p, p, sz, p], ctypes.c_int),
            "cider_int8_gemv": ([p, i64, i64, p, p, i32, i32, p, p], ctypes.c_int),
            "cider_linear": ([p, i32, i64, i64, i64, p, i32, p, i32, p, i32, p, sz, p],
                             ctypes.c_int),
            "cider_quantize_act_ex": ([p, i32, i64, i64, p, p, p], ctypes.c_int),
            "cider_a16_gemv": ([p, i32, i64, i64, p, i32, p, i32, p, i32, p], ctypes.c_int),
            "cider_quantize_weight_clipped": ([p, i32, i64, i64, i32, i32, ctypes.c_double, p,
                                               p, p], ctypes.c_int),
            "cider_w8a8_gemm_pc_noalloc": ([p, i64, i64, i64, p, p, p, p], ctypes.c_int),
            "cider_act_image": ([p, i64, i64, p, p, p], ctypes.c_int),
            "cider_weight_image": ([p, i64, i64, i32, p, p], ctypes.c_int),
            "cider_gemm_images": ([p, p, p, p, i64, i64, i64, i32, p, p], ctypes.c_int),
            "cider_test_gemm_s32": ([p, p, i64, i64, i64, i32, i32, p, p, sz, p], ctypes.c_int),
            "cider_device_status": ([p, ctypes.POINTER(ctypes.c_uint32)], ctypes.c_int),
            "cider_test_wait_timeout": ([i64, p], ctypes.c_int),
            "cider_test_int8_mma_loop": ([i32, i64, p, p], ctypes.c_int),
            "cider_test_read_bytes": ([p, i64, p, p], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().cider_status_string(int(status)).decode()


def abi_version() -> int:
    return int(load_library().cider_abi_version())


def _check(fn: str, status: int) -> None:
    if status != CIDER_OK:
        raise CiderError(fn, status)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _dev(t: torch.Tensor, dtype, name: str, ndim: int | None = None) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    return t.data_ptr()


def _check_weights(K: int, N: int, w: torch.Tensor, s_w: torch.Tensor, bits: int,
                   group_size: int) -> None:
    """The weights and scales must match the activations' K: the kernels read
    N x K codes (N x K/2 bytes packed) and the scale table the group size
    implies, so a smaller tensor would be read past its end."""
    if bits not in (8, 4):
        raise ValueError(f"bits must be 8 or 4, got {bits}")
    if w.dim() != 2 or w.shape[0] != N:
        raise ValueError(f"w must be 2-D with {N} rows, got shape {tuple(w.shape)}")
    if bits == 4 and K % 2:
        raise ValueError(f"packed INT4 weights need an even K, got {K}")
    cols = K if bits == 8 else K // 2
    if w.shape[1] != cols:
        raise ValueError(f"w has {w.shape[1]} columns; K = {K} with {bits}-bit codes "
                         f"needs {cols}")
    if group_size < 0 or (group_size and K % group_size):
        raise ValueError(f"group_size {group_size} must be 0 or a divisor of K = {K}")
    want = N if group_size == 0 else N * (K // group_size)
    if s_w.numel() != want:
        raise ValueError(f"s_w has {s_w.numel()} scales, {want} expected "
                         f"([N] per channel or [N, K/group_size] per group)")


def _check_out(out: torch.Tensor | None, shape: tuple, name: str = "out") -> None:
    """A caller's output tensor must have exactly the shape the call writes."""
    if out is not None and tuple(out.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(out.shape)}")


_ws_cache: dict = {}


def workspace_bytes(M: int, N: int, K: int, group_size: int = 0, bits: int = 8) -> int:
    """cider_workspace_bytes: arguments in the C order (M, N, K, group_size, bits)."""
    return int(load_library().cider_workspace_bytes(M, N, K, group_size, bits))


def _workspace(nbytes: int, device) -> torch.Tensor | None:
    """A per-device workspace buffer, grown on demand (stream-ordered reuse:
    calls on one stream may share it)."""
    if torch.device(device).type != "cuda":
        raise ValueError("the layer's tensors must be CUDA tensors")
    if nbytes == 0:
        return None
    key = torch.device(device).index
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


# ---------------------------------------------------------------------------
# quantization
# ---------------------------------------------------------------------------

def quantize_act(x: torch.Tensor):
    """Per-token INT8 activation quantization: x fp16 [M,K] -> (q int8 [M,K],
    s_a fp32 [M])."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    s = torch.empty((M,), dtype=torch.float32, device=x.device)
    lib = load_library()
    xp = _dev(x, torch.float16, "x", 2)
    if M == 0:  # no tokens: nothing to compute
        return q, s
    _check("cider_quantize_act", lib.cider_quantize_act(
        xp, M, K, q.data_ptr(), s.data_ptr(), _stream()))
    return q, s


def quantize_weight_int8(w: torch.Tensor, group_size: int = 0):
    """INT8 weight quantization: w fp16 [N,K] -> (wq int8 [N,K], s_w fp32
    [N] (group_size 0) or [N, K/group_size])."""
    N, K = w.shape
    wq = torch.empty((N, K), dtype=torch.int8, device=w.device)
    shape = (N,) if group_size == 0 else (N, K // group_size)
    s = torch.empty(shape, dtype=torch.float32, device=w.device)
    lib = load_library()
    wp = _dev(w, torch.float16, "w", 2)
    if N == 0:  # no output channels: nothing to compute
        return wq, s
    _check("cider_quantize_weight_int8", lib.cider_quantize_weight_int8(
        wp, N, K, group_size, wq.data_ptr(), s.data_ptr(), _stream()))
    return wq, s


def pack_weight_int4(w: torch.Tensor, group_size: int = 0):
    """INT4 weight quantization + packing: w fp16 [N,K] -> (wp uint8 [N,K/2],
    s_w fp32 [N] or [N, K/group_size])."""
    N, K = w.shape
    wp = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    shape = (N,) if group_size == 0 else (N, K // group_size)
    s = torch.empty(shape, dtype=torch.float32, device=w.device)
    lib = load_library()
    wd = _dev(w, torch.float16, "w", 2)
    if N == 0:  # no output channels: nothing to compute
        return wp, s
    _check("cider_pack_weight_int4", lib.cider_pack_weight_int4(
        wd, N, K, group_size, wp.data_ptr(), s.data_ptr(), _stream()))
    return wp, s


# ---------------------------------------------------------------------------
# linear layers
# ---------------------------------------------------------------------------

def w8a8_linear(x: torch.Tensor, wq: torch.Tensor, s_w: torch.Tensor, group_size: int = 0,
                out: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """W8A8 linear layer y = dequant(quant(x) . wq^T): per-channel for
    group_size 0 (s_w [N]), per-group otherwise (s_w [N, K/gs]). M == 1 runs
    the GEMV inside the library."""
    M, K = x.shape
    N = wq.shape[0]
    _check_weights(K, N, wq, s_w, 8, group_size)
    _check_out(out, (M, N))
    y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=x.device)
    need = workspace_bytes(M, N, K, group_size=group_size, bits=8)
    buf = ws if ws is not None else _workspace(need, x.device)
    wsp, wsn = (buf.data_ptr(), buf.numel()) if buf is not None else (None, 0)
    lib = load_library()
    xp = _dev(x, torch.float16, "x", 2)
    wp = _dev(wq, torch.int8, "wq", 2)
    sp = _dev(s_w, torch.float32, "s_w")
    yp = _dev(y, torch.float16, "y", 2)
    if M == 0 or N == 0:  # an empty output: nothing to compute
        return y
    if group_size == 0:
        st = lib.cider_w8a8_gemm_pc(xp, M, N, K, wp, sp, yp, wsp, wsn, _stream())
        _check("cider_w8a8_gemm_pc", st)
    else:
        st = lib.cider_w8a8_gemm_pg(xp, M, N, K, wp, sp, group_size, yp, wsp, wsn, _stream())
        _check("cider_w8a8_gemm_pg", st)
    return y


def linear(x: torch.Tensor, w: torch.Tensor, s_w: torch.Tensor, bits: int = 8,
           group_size: int = 0, out_dtype: torch.dtype | None = None,
           out: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """The quantized linear layer for fp16 or bf16 activations x [M,K]:
    w int8 [N,K] (bits 8) or packed uint8 [N,K/2] (bits 4), per-channel
    (group_size 0, s_w [N]) or per-group (s_w [N, K/gs]); y [M,N] in
    out_dtype (fp16 or bf16; default: x's dtype). M == 1 runs the GEMV."""
    if x.dtype not in _DTYPE_CODES:
        raise ValueError(f"x must be float16 or bfloat16, got {x.dtype}")
    out_dtype = out_dtype or x.dtype
    if out_dtype not in _DTYPE_CODES:
        raise ValueError(f"out_dtype must be float16 or bfloat16, got {out_dtype}")
    M, K = x.shape
    N = w.shape[0]
    _check_weights(K, N, w, s_w, bits, group_size)
    _check_out(out, (M, N))
    y = out if out is not None else torch.empty((M, N), dtype=out_dtype, device=x.device)
    need = workspace_bytes(M, N, K, group_size=group_size, bits=bits)
    buf = ws if ws is not None else _workspace(need, x.device)
    wsp, wsn = (buf.data_ptr(), buf.numel()) if buf is not None else (None, 0)
    wdt = torch.int8 if bits == 8 else torch.uint8
    lib = load_library()
    xp, wp = _dev(x, x.dtype, "x", 2), _dev(w, wdt, "w", 2)
    sp, yp = _dev(s_w, torch.float32, "s_w"), _dev(y, out_dtype, "y", 2)
    if M == 0 or N == 0:  # an empty output: nothing to compute
        return y
    st = lib.cider_linear(
        xp, _DTYPE_CODES[x.dtype], M, N, K, wp, bits, sp, group_size, yp,
        _DTYPE_CODES[out_dtype], wsp, wsn, _stream())
    _check("cider_linear", st)
    return y


def a16_gemv(x: torch.Tensor, w: torch.Tensor, s_w: torch.Tensor, bits: int = 8,
             group_size: int = 0, out_dtype: torch.dtype | None = None,
             out: torch.Tensor | None = None) -> torch.Tensor:
    """A16 decode product: x fp16/bf16 [K] (or [1,K]) used as it is against
    the dequantized weights (code * scale), fp32 accumulation; y [N]."""
    xv = x.reshape(-1)
    if xv.dtype not in _DTYPE_CODES:
        raise ValueError(f"x must be float16 or bfloat16, got {xv.dtype}")
    out_dtype = out_dtype or xv.dtype
    K = xv.numel()
    N = w.shape[0]
    _check_weights(K, N, w, s_w, bits, group_size)
    _check_out(out, (N,))
    y = out if out is not None else torch.empty((N,), dtype=out_dtype, device=x.device)
    wdt = torch.int8 if bits == 8 else torch.uint8
    lib = load_library()
    xp, wp = _dev(xv, xv.dtype, "x"), _dev(w, wdt, "w", 2)
    sp, yp = _dev(s_w, torch.float32, "s_w"), _dev(y, out_dtype, "y")
    if N == 0:  # no output channels: nothing to compute
        return y
    st = lib.cider_a16_gemv(
        xp, _DTYPE_CODES[xv.dtype], K, N, wp, bits, sp, group_size, yp,
        _DTYPE_CODES[out_dtype], _stream())
    _check("cider_a16_gemv", st)
    return y


def quantize_weight_clipped(w: torch.Tensor, group_size: int = 0, clip_percentile: float = 99.9,
                            bits: int = 8):
    """Weight preparation with percentile-clipped scales (fp16 or bf16 w
    [N,K]): returns (int8 [N,K] or packed uint8 [N,K/2], s_w fp32 [N] or
    [N, K/gs])."""
    if w.dtype not in _DTYPE_CODES:
        raise ValueError(f"w must be float16 or bfloat16, got {w.dtype}")
    N, K = w.shape
    G = 1 if group_size == 0 else K // group_size
    wq = torch.empty((N, K) if bits == 8 else (N, K // 2),
                     dtype=torch.int8 if bits == 8 else torch.uint8, device=w.device)
    s = torch.empty((N,) if group_size == 0 else (N, G), dtype=torch.float32, device=w.device)
    lib = load_library()
    wd = _dev(w, w.dtype, "w", 2)
    if N == 0:  # no output channels: nothing to compute
        return wq, s
    _check("cider_quantize_weight_clipped", lib.cider_quantize_weight_clipped(
        wd, _DTYPE_CODES[w.dtype], N, K, group_size, bits, float(clip_percentile),
        wq.data_ptr(), s.data_ptr(), _stream()))
    return wq, s


def quantize_act_any(x: torch.Tensor):
    """Per-token INT8 quantization of fp16 or bf16 activations: (q int8
    [M,K], s_a fp32 [M])."""
    if x.dtype not in _DTYPE_CODES:
        raise ValueError(f"x must be float16 or bfloat16, got {x.dtype}")
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    s = torch.empty((M,), dtype=torch.float32, device=x.device)
    lib = load_library()
    xp = _dev(x, x.dtype, "x", 2)
    if M == 0:  # no tokens: nothing to compute
        return q, s
    _check("cider_quantize_act_ex", lib.cider_quantize_act_ex(
        xp, _DTYPE_CODES[x.dtype], M, K, q.data_ptr(), s.data_ptr(), _stream()))
    return q, s


STATIC_SCRATCH_BYTES = 64 << 20


def w8a8_linear_noalloc(x: torch.Tensor, wq: torch.Tensor, s_w: torch.Tensor,
                        out: torch.Tensor) -> torch.Tensor:
    """W8A8 per-channel layer that allocates nothing: its scratch is a 64 MiB
    array inside the library, shared by all calls on the device (calls that
    overlap on the GPU race). ``out`` (fp16 [M,N]) must be provided."""
    M, K = x.shape
    N = wq.shape[0]
    _check_weights(K, N, wq, s_w, 8, 0)
    _check_out(out, (M, N))
    lib = load_library()
    xp, wp = _dev(x, torch.float16, "x", 2), _dev(wq, torch.int8, "wq", 2)
    sp, yp = _dev(s_w, torch.float32, "s_w"), _dev(out, torch.float16, "out", 2)
    if M == 0 or N == 0:  # an empty output: nothing to compute
        return out
    st = lib.cider_w8a8_gemm_pc_noalloc(xp, M, N, K, wp, sp, yp, _stream())
    _check("cider_w8a8_gemm_pc_noalloc", st)
    return out


def w4a8_linear(x: torch.Tensor, wp: torch.Tensor, s_w: torch.Tensor, group_size: int = 0,
                out: torch.Tensor | None = None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """W4A8 linear layer with packed INT4 weights wp [N, K/2]."""
    M, K = x.shape
    N = wp.shape[0]
    _check_weights(K, N, wp, s_w, 4, group_size)
    _check_out(out, (M, N))
    y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=x.device)
    need = workspace_bytes(M, N, K, group_size=group_size, bits=4)
    buf = ws if ws is not None else _workspace(need, x.device)
    wsp, wsn = (buf.data_ptr(), buf.numel()) if buf is not None else (None, 0)
    lib = load_library()
    xp, wpp = _dev(x, torch.float16, "x", 2), _dev(wp, torch.uint8, "wp", 2)
    sp, yp = _dev(s_w, torch.float32, "s_w"), _dev(y, torch.float16, "y", 2)
    if M == 0 or N == 0:  # an empty output: nothing to compute
        return y
    st = lib.cider_w4a8_gemm(xp, M, N, K, wpp, sp, group_size, yp, wsp, wsn,
                                        _stream())
    _check("cider_w4a8_gemm", st)
    return y


def int8_gemv(x: torch.Tensor, w: torch.Tensor, s_w: torch.Tensor, bits: int = 8,
              group_size: int = 0, out: torch.Tensor | None = None) -> torch.Tensor:
    """M = 1 GEMV: x fp16 [K] (or [1,K]); w int8 [N,K] (bits 8) or packed
    uint8 [N, K/2] (bits 4); returns y fp16 [N]."""
    xv = x.reshape(-1)
    K = xv.numel()
    N = w.shape[0]
    _check_weights(K, N, w, s_w, bits, group_size)
    _check_out(out, (N,))
    y = out if out is not None else torch.empty((N,), dtype=torch.float16, device=x.device)
    wdt = torch.int8 if bits == 8 else torch.uint8
    lib = load_library()
    xp, wp = _dev(xv, torch.float16, "x"), _dev(w, wdt, "w", 2)
    sp, yp = _dev(s_w, torch.float32, "s_w"), _dev(y, torch.float16, "y")
    if N == 0:  # no output channels: nothing to compute
        return y
    st = lib.cider_int8_gemv(xp, K, N, wp, sp, bits, group_size, yp, _stream())
    _check("cider_int8_gemv", st)
    return y


def act_image(x: torch.Tensor, a_img: torch.Tensor | None = None,
              s_a: torch.Tensor | None = None):
    """Stage 1 of the GEMM path: x fp16 [M,K] -> (codes as fp16 integers
    [M,K], s_a fp32 [M])."""
    M, K = x.shape
    _check_out(a_img, (M, K), "a_img")
    _check_out(s_a, (M,), "s_a")
    a_img = a_img if a_img is not None else torch.empty((M, K), dtype=torch.float16,
                                                        device=x.device)
    s_a = s_a if s_a is not None else torch.empty((M,), dtype=torch.float32, device=x.device)
    _check("cider_act_image", load_library().cider_act_image(
        _dev(x, torch.float16, "x", 2), M, K, _dev(a_img, torch.float16, "a_img", 2),
        _dev(s_a, torch.float32, "s_a"), _stream()))
    return a_img, s_a


def weight_image(w: torch.Tensor, K: int, bits: int = 8, b_img: torch.Tensor | None = None):
    """Stage 2: INT8 [N,K] or packed INT4 [N,K/2] codes -> fp16 integers [N,K]."""
    N = w.shape[0]
    if bits not in (8, 4) or w.dim() != 2 or w.shape[1] != (K if bits == 8 else K // 2) \
            or (bits == 4 and K % 2):
        raise ValueError(f"w of shape {tuple(w.shape)} does not hold {bits}-bit codes of "
                         f"K = {K}")
    _check_out(b_img, (N, K), "b_img")
    b_img = b_img if b_img is not None else torch.empty((N, K), dtype=torch.float16,
                                                        device=w.device)
    wdt = torch.int8 if bits == 8 else torch.uint8
    _check("cider_weight_image", load_library().cider_weight_image(
        _dev(w, wdt, "w", 2), N, K, bits, _dev(b_img, torch.float16, "b_img", 2), _stream()))
    return b_img


def gemm_images(a_img: torch.Tensor, s_a: torch.Tensor, b_img: torch.Tensor,
                s_w: torch.Tensor, group_size: int = 0,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """Stage 3: tensor-core GEMM + fused dequant on the fp16 code images."""
    M, K = a_img.shape
    N = b_img.shape[0]
    _check_out(s_a, (M,), "s_a")
    _check_weights(K, N, b_img, s_w, 8, group_size)  # the fp16 image is [N, K]
    _check_out(out, (M, N))
    y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=a_img.device)
    _check("cider_gemm_images", load_library().cider_gemm_images(
        _dev(a_img, torch.float16, "a_img", 2), _dev(s_a, torch.float32, "s_a"),
        _dev(b_img, torch.float16, "b_img", 2), _dev(s_w, torch.float32, "s_w"), M, N, K,
        group_size, _dev(y, torch.float16, "y", 2), _stream()))
    return y


def raw_gemm_s32(q: torch.Tensor, w: torch.Tensor, K: int, bits: int = 8,
                  group_size: int = 0) -> torch.Tensor:
    """Test hook: raw int32 products of the tensor-core engine on INT8 codes
    q [M,K] and weights (int8 [N,K] or packed [N,K/2]); [M,N] totals or
    [M,N,K/gs] per-group partials."""
    M = q.shape[0]
    N = w.shape[0]
    if q.dim() != 2 or q.shape[1] != K:
        raise ValueError(f"q must be [M, {K}], got shape {tuple(q.shape)}")
    if bits not in (8, 4) or w.dim() != 2 or w.shape[1] != (K if bits == 8 else K // 2):
        raise ValueError(f"w of shape {tuple(w.shape)} does not hold {bits}-bit codes of "
                         f"K = {K}")
    if group_size < 0 or (group_size and K % group_size):
        raise ValueError(f"group_size {group_size} must be 0 or a divisor of K = {K}")
    G = 1 if group_size == 0 else K // group_size
    out = torch.empty((M, N) if group_size == 0 else (M, N, G), dtype=torch.int32,
                      device=q.device)
    need = workspace_bytes(max(M, 2), N, K, group_size=group_size, bits=bits)
    buf = _workspace(need, q.device)
    wdt = torch.int8 if bits == 8 else torch.uint8
    st = load_library().cider_test_gemm_s32(
        _dev(q, torch.int8, "q", 2), _dev(w, wdt, "w", 2), M, N, K, bits, group_size,
        out.data_ptr(), buf.data_ptr(), buf.numel(), _stream())
    _check("cider_test_gemm_s32", st)
    return out


def device_status() -> tuple[int, int]:
    """Synchronizes the current stream; returns (status, wait site) of the
    device status word and clears it."""
    site = ctypes.c_uint32(0)
    st = load_library().cider_device_status(_stream(), ctypes.byref(site))
    return int(st), int(site.value)


def wait_timeout_probe(timeout_ns: int) -> None:
    """Test hook: a kernel whose bounded mbarrier wait is never satisfied."""
    _check("cider_test_wait_timeout",
           load_library().cider_test_wait_timeout(int(timeout_ns), _stream()))


# ---------------------------------------------------------------------------
# linears that read the same input (q/k/v, gate/up): one call
# ---------------------------------------------------------------------------

def int8_mma_loop(blocks: int, iters: int, device="cuda") -> torch.Tensor:
    """Measurement hook: `blocks` x 4 warps, each 8 * iters legacy INT8 MMAs
    (8192 operations each); returns the sink tensor (time it with events)."""
    sink = torch.empty(blocks * 128, dtype=torch.int32, device=device)
    _check("cider_test_int8_mma_loop",
           load_library().cider_test_int8_mma_loop(blocks, iters, sink.data_ptr(), _stream()))
    return sink


def read_bytes(t: torch.Tensor, sink: torch.Tensor) -> None:
    """Measurement hook: a plain streaming read of t's bytes, launched as the
    GEMV is; sink: uint32/int32 of at least 2 x (number of SMs) elements."""
    nbytes = t.numel() * t.element_size()
    _dev(t, t.dtype, "t")
    _check("cider_test_read_bytes",
           load_library().cider_test_read_bytes(t.data_ptr(), nbytes, sink.data_ptr(), _stream()))


def concat_linears(weights):
    """Offline, at weight-prep time: stacks the weight rows and scale rows of
    linears that read the same input (e.g. q, k, v) into one layer, so one
    call quantizes the input once and runs one GEMM with N = sum of the N's.
    Output channels are independent, so each linear's columns of the fused
    output equal that linear's own output bit for bit. `weights` is a list of
    (w, s_w) with the same K, bit width and group size. Returns (w, s_w,
    sizes); split_columns(y, sizes) recovers the per-linear outputs."""
    ws = [w for w, _ in weights]
    ss = [s for _, s in weights]
    if len({w.shape[1] for w in ws}) != 1 or len({w.dtype for w in ws}) != 1:
        raise ValueError("concat_linears: the linears must share K and the weight format")
    if len({tuple(s.shape[1:]) for s in ss}) != 1:
        raise ValueError("concat_linears: the linears must share the scale granularity")
    return torch.cat(ws, 0).contiguous(), torch.cat(ss, 0).contiguous(), [w.shape[0] for w in ws]


def split_columns(y: torch.Tensor, sizes):
    """The per-linear outputs of a fused call (column views of y)."""
    return list(torch.split(y, list(sizes), dim=1))


# ---------------------------------------------------------------------------
# column-parallel split (several GPUs, one process each)
# ---------------------------------------------------------------------------

def column_shard(N: int, world: int, rank: int, align: int = 128) -> tuple[int, int]:
    """Output channels [n0, n1) that rank `rank` of `world` owns when the
    layer is split by output channel (its weight rows and scale rows): a
    contiguous range, balanced in units of `align` channels (the GEMM's tile
    width), the remainder going to the first ranks; the last rank also takes
    the ragged end. Output channels are independent, so the split needs no
    reduction, only a gather of the columns when a consumer needs all of y."""
    if N <= 0 or world <= 0 or not 0 <= rank < world or align <= 0:
        raise ValueError("column_shard: bad N / world / rank / align")
    units = (N + align - 1) // align
    base, extra = divmod(units, world)
    u0 = rank * base + min(rank, extra)
    u1 = u0 + base + (1 if rank < extra else 0)
    return min(N, u0 * align), min(N, u1 * align)


def gather_columns(y_shard: torch.Tensor, N: int, world: int, align: int = 128,
                   group=None) -> torch.Tensor:
    """All-gathers the column shards of y ([M, n1 - n0] on every rank, split
    by column_shard) into the full [M, N] on every rank (torch.distributed;
    shards are padded to the widest for the collective)."""
    import torch.distributed as dist
    M = y_shard.shape[0]
    widths = [column_shard(N, world, r, align) for r in range(world)]
    wmax = max(n1 - n0 for n0, n1 in widths)
    pad = torch.zeros((M, wmax), dtype=y_shard.dtype, device=y_shard.device)
    pad[:, :y_shard.shape[1]] = y_shard
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad.contiguous(), group=group)
    return torch.cat([parts[r][:, :n1 - n0] for r, (n0, n1) in enumerate(widths)], dim=1)


def column_parallel_w8a8_linear(x: torch.Tensor, wq: torch.Tensor, s_w: torch.Tensor,
                                group_size: int = 0, world: int = 1, rank: int = 0,
                                group=None) -> torch.Tensor:
    """The W8A8 layer split by output channel over `world` ranks: this rank
    runs its weight rows (column_shard) through w8a8_linear and the shards
    are all-gathered into the full y. wq / s_w are the full tensors; only this
    rank's rows are read."""
    N = wq.shape[0]
    n0, n1 = column_shard(N, world, rank)
    if n1 > n0:
        y = w8a8_linear(x, wq[n0:n1], s_w[n0:n1], group_size)
    else:  # more ranks than 128-channel tiles: nothing to compute here
        y = torch.empty((x.shape[0], 0), dtype=torch.float16, device=x.device)
    return y if world == 1 else gather_columns(y, N, world, group=group)


# ---------------------------------------------------------------------------
# the pages' layer-level names (Cider README, "Layer-level API" and
# "Low-Level API"), over the calls above
# ---------------------------------------------------------------------------

def is_available() -> bool:
    """True when the library loads and a B300-class GPU (compute capability
    10.3, the target of the library's sm_103a kernels) is visible."""
    try:
        load_library()
    except (OSError, RuntimeError):
        return False
    return torch.cuda.is_available() and torch.cuda.get_device_capability() == (10, 3)


def perchannel_linear(x: torch.Tensor, w_int8: torch.Tensor, scale: torch.Tensor,
                      out: torch.Tensor | None = None) -> torch.Tensor:
    """Per-channel W8A8 linear layer: w8a8_linear with group size 0."""
    return w8a8_linear(x, w_int8, scale, 0, out=out)


class _QuantLinear(torch.nn.Module):
    """A linear layer without bias over pre-quantized weights: x [..., K]
    (fp16 or bf16) -> y [..., N] in x's dtype through `linear` (leading
    dimensions flattened into tokens; one token runs the GEMV)."""

    bits = 8

    def __init__(self, weights: torch.Tensor, scale_w: torch.Tensor, group_size: int = 0,
                 in_features: int | None = None, out_features: int | None = None):
        super().__init__()
        N = weights.shape[0]
        K = weights.shape[1] * (8 // self.bits)
        if in_features is not None and in_features != K:
            raise ValueError(f"in_features {in_features} != weight columns {K}")
        if out_features is not None and out_features != N:
            raise ValueError(f"out_features {out_features} != weight rows {N}")
        if group_size < 0 or (group_size and K % group_size):
            raise ValueError(f"group_size {group_size} does not divide in_features {K}")
        want_scales = (N,) if group_size == 0 else (N, K // group_size)
        if tuple(scale_w.shape) != want_scales:
            raise ValueError(f"scale_w must have shape {want_scales}, got {tuple(scale_w.shape)}")
        self.in_features, self.out_features, self.group_size = K, N, group_size
        self.register_buffer("weight", weights)
        self.register_buffer("scale_w", scale_w)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.shape[-1] != self.in_features:
            raise ValueError(f"x has {x.shape[-1]} features, the layer {self.in_features}")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features)
        if x2.shape[0] == 0:
            return x.new_empty(*lead, self.out_features)
        y = linear(x2.contiguous(), self.weight, self.scale_w, self.bits, self.group_size)
        return y.reshape(*lead, self.out_features)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"group_size={self.group_size}")


class W8A8Linear(_QuantLinear):
    """INT8 weights [N, K] (w_int8) with per-channel (group_size 0, scale_w
    [N]) or per-group (scale_w [N, K/group_size]) scales; activations
    quantized per token inside the call."""

    bits = 8

    def __init__(self, w_int8: torch.Tensor, scale_w: torch.Tensor, group_size: int = 0,
                 in_features: int | None = None, out_features: int | None = None):
        super().__init__(w_int8, scale_w, group_size, in_features, out_features)

    @classmethod
    def from_weights(cls, W: torch.Tensor, group_size: int = 0) -> "W8A8Linear":
        """Quantizes fp16 weights W [N, K] (on the GPU) and builds the layer."""
        wq, s = quantize_weight_int8(W, group_size)
        return cls(wq, s, group_size)


class W4A8Linear(_QuantLinear):
    """Packed INT4 weights [N, K/2] (two codes per byte) with per-column
    (group_size 0) or per-group scales; activations quantized per token."""

    bits = 4

    def __init__(self, packed_w4: torch.Tensor, scale_w: torch.Tensor, group_size: int = 0,
                 in_features: int | None = None, out_features: int | None = None):
        super().__init__(packed_w4, scale_w, group_size, in_features, out_features)

    @classmethod
    def from_weights(cls, W: torch.Tensor, group_size: int = 0) -> "W4A8Linear":
        """Quantizes and packs fp16 weights W [N, K] (on the GPU) and builds the layer."""
        wp, s = pack_weight_int4(W, group_size)
        return cls(wp, s, group_size)
