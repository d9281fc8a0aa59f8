"""Host-side checks of the C-ABI library that need no GPU: it loads, it
exports every symbol include/cider.h declares, and argument validation that
runs before any CUDA call answers as documented."""
import ctypes
import os
import re

import pytest

import w4a8_quantized_gemm_int8_b300 as cider
from w4a8_quantized_gemm_int8_b300 import build as cbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return cider.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "cider.h")).read()
    return sorted(set(re.findall(r"CIDER_API\s+[\w\s\*]*?\b(cider_\w+)\s*\(", src)))


def test_header_declares_binding_names():
    assert _declared() == sorted(cider.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    # nothing else leaks out as a C symbol with the prefix
    out = os.popen(f"nm -D --defined-only {cider.LIB_PATH}").read()
    exported = sorted(set(re.findall(r" T (cider_\w+)", out)))
    assert exported == _declared()


def test_status_strings_and_version(lib):
    assert cider.abi_version() == 3
    for code, name in [(0, "CIDER_OK"), (1, "CIDER_ERR_INVALID_ARG"),
                       (2, "CIDER_ERR_UNSUPPORTED"), (3, "CIDER_ERR_CUDA"),
                       (4, "CIDER_ERR_TIMEOUT"), (5, "CIDER_ERR_WORKSPACE"), (99, "CIDER_ERR_UNKNOWN")]:
        assert cider.status_string(code) == name


def test_workspace_bytes(lib):
    assert cider.workspace_bytes(1, 10240, 2560) == 0   # GEMV path
    assert cider.workspace_bytes(0, 16, 16) == 0
    assert cider.workspace_bytes(4, 16, 16, bits=3) == 0
    # per channel, SM pairs: activation image, token scales, fp16 weight image
    n = cider.workspace_bytes(4096, 10240, 2560)
    assert n == 2 * 4096 * 2560 + 4 * 4096 + 2 * 10240 * 2560
    assert n % 256 == 0
    # INT8 per group, SM pairs: the weights are widened on chip (no image)
    g = cider.workspace_bytes(4096, 2560, 10240, group_size=64, bits=8)
    assert g == 2 * 4096 * 10240 + 4 * 4096
    # W4A8 per group, SM pairs: weight image and a group-major copy of the scales
    w4 = cider.workspace_bytes(4096, 2560, 10240, group_size=128, bits=4)
    assert w4 == 2 * 4096 * 10240 + 4 * 4096 + 2 * 2560 * 10240 + 4 * 2560 * (10240 // 128)
    # few-token per-channel layers: activation image, token scales and the
    # stream-K partial tiles (2 per CTA, at most 160 CTAs, rows M rounded up to 32)
    a256 = lambda v: (v + 255) // 256 * 256
    assert cider.workspace_bytes(128, 10240, 2560) == \
        a256(128 * 2560 * 2) + a256(128 * 4) + a256(160 * 2 * 128 * 128 * 4)
    assert cider.workspace_bytes(40, 10240, 2560, bits=4) == \
        a256(40 * 2560 * 2) + a256(40 * 4) + a256(160 * 2 * 64 * 128 * 4)
    # few tokens, per group: activation image and the group-major scale copy
    s = cider.workspace_bytes(64, 2560, 10240, group_size=64, bits=8)
    assert s == 2 * 64 * 10240 + 256 + 4 * 2560 * (10240 // 64)
    assert cider.workspace_bytes(4096, 2560, 10240, group_size=100, bits=8) == 0  # 100 does not divide K


def test_null_and_size_checks_precede_cuda(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: checks fail first
    assert lib.cider_quantize_act(None, 4, 16, p, p, None) == 1
    assert lib.cider_quantize_act(p, 0, 16, p, p, None) == 1
    assert lib.cider_w8a8_gemm_pc(p, 4, 16, 16, None, p, p, p, 1 << 20, None) == 1
    assert lib.cider_w8a8_gemm_pc(p, -1, 16, 16, p, p, p, p, 1 << 20, None) == 1
    assert lib.cider_w8a8_gemm_pg(p, 4, 16, 128, p, p, 0, p, p, 1 << 20, None) == 1
    assert lib.cider_int8_gemv(p, 16, 16, p, p, 5, 0, p, None) == 1
    assert lib.cider_test_wait_timeout(0, None) == 1
    assert lib.cider_test_gemm_s32(p, p, 4, 4, 64, 7, 0, p, p, 1 << 20, None) == 1


def test_element_type_checks_precede_cuda(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: checks fail first
    # unknown activation / output element types, unknown weight width
    assert lib.cider_linear(p, 2, 4, 16, 16, p, 8, p, 0, p, 0, p, 1 << 20, None) == 1
    assert lib.cider_linear(p, 0, 4, 16, 16, p, 8, p, 0, p, -1, p, 1 << 20, None) == 1
    assert lib.cider_linear(p, 1, 4, 16, 16, p, 5, p, 0, p, 1, p, 1 << 20, None) == 1
    assert lib.cider_linear(None, 1, 4, 16, 16, p, 8, p, 0, p, 1, p, 1 << 20, None) == 1
    assert lib.cider_quantize_act_ex(p, 3, 4, 16, p, p, None) == 1
    assert lib.cider_quantize_act_ex(None, 1, 4, 16, p, p, None) == 1
    assert lib.cider_quantize_act_ex(p, 1, 0, 16, p, p, None) == 1


def test_a16_gemv_checks_precede_cuda(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: checks fail first
    assert lib.cider_a16_gemv(None, 0, 64, 16, p, 8, p, 0, p, 0, None) == 1
    assert lib.cider_a16_gemv(p, 0, 0, 16, p, 8, p, 0, p, 0, None) == 1
    assert lib.cider_a16_gemv(p, 0, 64, 16, p, 6, p, 0, p, 0, None) == 1
    assert lib.cider_a16_gemv(p, 2, 64, 16, p, 8, p, 0, p, 0, None) == 1
    assert lib.cider_a16_gemv(p, 0, 64, 16, p, 8, p, 0, p, 3, None) == 1


def test_clipped_weight_prep_checks_precede_cuda(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: checks fail first
    assert lib.cider_quantize_weight_clipped(p, 0, 4, 64, 0, 8, 0.0, p, p, None) == 1
    assert lib.cider_quantize_weight_clipped(p, 0, 4, 64, 0, 8, 100.5, p, p, None) == 1
    assert lib.cider_quantize_weight_clipped(p, 0, 4, 64, 0, 5, 99.9, p, p, None) == 1
    assert lib.cider_quantize_weight_clipped(None, 0, 4, 64, 0, 8, 99.9, p, p, None) == 1
    assert lib.cider_quantize_weight_clipped(p, 0, 4, 64, 60, 8, 99.9, p, p, None) == 2


_C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "cider.h"

int main(void) {
    /* host-only calls: version, status strings, workspace sizing, and the
       argument checks that answer before any CUDA call */
    /* arguments in the documented order: M, N, K, group_size, bits */
    size_t ws = cider_workspace_bytes(4096, 10240, 2560, 0, 8);
    size_t ws_pg = cider_workspace_bytes(4096, 2560, 10240, 64, 4);
    cider_status st = cider_w8a8_gemm_pc(NULL, 4, 8, 16, NULL, NULL, NULL, NULL, 0, NULL);
    printf("%d %s %zu %zu %d\n", cider_abi_version(), cider_status_string(CIDER_OK), ws, ws_pg,
           (int)st);
    return st == CIDER_ERR_INVALID_ARG ? 0 : 1;
}
"""


def test_header_is_plain_c_and_links(lib, tmp_path):
    """The header compiles as C99 (no C++ or CUDA types in the signatures),
    and a C program links against the library and calls it."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(_C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(cider.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lcider", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == lib.cider_abi_version()
    assert int(out[-3]) == cider.workspace_bytes(4096, 10240, 2560, group_size=0, bits=8)
    assert int(out[-2]) == cider.workspace_bytes(4096, 2560, 10240, group_size=64, bits=4)
    assert int(out[-2]) > int(out[-3]) > 0
    assert int(out[-1]) == cider.CIDER_ERR_INVALID_ARG
