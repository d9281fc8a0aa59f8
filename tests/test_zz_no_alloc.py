"""The no-allocation variant of the W8A8 per-channel layer.

cider_w8a8_gemm_pc_noalloc serves callers that cannot call cudaMalloc (for
example code under a framework that owns every device allocation, or a
latency-critical loop that must not synchronize on an allocation): its
scratch is a fixed 64 MiB array compiled into the library instead of a
caller workspace. These tests call it through the C ABI and check, on two
calls in a row with different problem sizes (so the second call runs over
the first call's leftovers in the shared array), that it produces the same
output as cider_w8a8_gemm_pc with a workspace, within the 1-ulp fp16 bar
the other parity tests use; and that a problem larger than the array is
refused before anything runs. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth
import w4a8_quantized_gemm_int8_b300 as cider
from gpu_helpers import f16_ulp_distance

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, x, wq, s_w, y):
    M, K = x.shape
    N = wq.shape[0]
    return lib.cider_w8a8_gemm_pc_noalloc(x.data_ptr(), M, N, K, wq.data_ptr(), s_w.data_ptr(),
                                          y.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = cider.load_library()
    torch.cuda.set_device(0)
    for M, N, K, seed in [(300, 1040, 2560, 11), (129, 264, 1088, 12)]:
        li = synth.linear_inputs(M, N, K, n_out=4, seed=seed)
        x = li.x.to("cuda:0")
        wq, s_w = cider.quantize_weight_int8(li.w.to("cuda:0"), 0)
        ws = torch.empty(cider.workspace_bytes(M, N, K, 8, 0), dtype=torch.uint8, device="cuda:0")
        y_ref = cider.w8a8_linear(x, wq, s_w, 0, ws=ws)
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda:0")
        assert _call_noalloc(lib, x, wq, s_w, y) == cider.CIDER_OK
        torch.cuda.synchronize()
        d = f16_ulp_distance(y.cpu().numpy(), y_ref.cpu().numpy())
        assert d.max() <= 1, f"M={M} N={N} K={K}: {int((d > 1).sum())} outputs beyond 1 ulp"
    st, site = cider.device_status()
    assert st == cider.CIDER_OK, f"device status {st} at {site:#x}"


def test_noalloc_rejects_problems_larger_than_the_array():
    lib = cider.load_library()
    torch.cuda.set_device(0)
    M, N, K = 16384, 256, 2560  # the activation image alone is 80 MiB (> 64 MiB)
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda:0")
    wq = torch.zeros((N, K), dtype=torch.int8, device="cuda:0")
    s_w = torch.ones((N,), dtype=torch.float32, device="cuda:0")
    y = torch.full((M, N), 7.0, dtype=torch.float16, device="cuda:0")
    assert _call_noalloc(lib, x, wq, s_w, y) == 5  # CIDER_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())  # nothing was enqueued
