"""The no-allocation variant of the W8A8 per-channel layer.

cider_w8a8_gemm_pc_noalloc serves callers that cannot call cudaMalloc (for
example code under a framework that owns every device allocation, or a
latency-critical loop that must not synchronize on an allocation): its
scratch is a fixed 64 MiB array compiled into the library instead of a
caller workspace. These tests call it through the C ABI on calls in a row of
different problem sizes (so each call runs over the previous call's leftovers
in the shared array), covering both GEMM engines (SM pairs for M > 128, one
SM for M <= 128) and M = 1 (the tensor-core GEMM, not the GEMV), and check
every output against the CPU oracle (bit-identical, the bar of the other
parity tests) and against cider_w8a8_gemm_pc with a workspace; and that a
problem larger than the array is refused before anything runs. This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a8_quantized_gemm_int8_b300 as cider
from gpu_helpers import assert_f16_within_1ulp

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, x, wq, s_w, y):
    M, K = x.shape
    N = wq.shape[0]
    return lib.cider_w8a8_gemm_pc_noalloc(x.data_ptr(), M, N, K, wq.data_ptr(), s_w.data_ptr(),
                                          y.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_oracle_and_workspace_entry_point_on_calls_in_a_row():
    lib = cider.load_library()
    torch.cuda.set_device(0)
    # SM pairs, single SM, M = 1, then SM pairs again over the leftovers
    for M, N, K, seed in [(300, 1040, 2560, 11), (64, 1040, 2560, 13), (1, 1040, 2560, 14),
                          (129, 264, 1088, 12)]:
        li = synth.linear_inputs(M, N, K, n_out=4, seed=seed)
        wq_h, s_h = oracle.quantize_weight_int8(li.w.numpy(), 0)
        ref = oracle.w8a8_linear(li.x.numpy(), wq_h, s_h, 0)
        x = li.x.to("cuda:0")
        wq, s_w = torch.from_numpy(wq_h).cuda(), torch.from_numpy(s_h).cuda()
        ws = torch.empty(max(1, cider.workspace_bytes(M, N, K, group_size=0, bits=8)),
                         dtype=torch.uint8, device="cuda:0")
        y_ws = cider.w8a8_linear(x, wq, s_w, 0, ws=ws)  # M = 1: the GEMV
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda:0")
        assert _call_noalloc(lib, x, wq, s_w, y) == cider.CIDER_OK
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert_f16_within_1ulp(got, ref, f"noalloc M={M} N={N} K={K}")
        assert np.array_equal(got.view(np.uint16), y_ws.cpu().numpy().view(np.uint16)), M
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
