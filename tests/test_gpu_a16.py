"""A16 decode matrix-vector product (weight-only dequantization, README
"Metal Kernel Pipeline", decode): CUDA path against the oracle's float64
value. The product is a floating-point sum, so the bar is an error bound
derived from the arithmetic instead of bit equality:

  |y_gpu - y| <= 0.5 ulp_out(|y| + E) + E,   E = (K + 2) 2^-24 S,
  S = sum_g |s_g| sum_{k in g} |x_k code_k|

(fp32 accumulation of K products in any order, one rounding for the scale
product and one for the group sum, then one rounding to the output type).
The tests also require almost every output within 1 ulp, a check that the
bound is not met by a loose kernel."""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a8_quantized_gemm_int8_b300 as cider
from gpu_helpers import cuda, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cider.load_library()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()
    st, site = cider.device_status()
    assert st == cider.CIDER_OK, f"device status {st} at site {site:#x}"


def _ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the output format at magnitude v (v >= 0)."""
    mant, emin = (10, -14) if dtype == "f16" else (7, -126)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** emin)))
    return 2.0 ** (np.maximum(e, emin) - mant)


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("xdt", ["f16", "bf16"])
@pytest.mark.parametrize("bits,gs", [(8, 0), (8, 64), (4, 0), (4, 128)])
@pytest.mark.parametrize("N,K", [(10240, 2560), (2560, 10240), (37, 512)])
def test_a16_gemv_within_bound(N, K, bits, gs, xdt, out):
    g = synth.generator(N + K + bits + gs)
    x32 = synth.activations(1, K, 4, g).float().numpy()[0] * 2
    w = synth.weights(N, K, g).numpy()
    if bits == 8:
        wdev, s = oracle.quantize_weight_int8(w, gs)
        codes = wdev.astype(np.float64)
    else:
        wdev, s = oracle.pack_weight_int4(w, gs)
        codes = oracle.unpack_int4(wdev, K).astype(np.float64)
    if xdt == "f16":
        xh = x32.astype(np.float16)
        xt, xv = torch.from_numpy(xh), xh.astype(np.float64)
        xo = xh
    else:
        xb = oracle.float_to_bf16(x32)
        xt = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
        xv = oracle.bf16_to_float(xb).astype(np.float64)
        xo = xb
    y = cider.a16_gemv(cuda(xt), cuda(torch.from_numpy(wdev)), cuda(torch.from_numpy(s)),
                       bits, gs, out_dtype=torch.float16 if out == "f16" else torch.bfloat16)
    yg = host(y.float()).astype(np.float64)
    ref = oracle.a16_gemv(xo, wdev, s, bits, gs, x_dtype=xdt)
    G = 1 if gs == 0 else K // gs
    sc = np.repeat(np.abs(np.asarray(s, np.float64).reshape(N, G)), K // G, axis=1)
    S = (np.abs(codes) * sc) @ np.abs(xv)
    E = (K + 2) * 2.0 ** -24 * S
    err = np.abs(yg - ref)
    bound = 0.5 * _ulp(np.abs(ref) + E, out) + E
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"
    within_1ulp = np.mean(err <= _ulp(np.abs(ref), out))
    assert within_1ulp >= 0.99, within_1ulp
