"""Weight preparation with percentile-clipped scales (README "LLM
Quantization" note, clip_percentile): GPU codes and scales against the
oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
import w4a8_quantized_gemm_int8_b300 as cider
from gpu_helpers import cuda, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wdt", ["f16", "bf16"])
@pytest.mark.parametrize("pct", [99.9, 99.0, 50.0, 100.0])
@pytest.mark.parametrize("bits,gs", [(8, 0), (8, 64), (8, 128), (4, 0), (4, 128)])
@pytest.mark.parametrize("N,K", [(300, 2560), (37, 1024)])
def test_clipped_weight_prep_bitexact(N, K, bits, gs, pct, wdt):
    w32 = synth.weights(N, K, synth.generator(N + K + gs)).float().numpy()
    w32[:, ::97] *= 30.0  # a few outliers per row for the clip to cut
    if wdt == "f16":
        wh = w32.astype(np.float16)
        wt, wo = torch.from_numpy(wh), wh
    else:
        wb = oracle.float_to_bf16(w32)
        wt, wo = torch.from_numpy(wb.view(np.int16)).view(torch.bfloat16), wb
    q, s = cider.quantize_weight_clipped(cuda(wt), gs, pct, bits)
    qo, so = oracle.quantize_weight_clipped(wo, gs, pct, bits, w_dtype=wdt)
    assert np.array_equal(host(s).view(np.uint32), np.asarray(so).view(np.uint32))
    assert np.array_equal(host(q), qo)


@pytest.mark.parametrize("bits,gs", [(8, 0), (8, 64), (4, 128)])
def test_clipped_blocks_whose_percentile_is_zero(bits, gs):
    """Blocks where more than p % of |w| is zero: the clip is 0, so the scale
    is 0 and every code 0, non-zero weights included (the oracle's pinned
    reading); the other blocks keep their ordinary clipped codes."""
    N, K = 64, 1024
    w = synth.weights(N, K, synth.generator(71 + gs)).float().numpy()
    keep = np.random.default_rng(5).random((N, K)) < 0.3
    keep[: N // 2] = True  # half the rows stay dense
    wh = np.where(keep, w, 0.0).astype(np.float16)
    q, s = cider.quantize_weight_clipped(cuda(torch.from_numpy(wh)), gs, 50.0, bits)
    qo, so = oracle.quantize_weight_clipped(wh, gs, 50.0, bits)
    assert (np.asarray(so)[N // 2:] == 0).all()  # the sparse rows' blocks clip to 0
    assert np.array_equal(host(s).view(np.uint32), np.asarray(so).view(np.uint32))
    assert np.array_equal(host(q), qo)
