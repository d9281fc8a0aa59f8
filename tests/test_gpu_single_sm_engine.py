"""The single-SM engine for per-channel layers of at most 128 tokens.

Layer calls of at most 128 tokens normally run on SM pairs (the weights as
the MMA's M side); CIDER_GEMM_ENGINE=single keeps them on one SM per CTA,
whose per-channel path splits the k-blocks of all tiles among the SMs
(stream-K) and sums shared tiles in a fix-up launch. The variable is read
once per process, so each case runs in a child process that writes its
output; the parent compares it with the oracle, bit for bit (the bar of the
other parity tests).
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import assert_f16_within_1ulp

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[2])
import synth, w4a8_quantized_gemm_int8_b300 as cider
M, N, K, bits = (int(v) for v in sys.argv[3:7])
wq = np.load(sys.argv[7]); s = np.load(sys.argv[8])
li = synth.linear_inputs(M, N, K, n_out=4, seed=M + K + bits)
x = li.x.cuda()
f = cider.w8a8_linear if bits == 8 else cider.w4a8_linear
y = f(x, torch.from_numpy(wq).cuda(), torch.from_numpy(s).cuda(), 0)
np.save(sys.argv[9], y.cpu().numpy())
"""


# Shapes where the single-SM engine takes stream-K (runs of about 17
# k-blocks crossing tile boundaries, tiles shared by two or three CTAs) and
# one where it keeps whole tiles.
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("M,N,K", [(32, 5120, 4096), (77, 2560, 8192), (128, 1280, 2560),
                                   (9, 10240, 1024)])
def test_single_sm_engine_per_channel(M, N, K, bits, tmp_path):
    li = synth.linear_inputs(M, N, K, n_out=4, seed=M + K + bits)
    x, w = li.x.numpy(), li.w.numpy()
    if bits == 8:
        wq, s = oracle.quantize_weight_int8(w, 0)
        ref = oracle.w8a8_linear(x, wq, s, 0)
    else:
        wq, s = oracle.pack_weight_int4(w, 0)
        ref = oracle.w4a8_linear(x, wq, s, 0)
    np.save(tmp_path / "wq.npy", wq)
    np.save(tmp_path / "s.npy", np.asarray(s))
    env = dict(os.environ, CIDER_GEMM_ENGINE="single")
    repo = os.path.dirname(HERE)
    r = subprocess.run([sys.executable, "-c", CHILD, HERE, repo, str(M), str(N), str(K),
                        str(bits), str(tmp_path / "wq.npy"), str(tmp_path / "s.npy"),
                        str(tmp_path / "y.npy")], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert_f16_within_1ulp(np.load(tmp_path / "y.npy"), ref, f"single-SM w{bits}")
