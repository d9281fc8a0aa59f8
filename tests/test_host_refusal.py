"""The product path has no CPU fallback: every public call refuses host
tensors with an error before any work, and a missing library raises instead
of degrading (no GPU needed)."""
import pytest
import torch

import w4a8_quantized_gemm_int8_b300 as cider


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cider.load_library()


M, N, K = 4, 32, 64
x = torch.zeros(M, K, dtype=torch.float16)
w = torch.zeros(N, K, dtype=torch.float16)
wq = torch.zeros(N, K, dtype=torch.int8)
wp = torch.zeros(N, K // 2, dtype=torch.uint8)
s_pc = torch.ones(N, dtype=torch.float32)
s_pg = torch.ones(N, K // 64, dtype=torch.float32)

CALLS = {
    "quantize_act": lambda: cider.quantize_act(x),
    "quantize_act_any": lambda: cider.quantize_act_any(x.bfloat16()),
    "quantize_weight_int8": lambda: cider.quantize_weight_int8(w, 64),
    "pack_weight_int4": lambda: cider.pack_weight_int4(w, 64),
    "quantize_weight_clipped": lambda: cider.quantize_weight_clipped(w, 64),
    "w8a8_linear_pc": lambda: cider.w8a8_linear(x, wq, s_pc),
    "w8a8_linear_pg": lambda: cider.w8a8_linear(x, wq, s_pg, 64),
    "w4a8_linear": lambda: cider.w4a8_linear(x, wp, s_pg, 64),
    "linear": lambda: cider.linear(x, wq, s_pc),
    "linear_bf16": lambda: cider.linear(x.bfloat16(), wq, s_pc),
    "w8a8_linear_noalloc": lambda: cider.w8a8_linear_noalloc(
        x, wq, s_pc, torch.empty(M, N, dtype=torch.float16)),
    "int8_gemv": lambda: cider.int8_gemv(x[0], wq, s_pc),
    "a16_gemv": lambda: cider.a16_gemv(x[0], wq, s_pc),
    "act_image": lambda: cider.act_image(x),
    "weight_image": lambda: cider.weight_image(wq, K),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused(name):
    with pytest.raises(ValueError, match="CUDA"):
        CALLS[name]()


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(cider, "LIB_PATH", str(tmp_path / "libcider.so"))
    monkeypatch.setattr(cider, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        cider.load_library()
    with pytest.raises(RuntimeError, match="missing"):
        cider.quantize_act(x)


# Shapes that disagree with the activations' K or the output's [M, N] are
# refused before any device work (a kernel would read or write past the
# tensor's end otherwise).
BAD_SHAPES = {
    "w8a8_short_weight_rows": lambda: cider.w8a8_linear(x, wq[:, :K - 16], s_pc),
    "w8a8_pc_scale_count": lambda: cider.w8a8_linear(x, wq, torch.ones(N - 1)),
    "w8a8_pg_scale_count": lambda: cider.w8a8_linear(x, wq, torch.ones(N, 2), 64),
    "w8a8_group_not_dividing_K": lambda: cider.w8a8_linear(x, wq, s_pg, 48),
    "w8a8_out_shape": lambda: cider.w8a8_linear(x, wq, s_pc,
                                                out=torch.empty(M, N - 8, dtype=torch.float16)),
    "w4a8_unpacked_weight": lambda: cider.w4a8_linear(x, wq.view(torch.uint8), s_pg, 64),
    "linear_bits": lambda: cider.linear(x, wq, s_pc, bits=2),
    "linear_int4_columns": lambda: cider.linear(x, wq.view(torch.uint8), s_pc, bits=4),
    "noalloc_out_shape": lambda: cider.w8a8_linear_noalloc(
        x, wq, s_pc, torch.empty(M + 1, N, dtype=torch.float16)),
    "gemv_weight_columns": lambda: cider.int8_gemv(torch.zeros(K + 16, dtype=torch.float16),
                                                   wq, s_pc),
    "gemv_out_shape": lambda: cider.int8_gemv(x[0], wq, s_pc,
                                              out=torch.empty(1, N, dtype=torch.float16)),
    "a16_scale_count": lambda: cider.a16_gemv(x[0], wq, s_pg, 8, 32),
    "act_image_buffer": lambda: cider.act_image(x, torch.empty(M, K - 8, dtype=torch.float16)),
    "weight_image_columns": lambda: cider.weight_image(wq, K + 16),
    "gemm_images_scales": lambda: cider.gemm_images(
        torch.empty(M, K, dtype=torch.float16), torch.ones(M), torch.empty(N, K,
                                                                           dtype=torch.float16),
        torch.ones(N + 1)),
    "raw_gemm_codes": lambda: cider.raw_gemm_s32(torch.zeros(M, K - 16, dtype=torch.int8), wq, K),
}


@pytest.mark.parametrize("name", sorted(BAD_SHAPES))
def test_mismatched_shapes_are_refused(name):
    with pytest.raises(ValueError) as e:
        BAD_SHAPES[name]()
    assert "CUDA" not in str(e.value), "refused for the device, not the shape"
