"""The layer-level names (W8A8Linear, W4A8Linear, perchannel_linear,
is_available) are argument marshalling over `linear` / `w8a8_linear`: checked
here on the CPU with a recording stand-in for the GPU call, and against the
real call's refusal of host tensors (no GPU needed)."""
import pytest
import torch

import w4a8_quantized_gemm_int8_b300 as cider

N, K = 48, 128


class _Recorder:
    def __init__(self):
        self.calls = []

    def __call__(self, x, w, s_w, bits=8, group_size=0, out_dtype=None, out=None, ws=None):
        self.calls.append((tuple(x.shape), x.is_contiguous(), tuple(w.shape), tuple(s_w.shape),
                           bits, group_size))
        return torch.full((x.shape[0], w.shape[0]), 1.0, dtype=x.dtype)


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    monkeypatch.setattr(cider, "linear", r)
    return r


def test_w8a8_layer_flattens_tokens_and_passes_its_weights(rec):
    layer = cider.W8A8Linear(torch.zeros(N, K, dtype=torch.int8), torch.ones(N), 0, K, N)
    y = layer(torch.zeros(2, 3, K, dtype=torch.float16))
    assert y.shape == (2, 3, N) and y.dtype == torch.float16
    assert rec.calls == [((6, K), True, (N, K), (N,), 8, 0)]


def test_w8a8_layer_per_group_and_noncontiguous_input(rec):
    layer = cider.W8A8Linear(torch.zeros(N, K, dtype=torch.int8), torch.ones(N, K // 64), 64)
    x = torch.zeros(K, 5, dtype=torch.bfloat16).t()   # non-contiguous [5, K]
    y = layer(x)
    assert y.shape == (5, N) and y.dtype == torch.bfloat16
    assert rec.calls == [((5, K), True, (N, K), (N, K // 64), 8, 64)]


def test_w4a8_layer_reads_packed_columns(rec):
    layer = cider.W4A8Linear(torch.zeros(N, K // 2, dtype=torch.uint8), torch.ones(N))
    assert (layer.in_features, layer.out_features, layer.group_size) == (K, N, 0)
    layer(torch.zeros(1, K, dtype=torch.float16))
    assert rec.calls == [((1, K), True, (N, K // 2), (N,), 4, 0)]


def test_empty_token_batch_gives_empty_output(rec):
    layer = cider.W8A8Linear(torch.zeros(N, K, dtype=torch.int8), torch.ones(N))
    y = layer(torch.zeros(0, K, dtype=torch.float16))
    assert y.shape == (0, N) and rec.calls == []


@pytest.mark.parametrize("kw", [dict(in_features=K + 1), dict(out_features=N + 1),
                                dict(group_size=48), dict(group_size=64, scale=(N,))])
def test_shape_mismatches_are_refused(kw):
    scale = torch.ones(*kw.pop("scale", (N,) if kw.get("group_size", 0) == 0
                                else (N, K // kw["group_size"])))
    with pytest.raises(ValueError):
        cider.W8A8Linear(torch.zeros(N, K, dtype=torch.int8), scale, **kw)


def test_wrong_feature_count_is_refused(rec):
    layer = cider.W8A8Linear(torch.zeros(N, K, dtype=torch.int8), torch.ones(N))
    with pytest.raises(ValueError):
        layer(torch.zeros(2, K + 16, dtype=torch.float16))


def test_layers_and_low_level_name_refuse_host_tensors():
    cider.load_library()
    layer = cider.W8A8Linear(torch.zeros(N, K, dtype=torch.int8), torch.ones(N))
    with pytest.raises(ValueError, match="CUDA"):
        layer(torch.zeros(4, K, dtype=torch.float16))
    with pytest.raises(ValueError, match="CUDA"):
        cider.perchannel_linear(torch.zeros(4, K, dtype=torch.float16),
                                torch.zeros(N, K, dtype=torch.int8), torch.ones(N))


def test_is_available_is_false_without_a_b300():
    if torch.cuda.is_available() and torch.cuda.get_device_capability() == (10, 3):
        pytest.skip("a B300 is visible")
    assert cider.is_available() is False
