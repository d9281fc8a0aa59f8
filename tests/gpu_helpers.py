"""Helpers shared by the GPU parity tests (no arithmetic of the method)."""
import numpy as np
import torch


def f16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units in the last place between two fp16 arrays, on the
    ordered integer line of binary16 (+0 and -0 coincide)."""
    ia = np.ascontiguousarray(a, dtype=np.float16).view(np.uint16).astype(np.int32)
    ib = np.ascontiguousarray(b, dtype=np.float16).view(np.uint16).astype(np.int32)
    oa = np.where(ia & 0x8000, -(ia & 0x7FFF), ia)
    ob = np.where(ib & 0x8000, -(ib & 0x7FFF), ib)
    return np.abs(oa - ob)


def assert_f16_within_1ulp(gpu: np.ndarray, ref: np.ndarray, what: str = "") -> int:
    """The acceptance bar for fp16 outputs: at most 1 ulp from the oracle.
    Returns the number of outputs that are not bit-identical."""
    d = f16_ulp_distance(gpu, ref)
    bad = np.argwhere(d > 1)
    assert bad.size == 0, (f"{what}: {len(bad)} outputs beyond 1 ulp, first at {bad[0].tolist()}: "
                           f"gpu={gpu[tuple(bad[0])]} oracle={ref[tuple(bad[0])]}")
    return int((d != 0).sum())


def cuda(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().to("cuda:0")


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()
