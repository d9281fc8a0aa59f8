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


def assert_f16_within_1ulp(gpu: np.ndarray, ref: np.ndarray, what: str = "",
                           identical: bool = True) -> int:
    """The acceptance bar for fp16 outputs: at most 1 ulp from the oracle.
    The kernels perform the oracle's operations in the oracle's order, so by
    default every output must also be bit-identical (the count of outputs
    that are not is reported in the message). Returns that count."""
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    d = f16_ulp_distance(gpu, ref)
    bad = np.argwhere(d > 1)
    assert bad.size == 0, (f"{what}: {len(bad)} outputs beyond 1 ulp, first at {bad[0].tolist()}: "
                           f"gpu={gpu[tuple(bad[0])]} oracle={ref[tuple(bad[0])]}")
    n_diff = int((d != 0).sum())
    if identical:
        first = np.argwhere(d != 0)[:1].tolist()
        assert n_diff == 0, (f"{what}: {n_diff} of {d.size} outputs 1 ulp from the oracle "
                             f"(not bit-identical), first at {first}")
    return n_diff


def cuda(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().to("cuda:0")


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def every_pair_rows(top: int, max_elems: int = 1 << 26):
    """Batches of uint16 rows covering every pair (x, a) of a 16-bit float
    format: for each positive finite bit pattern a in 1..top (ascending), one
    row holding every pattern 0..a and its negation (sign bit set), so that a
    is the row's absmax and every |x| <= a occurs with both signs; zero
    padded to the batch width (a multiple of 16). Each batch holds at most
    max_elems elements (the last absmax of a batch sets its width)."""
    a = 1
    while a <= top:
        width = 2 * (a + 1)
        width += (-width) % 16
        n = 1
        while a + n <= top:
            w = 2 * (a + n + 1)
            w += (-w) % 16
            if (n + 1) * w > max_elems:
                break
            n += 1
            width = w
        rows = np.zeros((n, width), np.uint16)
        for i in range(n):
            v = a + i
            xs = np.arange(v + 1, dtype=np.uint16)
            rows[i, :v + 1] = xs
            rows[i, v + 1:2 * v + 2] = xs | 0x8000
        yield rows
        a += n
