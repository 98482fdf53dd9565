"""Shared helpers for the tests: moving bit patterns between numpy and torch,
and the output tolerance used by every parity check.

Tolerance (stated once, used everywhere): a bf16 output y of the CUDA path
passes if it is within 1 bf16 ulp of the oracle's fp32 result rounded to bf16,
or -- where the fp32 sum cancels so that reordering it may move the last bit --
if |y - y64| <= bound + ulp(y)/2, with y64 the oracle's fp64 value and bound
its fp32 rounding-error bound for any summation order."""
import numpy as np
import torch

from w4a16_linear_layers_gb300 import synth


def to_dev_bits(a: np.ndarray, dtype: torch.dtype, device="cuda") -> torch.Tensor:
    """uint16 bit patterns -> a bf16/fp16 CUDA tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16))
    return t.view(dtype).to(device)


def from_dev_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(a)
    ulp = np.ldexp(1.0, e - 8)
    ulp[a == 0] = 2.0 ** -133
    return ulp


def compare_linear(y_bits: np.ndarray, ref: dict, label: str = "") -> dict:
    """Check the CUDA output against the oracle dict (y_bf16, y64, bound)."""
    g = synth.bf16_values(y_bits).astype(np.float64)
    o = synth.bf16_values(ref["y_bf16"]).astype(np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    diff_ulp = np.abs(g - o) / bf16_ulp(o)
    ok1 = diff_ulp <= 1.0
    ok2 = np.abs(g - ref["y64"]) <= ref["bound"] + 0.5 * bf16_ulp(g)
    bad = ~(ok1 | ok2)
    stats = {
        "n": int(g.size),
        "bit_exact": int(np.count_nonzero(y_bits == ref["y_bf16"])),
        "max_ulp": float(diff_ulp.max()) if g.size else 0.0,
        "by_bound": int(np.count_nonzero(~ok1 & ok2)),
    }
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(int(i) for i in ix), g[tuple(ix)], o[tuple(ix)], ref["y64"][tuple(ix)],
                   ref["bound"][tuple(ix)]) for ix in idx]
        raise AssertionError(f"{label}: {int(bad.sum())}/{g.size} outputs out of tolerance; "
                             f"first (index, gpu, oracle_bf16, y64, bound): {detail}; {stats}")
    return stats
