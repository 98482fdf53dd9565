"""Shared helpers for the tests: moving bit patterns between numpy and torch,
and the output tolerance used by every parity check.

Tolerance (stated once, used everywhere).  The bar is "within 1 bf16 ulp of
the oracle's fp32 result rounded to bf16".  A bf16 output y of the CUDA path
passes if

  (1) |y - bf16(y_f32)| <= 1 bf16 ulp of bf16(y_f32), y_f32 being the
      oracle's fp32 result; or
  (2) the output is a true cancellation, |y64| <= 2^-12 * S with
      S = sum |terms| (at least 12 bits of the terms cancel: the rounding
      errors of an fp32 evaluation scale with S, not with y, and only there
      can they reach a bf16 ulp of y), and |y - y64| <= B + ulp(y)/2, with
      y64 the oracle's fp64 value and B a bound on the kernel's own fp32
      evaluation order.

B per format:
  * W8A8: the group partials are exact integers and the kernel's fp32 chain
    is the oracle's (fma over ascending groups, then x s_a); a tile whose K
    is split across blocks adds a few partial sums.  The oracle's any-order
    bound (G + 2) * 2^-24 * S covers it.
  * W4A16 / W8A16: the tensor core accumulates the products in fp32 sixteen
    K values at a time (one MMA) into one of two accumulators (one per
    issuer, alternate 128-wide steps); the epilogue adds the two and any
    split partials: n = ceil(K/16) + 4 roundings of at most 2 ulps each.  A
    worst-case bound, linear in n, would excuse a whole dropped group at the
    drafter's K; the probabilistic bound for independent rounding errors,
    B = 4 * sqrt(n) * 2^-23 * S, is used instead.  (Higham and Mary,
    "A new approach to probabilistic rounding error analysis", SIAM J. Sci.
    Comput. 41 (2019): the error stays within a small multiple of
    sqrt(n) * u * S with high probability.)  A truncating accumulator adds
    a one-sided drift of at most about 2^-22 * S at these K, far inside B.

Outputs that needed clause (2) are counted (`by_bound`) and may be at most
1e-3 of the outputs (plus 2, for small checks); `max_ulp` is the largest
distance in bf16 ulps over all outputs."""
import numpy as np
import torch

from w4a16_linear_layers_gb300 import synth

CANCEL = 2.0 ** -12         # |y64| / S at or below which an output cancels
BY_BOUND_FRACTION = 1e-3    # most outputs that may need clause (2)


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


def kernel_bound(ref: dict, fmt: str, K: int) -> np.ndarray:
    """B of the module docstring for an oracle result of format `fmt`
    ('w8a8', 'w4a16' or 'w8a16') with reduction length K."""
    if fmt == "w8a8":
        return ref["bound"]
    if fmt in ("w4a16", "w8a16"):
        return 4.0 * np.sqrt(float(-(-K // 16)) + 4.0) * 2.0 ** -23 * ref["abs_sum"]
    raise ValueError(fmt)


def _clauses(y_bits, ref, fmt, K):
    g = synth.bf16_values(y_bits).astype(np.float64)
    o = synth.bf16_values(ref["y_bf16"]).astype(np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    diff_ulp = np.abs(g - o) / bf16_ulp(o)
    ok1 = diff_ulp <= 1.0
    cancel = np.abs(ref["y64"]) <= CANCEL * ref["abs_sum"]
    bound = kernel_bound(ref, fmt, K)
    ok2 = cancel & (np.abs(g - ref["y64"]) <= bound + 0.5 * bf16_ulp(g))
    return g, o, diff_ulp, ok1, ok2, cancel, bound


def check_linear(y_bits: np.ndarray, ref: dict, fmt: str = "w8a8", K: int = 0):
    """The tolerance of the module docstring, element by element: the mask of
    outputs that fail it, and the number that needed clause (2)."""
    _, _, _, ok1, ok2, _, _ = _clauses(y_bits, ref, fmt, K)
    return ~(ok1 | ok2), int(np.count_nonzero(~ok1 & ok2))


def compare_linear(y_bits: np.ndarray, ref: dict, label: str = "", fmt: str = "w8a8",
                   K: int = 0) -> dict:
    """Check the CUDA output against the oracle dict (y_bf16, y64, bound,
    abs_sum) under the tolerance of the module docstring."""
    g, o, diff_ulp, ok1, ok2, cancel, bound = _clauses(y_bits, ref, fmt, K)
    bad = ~(ok1 | ok2)
    by_bound = int(np.count_nonzero(~ok1 & ok2))
    stats = {
        "n": int(g.size),
        "bit_exact": int(np.count_nonzero(y_bits == ref["y_bf16"])),
        "max_ulp": float(diff_ulp.max()) if g.size else 0.0,
        "by_bound": by_bound,
        "cancelling": int(np.count_nonzero(cancel)),
    }
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(int(i) for i in ix), g[tuple(ix)], o[tuple(ix)], ref["y64"][tuple(ix)],
                   bound[tuple(ix)]) for ix in idx]
        raise AssertionError(f"{label}: {int(bad.sum())}/{g.size} outputs out of tolerance; "
                             f"first (index, gpu, oracle_bf16, y64, bound): {detail}; {stats}")
    limit = BY_BOUND_FRACTION * g.size + 2
    if by_bound > limit:
        raise AssertionError(f"{label}: {by_bound}/{g.size} outputs needed the cancellation "
                             f"clause (limit {limit:.0f}); {stats}")
    return stats
