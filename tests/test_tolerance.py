"""The output tolerance itself (tests/helpers.py), checked on the CPU.

A tolerance that passes everything proves nothing, and one that fails a
correct kernel stops the work.  So:
  * a planted mistake -- one 128-wide scale group of the weights dropped --
    must fail it at the drafter's longest reductions (down_proj, K = 17408,
    and the fc projection, K = 25600), in W4A16 and W8A8;
  * an evaluation of the same sums in another fp32 order, shaped like the
    kernel's (sixteen products per step, two interleaved accumulators, then
    their sum), must pass it.
The mistake is planted in the oracle's inputs; no GPU is involved."""
import numpy as np
import pytest

import oracle
from helpers import BY_BOUND_FRACTION, CANCEL, bf16_ulp, check_linear, compare_linear
from w4a16_linear_layers_gb300 import synth

M, N = 8, 64


def _w4a16_case(K, seed=0):
    xb = synth.activations(seed, f"tol/x/{K}", M, K, "normal")
    qwt, sb = synth.w4a16_weights(seed, f"tol/w4/{K}", K, N)
    qw, _, _ = oracle.pack_gptq(qwt, 4)
    return xb, qw, sb


def _assert_caught(wrong, ref, fmt, K):
    """Outputs the planted mistake moved by two bf16 ulps or more fail the
    tolerance: all of them outside true cancellation, at least 99% of them
    overall, and most outputs fail.  (With scales log-uniform over a factor
    of 30, a dropped group of small scales moves some outputs by less than an
    ulp: no tolerance at the 1-ulp bar can see those.  Inside cancellation,
    where |y64| <= 2^-12 S, a change smaller than the kernel bound B is
    excused.)"""
    bad, _ = check_linear(wrong["y_bf16"], ref, fmt, K)
    w = synth.bf16_values(wrong["y_bf16"]).astype(np.float64)
    r = synth.bf16_values(ref["y_bf16"]).astype(np.float64)
    moved = np.abs(w - r) >= 2.0 * bf16_ulp(r)
    cancel = np.abs(ref["y64"]) <= CANCEL * ref["abs_sum"]
    assert moved.sum() > 100
    assert bad[moved & ~cancel].all()
    assert bad[moved].mean() >= 0.99, (int(moved.sum()), int(bad[moved].sum()))
    assert bad.mean() > 0.5, bad.mean()


@pytest.mark.parametrize("K", [17408, 25600])
def test_a_dropped_scale_group_fails_w4a16(K):
    xb, qw, sb = _w4a16_case(K)
    ref = oracle.gemm_w4a16_g128(xb, qw, sb, K)
    planted = sb.copy()
    planted[(K // 128) // 2, :] = 0          # one group's scales -> +0.0
    wrong = oracle.gemm_w4a16_g128(xb, qw, planted, K)
    _assert_caught(wrong, ref, "w4a16", K)
    with pytest.raises(AssertionError):
        compare_linear(wrong["y_bf16"], ref, "planted", "w4a16", K)


@pytest.mark.parametrize("K", [17408, 25600])
def test_a_dropped_scale_group_fails_w8a8(K):
    xb = synth.activations(0, f"tol/x8/{K}", M, K, "outliers")
    qa, sa = oracle.act_quant_i8(xb)
    qwt, swb = synth.w8a8_weights(0, f"tol/w8/{K}", K, N)
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    ref = oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K)
    planted = swb.copy()
    planted[(K // 128) // 2, :] = 0
    wrong = oracle.gemm_w8a8_gs128(qa, sa, qw, planted, K)
    _assert_caught(wrong, ref, "w8a8", K)
    with pytest.raises(AssertionError):
        compare_linear(wrong["y_bf16"], ref, "planted", "w8a8", K)


def _kernel_shaped_fp32(xb, qw, sb, K):
    """The W4A16 sums in another fp32 order, shaped like the tensor-core
    path: products (exact in fp32), sixteen at a time summed in fp32, added
    into one of two accumulators (alternating every 128 K), the two added at
    the end.  Rounds to nearest, where the hardware may truncate; the point
    is a legitimate reordering, not a model of the hardware's bits."""
    w = synth.bf16_values(oracle.dequant_w4a16(qw, sb, K, qw.shape[1])).astype(np.float32)
    x = synth.bf16_values(xb).astype(np.float32)
    prod = x[:, :, None] * w[None, :, :]                      # [M, K, N], exact
    chunks = prod.reshape(x.shape[0], K // 16, 16, -1).sum(axis=2, dtype=np.float32)
    acc = np.zeros((2, x.shape[0], w.shape[1]), np.float32)
    for c in range(K // 16):
        i = (c // 8) & 1
        acc[i] = acc[i] + chunks[:, c, :]
    return synth.bf16_bits(acc[0] + acc[1])


@pytest.mark.parametrize("K", [5120, 17408, 25600])
def test_another_fp32_order_passes_w4a16(K):
    xb, qw, sb = _w4a16_case(K, seed=1)
    ref = oracle.gemm_w4a16_g128(xb, qw, sb, K)
    y = _kernel_shaped_fp32(xb, qw, sb, K)
    stats = compare_linear(y, ref, "reordered", "w4a16", K)
    assert stats["by_bound"] <= BY_BOUND_FRACTION * stats["n"] + 2
