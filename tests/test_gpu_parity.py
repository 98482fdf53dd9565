"""CUDA path vs the CPU oracle, through the C ABI (the ctypes binding).

Integer stages (quantized activations, activation scales, packed words, the
per-group integer partials) must be bit-exact; bf16 outputs must meet the
tolerance in tests/helpers.py.  Sizes span several tiles and a ragged tail;
the full-size workloads are checked on sampled columns (every row, since rows
are independent)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import bf16_ulp, compare_linear, from_dev_bits, to_dev, to_dev_bits
from w4a16_linear_layers_gb300 import qlin, synth
from w4a16_linear_layers_gb300 import build as qbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    qlin.load()
    oracle.build()
    assert qlin.device_status() == qlin.QLIN_OK
    yield
    assert qlin.device_status() == qlin.QLIN_OK


def _act_quant_gpu(xb):
    q, s = qlin.act_quant_i8(to_dev_bits(xb, torch.bfloat16))
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


# ------------------------------------------------------------- act-quant

@pytest.mark.parametrize("M,K,kind", [
    (1, 128, "normal"), (3, 5120, "outliers"), (8, 5120, "outliers"), (17, 4096, "normal2"),
    (96, 17408, "silu_mul"), (5, 25600, "normal2"), (4, 33024, "outliers"), (130, 640, "normal"),
    (300, 1280, "outliers"), (260, 40960, "normal"),   # more than 256 rows: 256-thread blocks
])
def test_act_quant_bit_exact(M, K, kind):
    xb = synth.activations(1, f"gpu/aq/{M}/{K}", M, K, kind)
    if M > 2:
        xb[0, : min(K, 256)] = 0         # a partly-zero row
        xb[1, :] = 0                     # an all-zero row
    q, s = _act_quant_gpu(xb)
    oq, os_ = oracle.act_quant_i8(xb)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(q, oq)


def test_act_quant_dense_sweep_near_rounding_boundaries():
    """Every row holds its maximum and 4095 bf16 values spread over
    [-amax, amax]: many quotients x / s land next to a half-integer, where the
    kernel's reciprocal shortcut must hand over to the IEEE divide."""
    rng = np.random.default_rng(7)
    M, K = 64, 4096
    amax = np.exp(rng.uniform(np.log(1e-3), np.log(1e3), M)).astype(np.float32)
    amax = synth.bf16_values(synth.bf16_bits(amax))
    x = np.linspace(-1.0, 1.0, K, dtype=np.float64)[None, :] * amax[:, None]
    x[:, 0] = amax
    xb = synth.bf16_bits(x)
    q, s = _act_quant_gpu(xb)
    oq, os_ = oracle.act_quant_i8(xb)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(q, oq)


def test_act_quant_ties_and_divide_cases():
    rows = [
        [127, 2.5, -3.5, 0.5, 1.5, -0.5, -1.5, 126.5],
        [254, 1, 3, -1, 5, -7, -254, 100],
        [0] * 8,
    ]
    x = np.zeros((3, 128), np.float32)
    for i, r in enumerate(rows):
        x[i, : len(r)] = r
    xb = synth.bf16_bits(x)
    q, s = _act_quant_gpu(xb)
    oq, os_ = oracle.act_quant_i8(xb)
    assert np.array_equal(q, oq) and np.array_equal(s, os_)
    assert q[0, :8].tolist() == [127, 2, -4, 0, 2, 0, -2, 126]
    # many random rows: elements near .5 boundaries included by volume
    xb = synth.activations(77, "gpu/aq/many", 512, 1024, "normal")
    q, s = _act_quant_gpu(xb)
    oq, os_ = oracle.act_quant_i8(xb)
    assert np.array_equal(q, oq) and np.array_equal(s, os_)


# ------------------------------------------------------------------ pack

@pytest.mark.parametrize("bits,K,N", [(8, 256, 40), (8, 5120, 1024), (4, 384, 72), (4, 5120, 1000)])
def test_pack_bit_exact(bits, K, N):
    lo, hi = (-128, 127) if bits == 8 else (-8, 7)
    q = synth.randint(2, f"gpu/pack/{bits}/{K}/{N}", (K, N), lo, hi)
    qw, qz = qlin.pack_gptq(to_dev(q), bits, with_qzeros=(N * bits) % 32 == 0)
    oqw, oqz, bad = oracle.pack_gptq(q, bits)
    assert bad == 0
    assert np.array_equal(qw.cpu().numpy(), oqw)
    if qz is not None:
        assert np.array_equal(qz.cpu().numpy(), oqz)
    assert qlin.device_status() == qlin.QLIN_OK


def test_pack_flags_out_of_range():
    q = np.zeros((128, 8), np.int8)
    q[5, 3] = 9
    qlin.pack_gptq(to_dev(q), 4)
    assert qlin.device_status() == qlin.QLIN_ERR_VALUE_RANGE
    assert qlin.device_status() == qlin.QLIN_OK      # the error word was cleared


# ---------------------------------------------------- W8A8 group partials

def _w8a8_inputs(seed, name, M, K, N, kind="outliers"):
    xb = synth.activations(seed, name + "/x", M, K, kind)
    qa, sa = oracle.act_quant_i8(xb)
    qwt, swb = synth.w8a8_weights(seed, name + "/w", K, N)
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    return xb, qa, sa, qwt, qw, swb


@pytest.mark.parametrize("M,K,N", [(1, 128, 128), (8, 640, 256), (17, 384, 200), (96, 256, 384),
                                   (130, 256, 136)])
def test_group_partials_bit_exact(M, K, N):
    _, qa, _, _, qw, _ = _w8a8_inputs(3, f"gpu/gp/{M}/{K}/{N}", M, K, N)
    P = qlin.debug_group_partials_i8(to_dev(qa), to_dev(qw))
    torch.cuda.synchronize()
    assert np.array_equal(P.cpu().numpy(), oracle.group_partials_i8(qa, qw, K))


def test_group_partials_extreme_magnitudes():
    """All +-127 operands: |P| = 128*127^2 = 2,064,512, the largest partial;
    fp16 operands with fp32 tensor-memory accumulation must stay exact."""
    M, K, N = 64, 512, 256
    sign_a = synth.randint(4, "gpu/gp/xa", (M, K), 0, 1) * 2 - 1
    sign_w = synth.randint(4, "gpu/gp/xw", (K, N), 0, 1) * 2 - 1
    qa = (127 * sign_a).astype(np.int8)
    qa[0] = 127
    qwt = (127 * sign_w).astype(np.int8)
    qwt[:, 0] = 127
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    P = qlin.debug_group_partials_i8(to_dev(qa), to_dev(qw)).cpu().numpy()
    ref = oracle.group_partials_i8(qa, qw, K)
    assert ref[:, 0, 0].tolist() == [128 * 127 * 127] * (K // 128)
    assert np.array_equal(P, ref)


# -------------------------------------------------------------- W8A8 GEMM

def _gemm_w8a8_gpu(qa, sa, qw, swb, workspace=None):
    y = qlin.gemm_w8a8_gs128(to_dev(qa), to_dev(sa), to_dev(qw), to_dev_bits(swb, torch.float16),
                             workspace=workspace)
    torch.cuda.synchronize()
    return from_dev_bits(y)


@pytest.mark.parametrize("M,K,N", [
    (1, 128, 128), (3, 256, 200), (8, 5120, 1024), (16, 1280, 384), (17, 640, 256),
    (64, 4096, 512), (96, 2560, 768), (100, 384, 136), (128, 512, 256), (257, 768, 264),
    (8, 128, 2048),   # one group: every step opens its own scale chunk
])
def test_w8a8_matches_oracle(M, K, N):
    _, qa, sa, _, qw, swb = _w8a8_inputs(5, f"gpu/w8/{M}/{K}/{N}", M, K, N)
    y = _gemm_w8a8_gpu(qa, sa, qw, swb)
    compare_linear(y, oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K), f"w8a8 {M}x{K}x{N}")


def test_w8a8_extreme_fp16_scales():
    """Weight scales over the whole positive fp16 range, subnormals to 65504,
    mixed per group and column: the fp32 rescale chain must still match."""
    M, K, N = 8, 1024, 384
    _, qa, sa, _, qw, _ = _w8a8_inputs(21, "gpu/w8/extreme", M, K, N)
    rng = np.random.default_rng(21)
    exps = rng.uniform(-24.0, 15.9, size=(K // 128, N))
    scales = np.clip(np.exp2(exps), 2.0 ** -24, 65504.0)
    swb = synth.f16_bits(scales)
    y = _gemm_w8a8_gpu(qa, sa, qw, swb)
    compare_linear(y, oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K), "w8a8 extreme scales")


def test_w4a16_wide_range_bf16_scales():
    """bf16 weight scales from 2^-30 to 2^30, mixed per group and column."""
    M, K, N = 8, 1024, 384
    xb, _, qw, _ = _w4a16_inputs(22, "gpu/w4/wide", M, K, N)
    rng = np.random.default_rng(22)
    sb = synth.bf16_bits(np.exp2(rng.uniform(-30.0, 30.0, size=(K // 128, N))))
    y = _gemm_w4a16_gpu(xb, qw, sb)
    compare_linear(y, oracle.gemm_w4a16_g128(xb, qw, sb, K), "w4a16 wide scales", "w4a16", K)


def test_w8a8_identity_probe():
    """Feeding I_K recovers the effective weight q*s (single nonzero group per
    row, so every split of K gives the oracle's exact fp32 chain)."""
    K, N = 384, 256
    xb = synth.bf16_bits(np.eye(K, dtype=np.float32))
    qa, sa = oracle.act_quant_i8(xb)
    qwt, swb = synth.w8a8_weights(6, "gpu/w8/probe", K, N)
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    y = _gemm_w8a8_gpu(qa, sa, qw, swb)
    ref = oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K)
    assert np.array_equal(y, ref["y_bf16"])


def test_w8a8_deterministic_and_workspace_reuse():
    M, K, N = 8, 5120, 1024
    _, qa, sa, _, qw, swb = _w8a8_inputs(7, "gpu/w8/det", M, K, N)
    ws = qlin.Workspace()
    y1 = _gemm_w8a8_gpu(qa, sa, qw, swb, ws)
    y2 = _gemm_w8a8_gpu(qa, sa, qw, swb, ws)
    assert np.array_equal(y1, y2)
    counters = ws.buf[:4096].view(torch.int32).cpu().numpy()
    assert not counters.any(), "split-K counters must return to zero"


def test_shared_workspace_across_shapes():
    """One workspace, many shapes in a row, never re-zeroed by the caller:
    each call's partials must not disturb the next call's counters."""
    ws = qlin.Workspace()
    shapes = [(96, 2560, 768), (8, 640, 5120), (64, 1280, 2048), (8, 1280, 4352), (17, 384, 1000)]
    for i, (M, K, N) in enumerate(shapes * 2):
        _, qa, sa, _, qw, swb = _w8a8_inputs(40 + i, f"gpu/w8/shared/{i}", M, K, N)
        y = _gemm_w8a8_gpu(qa, sa, qw, swb, ws)
        compare_linear(y, oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K), f"shared ws w8a8 {i}")
        xb, _, qw4, sb = _w4a16_inputs(60 + i, f"gpu/w4/shared/{i}", M, K, N)
        y4 = _gemm_w4a16_gpu(xb, qw4, sb, ws)
        compare_linear(y4, oracle.gemm_w4a16_g128(xb, qw4, sb, K), f"shared ws w4a16 {i}", "w4a16", K)
    assert not ws.buf[:4096].view(torch.int32).cpu().numpy().any()


# ------------------------------------------------------------- W4A16 GEMM

def _w4a16_inputs(seed, name, M, K, N, kind="normal"):
    xb = synth.activations(seed, name + "/x", M, K, kind)
    qwt, sb = synth.w4a16_weights(seed, name + "/w", K, N)
    qw, _, _ = oracle.pack_gptq(qwt, 4)
    return xb, qwt, qw, sb


def _gemm_w4a16_gpu(xb, qw, sb, workspace=None):
    y = qlin.gemm_w4a16_g128(to_dev_bits(xb, torch.bfloat16), to_dev(qw),
                             to_dev_bits(sb, torch.bfloat16), workspace=workspace)
    torch.cuda.synchronize()
    return from_dev_bits(y)


@pytest.mark.parametrize("M,K,N", [
    (1, 128, 128), (3, 256, 200), (8, 5120, 1024), (17, 640, 256), (64, 4096, 512),
    (96, 1280, 384), (130, 512, 264),
    # one (two-group) step per tile: every step opens its own scale chunk
    (8, 128, 2048), (8, 256, 2048), (64, 256, 4096),
    # one-group tiles on every SM, many chunks per block: 16-, 32- and
    # 64-token tiles, where a converter group could run chunks ahead
    (8, 128, 40960), (32, 128, 40960), (64, 128, 40960), (64, 256, 40960),
])
def test_w4a16_matches_oracle(M, K, N):
    xb, _, qw, sb = _w4a16_inputs(9, f"gpu/w4/{M}/{K}/{N}", M, K, N)
    y = _gemm_w4a16_gpu(xb, qw, sb)
    compare_linear(y, oracle.gemm_w4a16_g128(xb, qw, sb, K), f"w4a16 {M}x{K}x{N}", "w4a16", K)


@pytest.mark.parametrize("fmt,M", [("w8a8", 8), ("w8a8", 64), ("w8a8", 96), ("w4a16", 8), ("w4a16", 64)])
def test_fused_projections_match_each_oracle(fmt, M):
    """Projections that read one input (q/k/v, gate/up) run as one GEMM over
    their packed weights and scales concatenated along N; each column block
    of the output must match the oracle of its own projection."""
    K, Ns = 640, (256, 128, 136)
    xb = synth.activations(12, f"gpu/fused/{fmt}/{M}/x", M, K, "outliers" if fmt == "w8a8" else "normal")
    parts = []
    for i, N in enumerate(Ns):
        if fmt == "w8a8":
            qwt, sc = synth.w8a8_weights(12, f"gpu/fused/{fmt}/w{i}", K, N)
            qw, _, _ = oracle.pack_gptq(qwt, 8)
        else:
            qwt, sc = synth.w4a16_weights(12, f"gpu/fused/{fmt}/w{i}", K, N)
            qw, _, _ = oracle.pack_gptq(qwt, 4)
        parts.append((qw, sc))
    qw_cat = np.concatenate([p[0] for p in parts], axis=1)
    sc_cat = np.concatenate([p[1] for p in parts], axis=1)
    if fmt == "w8a8":
        qa, sa = oracle.act_quant_i8(xb)
        y = _gemm_w8a8_gpu(qa, sa, qw_cat, sc_cat)
    else:
        y = _gemm_w4a16_gpu(xb, qw_cat, sc_cat)
    off = 0
    for i, ((qw, sc), N) in enumerate(zip(parts, Ns)):
        ref = (oracle.gemm_w8a8_gs128(qa, sa, qw, sc, K) if fmt == "w8a8"
               else oracle.gemm_w4a16_g128(xb, qw, sc, K))
        compare_linear(np.ascontiguousarray(y[:, off:off + N]), ref, f"fused {fmt} M={M} part {i}",
                       fmt, K)
        off += N


def test_w4a16_identity_probe_bit_exact():
    K, N = 256, 384
    _, qwt, qw, sb = _w4a16_inputs(10, "gpu/w4/probe", 1, K, N)
    xb = synth.bf16_bits(np.eye(K, dtype=np.float32))
    y = _gemm_w4a16_gpu(xb, qw, sb)
    assert np.array_equal(y, oracle.dequant_w4a16(qw, sb, K, N))


def test_w4a16_full_nibble_range():
    """q = -8 (nibble 0) decodes to -8 as well."""
    M, K, N = 8, 256, 128
    xb = synth.activations(11, "gpu/w4/nib/x", M, K, "normal")
    qwt = synth.randint(11, "gpu/w4/nib/w", (K, N), -8, 7)
    qw, _, _ = oracle.pack_gptq(qwt, 4)
    sb = synth.bf16_bits(synth.log_uniform(11, "gpu/w4/nib/s", (K // 128, N), 1e-3, 3e-2))
    y = _gemm_w4a16_gpu(xb, qw, sb)
    compare_linear(y, oracle.gemm_w4a16_g128(xb, qw, sb, K), "w4a16 nibble range", "w4a16", K)


# ------------------------------------------------------------ host checks

def test_argument_errors_return_status():
    lib = qlin.load()
    x = torch.zeros((8, 256), dtype=torch.int8, device="cuda")
    s = torch.zeros(8, dtype=torch.float32, device="cuda")
    qw = torch.zeros((64, 128), dtype=torch.int32, device="cuda")
    sc = torch.zeros((2, 128), dtype=torch.float16, device="cuda")
    y = torch.zeros((8, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(qlin.workspace_bytes(8, 128, 256), dtype=torch.uint8, device="cuda")
    P = lambda t: t.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    f = lib.qlin_gemm_w8a8_gs128
    assert f(None, P(s), P(qw), P(sc), 8, 128, 256, P(y), P(ws), ws.numel(), st) == qlin.QLIN_ERR_NULL
    assert f(P(x), P(s), P(qw), P(sc), 8, 128, 200, P(y), P(ws), ws.numel(), st) == qlin.QLIN_ERR_SHAPE
    assert f(P(x), P(s), P(qw), P(sc), 8, 124, 256, P(y), P(ws), ws.numel(), st) == qlin.QLIN_ERR_SHAPE
    assert f(P(x) + 1, P(s), P(qw), P(sc), 8, 128, 256, P(y), P(ws), ws.numel(), st) == qlin.QLIN_ERR_ALIGN
    assert f(P(x), P(s), P(qw), P(sc), 8, 128, 256, P(y), P(ws), 16, st) == qlin.QLIN_ERR_WORKSPACE
    assert f(P(x), P(s), P(qw), P(sc), 0, 128, 256, P(y), P(ws), ws.numel(), st) == qlin.QLIN_OK
    assert lib.qlin_pack_gptq(P(x), 256, 8, 5, P(qw), None, st) == qlin.QLIN_ERR_BITS
    assert lib.qlin_act_quant_i8(P(y), 8, 100, P(x), P(s), st) == qlin.QLIN_ERR_SHAPE
    assert qlin.device_status() == qlin.QLIN_OK


def test_bounded_wait_reports_timeout_and_context_survives():
    qlin.debug_wait_timeout(2_000_000)      # 2 ms limit on a barrier nothing completes
    assert qlin.device_status() == qlin.QLIN_ERR_DEVICE_TIMEOUT
    assert qlin.device_status() == qlin.QLIN_OK
    # the context still works
    xb = synth.activations(1, "gpu/after-timeout", 4, 256, "normal")
    q, s = _act_quant_gpu(xb)
    oq, _ = oracle.act_quant_i8(xb)
    assert np.array_equal(q, oq)


# ---------------------------------------------------- fused greedy argmax

def _argmax_case(fmt, M, K, N, seed=13):
    if fmt == "w8a8":
        xb, qa, sa, _, qw, sc = _w8a8_inputs(seed, f"gpu/amax/{M}/{K}/{N}", M, K, N)
        y = _gemm_w8a8_gpu(qa, sa, qw, sc)
        idx = qlin.gemm_w8a8_gs128_argmax(to_dev(qa), to_dev(sa), to_dev(qw),
                                          to_dev_bits(sc, torch.float16))
        ref = oracle.gemm_w8a8_gs128(qa, sa, qw, sc, K)
    else:
        xb, _, qw, sc = _w4a16_inputs(seed, f"gpu/amax4/{M}/{K}/{N}", M, K, N)
        y = _gemm_w4a16_gpu(xb, qw, sc)
        idx = qlin.gemm_w4a16_g128_argmax(to_dev_bits(xb, torch.bfloat16), to_dev(qw),
                                          to_dev_bits(sc, torch.bfloat16))
        ref = oracle.gemm_w4a16_g128(xb, qw, sc, K)
    torch.cuda.synchronize()
    return y, idx.cpu().numpy(), ref


@pytest.mark.parametrize("fmt,M,K,N", [("w8a8", 8, 512, 2000), ("w8a8", 96, 640, 3000),
                                       ("w8a8", 1, 256, 136), ("w4a16", 8, 512, 2000),
                                       ("w4a16", 64, 384, 1000)])
def test_greedy_argmax_matches_gemm_and_oracle(fmt, M, K, N):
    y, idx, ref = _argmax_case(fmt, M, K, N)
    # the fused reduction sees the same bf16 values the plain call writes
    assert np.array_equal(idx, oracle.argmax_bf16_rows(y))
    # and picks a maximum of the oracle's output, up to the output tolerance:
    # where the oracle's argmax differs, both columns' exact values lie within
    # their error bounds (plus half an ulp each) of each other
    want = oracle.argmax_bf16_rows(ref["y_bf16"])
    rows = np.arange(M)
    g, w = ref["y64"][rows, idx], ref["y64"][rows, want]
    slack = ref["bound"][rows, idx] + ref["bound"][rows, want] + \
        bf16_ulp(synth.bf16_values(ref["y_bf16"][rows, want]).astype(np.float64))
    assert np.all((idx == want) | (np.abs(g - w) <= slack)), (idx, want)


def test_greedy_argmax_ties_take_lowest_index():
    M, K, N = 8, 256, 512
    xb = synth.bf16_bits(np.abs(synth.bf16_values(
        synth.activations(14, "gpu/amax/ties/x", M, K, "normal"))).astype(np.float32))
    qa, sa = oracle.act_quant_i8(xb)
    qwt = np.zeros((K, N), np.int8)
    qwt[:, 300] = 1
    qwt[:, 260] = 1                      # same 128-column tile: identical values
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    sc = synth.f16_bits(np.full((K // 128, N), 0.01, np.float32))
    idx = qlin.gemm_w8a8_gs128_argmax(to_dev(qa), to_dev(sa), to_dev(qw),
                                      to_dev_bits(sc, torch.float16)).cpu().numpy()
    assert idx.tolist() == [260] * M
    # all outputs zero: the first column
    qw0, _, _ = oracle.pack_gptq(np.zeros((K, N), np.int8), 8)
    idx0 = qlin.gemm_w8a8_gs128_argmax(to_dev(qa), to_dev(sa), to_dev(qw0),
                                       to_dev_bits(sc, torch.float16)).cpu().numpy()
    assert idx0.tolist() == [0] * M


# ---------------------------------------- [N, K/8] ingest (compressed-tensors)

def _pack_rows(q: np.ndarray, bits: int) -> np.ndarray:
    """Per-output-row packing of q (the compressed-tensors orientation), from
    the oracle's GPTQ words: word (n, kk) = GPTQ word (kk, n)."""
    qw, _, _ = oracle.pack_gptq(q, bits)
    return np.ascontiguousarray(qw.T)


@pytest.mark.parametrize("bits,K,N", [(4, 384, 72), (4, 5120, 1000), (8, 256, 40), (8, 1280, 2056)])
def test_ingest_nk_bit_exact(bits, K, N):
    rng = np.random.default_rng(bits * 7 + N)
    lim = (1 << (bits - 1)) - 1
    q = rng.integers(-lim, lim + 1, size=(K, N)).astype(np.int8)
    scales_ng = rng.integers(0, 65536, size=(N, K // 128)).astype(np.uint16)
    packed = _pack_rows(q, bits)
    want_w, want_s = oracle.ingest_nk(packed, scales_ng, K, N, bits)
    qw, sc = qlin.ingest_nk(to_dev(packed), to_dev_bits(scales_ng, torch.bfloat16), K, bits)
    torch.cuda.synchronize()
    assert np.array_equal(qw.cpu().numpy(), want_w)
    assert np.array_equal(from_dev_bits(sc), want_s)


def test_w4a16_from_ingested_weights_matches_oracle():
    """End to end: compressed-tensors weights ingested on the device, then the
    W4A16 GEMM, against the oracle on the GPTQ-oriented words."""
    M, K, N = 17, 640, 264
    xb, _, qw, sb = _w4a16_inputs(15, "gpu/ingest/w4", M, K, N)
    packed = np.ascontiguousarray(qw.T)
    sb_ng = np.ascontiguousarray(sb.T)
    qw_d, sb_d = qlin.ingest_nk(to_dev(packed), to_dev_bits(sb_ng, torch.bfloat16), K, 4)
    y = qlin.gemm_w4a16_g128(to_dev_bits(xb, torch.bfloat16), qw_d, sb_d)
    torch.cuda.synchronize()
    compare_linear(from_dev_bits(y), oracle.gemm_w4a16_g128(xb, qw, sb, K), "ingested w4a16",
                   "w4a16", K)


# ------------------------------------------------------ W8A16 (int8 weight-only)

def _w8a16_inputs(seed, name, M, K, N, gs):
    xb = synth.activations(seed, name + "/x", M, K, "normal")
    qwt, sb = synth.w8a16_weights(seed, name + "/w", K, N, gs)
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    return xb, qw, sb


@pytest.mark.parametrize("gs", [32, 128, 0])
@pytest.mark.parametrize("M,K,N", [(1, 128, 128), (8, 5120, 1024), (17, 640, 264), (64, 1280, 384),
                                   (96, 384, 136), (130, 256, 200), (8, 128, 2048),
                                   (8, 128, 40960), (64, 256, 40960)])
def test_w8a16_matches_oracle(M, K, N, gs):
    xb, qw, sb = _w8a16_inputs(16, f"gpu/w8a16/{M}/{K}/{N}/{gs}", M, K, N, gs)
    y = qlin.gemm_w8a16(to_dev_bits(xb, torch.bfloat16), to_dev(qw), to_dev_bits(sb, torch.bfloat16), gs)
    torch.cuda.synchronize()
    compare_linear(from_dev_bits(y), oracle.gemm_w8a16(xb, qw, sb, K, gs), f"w8a16 g{gs} {M}x{K}x{N}",
                   "w8a16", K)


@pytest.mark.parametrize("gs", [32, 0])
def test_w8a16_identity_probe_bit_exact(gs):
    """Feeding I_K recovers w = bf16(q * s) bit for bit (one nonzero product
    per output, so any summation order gives the same value)."""
    K, N = 256, 384
    xb = synth.bf16_bits(np.eye(K, dtype=np.float32))
    _, qw, sb = _w8a16_inputs(17, f"gpu/w8a16/probe/{gs}", K, K, N, gs)
    y = qlin.gemm_w8a16(to_dev_bits(xb, torch.bfloat16), to_dev(qw), to_dev_bits(sb, torch.bfloat16), gs)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_bits(y), oracle.gemm_w8a16(xb, qw, sb, K, gs)["y_bf16"])


def test_w8a16_rejects_other_group_sizes():
    x = torch.zeros((8, 256), dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros((64, 128), dtype=torch.int32, device="cuda")
    sc = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qlin.QlinError) as e:
        qlin.gemm_w8a16(x, qw, sc, 64)
    assert e.value.status == qlin.QLIN_ERR_SHAPE


# ------------------------------------------------- repeated back-to-back launches

@pytest.mark.parametrize("fmt,M,K,N", [("w4a16", 8, 5120, 17408), ("w4a16", 8, 4096, 5120),
                                       ("w4a16", 64, 17408, 5120), ("w8a8", 8, 5120, 17408),
                                       ("w8a8", 96, 5120, 6144), ("w8a16", 8, 5120, 6144),
                                       # tiles of one K group: every scale chunk is one step
                                       ("w4a16", 8, 128, 622592), ("w4a16", 64, 128, 622592),
                                       ("w8a16", 8, 128, 622592)])
def test_repeated_launches_are_identical(fmt, M, K, N):
    """Hundreds of launches of one full-size linear, back to back on one
    stream with one workspace: no bounded wait may run out, and every launch
    must reproduce the first one's output bit for bit (the split-tile fix-up
    sums in a fixed order)."""
    reps = 300
    if fmt == "w8a8":
        _, qa, sa, _, qw, swb = _w8a8_inputs(20, f"gpu/rep/{M}/{K}/{N}", M, K, N)
        args = (to_dev(qa), to_dev(sa), to_dev(qw), to_dev_bits(swb, torch.float16))
        fn = qlin.gemm_w8a8_gs128
    elif fmt == "w4a16":
        xb, _, qw, sb = _w4a16_inputs(20, f"gpu/rep4/{M}/{K}/{N}", M, K, N)
        args = (to_dev_bits(xb, torch.bfloat16), to_dev(qw), to_dev_bits(sb, torch.bfloat16))
        fn = qlin.gemm_w4a16_g128
    else:
        xb, qw, sb = _w8a16_inputs(20, f"gpu/rep8/{M}/{K}/{N}", M, K, N, 32)
        args = (to_dev_bits(xb, torch.bfloat16), to_dev(qw), to_dev_bits(sb, torch.bfloat16), 32)
        fn = qlin.gemm_w8a16
    ws = torch.zeros(qlin.workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    first = fn(*args, workspace=ws)
    torch.cuda.synchronize()
    y = torch.empty_like(first)
    mismatches = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(reps):
        fn(*args, y=y, workspace=ws)
        mismatches += (y.view(torch.int16) != first.view(torch.int16)).sum()
    st, where, block = qlin.device_error_detail()
    qlin.device_status()
    assert st == qlin.QLIN_OK, f"{qlin.status_string(st)} (wait {where}, block {block})"
    assert int(mismatches) == 0


# ------------------------------------------- fused producers + act-quant

def _bf16_steps_apart(a_bits, b_bits):
    """Distance in bf16 steps between two bit-pattern arrays (+0 and -0 equal)."""
    def ordered(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def _check_producer(q_d, s_d, y_d, ref, what):
    """The kernel's bf16 producer output z, its INT8 codes q and its scales
    s_a against the oracle's chain from the same input (producer in fp64,
    rounded once to bf16, then act-quant): all bit-exact.  The kernel forms
    z in fp32 and re-forms in fp64 the values whose fp32 error could move
    them across a bf16 rounding boundary."""
    q_ref, s_ref, z_ref = ref
    z = from_dev_bits(y_d)
    d = _bf16_steps_apart(z, z_ref)
    assert d.max() == 0, (f"{what}: {int((d > 0).sum())}/{d.size} producer outputs differ, "
                          f"by up to {d.max()} bf16 steps")
    assert np.array_equal(q_d.cpu().numpy(), q_ref), what
    assert np.array_equal(s_d.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), what


@pytest.mark.parametrize("M,K,kind", [(1, 128, "normal"), (8, 5120, "outliers"), (96, 5120, "normal2"),
                                      (130, 640, "outliers"), (2048, 5120, "outliers"),
                                      (3, 40960, "normal")])
def test_rmsnorm_act_quant_matches_oracle(M, K, kind):
    x = synth.activations(30, f"gpu/rms/{M}/{K}", M, K, kind)
    if M > 2:
        x[M // 2] = 0          # an all-zero row: z = 0, s_a = 0, q = 0
    g = synth.bf16_bits(1.0 + 0.1 * synth.normal(30, f"gpu/rms/{K}/gamma", (K,)))
    eps = 1e-6
    xd, gd = to_dev_bits(x, torch.bfloat16), to_dev_bits(g, torch.bfloat16)
    y = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    q, s = qlin.rmsnorm_act_quant_i8(xd, gd, eps, y=y)
    q2, s2 = qlin.rmsnorm_act_quant_i8(xd, gd, eps)           # without the bf16 output
    torch.cuda.synchronize()
    _check_producer(q, s, y, oracle.rmsnorm_act_quant_i8(x, g, eps), f"rmsnorm {M}x{K}")
    assert torch.equal(q, q2) and torch.equal(s, s2)


@pytest.mark.parametrize("M,I", [(1, 128), (8, 17408), (96, 17408), (130, 384), (512, 17408),
                                 (2, 34816)])
def test_silu_mul_act_quant_matches_oracle(M, I):
    gu = synth.activations(31, f"gpu/silu/{M}/{I}", M, 2 * I, "normal2")
    if M > 2:
        gu[M // 2, :I] = 0     # SiLU(0) = 0: an all-zero output row
    gud = to_dev_bits(gu, torch.bfloat16)
    y = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    q, s = qlin.silu_mul_act_quant_i8(gud, y=y)
    q2, s2 = qlin.silu_mul_act_quant_i8(gud)
    torch.cuda.synchronize()
    _check_producer(q, s, y, oracle.silu_mul_act_quant_i8(gu), f"silu_mul {M}x{I}")
    assert torch.equal(q, q2) and torch.equal(s, s2)


def test_fused_producers_reject_bad_shapes():
    x = torch.zeros((4, 200), dtype=torch.bfloat16, device="cuda")
    g = torch.ones((200,), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qlin.QlinError):
        qlin.rmsnorm_act_quant_i8(x, g, 1e-6)                 # K not a multiple of 128
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    g = torch.ones((256,), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qlin.QlinError):
        qlin.rmsnorm_act_quant_i8(x, g, -1.0)                 # negative eps
    with pytest.raises(qlin.QlinError):
        qlin.silu_mul_act_quant_i8(torch.zeros((4, 200), dtype=torch.bfloat16, device="cuda"))


def test_empty_batch_is_a_no_op_everywhere():
    """M = 0 through every call of the binding: empty outputs, QLIN_OK, no
    device error (the batch-sized buffers of an empty batch are NULL)."""
    K, N = 256, 128
    dev = "cuda"
    x = torch.empty((0, K), dtype=torch.bfloat16, device=dev)
    q, s = qlin.act_quant_i8(x)
    assert q.shape == (0, K) and s.shape == (0,)
    g = torch.ones((K,), dtype=torch.bfloat16, device=dev)
    q, s = qlin.rmsnorm_act_quant_i8(x, g, 1e-6)
    assert q.shape == (0, K)
    q, s = qlin.silu_mul_act_quant_i8(torch.empty((0, 2 * K), dtype=torch.bfloat16, device=dev))
    assert q.shape == (0, K)
    qa = torch.empty((0, K), dtype=torch.int8, device=dev)
    sa = torch.empty((0,), dtype=torch.float32, device=dev)
    qw8 = torch.zeros((K // 4, N), dtype=torch.int32, device=dev)
    qw4 = torch.zeros((K // 8, N), dtype=torch.int32, device=dev)
    s16 = torch.ones((K // 128, N), dtype=torch.float16, device=dev)
    sb16 = torch.ones((K // 128, N), dtype=torch.bfloat16, device=dev)
    assert qlin.gemm_w8a8_gs128(qa, sa, qw8, s16).shape == (0, N)
    assert qlin.gemm_w8a8_gs128_noalloc(qa, sa, qw8, s16).shape == (0, N)
    assert qlin.gemm_w4a16_g128(x, qw4, sb16).shape == (0, N)
    assert qlin.gemm_w8a16(x, qw8, sb16, 128).shape == (0, N)
    assert qlin.gemm_w8a8_gs128_argmax(qa, sa, qw8, s16).shape == (0,)
    assert qlin.gemm_w4a16_g128_argmax(x, qw4, sb16).shape == (0,)
    torch.cuda.synchronize()
    assert qlin.device_status() == qlin.QLIN_OK


# ------------------------------------------------ weights in the tile layout

@pytest.mark.parametrize("K,N,bits", [(128, 136, 8), (5120, 1024, 8), (640, 3000, 4), (256, 8, 4)])
def test_pack_tiles_bit_exact(K, N, bits):
    rng = np.random.default_rng(K * N + bits)
    qw = rng.integers(-2**31, 2**31 - 1, size=(K * bits // 32, N), dtype=np.int64).astype(np.int32)
    t = qlin.pack_tiles(to_dev(qw), K, bits)
    torch.cuda.synchronize()
    assert np.array_equal(t.data.cpu().numpy(), oracle.pack_tiles(qw, K, bits))


@pytest.mark.parametrize("M,K,N", [(8, 5120, 1024), (17, 640, 264), (64, 4096, 512), (96, 2560, 776),
                                   (130, 512, 256), (8, 128, 40960), (1, 256, 136)])
def test_tiled_w8a8_equals_plain_call(M, K, N):
    """The tile layout changes only how the weight stream reads the words:
    the outputs are those of the plain call, bit for bit, and so within the
    tolerance of the oracle."""
    _, qa, sa, _, qw, swb = _w8a8_inputs(31, f"gpu/tiles8/{M}/{K}/{N}", M, K, N)
    args = (to_dev(qa), to_dev(sa))
    sc = to_dev_bits(swb, torch.float16)
    y_plain = qlin.gemm_w8a8_gs128(*args, to_dev(qw), sc)
    y_tiled = qlin.gemm_w8a8_gs128_tiled(*args, qlin.pack_tiles(to_dev(qw), K, 8), sc)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_bits(y_tiled), from_dev_bits(y_plain))
    compare_linear(from_dev_bits(y_tiled), oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K),
                   f"tiled w8a8 {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", [(8, 5120, 1024), (17, 640, 264), (64, 4096, 512), (96, 1280, 392),
                                   (8, 128, 40960), (64, 256, 4096)])
def test_tiled_w4a16_equals_plain_call(M, K, N):
    xb, _, qw, sb = _w4a16_inputs(32, f"gpu/tiles4/{M}/{K}/{N}", M, K, N)
    x, sc = to_dev_bits(xb, torch.bfloat16), to_dev_bits(sb, torch.bfloat16)
    y_plain = qlin.gemm_w4a16_g128(x, to_dev(qw), sc)
    y_tiled = qlin.gemm_w4a16_g128_tiled(x, qlin.pack_tiles(to_dev(qw), K, 4), sc)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_bits(y_tiled), from_dev_bits(y_plain))
    compare_linear(from_dev_bits(y_tiled), oracle.gemm_w4a16_g128(xb, qw, sb, K),
                   f"tiled w4a16 {M}x{K}x{N}", "w4a16", K)


# ------------------------------------------- many token tiles: banded whole tiles

@pytest.mark.parametrize("M,K,N", [(600, 384, 776), (1000, 256, 264), (1500, 17408, 136)])
def test_banded_tile_schedule_w8a8(M, K, N):
    """Batches of six or more token tiles take whole tiles in bands of token
    tiles (one band at K = 384 and 256; at K = 17408 the bands hold 14 token
    tiles, so the 16 token tiles make a full band and a ragged one).  No tile
    is split, every output is written once, and the fp32 chain is the
    oracle's."""
    _, qa, sa, _, qw, swb = _w8a8_inputs(33, f"gpu/band8/{M}/{K}/{N}", M, K, N)
    y = _gemm_w8a8_gpu(qa, sa, qw, swb)
    rows = np.concatenate([np.arange(0, M, 7), [M - 1]])
    ref = oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K, rows)
    compare_linear(np.ascontiguousarray(y[rows]), ref, f"banded w8a8 {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", [(600, 384, 776), (1500, 17408, 136)])
def test_banded_tile_schedule_w4a16(M, K, N):
    xb, _, qw, sb = _w4a16_inputs(34, f"gpu/band4/{M}/{K}/{N}", M, K, N)
    y = _gemm_w4a16_gpu(xb, qw, sb)
    rows = np.concatenate([np.arange(0, M, 7), [M - 1]])
    ref = oracle.gemm_w4a16_g128(xb, qw, sb, K, rows)
    compare_linear(np.ascontiguousarray(y[rows]), ref, f"banded w4a16 {M}x{K}x{N}", "w4a16", K)


# -------------------------------------------- activation codes stored as fp16

def _codes_as_i8(q16):
    """fp16 codes -> int8, asserting that every code is an integer in range."""
    f = q16.float().cpu().numpy()
    assert np.array_equal(f, np.rint(f)) and np.abs(f).max(initial=0) <= 127
    return f.astype(np.int8)


@pytest.mark.parametrize("M,K,kind", [(1, 128, "normal"), (8, 5120, "outliers"), (33, 4096, "normal2"),
                                      (96, 17408, "silu_mul"), (300, 1280, "outliers"),
                                      (4, 33024, "outliers")])
def test_act_quant_c16_holds_the_int8_codes(M, K, kind):
    xb = synth.activations(40, f"gpu/aq16/{M}/{K}", M, K, kind)
    if M > 2:
        xb[1, :] = 0                     # an all-zero row
    x = to_dev_bits(xb, torch.bfloat16)
    q16, s16 = qlin.act_quant_c16(x)
    torch.cuda.synchronize()
    oq, os_ = oracle.act_quant_i8(xb)
    assert np.array_equal(_codes_as_i8(q16), oq)
    assert np.array_equal(s16.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("M,K", [(1, 128), (64, 5120), (130, 640), (3, 40960)])
def test_rmsnorm_act_quant_c16_holds_the_int8_codes(M, K):
    x = synth.activations(41, f"gpu/rms16/{M}/{K}", M, K, "outliers")
    g = synth.bf16_bits(1.0 + 0.1 * synth.normal(41, f"gpu/rms16/{K}/gamma", (K,)))
    xd, gd = to_dev_bits(x, torch.bfloat16), to_dev_bits(g, torch.bfloat16)
    y = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    q16, s16 = qlin.rmsnorm_act_quant_c16(xd, gd, 1e-6, y=y)
    q8, s8 = qlin.rmsnorm_act_quant_i8(xd, gd, 1e-6)
    torch.cuda.synchronize()
    q_ref, s_ref, z_ref = oracle.rmsnorm_act_quant_i8(x, g, 1e-6)
    assert np.array_equal(_codes_as_i8(q16), q_ref)
    assert np.array_equal(q8.cpu().numpy(), q_ref)
    assert np.array_equal(s16.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert torch.equal(s16, s8)
    assert np.array_equal(from_dev_bits(y), z_ref)


@pytest.mark.parametrize("M,I", [(1, 128), (96, 17408), (130, 384), (2, 34816)])
def test_silu_mul_act_quant_c16_holds_the_int8_codes(M, I):
    gu = synth.activations(42, f"gpu/silu16/{M}/{I}", M, 2 * I, "normal2")
    gud = to_dev_bits(gu, torch.bfloat16)
    q16, s16 = qlin.silu_mul_act_quant_c16(gud)
    q8, s8 = qlin.silu_mul_act_quant_i8(gud)
    torch.cuda.synchronize()
    q_ref, s_ref, _ = oracle.silu_mul_act_quant_i8(gu)
    assert np.array_equal(_codes_as_i8(q16), q_ref)
    assert np.array_equal(q8.cpu().numpy(), q_ref)
    assert torch.equal(s16, s8)


@pytest.mark.parametrize("M,K,N", [(1, 256, 136), (8, 5120, 1024), (17, 640, 264), (32, 1280, 776),
                                   (33, 384, 200), (64, 4096, 512), (65, 640, 264), (96, 2560, 776),
                                   (130, 512, 256), (600, 384, 776), (8, 128, 40960)])
def test_gemm_w8a8_c16_equals_int8_call(M, K, N):
    """The fp16-code entry computes what the int8 entry computes, bit for
    bit, on every token-tile size: 16 and 32 (codes narrowed to int8 in the
    workspace), 64 and 96 (the codes are the tensor-core operand), the banded
    schedule (600 rows), and so within the tolerance of the oracle."""
    _, qa, sa, _, qw, swb = _w8a8_inputs(43, f"gpu/c16/{M}/{K}/{N}", M, K, N)
    qad, sad = to_dev(qa), to_dev(sa)
    q16 = qad.to(torch.float16)            # exact: every int8 value is an fp16 integer
    sc, qwd = to_dev_bits(swb, torch.float16), to_dev(qw)
    y8 = qlin.gemm_w8a8_gs128(qad, sad, qwd, sc)
    y16 = qlin.gemm_w8a8_gs128_c16(q16, sad, qwd, sc)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev_bits(y16), from_dev_bits(y8))
    rows = np.arange(M) if M <= 130 else np.concatenate([np.arange(0, M, 7), [M - 1]])
    ref = oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K, rows if M > 130 else None)
    got = from_dev_bits(y16)
    compare_linear(np.ascontiguousarray(got[rows]) if M > 130 else got, ref,
                   f"w8a8 c16 {M}x{K}x{N}")


def test_c16_chain_equals_int8_chain():
    """Producer -> GEMM through fp16 codes gives the int8 chain's output bit
    for bit (norm -> q/k/v-like GEMM at 96 tokens, SiLU -> down-like GEMM at
    8 tokens)."""
    M, K, N = 96, 1280, 512
    x = synth.activations(44, "gpu/chain16/x", M, K, "outliers")
    g = synth.bf16_bits(1.0 + 0.1 * synth.normal(44, "gpu/chain16/g", (K,)))
    _, _, _, _, qw, swb = _w8a8_inputs(44, "gpu/chain16/w", 1, K, N)
    xd, gd = to_dev_bits(x, torch.bfloat16), to_dev_bits(g, torch.bfloat16)
    sc, qwd = to_dev_bits(swb, torch.float16), to_dev(qw)
    a8 = qlin.gemm_w8a8_gs128(*qlin.rmsnorm_act_quant_i8(xd, gd, 1e-6), qwd, sc)
    a16 = qlin.gemm_w8a8_gs128_c16(*qlin.rmsnorm_act_quant_c16(xd, gd, 1e-6), qwd, sc)
    gu = to_dev_bits(synth.activations(44, "gpu/chain16/gu", 8, 2 * K, "normal2"), torch.bfloat16)
    b8 = qlin.gemm_w8a8_gs128(*qlin.silu_mul_act_quant_i8(gu), qwd, sc)
    b16 = qlin.gemm_w8a8_gs128_c16(*qlin.silu_mul_act_quant_c16(gu), qwd, sc)
    torch.cuda.synchronize()
    assert torch.equal(a8, a16) and torch.equal(b8, b16)


def test_c16_empty_batch_and_bad_arguments():
    K, N, dev = 256, 128, "cuda"
    x = torch.empty((0, K), dtype=torch.bfloat16, device=dev)
    q, s = qlin.act_quant_c16(x)
    assert q.shape == (0, K) and q.dtype == torch.float16
    g = torch.ones((K,), dtype=torch.bfloat16, device=dev)
    assert qlin.rmsnorm_act_quant_c16(x, g, 1e-6)[0].shape == (0, K)
    assert qlin.silu_mul_act_quant_c16(torch.empty((0, 2 * K), dtype=torch.bfloat16,
                                                   device=dev))[0].shape == (0, K)
    qw8 = torch.zeros((K // 4, N), dtype=torch.int32, device=dev)
    s16 = torch.ones((K // 128, N), dtype=torch.float16, device=dev)
    assert qlin.gemm_w8a8_gs128_c16(torch.empty((0, K), dtype=torch.float16, device=dev),
                                    torch.empty((0,), dtype=torch.float32, device=dev),
                                    qw8, s16).shape == (0, N)
    lib = qlin.load()
    # K not a multiple of 128; a misaligned code pointer
    assert lib.qlin_act_quant_c16(None, 0, 200, None, None, None) == qlin.QLIN_ERR_SHAPE
    xa = torch.zeros((2, K), dtype=torch.bfloat16, device=dev)
    qb = torch.zeros((2 * K + 8,), dtype=torch.float16, device=dev)
    sb = torch.zeros((2,), dtype=torch.float32, device=dev)
    assert lib.qlin_act_quant_c16(xa.data_ptr(), 2, K, qb.data_ptr() + 2, sb.data_ptr(),
                                  None) == qlin.QLIN_ERR_ALIGN
    torch.cuda.synchronize()
    assert qlin.device_status() == qlin.QLIN_OK
