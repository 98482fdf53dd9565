"""Full-size workloads through the C ABI, checked against the oracle on
sampled columns (all rows, or sampled rows at M = 8192).  Shapes: the drafter
layer's seven projections and the fc projection (hidden 5120, intermediate
17408, 32 query / 8 key-value heads of 128, fc 25600 -> 5120), the 5120 ->
248320 vocabulary head, at the decode, prefill and verification token counts
of the serving recipes.  Inputs are synthetic (seeded), drawn as the
workload recipe in the design notes states."""
import numpy as np
import pytest
import torch

import oracle
from helpers import compare_linear, from_dev_bits, to_dev, to_dev_bits
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
    yield
    assert qlin.device_status() == qlin.QLIN_OK


def sample_cols(N, seed, blocks=2):
    """All columns for N <= 1024; else `blocks` random 128-wide blocks plus the
    last 128 columns (the tail tile)."""
    if N <= 1024:
        return np.arange(N)
    nb = N // 128
    pick = synth.choice_without_replacement(seed, f"cols/{N}", nb - 1, blocks)
    cols = [np.arange(b * 128, b * 128 + 128) for b in pick]
    cols.append(np.arange(N - 128, N))
    return np.concatenate(cols)


def sample_rows(M, seed, limit=96):
    if M <= limit:
        return np.arange(M)
    rows = synth.choice_without_replacement(seed, f"rows/{M}", M - 2, limit - 2)
    return np.concatenate([[0], rows + 1, [M - 1]])


def run_w8a8(name, M, K, N, kind, seed=0, argmax=False):
    xb = synth.activations(seed, synth.shared_input_name(name) + f"/M{M}", M, K, kind)
    qwt, swb = synth.w8a8_weights(seed, name, K, N)
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    del qwt
    x_d = to_dev_bits(xb, torch.bfloat16)
    qa_d, sa_d = qlin.act_quant_i8(x_d)
    qw_d, sw_d = to_dev(qw), to_dev_bits(swb, torch.float16)
    y_d = qlin.gemm_w8a8_gs128(qa_d, sa_d, qw_d, sw_d)
    if argmax:
        # the fused greedy argmax must pick, per row, the first maximum of the
        # very outputs the plain call wrote
        idx = qlin.gemm_w8a8_gs128_argmax(qa_d, sa_d, qw_d, sw_d)
        want = y_d.float().argmax(dim=1).to(torch.int32)
        assert torch.equal(idx, want), f"{name} M={M}: fused argmax differs"
    torch.cuda.synchronize()
    qa, sa = oracle.act_quant_i8(xb)
    assert np.array_equal(qa_d.cpu().numpy(), qa) and np.array_equal(sa_d.cpu().numpy(), sa)
    rows, cols = sample_rows(M, seed), sample_cols(N, seed)
    y = from_dev_bits(y_d)[np.ix_(rows, cols)]
    ref = oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K, rows, cols)
    return compare_linear(y, ref, f"{name} M={M}")


def run_w4a16(name, M, K, N, seed=0):
    xb = synth.activations(seed, synth.shared_input_name(name) + f"/w4/M{M}", M, K, "normal")
    qwt, sb = synth.w4a16_weights(seed, name + "/w4", K, N)
    qw, _, _ = oracle.pack_gptq(qwt, 4)
    del qwt
    y_d = qlin.gemm_w4a16_g128(to_dev_bits(xb, torch.bfloat16), to_dev(qw),
                               to_dev_bits(sb, torch.bfloat16))
    torch.cuda.synchronize()
    rows, cols = sample_rows(M, seed), sample_cols(N, seed)
    y = from_dev_bits(y_d)[np.ix_(rows, cols)]
    ref = oracle.gemm_w4a16_g128(xb, qw, sb, K, rows, cols)
    return compare_linear(y, ref, f"{name} w4a16 M={M}", "w4a16", K)


def test_single_w8a8_linear_all_outputs():
    """5120 -> 1024 at M = 8, every output checked."""
    st = run_w8a8("single", 8, 5120, 1024, "outliers")
    assert st["n"] == 8 * 1024


@pytest.mark.parametrize("M", [8, 64, 96])
def test_drafter_layer_w8a8(M):
    for name, K, N, kind in synth.DRAFTER_LAYER:
        run_w8a8(f"layers.0.{name}", M, K, N, kind)


def test_fc_projection_w8a8():
    name, K, N, kind = synth.FC
    run_w8a8(name, 96, K, N, kind)


@pytest.mark.parametrize("M", [8, 64])
def test_drafter_w4a16(M):
    for name, K, N, _ in synth.DRAFTER_LAYER + (synth.FC,):
        run_w4a16(name, M, K, N)


@pytest.mark.parametrize("M", [128, 512, 2048, 8192])
def test_prefill_mlp_w8a8(M):
    run_w8a8("layers.0.gate_proj", M, 5120, 17408, "outliers")
    run_w8a8("layers.0.down_proj", M, 17408, 5120, "silu_mul")


@pytest.mark.parametrize("M", [8, 96])
def test_vocab_head_w8a8(M):
    run_w8a8("lm_head", M, 5120, 248320, "outliers", argmax=True)


@pytest.mark.parametrize("M", [8, 96])
def test_vocab_head_w4a16_argmax(M):
    """The INT4 g128 vocabulary head of the DFlash2 decoding recipe at full
    size (5120 -> 248320), plain and with the fused greedy argmax.  The 1.27 G
    weights are drawn on the device from the generator's stream (bit for bit
    the host's) and packed there; the oracle takes the sampled columns'
    weights from the host generator and packs them itself."""
    name, K, N, seed = "lm_head", 5120, 248320, 0
    xb = synth.activations(seed, f"{name}/w4/M{M}", M, K, "normal")
    q_d = synth.randint_device(seed, name + "/w4/qw", (K, N), -7, 7, "cuda")
    qw_d, _ = qlin.pack_gptq(q_d, 4, with_qzeros=False)
    del q_d
    sb = synth.bf16_bits(synth.log_uniform(seed, name + "/w4/sw", (K // 128, N), 1e-3, 3e-2))
    x_d, sb_d = to_dev_bits(xb, torch.bfloat16), to_dev_bits(sb, torch.bfloat16)
    y_d = qlin.gemm_w4a16_g128(x_d, qw_d, sb_d)
    idx = qlin.gemm_w4a16_g128_argmax(x_d, qw_d, sb_d)
    want = y_d.float().argmax(dim=1).to(torch.int32)
    torch.cuda.synchronize()
    assert torch.equal(idx, want), f"M={M}: fused W4A16 argmax differs from the plain call's"
    rows, cols = sample_rows(M, seed), sample_cols(N, seed)
    q_cols = synth.randint_at(seed, name + "/w4/qw", N, np.arange(K), cols, -7, 7)
    qw_cols, _, _ = oracle.pack_gptq(np.ascontiguousarray(q_cols), 4)
    ref = oracle.gemm_w4a16_g128(xb, qw_cols, np.ascontiguousarray(sb[:, cols]), K, rows)
    y = from_dev_bits(y_d)[np.ix_(rows, cols)]
    compare_linear(y, ref, f"lm_head w4a16 M={M}", "w4a16", K)


@pytest.mark.parametrize("M", [8, 64, 96])
def test_fused_gate_up_full_size_w8a8(M):
    """gate_proj and up_proj as one GEMM over their weights concatenated along
    N (5120 -> 2 x 17408), as the benchmark runs them: sampled columns of each
    half against the oracle of its own projection."""
    K, I = 5120, 17408
    xb = synth.activations(0, f"layers.0.gate_proj/M{M}", M, K, "outliers")
    qa, sa = oracle.act_quant_i8(xb)
    parts = [synth.w8a8_weights(0, f"layers.0.{n}", K, I) for n in ("gate_proj", "up_proj")]
    packed = [oracle.pack_gptq(q, 8)[0] for q, _ in parts]
    qw_cat = np.ascontiguousarray(np.concatenate(packed, axis=1))
    sw_cat = np.ascontiguousarray(np.concatenate([s for _, s in parts], axis=1))
    y_d = qlin.gemm_w8a8_gs128(to_dev(qa), to_dev(sa), to_dev(qw_cat),
                               to_dev_bits(sw_cat, torch.float16))
    torch.cuda.synchronize()
    y = from_dev_bits(y_d)
    rows = sample_rows(M, 0)
    for half, (qw, (_, sw)) in enumerate(zip(packed, parts)):
        cols = sample_cols(I, half)
        ref = oracle.gemm_w8a8_gs128(qa, sa, qw, sw, K, rows, cols)
        compare_linear(y[np.ix_(rows, cols + half * I)], ref, f"gate_up half {half} M={M}")


def run_w8a16(name, M, K, N, seed=0, gs=32):
    xb = synth.activations(seed, synth.shared_input_name(name) + f"/w8a16/M{M}", M, K, "normal")
    qwt, sb = synth.w8a16_weights(seed, name + "/w8a16", K, N, gs)
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    del qwt
    y_d = qlin.gemm_w8a16(to_dev_bits(xb, torch.bfloat16), to_dev(qw),
                          to_dev_bits(sb, torch.bfloat16), gs)
    torch.cuda.synchronize()
    rows, cols = sample_rows(M, seed), sample_cols(N, seed)
    y = from_dev_bits(y_d)[np.ix_(rows, cols)]
    ref = oracle.gemm_w8a16(xb, qw, sb, K, gs, rows, cols)
    return compare_linear(y, ref, f"{name} w8a16 M={M}", "w8a16", K)


@pytest.mark.parametrize("M", [8, 64])
def test_drafter_layer_w8a16_group32(M):
    for name, K, N, _ in synth.DRAFTER_LAYER:
        run_w8a16(f"layers.0.{name}", M, K, N)
