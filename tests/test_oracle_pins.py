"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- hand-worked values, exact rational arithmetic, library routines
(numpy integer/fp64 matmul, numpy fp16, torch bf16 rounding), brute force and
invariants.  None of these needs a GPU."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from w4a16_linear_layers_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_bf16_bits(values_f32: np.ndarray) -> np.ndarray:
    """Library rounding fp32 -> bf16 (torch, round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(values_f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_of(values) -> np.ndarray:
    return torch_bf16_bits(np.asarray(values, np.float32))


# ------------------------------------------------------------------ formats

def test_f16_decode_all_patterns(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    got = np.array([oracle_lib.f16_to_f32(int(p)) for p in pats], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_rounding_matches_torch(oracle_lib):
    rng = np.random.default_rng(1)
    vals = rng.standard_normal(20000).astype(np.float32) * np.float32(1000.0)
    bits = vals.view(np.uint32)
    # exact ties (lower 16 bits == 0x8000), both parities, plus carries into the exponent
    ties = ((bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    carry = np.array([0x3F7FFFFF, 0x3F7F8000, 0x477F8000, 0xBF7FC000], np.uint32).view(np.float32)
    allv = np.concatenate([vals, ties[:5000], carry, np.float32([0.0, -0.0, 1e-40, -3e-39])])
    ref = bf16_of(allv)
    got = np.array([oracle_lib.f32_to_bf16(float(v)) for v in allv], np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([oracle_lib.bf16_to_f32(int(b)) for b in ref[:1000]], np.float32)
    assert np.array_equal(back.view(np.uint32), ref[:1000].astype(np.uint32) << 16)


# --------------------------------------------------------------- act-quant

def _read_act_golden():
    rows = []
    with open(os.path.join(GOLDEN, "act_quant_hand.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            xs, ss, qs = line.split("|")
            x = [float(v) for v in xs.split(":")[1].split()]
            s = float.fromhex(ss.split(":")[1].strip())
            q = [int(v) for v in qs.split(":")[1].split()]
            rows.append((x, s, q))
    return rows


def test_act_quant_hand_rows(oracle_lib):
    for x, s, q in _read_act_golden():
        xb = bf16_of(x)[None, :]
        assert np.array_equal(synth.bf16_values(xb)[0], np.float32(x)), "fixture not exact in bf16"
        gq, gs = oracle_lib.act_quant_i8(xb)
        assert gs[0] == np.float32(s)
        assert gq[0].tolist() == q


def _rn32(v: Fraction) -> Fraction:
    """Exact round-to-nearest-even of a rational to binary32 (normal range)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    t = a / ulp
    fl = t.numerator // t.denominator
    rem = t - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def _rint_even(v: Fraction) -> int:
    fl = v.numerator // v.denominator
    rem = v - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def test_act_quant_exact_rational(oracle_lib):
    """Every q equals rint(RN32(x / RN32(amax / 127))) evaluated in exact
    rational arithmetic (round half to even at both steps)."""
    M, K = 6, 512
    xb = synth.activations(11, "pin/act", M, K, "outliers")
    q, s = oracle_lib.act_quant_i8(xb)
    x = synth.bf16_values(xb)
    for m in range(M):
        amax = Fraction(float(np.max(np.abs(x[m]))))
        sm = _rn32(amax / 127)
        assert Fraction(float(s[m])) == sm
        for k in range(K):
            xv = Fraction(float(x[m, k]))
            want = max(-127, min(127, _rint_even(_rn32(xv / sm))))
            assert int(q[m, k]) == want, (m, k)


def test_act_quant_divide_not_reciprocal(oracle_lib):
    """Search for an element whose x/s and x*(127/amax) round to different
    integers; the oracle must follow the IEEE divide (checked exactly)."""
    found = None
    for trial in range(200):
        xb = synth.activations(100 + trial, "pin/divform", 1, 1024, "normal")
        x = synth.bf16_values(xb)[0]
        amax = np.float32(np.max(np.abs(x)))
        sf = np.float32(amax / np.float32(127.0))
        div = np.rint(x / sf)
        mul = np.rint(x * (np.float32(127.0) / amax))
        idx = np.nonzero(div != mul)[0]
        if idx.size:
            found = (xb, int(idx[0]))
            break
    assert found is not None, "no divide-sensitive element found"
    xb, k = found
    q, s = oracle_lib.act_quant_i8(xb)
    x = synth.bf16_values(xb)[0]
    sm = _rn32(Fraction(float(np.max(np.abs(x)))) / 127)
    assert int(q[0, k]) == _rint_even(_rn32(Fraction(float(x[k])) / sm))


def test_act_quant_invariants(oracle_lib):
    M, K = 16, 1024
    for kind in ("outliers", "normal", "silu_mul", "normal2"):
        xb = synth.activations(3, "pin/inv/" + kind, M, K, kind)
        q, s = oracle_lib.act_quant_i8(xb)
        x = synth.bf16_values(xb).astype(np.float64)
        sd = s.astype(np.float64)[:, None]
        assert np.all(np.abs(q.astype(np.int32)) <= 127)
        assert np.all(np.max(np.abs(q.astype(np.int32)), axis=1) == 127)
        # |x/s - q| <= 1/2 up to the rounding of the fp32 quotient
        err = np.abs(x / sd - q)
        assert np.all(err <= 0.5 + 127 * 2.0**-23)


def test_act_quant_zero_and_tiny_rows(oracle_lib):
    xb = np.zeros((3, 256), np.uint16)
    xb[1, 7] = bf16_of([1e-30])[0]          # tiny but normal
    xb[2, :] = bf16_of(np.full(256, -3.0))
    q, s = oracle_lib.act_quant_i8(xb)
    assert s[0] == 0 and not q[0].any()
    assert q[1, 7] == 127 and np.count_nonzero(q[1]) == 1
    assert np.all(q[2] == -127)


# -------------------------------------------------------------------- pack

def _read_pack_golden():
    out = []
    with open(os.path.join(GOLDEN, "pack_words.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            b, qs, w = line.split("|")
            out.append((int(b), [int(v) for v in qs.split()], int(w.strip(), 16)))
    return out


def test_pack_hand_words(oracle_lib):
    for bits, qs, word in _read_pack_golden():
        per = 32 // bits
        q = np.zeros((128, 8), np.int8)
        q[:per, 1] = qs
        qw, qz, bad = oracle_lib.pack_gptq(q, bits)
        assert bad == 0
        assert int(qw[0, 1]) & 0xFFFFFFFF == word
        zero_word = 0x80808080 if bits == 8 else 0x88888888
        assert np.all(qz.view(np.uint32) == zero_word)
        assert int(qw[0, 0]) & 0xFFFFFFFF == zero_word


def test_pack_roundtrip_and_range(oracle_lib):
    for bits, lo, hi in ((8, -128, 127), (4, -8, 7)):
        q = synth.randint(5, f"pin/pack{bits}", (512, 40), lo, hi, np.int8)
        qw, qz, bad = oracle_lib.pack_gptq(q, bits)
        assert bad == 0 and qw.shape == (512 * bits // 32, 40)
        assert np.array_equal(oracle_lib.unpack_gptq(qw, 512, 40, bits), q)
        # an independent numpy unpack of the same words
        per = 32 // bits
        u = qw.view(np.uint32)
        ref = np.empty_like(q)
        for i in range(per):
            ref[i::per] = ((u >> np.uint32(bits * i)) & np.uint32((1 << bits) - 1)).astype(np.int32) - (1 << (bits - 1))
        assert np.array_equal(ref, q)
    q = np.zeros((128, 4), np.int8)
    q[3, 2] = 9        # outside int4
    q[5, 1] = -9
    _, _, bad = oracle_lib.pack_gptq(q, 4)
    assert bad == 2


# ------------------------------------------------------------------ W8A8

def test_group_partials_brute_force_all_pairs(oracle_lib):
    """All 255^2 (a, w) pairs on a 128-long group: P = 128 * a * w."""
    vals = np.arange(-127, 128, dtype=np.int8)
    qa = np.repeat(vals[:, None], 128, axis=1)            # row i constant a_i
    qwt = np.repeat(vals[None, :], 128, axis=0)          # column j constant w_j
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    P = oracle_lib.group_partials_i8(qa, qw, 128)
    want = 128 * vals.astype(np.int64)[:, None] * vals.astype(np.int64)[None, :]
    assert P.shape == (1, 255, 255)
    assert np.array_equal(P[0].astype(np.int64), want)


def test_group_partials_vs_numpy_matmul(oracle_lib):
    M, K, N = 5, 640, 33
    qa = synth.randint(7, "pin/gp/a", (M, K), -127, 127)
    qwt = synth.randint(7, "pin/gp/w", (K, N), -127, 127)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    P = oracle_lib.group_partials_i8(qa, qw, K)
    for g in range(K // 128):
        sl = slice(128 * g, 128 * (g + 1))
        ref = qa[:, sl].astype(np.int64) @ qwt[sl].astype(np.int64)
        assert np.array_equal(P[g].astype(np.int64), ref)
    # extreme magnitudes: all +-127 stays exact and within int32
    qa2 = np.full((2, 128), 127, np.int8)
    qa2[1] = -127
    qw2, _, _ = oracle_lib.pack_gptq(np.full((128, 2), -127, np.int8), 8)
    P2 = oracle_lib.group_partials_i8(qa2, qw2, 128)
    assert P2[0, 0, 0] == -128 * 127 * 127 and P2[0, 1, 1] == 128 * 127 * 127


def test_w8a8_hand_fixture(oracle_lib):
    rows = []
    with open(os.path.join(GOLDEN, "w8a8_hand.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            c, ps, yf, yb = line.split("|")
            rows.append((int(c), [int(v) for v in ps.split()], float(yf), int(yb.strip(), 16)))
    K = 256
    qa = np.ones((1, K), np.int8)
    qa[0, 128:] = -1
    qwt = np.zeros((K, 2), np.int8)
    qwt[:128, 0], qwt[128:, 0] = 2, 3
    qwt[:128, 1], qwt[128:, 1] = -127, 127
    sw = np.array([[0.5, 2.0**-7], [0.25, 1.0]])
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    out = oracle_lib.gemm_w8a8_gs128(qa, np.float32([0.25]), qw, synth.f16_bits(sw), K)
    P = oracle_lib.group_partials_i8(qa, qw, K)
    for c, ps, yf, yb in rows:
        assert [int(P[0, 0, c]), int(P[1, 0, c])] == ps
        assert out["y_f32"][0, c] == np.float32(yf)
        assert int(out["y_bf16"][0, c]) == yb


def test_w8a8_unit_scales_is_integer_matmul(oracle_lib):
    """All scales 1: y = bf16(integer matmul), exact in fp32 for these sizes."""
    M, K, N = 7, 384, 19
    qa = synth.randint(9, "pin/unit/a", (M, K), -127, 127)
    qwt = synth.randint(9, "pin/unit/w", (K, N), -127, 127)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    ones = np.full((K // 128, N), 0x3C00, np.uint16)       # fp16 1.0
    out = oracle_lib.gemm_w8a8_gs128(qa, np.ones(M, np.float32), qw, ones, K)
    ref = qa.astype(np.int64) @ qwt.astype(np.int64)
    assert np.all(np.abs(ref) < 2**24)
    assert np.array_equal(out["y_f32"], ref.astype(np.float32))
    assert np.array_equal(out["y_bf16"], bf16_of(ref.astype(np.float32)))


def test_w8a8_fp64_invariant(oracle_lib):
    """y64 is the dequantize-then-fp64-matmul value (numpy route from the
    generator's unpacked weights) and the fp32 chain lies within the bound."""
    M, K, N = 9, 1280, 70
    xb = synth.activations(21, "pin/f64/x", M, K, "outliers")
    qa, sa = oracle_lib.act_quant_i8(xb)
    qwt, swb = synth.w8a8_weights(21, "pin/f64/w", K, N)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    out = oracle_lib.gemm_w8a8_gs128(qa, sa, qw, swb, K)
    sw = swb.view(np.float16).astype(np.float64)
    w_dq = qwt.astype(np.float64) * np.repeat(sw, 128, axis=0)
    a_dq = qa.astype(np.float64) * sa.astype(np.float64)[:, None]
    ref = a_dq @ w_dq
    assert np.allclose(out["y64"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.all(np.abs(out["y_f32"].astype(np.float64) - out["y64"]) <= out["bound"])
    # bf16 output is the round-to-nearest-even image of the fp32 chain
    assert np.array_equal(out["y_bf16"], bf16_of(out["y_f32"]))
    # sub-grid evaluation agrees with the full one
    rows, cols = np.array([8, 0, 3]), np.array([69, 1, 40])
    sub = oracle_lib.gemm_w8a8_gs128(qa, sa, qw, swb, K, rows, cols)
    assert np.array_equal(sub["y_bf16"], out["y_bf16"][np.ix_(rows, cols)])


def test_w8a8_identity_probe(oracle_lib):
    """Identity probe: feeding I_K through the W8A8 linear recovers q*s
    within two fp32 roundings (plus the bf16 output rounding)."""
    K, N = 256, 24
    xb = bf16_of(np.eye(K, dtype=np.float32))
    qa, sa = oracle_lib.act_quant_i8(xb)
    assert np.all(np.diag(qa) == 127) and np.count_nonzero(qa) == K
    qwt, swb = synth.w8a8_weights(4, "pin/probe8", K, N)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    out = oracle_lib.gemm_w8a8_gs128(qa, sa, qw, swb, K)
    w_dq = qwt.astype(np.float64) * np.repeat(swb.view(np.float16).astype(np.float64), 128, axis=0)
    assert np.all(np.abs(out["y_f32"] - w_dq) <= 2.0**-21 * np.abs(w_dq))


# ----------------------------------------------------------------- W4A16

def test_w4a16_identity_probe_bit_exact(oracle_lib):
    """Identity probe: y = bf16(q * s) exactly (library rounding of the exact
    fp32 product)."""
    K, N = 256, 40
    qwt, sb = synth.w4a16_weights(8, "pin/probe4", K, N)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 4)
    xb = bf16_of(np.eye(K, dtype=np.float32))
    out = oracle_lib.gemm_w4a16_g128(xb, qw, sb, K)
    s = np.repeat(synth.bf16_values(sb), 128, axis=0)
    want = bf16_of(qwt.astype(np.float32) * s)
    assert np.array_equal(out["y_bf16"], want)
    assert np.array_equal(oracle_lib.dequant_w4a16(qw, sb, K, N), want)


def test_w4a16_unit_scales_integer(oracle_lib):
    M, K, N = 4, 512, 9
    x_int = synth.randint(12, "pin/w4unit/x", (M, K), -3, 3).astype(np.float32)
    xb = bf16_of(x_int)
    qwt = synth.randint(12, "pin/w4unit/w", (K, N), -8, 7)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 4)
    ones = np.full((K // 128, N), 0x3F80, np.uint16)      # bf16 1.0
    out = oracle_lib.gemm_w4a16_g128(xb, qw, ones, K)
    ref = x_int.astype(np.int64) @ qwt.astype(np.int64)
    assert np.array_equal(out["y_f32"], ref.astype(np.float32))


def test_w4a16_fp64_invariant(oracle_lib):
    M, K, N = 6, 1152, 50
    xb = synth.activations(13, "pin/w4f64/x", M, K, "normal")
    qwt, sb = synth.w4a16_weights(13, "pin/w4f64/w", K, N)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 4)
    out = oracle_lib.gemm_w4a16_g128(xb, qw, sb, K)
    s = np.repeat(synth.bf16_values(sb), 128, axis=0)
    w = synth.bf16_values(bf16_of(qwt.astype(np.float32) * s)).astype(np.float64)
    ref = synth.bf16_values(xb).astype(np.float64) @ w
    assert np.allclose(out["y64"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.all(np.abs(out["y_f32"].astype(np.float64) - out["y64"]) <= out["bound"])
    assert np.array_equal(out["y_bf16"], bf16_of(out["y_f32"]))


# ------------------------------------------------------------- greedy argmax

def test_argmax_rows_hand_cases(oracle_lib):
    """Largest value per row, lowest index on ties; -0 and +0 are equal."""
    y = synth.bf16_bits(np.array([
        [-1.0, -0.5, -0.5, -2.0],     # tie between 1 and 2 -> 1
        [2.0, 2.0, 1.0, 2.0],         # three-way tie -> 0
        [-0.0, 0.0, -0.0, 0.0],       # signed zeros compare equal -> 0
        [-3.0, -2.0, -7.0, -2.0],     # all negative -> 1
        [1.0, 1.0078125, 1.0, 0.5],   # one bf16 ulp above 1 -> 1
    ], np.float32))
    assert oracle_lib.argmax_bf16_rows(y).tolist() == [1, 0, 0, 1, 1]


def test_argmax_rows_matches_numpy_first_max(oracle_lib):
    """Against numpy's argmax of the decoded values (first maximum), on rows
    with many exact ties (few distinct values)."""
    rng = np.random.default_rng(3)
    vals = rng.integers(-4, 5, size=(64, 1000)).astype(np.float32) * 0.25
    y = synth.bf16_bits(vals)
    want = np.argmax(synth.bf16_values(y).astype(np.float64), axis=1)
    assert np.array_equal(oracle_lib.argmax_bf16_rows(y), want.astype(np.int32))


# ------------------------------------------------- [N, K/8] ingest (compressed-tensors)

def _pack_rows_numpy(q: np.ndarray, bits: int) -> np.ndarray:
    """Independent packer for the per-output-row orientation: word (n, kk)
    field i = q[(32/bits) kk + i, n] + 2^(bits-1), least significant first."""
    K, N = q.shape
    per = 32 // bits
    u = (q.astype(np.int64) + (1 << (bits - 1))).T.reshape(N, K // per, per)
    words = np.zeros((N, K // per), np.int64)
    for i in range(per):
        words |= (u[:, :, i] & ((1 << bits) - 1)) << (bits * i)
    return words.astype(np.uint32).view(np.int32)


@pytest.mark.parametrize("bits", [4, 8])
def test_ingest_nk_matches_gptq_packing(oracle_lib, bits):
    """The row-oriented words of q, ingested, equal the GPTQ words of q; the
    scales are transposed unchanged."""
    rng = np.random.default_rng(5 + bits)
    lim = (1 << (bits - 1)) - 1
    K, N = 256, 72
    q = rng.integers(-lim, lim + 1, size=(K, N)).astype(np.int8)
    scales_ng = rng.integers(0, 65536, size=(N, K // 128)).astype(np.uint16)
    qw, sc = oracle_lib.ingest_nk(_pack_rows_numpy(q, bits), scales_ng, K, N, bits)
    want, _, _ = oracle_lib.pack_gptq(q, bits)
    assert np.array_equal(qw, want)
    assert np.array_equal(sc, scales_ng.T)


def test_ingest_nk_hand_word(oracle_lib):
    """One 4-bit column: q[0..7, 0] = -8..-1 -> nibbles 0..7 -> 0x76543210."""
    q = np.zeros((128, 1), np.int8)
    q[:8, 0] = np.arange(-8, 0)
    packed = _pack_rows_numpy(q, 4)
    assert packed[0, 0] == 0x76543210
    qw, _ = oracle_lib.ingest_nk(packed, np.zeros((1, 1), np.uint16), 128, 1, 4)
    assert qw[0, 0] == 0x76543210


# ------------------------------------------------------ W8A16 (int8 weight-only)

def _expand_scales(sb, K, gs):
    v = synth.bf16_values(sb)
    return np.repeat(v, K, axis=0) if gs == 0 else np.repeat(v, gs, axis=0)


@pytest.mark.parametrize("gs", [32, 128, 0])
def test_w8a16_identity_probe_bit_exact(oracle_lib, gs):
    """Identity probe: y = bf16(q * s) exactly (library rounding of the exact
    fp32 product), for group-32, group-128 and per-column scales."""
    K, N = 256, 40
    qwt, sb = synth.w8a16_weights(8, f"pin/probe8/{gs}", K, N, gs)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    xb = bf16_of(np.eye(K, dtype=np.float32))
    out = oracle_lib.gemm_w8a16(xb, qw, sb, K, gs)
    want = bf16_of(qwt.astype(np.float32) * _expand_scales(sb, K, gs))
    assert np.array_equal(out["y_bf16"], want)


def test_w8a16_unit_scales_integer(oracle_lib):
    M, K, N = 4, 512, 9
    x_int = synth.randint(12, "pin/w8unit/x", (M, K), -3, 3).astype(np.float32)
    qwt = synth.randint(12, "pin/w8unit/w", (K, N), -127, 127)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    ones = np.full((K // 32, N), 0x3F80, np.uint16)       # bf16 1.0
    out = oracle_lib.gemm_w8a16(bf16_of(x_int), qw, ones, K, 32)
    ref = x_int.astype(np.int64) @ qwt.astype(np.int64)
    assert np.array_equal(out["y_f32"], ref.astype(np.float32))


@pytest.mark.parametrize("gs", [32, 0])
def test_w8a16_fp64_invariant(oracle_lib, gs):
    M, K, N = 6, 1152, 50
    xb = synth.activations(13, f"pin/w8f64/{gs}/x", M, K, "normal")
    qwt, sb = synth.w8a16_weights(13, f"pin/w8f64/{gs}/w", K, N, gs)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    out = oracle_lib.gemm_w8a16(xb, qw, sb, K, gs)
    w = synth.bf16_values(bf16_of(qwt.astype(np.float32) * _expand_scales(sb, K, gs))).astype(np.float64)
    ref = synth.bf16_values(xb).astype(np.float64) @ w
    assert np.allclose(out["y64"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.all(np.abs(out["y_f32"].astype(np.float64) - out["y64"]) <= out["bound"])
    assert np.array_equal(out["y_bf16"], bf16_of(out["y_f32"]))


# ------------------------------------------------------------ fused producers

def _bf16_value(bits: int) -> Fraction:
    """Exact value of a finite bf16 bit pattern."""
    return Fraction(float(np.array([int(bits) << 16], np.uint32).view(np.float32)[0]))


def _round_bf16_brute(v: Fraction) -> int:
    """Nearest bf16 to an exact rational (ties to the even pattern), found by
    testing the neighbours of torch's rounding of the nearest float32."""
    approx = int(bf16_of([float(v)])[0])
    best = None
    for b in (approx - 1, approx, approx + 1):
        if b < 0 or (b & 0x7F80) == 0x7F80:
            continue
        if (b >> 15) != (approx >> 15) and v != 0:
            continue
        d = abs(_bf16_value(b) - v)
        if best is None or d < best[0] or (d == best[0] and b % 2 == 0):
            best = (d, b)
    return best[1]


def test_f64_to_bf16_matches_exact_rounding(oracle_lib):
    rng = np.random.default_rng(11)
    vals = list(rng.standard_normal(3000) * np.exp(rng.uniform(-60, 60, 3000)))
    # doubles just off bf16 ties, which a double rounding through fp32 would get wrong
    for base in (1.0, 1.5, 3.0, 0.8125, 1e-20, 7e30):
        m, e = np.frexp(base)
        ulp = 2.0 ** (e - 8)
        tie = (np.floor(base / ulp) + 0.5) * ulp
        vals += [tie, tie + tie * 2 ** -40, tie - tie * 2 ** -40, -tie]
    for v in vals:
        got = oracle_lib.f64_to_bf16(float(v))
        assert got == _round_bf16_brute(Fraction(float(v))), (v, hex(got))
    assert oracle_lib.f64_to_bf16(0.0) == 0 and oracle_lib.f64_to_bf16(-0.0) == 0x8000
    assert oracle_lib.f64_to_bf16(1e39) == 0x7F80 and oracle_lib.f64_to_bf16(-1e39) == 0xFF80


def test_rmsnorm_constant_rows_give_gamma(oracle_lib):
    """x = c on a whole row: mean x^2 = c^2, so z = gamma exactly (eps = 0)."""
    K = 256
    cs = [3.0, -0.15625, 1024.0, 2.0 ** -20]
    x = np.stack([bf16_of(np.full(K, c)) for c in cs])
    g = bf16_of(np.linspace(-2.0, 2.0, K))
    z = oracle_lib.rmsnorm_bf16(x, g, 0.0)
    for i, c in enumerate(cs):
        want = g if c > 0 else g ^ np.uint16(0x8000)
        nz = g != 0
        assert np.array_equal(z[i][nz], want[nz]), c


def test_rmsnorm_hand_row(oracle_lib):
    """[3, 4, 0, 0]: mean of squares 25/4, rstd = 2/5, t = (6/5, 8/5, 0, 0)."""
    x = bf16_of([3.0, 4.0, 0.0, 0.0])[None, :]
    g = bf16_of([1.0, 2.0, 0.5, 4.0])
    z = oracle_lib.rmsnorm_bf16(x, g, 0.0)[0]
    t0 = _round_bf16_brute(Fraction(6, 5))
    t1 = _round_bf16_brute(Fraction(8, 5))
    assert z[0] == _round_bf16_brute(_bf16_value(t0))
    assert z[1] == _round_bf16_brute(2 * _bf16_value(t1))
    assert z[2] == 0 and z[3] == 0


def test_rmsnorm_eps_under_the_root(oracle_lib):
    """K = 1, x = 1, eps = 3: 1 / sqrt(1 + 3) = 1/2; an all-zero row stays 0."""
    g = bf16_of([3.0])
    z = oracle_lib.rmsnorm_bf16(bf16_of([[1.0], [0.0]]), g, 3.0)
    assert z[0, 0] == bf16_of([1.5])[0] and z[1, 0] == 0


def test_rmsnorm_power_of_two_scale_invariance(oracle_lib):
    x = synth.activations(3, "pins/rms", 6, 640, "outliers")
    g = synth.bf16_bits(1.0 + 0.1 * synth.normal(3, "pins/rms/g", (640,)))
    z = oracle_lib.rmsnorm_bf16(x, g, 0.0)
    for j in (-7, 3, 20):
        xs = bf16_of(synth.bf16_values(x) * np.float32(2.0 ** j))
        assert np.array_equal(oracle_lib.rmsnorm_bf16(xs, g, 0.0), z)


def test_silu_mul_hand_values_and_layout(oracle_lib):
    """Row [gate | up] = [1, 0, -30, 30 | 2, 5, 1, 3]."""
    gu = bf16_of([1.0, 0.0, -30.0, 30.0, 2.0, 5.0, 1.0, 3.0])[None, :]
    z = oracle_lib.silu_mul_bf16(gu)[0]
    e1 = Fraction(np.exp(-1.0))
    assert z[0] == _round_bf16_brute(2 / (1 + e1))
    assert z[1] == 0
    e30 = Fraction(np.exp(-30.0))
    assert z[2] == _round_bf16_brute(Fraction(-30) / (1 + 1 / e30))
    assert z[3] == bf16_of([90.0])[0]      # SiLU(30) = 30 - 2.8e-12 -> 30, times 3


def test_silu_odd_identity(oracle_lib):
    """SiLU(g) - SiLU(-g) = g: with up = 1 the two rounded outputs differ by g
    up to their roundings."""
    gs = np.linspace(-12.0, 12.0, 97)
    gate = bf16_of(gs)
    g_vals = synth.bf16_values(gate).astype(np.float64)
    gu_pos = np.concatenate([gate, bf16_of(np.ones_like(gs))])[None, :]
    gu_neg = np.concatenate([gate ^ np.uint16(0x8000), bf16_of(np.ones_like(gs))])[None, :]
    zp = synth.bf16_values(oracle_lib.silu_mul_bf16(gu_pos)[0]).astype(np.float64)
    zn = synth.bf16_values(oracle_lib.silu_mul_bf16(gu_neg)[0]).astype(np.float64)
    tol = 2.0 ** -8 * (np.abs(zp) + np.abs(zn)) + 1e-30
    assert np.all(np.abs(zp - zn - g_vals) <= tol)


def test_fused_producers_compose_with_act_quant(oracle_lib):
    x = synth.activations(4, "pins/fp", 5, 384, "normal")
    g = synth.bf16_bits(1.0 + 0.1 * synth.normal(4, "pins/fp/g", (384,)))
    q, s, z = oracle_lib.rmsnorm_act_quant_i8(x, g, 1e-6)
    q2, s2 = oracle_lib.act_quant_i8(z)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    gu = synth.activations(4, "pins/fp/gu", 5, 2 * 384, "normal")
    q, s, z = oracle_lib.silu_mul_act_quant_i8(gu)
    q2, s2 = oracle_lib.act_quant_i8(z)
    assert np.array_equal(q, q2) and np.array_equal(s, s2) and z.shape == (5, 384)


# ------------------------------------------------------------ equivariance

def test_act_quant_power_of_two_and_sign_equivariance(oracle_lib):
    """Scaling a row by 2^j scales s by 2^j and keeps q (every step is exact
    under a power of two); negating a row negates q and keeps s."""
    xb = synth.activations(5, "pin/eqv", 12, 640, "outliers")
    q, s = oracle_lib.act_quant_i8(xb)
    x = synth.bf16_values(xb)
    for j in (-9, 4, 30):
        q2, s2 = oracle_lib.act_quant_i8(bf16_of(x * np.float32(2.0 ** j)))
        assert np.array_equal(q2, q)
        assert np.array_equal(s2, (s * np.float32(2.0 ** j)).astype(np.float32))
    qn, sn = oracle_lib.act_quant_i8(xb ^ np.uint16(0x8000))
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)


def test_w8a8_scale_and_sign_equivariance(oracle_lib):
    """Doubling every weight scale doubles the fp32 chain exactly; negating
    every weight negates it exactly (round-to-nearest is symmetric)."""
    M, K, N = 5, 768, 96
    xb = synth.activations(6, "pin/eqv8/x", M, K, "normal")
    qa, sa = oracle_lib.act_quant_i8(xb)
    qwt, swb = synth.w8a8_weights(6, "pin/eqv8/w", K, N)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 8)
    base = oracle_lib.gemm_w8a8_gs128(qa, sa, qw, swb, K)
    sw2 = synth.f16_bits(swb.view(np.float16).astype(np.float64) * 2.0)
    dbl = oracle_lib.gemm_w8a8_gs128(qa, sa, qw, sw2, K)
    assert np.array_equal(dbl["y_f32"], base["y_f32"] * np.float32(2.0))
    qwn, _, _ = oracle_lib.pack_gptq((-qwt.astype(np.int16)).astype(np.int8), 8)
    neg = oracle_lib.gemm_w8a8_gs128(qa, sa, qwn, swb, K)
    assert np.array_equal(neg["y_f32"], -base["y_f32"])


def test_w4a16_scale_equivariance(oracle_lib):
    """Doubling every bf16 scale doubles each dequantized weight exactly, and
    so the fp32 accumulation."""
    M, K, N = 4, 512, 72
    xb = synth.activations(7, "pin/eqv4/x", M, K, "normal")
    qwt, sb = synth.w4a16_weights(7, "pin/eqv4/w", K, N)
    qw, _, _ = oracle_lib.pack_gptq(qwt, 4)
    base = oracle_lib.gemm_w4a16_g128(xb, qw, sb, K)
    sb2 = bf16_of(synth.bf16_values(sb) * np.float32(2.0))
    dbl = oracle_lib.gemm_w4a16_g128(xb, qw, sb2, K)
    assert np.array_equal(dbl["y_f32"], base["y_f32"] * np.float32(2.0))


# ------------------------------------------------------------ tile layout

@pytest.mark.parametrize("K,N,bits", [(128, 128, 8), (256, 200, 8), (384, 130, 4), (128, 8, 4),
                                      (512, 384, 8)])
def test_pack_tiles_matches_a_reshape_of_the_words(oracle_lib, K, N, bits):
    """The oracle's tile layout equals the GPTQ words padded to a multiple of
    128 columns and viewed as [G, W, F, 128] with the feature-tile axis moved
    first (an independent numpy formulation: reshape and transpose)."""
    W = 128 * bits // 32
    rng = np.random.default_rng(K + N + bits)
    qw = rng.integers(-2**31, 2**31 - 1, size=(K * bits // 32, N), dtype=np.int64).astype(np.int32)
    F = -(-N // 128)
    padded = np.zeros((K * bits // 32, F * 128), np.int32)
    padded[:, :N] = qw
    want = padded.reshape(K // 128, W, F, 128).transpose(2, 0, 1, 3).reshape(-1)
    got = oracle_lib.pack_tiles(qw, K, bits)
    assert np.array_equal(got, want)


def test_pack_tiles_hand_words(oracle_lib):
    """K = 256 (two groups), N = 130 (two feature tiles, the second with two
    live columns), 8-bit: W = 32 words per tile column.  Tile (f=1, g=1) starts
    at word (1 * 2 + 1) * 32 * 128; its word (kk=5, j=1) is GPTQ word
    (32 + 5, 129), and its column j = 2 is past N."""
    K, N = 256, 130
    qw = (np.arange(64)[:, None] * 1000 + np.arange(N)[None, :]).astype(np.int32)
    t = oracle_lib.pack_tiles(qw, K, 8)
    assert t.size == 2 * 2 * 32 * 128
    base = (1 * 2 + 1) * 32 * 128
    assert t[base + 5 * 128 + 1] == 37 * 1000 + 129
    assert t[base + 5 * 128 + 2] == 0
    assert t[(0 * 2 + 1) * 32 * 128 + 0 * 128 + 127] == 32 * 1000 + 127     # tile (0, 1)


# ------------------------------------------------------------ input generator

@pytest.mark.parametrize("shape,lo,hi", [((64, 130), -127, 127), ((257,), -7, 7), ((3, 5, 7), -127, 127)])
def test_device_draw_equals_the_host_draw(shape, lo, hi):
    """synth.randint_device (torch, used for gigabyte weight matrices) draws
    the host generator's integers bit for bit; run here with torch on the
    CPU, which computes the same int64 arithmetic."""
    host = synth.randint(7, "pins/device_draw", shape, lo, hi)
    dev = synth.randint_device(7, "pins/device_draw", shape, lo, hi, "cpu")
    assert np.array_equal(dev.numpy().reshape(host.shape), host)
