"""CPU oracle for the group-wise quantized linear layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and this
package never imports the product: the two share no code.  The arithmetic lives
in ``qlin_oracle.c`` (plain C, built with gcc); this module only compiles it,
loads it with ctypes and marshals numpy arrays.

Functions (all numpy in, numpy out; bf16 and fp16 travel as their uint16 bit
patterns):

* ``act_quant_i8(x_bits)``            -> (q int8 [M,K], s float32 [M])
* ``pack_gptq(q, bits)``              -> (qweight int32, qzeros int32, n_out_of_range)
* ``unpack_gptq(qweight, K, N, bits)``-> q int8 [K,N]
* ``group_partials_i8(qa, qweight, K)``-> P int32 [G,M,N]
* ``gemm_w8a8_gs128(...)``            -> dict of y_bf16 / y_f32 / y64 / bound / abs_sum
* ``pack_tiles(qweight, K, bits)``      -> the GEMMs' tile layout of the words
* ``gemm_w4a16_g128(...)``            -> same dict
* ``gemm_w8a16(..., group_size)``     -> same dict (int8 weight-only; g32, g128 or per channel)
* ``dequant_w4a16(qweight, scales, K, N)`` -> w bf16 bits [K,N]
* ``argmax_bf16_rows(y_bits)``        -> int32 [M], greedy token per row
* ``ingest_nk(packed_nk, scales_ng, K, N, bits)`` -> (qweight [K*bits/32,N], scales [K/128,N])
* ``rmsnorm_bf16(x_bits, gamma_bits, eps)`` -> z bf16 bits [M,K] (decoder RMSNorm)
* ``silu_mul_bf16(gate_up_bits)``      -> z bf16 bits [M,I] (SiLU(gate) * up)
* ``rmsnorm_act_quant_i8`` / ``silu_mul_act_quant_i8`` -> (q, s, z): the producer, then act-quant
* ``f64_to_bf16(v)``                   -> bf16 bits of one binary64 value
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qlin_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no fused multiply-adds)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f32.restype = ctypes.c_float
            lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_bf16.restype = ctypes.c_uint16
            lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f32.restype = ctypes.c_float
            lib.orc_act_quant_i8.argtypes = [P, I, I, P, P]
            lib.orc_act_quant_i8.restype = None
            lib.orc_pack_gptq.argtypes = [P, I, I, ctypes.c_int, P, P]
            lib.orc_pack_gptq.restype = I
            lib.orc_unpack_gptq.argtypes = [P, I, I, ctypes.c_int, P]
            lib.orc_unpack_gptq.restype = None
            lib.orc_group_partials_i8.argtypes = [P, P, I, I, I, P]
            lib.orc_group_partials_i8.restype = None
            gemm_args = [P, P, P, P, I, I, I, P, I, P, I, P, P, P, P, P]
            lib.orc_gemm_w8a8_gs128.argtypes = gemm_args
            lib.orc_gemm_w8a8_gs128.restype = None
            lib.orc_gemm_w4a16_g128.argtypes = [P, P, P, I, I, I, P, I, P, I, P, P, P, P, P]
            lib.orc_gemm_w4a16_g128.restype = None
            lib.orc_dequant_w4a16.argtypes = [P, P, I, I, P]
            lib.orc_dequant_w4a16.restype = None
            lib.orc_argmax_bf16_rows.argtypes = [P, I, I, P]
            lib.orc_argmax_bf16_rows.restype = None
            lib.orc_ingest_nk.argtypes = [P, P, I, I, ctypes.c_int, P, P]
            lib.orc_ingest_nk.restype = None
            lib.orc_pack_tiles.argtypes = [P, I, I, ctypes.c_int, P]
            lib.orc_pack_tiles.restype = None
            lib.orc_gemm_w8a16.argtypes = [P, P, P, I, I, I, I, P, I, P, I, P, P, P, P, P]
            lib.orc_gemm_w8a16.restype = None
            lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.orc_f64_to_bf16.restype = ctypes.c_uint16
            lib.orc_rmsnorm_bf16.argtypes = [P, P, ctypes.c_double, I, I, P]
            lib.orc_rmsnorm_bf16.restype = None
            lib.orc_silu_mul_bf16.argtypes = [P, I, I, P]
            lib.orc_silu_mul_bf16.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------ scalar formats

def bf16_to_f32(bits: int) -> float:
    return float(_load().orc_bf16_to_f32(int(bits)))


def f32_to_bf16(value: float) -> int:
    return int(_load().orc_f32_to_bf16(float(value)))


def f16_to_f32(bits: int) -> float:
    return float(_load().orc_f16_to_f32(int(bits)))


# --------------------------------------------------------------- operations

def act_quant_i8(x_bits: np.ndarray):
    """x_bits: uint16 bf16 bit patterns [M, K] -> (q int8 [M,K], s float32 [M])."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    _load().orc_act_quant_i8(_ptr(x), M, K, _ptr(q), _ptr(s))
    return q, s


def pack_gptq(q: np.ndarray, bits: int):
    """q int8 [K, N] -> (qweight int32 [K*bits/32, N], qzeros int32 [K/128, N*bits/32], n_bad)."""
    q = _c(q, np.int8)
    K, N = q.shape
    per = 32 // bits
    qweight = np.empty((K // per, N), np.int32)
    qzeros = np.empty((K // 128, N // per), np.int32)
    bad = _load().orc_pack_gptq(_ptr(q), K, N, bits, _ptr(qweight), _ptr(qzeros))
    return qweight, qzeros, int(bad)


def unpack_gptq(qweight: np.ndarray, K: int, N: int, bits: int) -> np.ndarray:
    qw = _c(qweight, np.int32)
    q = np.empty((K, N), np.int8)
    _load().orc_unpack_gptq(_ptr(qw), K, N, bits, _ptr(q))
    return q


def group_partials_i8(qa: np.ndarray, qweight: np.ndarray, K: int) -> np.ndarray:
    qa = _c(qa, np.int8)
    qw = _c(qweight, np.int32)
    M = qa.shape[0]
    N = qw.shape[1]
    P = np.empty((K // 128, M, N), np.int32)
    _load().orc_group_partials_i8(_ptr(qa), _ptr(qw), M, N, K, _ptr(P))
    return P


def _index(idx, limit):
    if idx is None:
        return np.arange(limit, dtype=np.int64)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= limit):
        raise IndexError("index out of range")
    return idx


def _outputs(nr, nc):
    return {
        "y_bf16": np.empty((nr, nc), np.uint16),
        "y_f32": np.empty((nr, nc), np.float32),
        "y64": np.empty((nr, nc), np.float64),
        "bound": np.empty((nr, nc), np.float64),
        "abs_sum": np.empty((nr, nc), np.float64),
    }


def gemm_w8a8_gs128(qa, sa, qweight, scales_f16_bits, K, rows=None, cols=None):
    """W8A8 GS128 linear on a sub-grid of outputs.

    qa int8 [M,K], sa float32 [M], qweight int32 [K/4,N], scales fp16 bits
    uint16 [K/128,N].  rows/cols: optional index lists (default: all)."""
    qa = _c(qa, np.int8)
    sa = _c(sa, np.float32)
    qw = _c(qweight, np.int32)
    sc = _c(scales_f16_bits, np.uint16)
    M = qa.shape[0]
    N = qw.shape[1]
    r = _index(rows, M)
    c = _index(cols, N)
    out = _outputs(r.size, c.size)
    _load().orc_gemm_w8a8_gs128(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sc), M, N, K,
                                _ptr(r), r.size, _ptr(c), c.size,
                                _ptr(out["y_bf16"]), _ptr(out["y_f32"]),
                                _ptr(out["y64"]), _ptr(out["bound"]),
                                _ptr(out["abs_sum"]))
    return out


def gemm_w4a16_g128(x_bits, qweight, scales_bf16_bits, K, rows=None, cols=None):
    """W4A16 g128 linear on a sub-grid of outputs.

    x bf16 bits uint16 [M,K], qweight int32 [K/8,N], scales bf16 bits uint16
    [K/128,N].  rows/cols: optional index lists (default: all)."""
    x = _c(x_bits, np.uint16)
    qw = _c(qweight, np.int32)
    sc = _c(scales_bf16_bits, np.uint16)
    M = x.shape[0]
    N = qw.shape[1]
    r = _index(rows, M)
    c = _index(cols, N)
    out = _outputs(r.size, c.size)
    _load().orc_gemm_w4a16_g128(_ptr(x), _ptr(qw), _ptr(sc), M, N, K,
                                _ptr(r), r.size, _ptr(c), c.size,
                                _ptr(out["y_bf16"]), _ptr(out["y_f32"]),
                                _ptr(out["y64"]), _ptr(out["bound"]),
                                _ptr(out["abs_sum"]))
    return out


def gemm_w8a16(x_bits, qweight, scales_bf16_bits, K, group_size, rows=None, cols=None):
    """W8A16 weight-only int8 linear on a sub-grid of outputs.

    x bf16 bits [M,K], qweight int32 [K/4,N] (8-bit GPTQ words), scales bf16
    bits [K/group_size, N], or [1, N] for group_size 0 (one scale per column)."""
    x = _c(x_bits, np.uint16)
    qw = _c(qweight, np.int32)
    sc = _c(scales_bf16_bits, np.uint16)
    M = x.shape[0]
    N = qw.shape[1]
    r = _index(rows, M)
    c = _index(cols, N)
    out = _outputs(r.size, c.size)
    _load().orc_gemm_w8a16(_ptr(x), _ptr(qw), _ptr(sc), M, N, K, int(group_size),
                           _ptr(r), r.size, _ptr(c), c.size,
                           _ptr(out["y_bf16"]), _ptr(out["y_f32"]),
                           _ptr(out["y64"]), _ptr(out["bound"]),
                                _ptr(out["abs_sum"]))
    return out


def dequant_w4a16(qweight, scales_bf16_bits, K: int, N: int) -> np.ndarray:
    qw = _c(qweight, np.int32)
    sc = _c(scales_bf16_bits, np.uint16)
    w = np.empty((K, N), np.uint16)
    _load().orc_dequant_w4a16(_ptr(qw), _ptr(sc), K, N, _ptr(w))
    return w


def argmax_bf16_rows(y_bits) -> np.ndarray:
    """Greedy token per row of a bf16 output: index of the largest value,
    the lowest index on ties."""
    y = _c(y_bits, np.uint16)
    M, N = y.shape
    idx = np.empty(M, np.int32)
    _load().orc_argmax_bf16_rows(_ptr(y), M, N, _ptr(idx))
    return idx


def ingest_nk(packed_nk, scales_ng_bits, K: int, N: int, bits: int):
    """compressed-tensors orientation (words [N, K*bits/32], scales [N, K/128])
    -> the GEMMs' orientation (words [K*bits/32, N], scales [K/128, N])."""
    pk = _c(packed_nk, np.int32)
    sc = _c(scales_ng_bits, np.uint16)
    qw = np.empty((K * bits // 32, N), np.int32)
    so = np.empty((K // 128, N), np.uint16)
    _load().orc_ingest_nk(_ptr(pk), _ptr(sc), K, N, bits, _ptr(qw), _ptr(so))
    return qw, so


def pack_tiles(qweight, K: int, bits: int) -> np.ndarray:
    """GPTQ words [K*bits/32, N] -> the flat int32 tile layout (tile (f, g) =
    W x 128 words of features 128f.. and K group g, by f then g; 0 past N)."""
    qw = _c(qweight, np.int32)
    N = qw.shape[1]
    F = (N + 127) // 128
    out = np.empty(F * (K // 128) * (128 * bits // 32) * 128, np.int32)
    _load().orc_pack_tiles(_ptr(qw), K, N, bits, _ptr(out))
    return out


# ------------------------------------------------------------ fused producers

def f64_to_bf16(v: float) -> int:
    """One binary64 value -> bf16 bits, rounded once (ties to even)."""
    return int(_load().orc_f64_to_bf16(float(v)))


def rmsnorm_bf16(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of bf16 rows [M, K] with bf16 weight [K] -> bf16 bits [M, K]."""
    x = _c(x_bits, np.uint16)
    g = _c(gamma_bits, np.uint16)
    M, K = x.shape
    assert g.shape == (K,)
    z = np.empty((M, K), np.uint16)
    _load().orc_rmsnorm_bf16(_ptr(x), _ptr(g), float(eps), M, K, _ptr(z))
    return z


def silu_mul_bf16(gate_up_bits: np.ndarray) -> np.ndarray:
    """bf16 [M, 2I] (gate columns first, then up) -> bf16 bits [M, I]."""
    gu = _c(gate_up_bits, np.uint16)
    M, I2 = gu.shape
    assert I2 % 2 == 0
    z = np.empty((M, I2 // 2), np.uint16)
    _load().orc_silu_mul_bf16(_ptr(gu), M, I2 // 2, _ptr(z))
    return z


def rmsnorm_act_quant_i8(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float):
    """RMSNorm, then dynamic per-token INT8 quantization of its bf16 output:
    (q int8 [M,K], s float32 [M], z bf16 bits [M,K])."""
    z = rmsnorm_bf16(x_bits, gamma_bits, eps)
    q, s = act_quant_i8(z)
    return q, s, z


def silu_mul_act_quant_i8(gate_up_bits: np.ndarray):
    """SiLU(gate) * up, then dynamic per-token INT8 quantization of its bf16
    output: (q int8 [M,I], s float32 [M], z bf16 bits [M,I])."""
    z = silu_mul_bf16(gate_up_bits)
    q, s = act_quant_i8(z)
    return q, s, z
