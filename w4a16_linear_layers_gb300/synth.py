"""Seeded synthetic inputs for the quantized linear layer.

This module only draws numbers: it holds none of the layer's arithmetic (no
quantization, no packing, no products).  Tests, the benchmark and the oracle
checks all take their inputs from here, so the CUDA path and the oracle see the
same bytes.

Generator: counter-based splitmix64.  Word i of stream ``name`` under ``seed``
is ``mix64(base(seed, name) + (i + 1) * 0x9E3779B97F4A7C15)``, where ``mix64`` is
the splitmix64 output function and ``base`` mixes the seed with the CRC-32 of
the stream name.  Every tensor draws from its own named stream, so adding a
tensor never shifts another one.

Derived draws:
* uniform(0,1]: ``((w >> 11) + 1) * 2^-53``;
* integers in [lo, hi]: ``lo + (w >> 11) % (hi - lo + 1)`` (modulo bias < 2^-44);
* normals: Box-Muller in fp64 on two uniforms, ``sqrt(-2 ln u1) cos(2 pi u2)``;
* log-uniform in [a, b]: ``exp(ln a + u (ln b - ln a))`` in fp64;
* bf16 / fp16 values are the round-to-nearest-even images of those fp64 draws
  (fp64 -> fp32 -> bf16 for bf16; numpy's fp64 -> fp16 for fp16).

Large draws are produced in chunks on a thread pool (numpy releases the GIL).
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _base(seed: int, name: str) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(int(seed) * 0x100000001B3 + zlib.crc32(name.encode())) & (2**64 - 1)],
                     dtype=np.uint64)
        return _mix64(s)[0]


def _words(base: np.uint64, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(base + idx * _GOLDEN)


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(16, os.cpu_count() or 1))


def _fill(total: int, fn, out: np.ndarray) -> np.ndarray:
    """Run fn(start, count) -> array over chunks, writing into out.ravel()."""
    flat = out.reshape(-1)
    spans = [(s, min(_CHUNK, total - s)) for s in range(0, total, _CHUNK)]
    if len(spans) <= 1:
        for s, c in spans:
            flat[s:s + c] = fn(s, c)
        return out

    def work(span):
        s, c = span
        flat[s:s + c] = fn(s, c)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, spans))
    return out


def _count(shape) -> int:
    return int(np.prod(shape, dtype=np.int64)) if len(shape) else 1


def uniform01(seed: int, name: str, shape) -> np.ndarray:
    """fp64 uniform draws in (0, 1]."""
    base = _base(seed, name)
    n = _count(shape)
    out = np.empty(shape, np.float64)

    def fn(s, c):
        return ((_words(base, s, c) >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53

    return _fill(n, fn, out)


def randint(seed: int, name: str, shape, lo: int, hi: int, dtype=np.int8) -> np.ndarray:
    """Integers uniform on [lo, hi] (inclusive)."""
    base = _base(seed, name)
    span = np.uint64(hi - lo + 1)
    out = np.empty(shape, dtype)

    def fn(s, c):
        return ((_words(base, s, c) >> np.uint64(11)) % span).astype(np.int64) + lo

    return _fill(_count(shape), fn, out)


def normal(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    """fp64 normals N(0, std^2) by Box-Muller (two words per draw)."""
    base1 = _base(seed, name + "/u1")
    base2 = _base(seed, name + "/u2")
    out = np.empty(shape, np.float64)

    def fn(s, c):
        u1 = ((_words(base1, s, c) >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
        u2 = ((_words(base2, s, c) >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
        return std * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    return _fill(_count(shape), fn, out)


def log_uniform(seed: int, name: str, shape, lo: float, hi: float) -> np.ndarray:
    u = uniform01(seed, name, shape)
    return np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))


def randint_at(seed: int, name: str, ncols: int, rows, cols, lo: int, hi: int,
               dtype=np.int8) -> np.ndarray:
    """The entries [rows][:, cols] of randint(seed, name, (R, ncols), lo, hi):
    element (r, c) is word r * ncols + c of the stream, so a sub-grid costs
    only its own words."""
    base = _base(seed, name)
    r = np.asarray(rows, np.uint64)[:, None]
    c = np.asarray(cols, np.uint64)[None, :]
    idx = r * np.uint64(ncols) + c + np.uint64(1)
    with np.errstate(over="ignore"):
        w = _mix64(base + idx * _GOLDEN)
    return (((w >> np.uint64(11)) % np.uint64(hi - lo + 1)).astype(np.int64) + lo).astype(dtype)


def log_uniform_at(seed: int, name: str, ncols: int, rows, cols, lo: float, hi: float) -> np.ndarray:
    """The entries [rows][:, cols] of log_uniform(seed, name, (R, ncols), lo, hi)."""
    base = _base(seed, name)
    r = np.asarray(rows, np.uint64)[:, None]
    c = np.asarray(cols, np.uint64)[None, :]
    idx = r * np.uint64(ncols) + c + np.uint64(1)
    with np.errstate(over="ignore"):
        w = _mix64(base + idx * _GOLDEN)
    u = ((w >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
    return np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo)))


def randint_device(seed: int, name: str, shape, lo: int, hi: int, device):
    """randint(seed, name, shape, lo, hi, int8) drawn by torch on `device`,
    bit for bit the same integers (the words are formed in int64 with
    two's-complement wraparound, and logical shifts are arithmetic shifts
    masked to the unsigned width).  Used for weight matrices of gigabytes,
    which the numpy path would take minutes to draw."""
    import torch

    def s64(v):                      # uint64 constant -> the int64 with its bits
        return v - (1 << 64) if v >= (1 << 63) else v

    def shr(z, k):
        return (z >> k) & ((1 << (64 - k)) - 1)

    golden, m1, m2 = s64(int(_GOLDEN)), s64(int(_M1)), s64(int(_M2))
    base = s64(int(_base(seed, name)))
    n = _count(shape)
    out = torch.empty(n, dtype=torch.int8, device=device)
    step = 1 << 25
    for s in range(0, n, step):
        c = min(step, n - s)
        z = torch.arange(s + 1, s + c + 1, dtype=torch.int64, device=device)
        z = z * golden + base
        z = z ^ shr(z, 30)
        z = z * m1
        z = z ^ shr(z, 27)
        z = z * m2
        z = z ^ shr(z, 31)
        out[s:s + c] = (torch.remainder(shr(z, 11), hi - lo + 1) + lo).to(torch.int8)
    return out.view(*shape)


def choice_without_replacement(seed: int, name: str, n: int, k: int) -> np.ndarray:
    """k distinct indices of range(n): the k smallest of n random keys."""
    keys = _words(_base(seed, name), 0, n)
    return np.sort(np.argsort(keys, kind="stable")[:k]).astype(np.int64)


# --------------------------------------------------------------- encodings

def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp64/fp32 values -> bf16 bit patterns (uint16), round to nearest even
    from the fp32 image of the value."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lower = u & np.uint64(0xFFFF)
    upper = u >> np.uint64(16)
    up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & np.uint64(1)) == 1))
    return (upper + up.astype(np.uint64)).astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f16_bits(a: np.ndarray) -> np.ndarray:
    """fp64 values -> IEEE fp16 bit patterns (numpy's round to nearest even)."""
    return np.ascontiguousarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------- workload recipes

def activations(seed: int, name: str, M: int, K: int, kind: str = "outliers") -> np.ndarray:
    """bf16 bits [M, K] of one linear's input.

    kind = "normal"   : x ~ N(0, 1)
           "outliers" : x ~ N(0, 1) with 8 channels (chosen without replacement)
                        multiplied by 20
           "silu_mul" : SiLU(a) * b with a, b ~ N(0, 1) independent
           "normal2"  : x ~ N(0, 2) (standard deviation sqrt(2))
    """
    if kind == "normal":
        x = normal(seed, name + "/x", (M, K))
    elif kind == "outliers":
        x = normal(seed, name + "/x", (M, K))
        ch = choice_without_replacement(seed, name + "/outlier_channels", K, min(8, K))
        x[:, ch] *= 20.0
    elif kind == "silu_mul":
        a = normal(seed, name + "/a", (M, K))
        b = normal(seed, name + "/b", (M, K))
        x = a / (1.0 + np.exp(-a)) * b
    elif kind == "normal2":
        x = normal(seed, name + "/x", (M, K), std=np.sqrt(2.0))
    else:
        raise ValueError(f"unknown activation kind {kind!r}")
    return bf16_bits(x)


def w8a8_weights(seed: int, name: str, K: int, N: int, scale_lo: float = 1e-3,
                 scale_hi: float = 1e-2):
    """Symmetric int8 weights q [K, N] uniform on [-127, 127] and fp16 group
    scales [K/128, N] log-uniform on [scale_lo, scale_hi] (bits)."""
    q = randint(seed, name + "/qw", (K, N), -127, 127, np.int8)
    s = f16_bits(log_uniform(seed, name + "/sw", (K // 128, N), scale_lo, scale_hi))
    return q, s


def w4a16_weights(seed: int, name: str, K: int, N: int, scale_lo: float = 1e-3,
                  scale_hi: float = 3e-2):
    """Symmetric int4 weights q [K, N] uniform on [-7, 7] and bf16 group scales
    [K/128, N] log-uniform on [scale_lo, scale_hi] (bits)."""
    q = randint(seed, name + "/qw", (K, N), -7, 7, np.int8)
    s = bf16_bits(log_uniform(seed, name + "/sw", (K // 128, N), scale_lo, scale_hi))
    return q, s


def w8a16_weights(seed: int, name: str, K: int, N: int, group_size: int,
                  scale_lo: float = 1e-3, scale_hi: float = 1e-2):
    """Symmetric int8 weights q [K, N] uniform on [-127, 127] and bf16 scales
    log-uniform on [scale_lo, scale_hi] (bits): [K/group_size, N], or [1, N]
    (one scale per output column) for group_size 0."""
    q = randint(seed, name + "/qw", (K, N), -127, 127, np.int8)
    rows = 1 if group_size == 0 else K // group_size
    s = bf16_bits(log_uniform(seed, name + "/sw", (rows, N), scale_lo, scale_hi))
    return q, s


# The drafter layer's seven projections (hidden 5120, intermediate 17408,
# 32 query heads and 8 key/value heads of dimension 128) and the target-hidden
# projection fc (5 x 5120 -> 5120).  (name, K, N, activation kind)
DRAFTER_LAYER = (
    ("q_proj", 5120, 4096, "outliers"),
    ("k_proj", 5120, 1024, "outliers"),
    ("v_proj", 5120, 1024, "outliers"),
    ("o_proj", 4096, 5120, "outliers"),
    ("gate_proj", 5120, 17408, "outliers"),
    ("up_proj", 5120, 17408, "outliers"),
    ("down_proj", 17408, 5120, "silu_mul"),
)
FC = ("fc", 25600, 5120, "normal2")


def drafter_linears(num_layers: int = 5, with_fc: bool = True):
    """The linears of the full drafter: 5 layers x 7 projections (+ fc)."""
    out = []
    for layer in range(num_layers):
        for name, K, N, kind in DRAFTER_LAYER:
            out.append((f"layers.{layer}.{name}", K, N, kind))
    if with_fc:
        out.append(FC)
    return out


def shared_input_name(linear_name: str) -> str:
    """Projections that read the same tensor share one input stream:
    q/k/v read the attention input, gate/up the MLP input."""
    for a, b in (("k_proj", "q_proj"), ("v_proj", "q_proj"), ("up_proj", "gate_proj")):
        if linear_name.endswith(a):
            return linear_name[: -len(a)] + b
    return linear_name
