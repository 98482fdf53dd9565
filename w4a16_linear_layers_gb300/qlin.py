"""Python binding of libqlin (ctypes).  Argument marshalling only: every step
of the computation runs in the library's CUDA kernels; PyTorch supplies device
memory and the current stream.

Names follow the C ABI (include/qlin.h) without the ``qlin_`` prefix.  Tensors
must be CUDA tensors, contiguous, of the dtypes listed per call; outputs are
allocated with ``torch.empty`` when not given.  A non-zero status raises
``QlinError``.  If the shared library has not been built the first call raises
``QlinError`` -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

QLIN_OK = 0
QLIN_ERR_NULL = -1
QLIN_ERR_SHAPE = -2
QLIN_ERR_ALIGN = -3
QLIN_ERR_WORKSPACE = -4
QLIN_ERR_BITS = -5
QLIN_ERR_DEVICE = -6
QLIN_ERR_TOO_LARGE = -7
QLIN_ERR_CUDA = -10
QLIN_ERR_DEVICE_TIMEOUT = -20
QLIN_ERR_VALUE_RANGE = -21

EXPORTS = (
    "qlin_act_quant_i8",
    "qlin_rmsnorm_act_quant_i8",
    "qlin_silu_mul_act_quant_i8",
    "qlin_act_quant_c16",
    "qlin_rmsnorm_act_quant_c16",
    "qlin_silu_mul_act_quant_c16",
    "qlin_gemm_w8a8_gs128",
    "qlin_gemm_w8a8_gs128_c16",
    "qlin_gemm_w8a8_gs128_noalloc",
    "qlin_gemm_w4a16_g128",
    "qlin_gemm_w8a8_gs128_tiled",
    "qlin_gemm_w4a16_g128_tiled",
    "qlin_tiles_bytes",
    "qlin_pack_tiles",
    "qlin_gemm_w8a16",
    "qlin_gemm_w8a8_gs128_argmax",
    "qlin_gemm_w4a16_g128_argmax",
    "qlin_pack_gptq",
    "qlin_ingest_nk",
    "qlin_workspace_bytes",
    "qlin_debug_group_partials_i8",
    "qlin_debug_wait_timeout",
    "qlin_device_status",
    "qlin_device_error_detail",
    "qlin_status_string",
    "qlin_version",
)


class QlinError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"qlin status {status}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load libqlin.so (built in-tree by ``w4a16_linear_layers_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise QlinError(QLIN_ERR_CUDA, f"{path} is not built; run "
                            "`python -m w4a16_linear_layers_gb300.build` (or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sig = {
            "qlin_act_quant_i8": ([P, I64, I64, P, P, P], I),
            "qlin_rmsnorm_act_quant_i8": ([P, P, ctypes.c_float, I64, I64, P, P, P, P], I),
            "qlin_silu_mul_act_quant_i8": ([P, I64, I64, P, P, P, P], I),
            "qlin_act_quant_c16": ([P, I64, I64, P, P, P], I),
            "qlin_rmsnorm_act_quant_c16": ([P, P, ctypes.c_float, I64, I64, P, P, P, P], I),
            "qlin_silu_mul_act_quant_c16": ([P, I64, I64, P, P, P, P], I),
            "qlin_gemm_w8a8_gs128": ([P, P, P, P, I64, I64, I64, P, P, SZ, P], I),
            "qlin_gemm_w8a8_gs128_c16": ([P, P, P, P, I64, I64, I64, P, P, SZ, P], I),
            "qlin_gemm_w8a8_gs128_noalloc": ([P, P, P, P, I64, I64, I64, P, P], I),
            "qlin_gemm_w4a16_g128": ([P, P, P, I64, I64, I64, P, P, SZ, P], I),
            "qlin_gemm_w8a16": ([P, P, P, I64, I64, I64, I, P, P, SZ, P], I),
            "qlin_gemm_w8a8_gs128_tiled": ([P, P, P, P, I64, I64, I64, P, P, SZ, P], I),
            "qlin_gemm_w4a16_g128_tiled": ([P, P, P, I64, I64, I64, P, P, SZ, P], I),
            "qlin_tiles_bytes": ([I64, I64, I], SZ),
            "qlin_pack_tiles": ([P, I64, I64, I, P, P], I),
            "qlin_gemm_w8a8_gs128_argmax": ([P, P, P, P, I64, I64, I64, P, P, SZ, P], I),
            "qlin_gemm_w4a16_g128_argmax": ([P, P, P, I64, I64, I64, P, P, SZ, P], I),
            "qlin_pack_gptq": ([P, I64, I64, I, P, P, P], I),
            "qlin_ingest_nk": ([P, P, I64, I64, I, P, P, P], I),
            "qlin_workspace_bytes": ([I64, I64, I64], SZ),
            "qlin_debug_group_partials_i8": ([P, P, I64, I64, I64, P, P, SZ, P], I),
            "qlin_debug_wait_timeout": ([I64, P], I),
            "qlin_device_status": ([P], I),
            "qlin_device_error_detail": ([P, P, P], I),
            "qlin_status_string": ([I], ctypes.c_char_p),
            "qlin_version": ([], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().qlin_status_string(int(status)).decode()


def _check(status: int) -> None:
    if status != QLIN_OK:
        raise QlinError(status, status_string(status))


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------- calls

def _quant_outputs(M, K, device, q, s_a, code_dtype=torch.int8):
    if q is None:
        q = torch.empty((M, K), dtype=code_dtype, device=device)
    if s_a is None:
        s_a = torch.empty((M,), dtype=torch.float32, device=device)
    _need(q, "q", code_dtype, 2)
    _need(s_a, "s_a", torch.float32, 1)
    if tuple(q.shape) != (M, K) or tuple(s_a.shape) != (M,):
        raise ValueError("q must be [M, K] and s_a [M]")
    return q, s_a


def _act_quant(fn, code_dtype, x, q, s_a, stream):
    _need(x, "x", torch.bfloat16, 2)
    M, K = x.shape
    q, s_a = _quant_outputs(M, K, x.device, q, s_a, code_dtype)
    _check(fn(_ptr(x), M, K, _ptr(q), _ptr(s_a), _stream_handle(stream)))
    return q, s_a


def act_quant_i8(x: torch.Tensor, q: torch.Tensor | None = None, s_a: torch.Tensor | None = None,
                 stream=None):
    """x bf16 [M,K] -> (q int8 [M,K], s_a fp32 [M])."""
    return _act_quant(load().qlin_act_quant_i8, torch.int8, x, q, s_a, stream)


def act_quant_c16(x: torch.Tensor, q: torch.Tensor | None = None, s_a: torch.Tensor | None = None,
                  stream=None):
    """act_quant_i8 with the codes as fp16: -> (q fp16 [M,K] holding the same
    integers, s_a fp32 [M])."""
    return _act_quant(load().qlin_act_quant_c16, torch.float16, x, q, s_a, stream)


def _rmsnorm_act_quant(fn, code_dtype, x, gamma, eps, q, s_a, y, stream):
    _need(x, "x", torch.bfloat16, 2)
    _need(gamma, "gamma", torch.bfloat16, 1)
    M, K = x.shape
    if tuple(gamma.shape) != (K,):
        raise ValueError("gamma must be [K]")
    q, s_a = _quant_outputs(M, K, x.device, q, s_a, code_dtype)
    if y is not None:
        _need(y, "y", torch.bfloat16, 2)
        if tuple(y.shape) != (M, K):
            raise ValueError("y must be [M, K]")
    _check(fn(_ptr(x), _ptr(gamma), float(eps), M, K, _ptr(q), _ptr(s_a),
              _ptr(y) if y is not None else None, _stream_handle(stream)))
    return q, s_a


def rmsnorm_act_quant_i8(x: torch.Tensor, gamma: torch.Tensor, eps: float, q=None, s_a=None,
                         y=None, stream=None):
    """RMSNorm of x bf16 [M,K] with weight gamma bf16 [K], then per-token INT8
    act-quant -> (q int8 [M,K], s_a fp32 [M]).  If y (bf16 [M,K]) is given
    the norm's bf16 output is written there too."""
    return _rmsnorm_act_quant(load().qlin_rmsnorm_act_quant_i8, torch.int8, x, gamma, eps, q, s_a,
                              y, stream)


def rmsnorm_act_quant_c16(x: torch.Tensor, gamma: torch.Tensor, eps: float, q=None, s_a=None,
                          y=None, stream=None):
    """rmsnorm_act_quant_i8 with the codes as fp16 (q fp16 [M,K])."""
    return _rmsnorm_act_quant(load().qlin_rmsnorm_act_quant_c16, torch.float16, x, gamma, eps, q,
                              s_a, y, stream)


def _silu_mul_act_quant(fn, code_dtype, gate_up, q, s_a, y, stream):
    _need(gate_up, "gate_up", torch.bfloat16, 2)
    M, I2 = gate_up.shape
    if I2 % 2:
        raise ValueError("gate_up must have an even number of columns")
    q, s_a = _quant_outputs(M, I2 // 2, gate_up.device, q, s_a, code_dtype)
    if y is not None:
        _need(y, "y", torch.bfloat16, 2)
        if tuple(y.shape) != (M, I2 // 2):
            raise ValueError("y must be [M, I]")
    _check(fn(_ptr(gate_up), M, I2 // 2, _ptr(q), _ptr(s_a), _ptr(y) if y is not None else None,
              _stream_handle(stream)))
    return q, s_a


def silu_mul_act_quant_i8(gate_up: torch.Tensor, q=None, s_a=None, y=None, stream=None):
    """SiLU(gate) * up of gate_up bf16 [M, 2I] (gate columns first), then
    per-token INT8 act-quant -> (q int8 [M,I], s_a fp32 [M]).  If y (bf16
    [M,I]) is given the activation's bf16 output is written there too."""
    return _silu_mul_act_quant(load().qlin_silu_mul_act_quant_i8, torch.int8, gate_up, q, s_a, y,
                               stream)


def silu_mul_act_quant_c16(gate_up: torch.Tensor, q=None, s_a=None, y=None, stream=None):
    """silu_mul_act_quant_i8 with the codes as fp16 (q fp16 [M,I])."""
    return _silu_mul_act_quant(load().qlin_silu_mul_act_quant_c16, torch.float16, gate_up, q, s_a,
                               y, stream)


def workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().qlin_workspace_bytes(int(M), int(N), int(K)))


class Workspace:
    """A zero-initialised device buffer for the GEMMs' split-K partials and
    counters, grown on demand.  The kernels return the counters to zero, so one
    Workspace serves any number of calls ordered on one stream."""

    def __init__(self, device=None, nbytes: int = 0):
        self.device = torch.device(device if device is not None else "cuda")
        self.buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)

    def get(self, M: int, N: int, K: int) -> torch.Tensor:
        need = workspace_bytes(M, N, K)
        if need > self.buf.numel():
            self.buf = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _workspace(ws, M, N, K, device):
    if ws is None:
        key = (device.index if device.index is not None else torch.cuda.current_device())
        ws = _default_ws.get(key)
        if ws is None:
            ws = _default_ws[key] = Workspace(device)
    if isinstance(ws, Workspace):
        return ws.get(M, N, K)
    return ws


def _gemm_w8a8(fn, code_dtype, q_a, s_a, qweight, scales, y, workspace, stream):
    _need(q_a, "q_a", code_dtype, 2)
    _need(s_a, "s_a", torch.float32, 1)
    _need(qweight, "qweight", torch.int32, 2)
    _need(scales, "scales", torch.float16, 2)
    M, K = q_a.shape
    N = qweight.shape[1]
    if qweight.shape[0] * 4 != K or scales.shape != (K // 128, N) or s_a.shape[0] != M:
        raise ValueError("inconsistent W8A8 shapes")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=q_a.device)
    _need(y, "y", torch.bfloat16, 2)
    ws = _workspace(workspace, M, N, K, q_a.device)
    _check(fn(_ptr(q_a), _ptr(s_a), _ptr(qweight), _ptr(scales), M, N, K, _ptr(y), _ptr(ws),
              ws.numel(), _stream_handle(stream)))
    return y


def gemm_w8a8_gs128(q_a: torch.Tensor, s_a: torch.Tensor, qweight: torch.Tensor,
                    scales: torch.Tensor, y: torch.Tensor | None = None, workspace=None,
                    stream=None) -> torch.Tensor:
    """q_a int8 [M,K], s_a fp32 [M], qweight int32 [K/4,N], scales fp16 [K/128,N]
    -> y bf16 [M,N]."""
    return _gemm_w8a8(load().qlin_gemm_w8a8_gs128, torch.int8, q_a, s_a, qweight, scales, y,
                      workspace, stream)


def gemm_w8a8_gs128_c16(q_a: torch.Tensor, s_a: torch.Tensor, qweight: torch.Tensor,
                        scales: torch.Tensor, y: torch.Tensor | None = None, workspace=None,
                        stream=None) -> torch.Tensor:
    """gemm_w8a8_gs128 with the activation codes as fp16 (q_a fp16 [M,K], the
    output of the *_c16 producers)."""
    return _gemm_w8a8(load().qlin_gemm_w8a8_gs128_c16, torch.float16, q_a, s_a, qweight, scales,
                      y, workspace, stream)


def gemm_w8a8_gs128_noalloc(q_a: torch.Tensor, s_a: torch.Tensor, qweight: torch.Tensor,
                            scales: torch.Tensor, y: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """W8A8 GS128 linear that allocates nothing inside the library: its split-K
    scratch is the library's built-in 24 MiB device array (for callers that
    cannot allocate; see include/qlin.h).  Same arguments and result as
    gemm_w8a8_gs128 without the workspace.  Calls that overlap on the GPU
    race on the shared array."""
    _need(q_a, "q_a", torch.int8, 2)
    _need(s_a, "s_a", torch.float32, 1)
    _need(qweight, "qweight", torch.int32, 2)
    _need(scales, "scales", torch.float16, 2)
    M, K = q_a.shape
    N = qweight.shape[1]
    if qweight.shape[0] * 4 != K or scales.shape != (K // 128, N) or s_a.shape[0] != M:
        raise ValueError("inconsistent W8A8 shapes")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=q_a.device)
    _need(y, "y", torch.bfloat16, 2)
    _check(load().qlin_gemm_w8a8_gs128_noalloc(_ptr(q_a), _ptr(s_a), _ptr(qweight), _ptr(scales),
                                               M, N, K, _ptr(y), _stream_handle(stream)))
    return y


def gemm_w4a16_g128(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                    y: torch.Tensor | None = None, workspace=None, stream=None) -> torch.Tensor:
    """x bf16 [M,K], qweight int32 [K/8,N], scales bf16 [K/128,N] -> y bf16 [M,N]."""
    _need(x, "x", torch.bfloat16, 2)
    _need(qweight, "qweight", torch.int32, 2)
    _need(scales, "scales", torch.bfloat16, 2)
    M, K = x.shape
    N = qweight.shape[1]
    if qweight.shape[0] * 8 != K or scales.shape != (K // 128, N):
        raise ValueError("inconsistent W4A16 shapes")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, 2)
    ws = _workspace(workspace, M, N, K, x.device)
    _check(load().qlin_gemm_w4a16_g128(_ptr(x), _ptr(qweight), _ptr(scales), M, N, K, _ptr(y),
                                       _ptr(ws), ws.numel(), _stream_handle(stream)))
    return y


class Tiles:
    """Weights in the tile layout of qlin_pack_tiles: the flat int32 device
    tensor and the shape of the matrix it holds (K, N, bits)."""

    def __init__(self, data: torch.Tensor, K: int, N: int, bits: int):
        self.data, self.K, self.N, self.bits = data, int(K), int(N), int(bits)


def tiles_bytes(K: int, N: int, bits: int) -> int:
    return int(load().qlin_tiles_bytes(int(K), int(N), int(bits)))


def pack_tiles(qweight: torch.Tensor, K: int, bits: int, stream=None) -> Tiles:
    """GPTQ words [K*bits/32, N] -> the tile layout (one contiguous block per
    128-feature x 128-K tile)."""
    _need(qweight, "qweight", torch.int32, 2)
    N = qweight.shape[1]
    if qweight.shape[0] * (32 // bits) != K:
        raise ValueError("qweight rows do not match K and bits")
    nbytes = tiles_bytes(K, N, bits)
    if nbytes == 0:
        raise ValueError("invalid shape or bits for the tile layout")
    data = torch.empty(nbytes // 4, dtype=torch.int32, device=qweight.device)
    _check(load().qlin_pack_tiles(_ptr(qweight), K, N, bits, _ptr(data), _stream_handle(stream)))
    return Tiles(data, K, N, bits)


def gemm_w8a8_gs128_tiled(q_a: torch.Tensor, s_a: torch.Tensor, tiles: Tiles,
                          scales: torch.Tensor, y: torch.Tensor | None = None, workspace=None,
                          stream=None) -> torch.Tensor:
    """gemm_w8a8_gs128 with the weights in the tile layout (pack_tiles, bits 8)."""
    _need(q_a, "q_a", torch.int8, 2)
    _need(s_a, "s_a", torch.float32, 1)
    _need(scales, "scales", torch.float16, 2)
    M, K = q_a.shape
    N = tiles.N
    if tiles.bits != 8 or tiles.K != K or scales.shape != (K // 128, N) or s_a.shape[0] != M:
        raise ValueError("inconsistent W8A8 shapes")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=q_a.device)
    _need(y, "y", torch.bfloat16, 2)
    ws = _workspace(workspace, M, N, K, q_a.device)
    _check(load().qlin_gemm_w8a8_gs128_tiled(_ptr(q_a), _ptr(s_a), _ptr(tiles.data), _ptr(scales),
                                             M, N, K, _ptr(y), _ptr(ws), ws.numel(),
                                             _stream_handle(stream)))
    return y


def gemm_w4a16_g128_tiled(x: torch.Tensor, tiles: Tiles, scales: torch.Tensor,
                          y: torch.Tensor | None = None, workspace=None, stream=None) -> torch.Tensor:
    """gemm_w4a16_g128 with the weights in the tile layout (pack_tiles, bits 4)."""
    _need(x, "x", torch.bfloat16, 2)
    _need(scales, "scales", torch.bfloat16, 2)
    M, K = x.shape
    N = tiles.N
    if tiles.bits != 4 or tiles.K != K or scales.shape != (K // 128, N):
        raise ValueError("inconsistent W4A16 shapes")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, 2)
    ws = _workspace(workspace, M, N, K, x.device)
    _check(load().qlin_gemm_w4a16_g128_tiled(_ptr(x), _ptr(tiles.data), _ptr(scales), M, N, K,
                                             _ptr(y), _ptr(ws), ws.numel(), _stream_handle(stream)))
    return y


def gemm_w8a16(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, group_size: int,
               y: torch.Tensor | None = None, workspace=None, stream=None) -> torch.Tensor:
    """x bf16 [M,K], qweight int32 [K/4,N] (8-bit GPTQ words), scales bf16
    [K/group_size,N] ([1,N] for group_size 0) -> y bf16 [M,N]."""
    _need(x, "x", torch.bfloat16, 2)
    _need(qweight, "qweight", torch.int32, 2)
    _need(scales, "scales", torch.bfloat16, 2)
    M, K = x.shape
    N = qweight.shape[1]
    rows = 1 if group_size == 0 else K // group_size
    if qweight.shape[0] * 4 != K or scales.shape != (rows, N):
        raise ValueError("inconsistent W8A16 shapes")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, 2)
    ws = _workspace(workspace, M, N, K, x.device)
    _check(load().qlin_gemm_w8a16(_ptr(x), _ptr(qweight), _ptr(scales), M, N, K, int(group_size),
                                  _ptr(y), _ptr(ws), ws.numel(), _stream_handle(stream)))
    return y


def gemm_w8a8_gs128_argmax(q_a: torch.Tensor, s_a: torch.Tensor, qweight: torch.Tensor,
                           scales: torch.Tensor, out: torch.Tensor | None = None,
                           workspace=None, stream=None) -> torch.Tensor:
    """Greedy token per row of the W8A8 GS128 linear (M <= 96): int32 [M],
    the index of the largest bf16 output, lowest index on ties."""
    _need(q_a, "q_a", torch.int8, 2)
    _need(s_a, "s_a", torch.float32, 1)
    _need(qweight, "qweight", torch.int32, 2)
    _need(scales, "scales", torch.float16, 2)
    M, K = q_a.shape
    N = qweight.shape[1]
    if qweight.shape[0] * 4 != K or scales.shape != (K // 128, N) or s_a.shape[0] != M:
        raise ValueError("inconsistent W8A8 shapes")
    if out is None:
        out = torch.empty((M,), dtype=torch.int32, device=q_a.device)
    _need(out, "out", torch.int32, 1)
    ws = _workspace(workspace, M, N, K, q_a.device)
    _check(load().qlin_gemm_w8a8_gs128_argmax(_ptr(q_a), _ptr(s_a), _ptr(qweight), _ptr(scales),
                                              M, N, K, _ptr(out), _ptr(ws), ws.numel(),
                                              _stream_handle(stream)))
    return out


def gemm_w4a16_g128_argmax(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor,
                           out: torch.Tensor | None = None, workspace=None,
                           stream=None) -> torch.Tensor:
    """Greedy token per row of the W4A16 g128 linear (M <= 96)."""
    _need(x, "x", torch.bfloat16, 2)
    _need(qweight, "qweight", torch.int32, 2)
    _need(scales, "scales", torch.bfloat16, 2)
    M, K = x.shape
    N = qweight.shape[1]
    if qweight.shape[0] * 8 != K or scales.shape != (K // 128, N):
        raise ValueError("inconsistent W4A16 shapes")
    if out is None:
        out = torch.empty((M,), dtype=torch.int32, device=x.device)
    _need(out, "out", torch.int32, 1)
    ws = _workspace(workspace, M, N, K, x.device)
    _check(load().qlin_gemm_w4a16_g128_argmax(_ptr(x), _ptr(qweight), _ptr(scales), M, N, K,
                                              _ptr(out), _ptr(ws), ws.numel(),
                                              _stream_handle(stream)))
    return out


def ingest_nk(packed_nk: torch.Tensor, scales_ng: torch.Tensor, K: int, bits: int,
              stream=None):
    """compressed-tensors orientation (words int32 [N, K*bits/32], 16-bit scales
    [N, K/128]) -> the GEMMs' orientation (qweight [K*bits/32, N], scales
    [K/128, N], same dtype as scales_ng)."""
    _need(packed_nk, "packed_nk", torch.int32, 2)
    if scales_ng.dtype not in (torch.float16, torch.bfloat16) or scales_ng.dim() != 2:
        raise ValueError("scales_ng must be a 2-D fp16 or bf16 tensor")
    N = packed_nk.shape[0]
    if packed_nk.shape[1] * 32 != K * bits or scales_ng.shape != (N, K // 128):
        raise ValueError("inconsistent ingest shapes")
    qweight = torch.empty((K * bits // 32, N), dtype=torch.int32, device=packed_nk.device)
    scales = torch.empty((K // 128, N), dtype=scales_ng.dtype, device=packed_nk.device)
    _check(load().qlin_ingest_nk(_ptr(packed_nk.contiguous()), _ptr(scales_ng.contiguous()), K, N,
                                 bits, _ptr(qweight), _ptr(scales), _stream_handle(stream)))
    return qweight, scales


def pack_gptq(q: torch.Tensor, bits: int, qweight: torch.Tensor | None = None,
              qzeros: torch.Tensor | None = None, with_qzeros: bool = True, stream=None):
    """q int8 [K,N] -> (qweight int32 [K*bits/32,N], qzeros int32 [K/128,N*bits/32] or None)."""
    _need(q, "q", torch.int8, 2)
    K, N = q.shape
    per = 32 // bits if bits in (4, 8) else 1
    if qweight is None:
        qweight = torch.empty((K // per, N), dtype=torch.int32, device=q.device)
    if qzeros is None and with_qzeros:
        qzeros = torch.empty((K // 128, N // per), dtype=torch.int32, device=q.device)
    _need(qweight, "qweight", torch.int32, 2)
    zp = ctypes.c_void_p(0)
    if qzeros is not None:
        _need(qzeros, "qzeros", torch.int32, 2)
        zp = _ptr(qzeros)
    _check(load().qlin_pack_gptq(_ptr(q), K, N, int(bits), _ptr(qweight), zp,
                                 _stream_handle(stream)))
    return qweight, qzeros


def debug_group_partials_i8(q_a: torch.Tensor, qweight: torch.Tensor, P: torch.Tensor | None = None,
                            workspace=None, stream=None) -> torch.Tensor:
    """Exact per-group integer partials P int32 [K/128, M, N] of the W8A8 path."""
    _need(q_a, "q_a", torch.int8, 2)
    _need(qweight, "qweight", torch.int32, 2)
    M, K = q_a.shape
    N = qweight.shape[1]
    if P is None:
        P = torch.empty((K // 128, M, N), dtype=torch.int32, device=q_a.device)
    _need(P, "P", torch.int32, 3)
    ws = _workspace(workspace, M, N, K, q_a.device)
    _check(load().qlin_debug_group_partials_i8(_ptr(q_a), _ptr(qweight), M, N, K, _ptr(P),
                                               _ptr(ws), ws.numel(), _stream_handle(stream)))
    return P


def debug_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load().qlin_debug_wait_timeout(int(limit_ns), _stream_handle(stream)))


def device_error_detail(stream=None):
    """(status, where, block) of the device error word, without clearing it."""
    w = ctypes.c_int32(0)
    b = ctypes.c_int32(0)
    st = int(load().qlin_device_error_detail(_stream_handle(stream), ctypes.byref(w), ctypes.byref(b)))
    return st, int(w.value), int(b.value)


def device_status(stream=None) -> int:
    """Synchronize the stream, read and clear the device error word; returns the status."""
    return int(load().qlin_device_status(_stream_handle(stream)))


def version() -> int:
    return int(load().qlin_version())
