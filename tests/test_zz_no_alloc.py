"""The no-allocation W8A8 entry point, qlin_gemm_w8a8_gs128_noalloc.

Callers that cannot allocate device memory (allocator or memory-pool
callbacks, plugins whose host framework owns all device memory, processes
that must not grow their footprint while serving) use this entry point: it
takes its scratch from the library's built-in 24 MiB device array
instead of a caller-provided workspace.  This file is collected last so that a
run stopping at the first failure has already run every other test.  It is
self-contained: it passes alone in a fresh process and after the others."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import compare_linear, from_dev_bits, to_dev, to_dev_bits
from w4a16_linear_layers_gb300 import build as qbuild
from w4a16_linear_layers_gb300 import qlin, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qbuild.build()
    oracle.build()
    return qlin.load()


def _inputs(seed, M, K, N):
    xb = synth.activations(seed, f"noalloc/x/{M}/{K}", M, K, "outliers")
    qa, sa = oracle.act_quant_i8(xb)
    qwt, swb = synth.w8a8_weights(seed, f"noalloc/w/{K}/{N}", K, N)
    qw, _, _ = oracle.pack_gptq(qwt, 8)
    return qa, sa, qw, swb


def _call_noalloc(lib, qa_d, sa_d, qw_d, sc_d, y_d, M, N, K):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.qlin_gemm_w8a8_gs128_noalloc(P(qa_d), P(sa_d), P(qw_d), P(sc_d), M, N, K, P(y_d),
                                            stream)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(lib):
    # Two calls back to back on the shared scratch array: a split-K decode
    # shape, then a different shape that splits its tiles differently, so
    # anything left behind by the first call would show up in the second.
    for seed, (M, K, N) in enumerate([(8, 5120, 1024), (96, 2560, 768)]):
        qa, sa, qw, swb = _inputs(seed, M, K, N)
        qa_d, sa_d, qw_d = to_dev(qa), to_dev(sa), to_dev(qw)
        sc_d = to_dev_bits(swb, torch.float16)
        y_na = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        st = _call_noalloc(lib, qa_d, sa_d, qw_d, sc_d, y_na, M, N, K)
        assert st == qlin.QLIN_OK, qlin.status_string(st)
        y_ws = qlin.gemm_w8a8_gs128(qa_d, sa_d, qw_d, sc_d)
        torch.cuda.synchronize()
        # the same kernel with the same plan and the same split of K: the
        # outputs must be identical bit for bit (a stale partial or counter
        # left in the shared array would show here)
        assert np.array_equal(from_dev_bits(y_na), from_dev_bits(y_ws)), \
            f"call {seed}: no-alloc differs from workspace entry"
        compare_linear(from_dev_bits(y_na), oracle.gemm_w8a8_gs128(qa, sa, qw, swb, K),
                       f"no-alloc call {seed}")
    assert qlin.device_status() == qlin.QLIN_OK


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 96-token tiles: the 16 MiB fp16 activation image plus the per-block
    # split partials (about 15 MB on 152 SMs) exceed the 24 MiB array
    M, K, N = 8192, 1024, 1024
    assert qlin.workspace_bytes(M, N, K) > 24 * 1024 * 1024
    qa_d = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sa_d = torch.zeros(M, dtype=torch.float32, device="cuda")
    qw_d = torch.zeros((K // 4, N), dtype=torch.int32, device="cuda")
    sc_d = torch.zeros((K // 128, N), dtype=torch.float16, device="cuda")
    y_d = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = _call_noalloc(lib, qa_d, sa_d, qw_d, sc_d, y_d, M, N, K)
    assert st == qlin.QLIN_ERR_TOO_LARGE
    assert "24 MiB" in qlin.status_string(st)
