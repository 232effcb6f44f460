"""The allocation-free tensor-core entry point, called through the C ABI.

w4a16_linear_gemm_noalloc serves callers that may not allocate device memory
while they run the layer (an engine that reserves its whole memory budget at
start-up and forbids later allocations, so a running model never fails
half-way on an out-of-memory error): its FP16 copy of x sits in one fixed
device array shared by every call.  These tests check that two calls in
a row (different shapes, so the second overwrites what the first left in the
array) each match the allocating entry point w4a16_linear_gemm within the
output tolerance of helpers.py, and that a problem too large for the array is
refused before anything runs.  The file is named so that pytest collects it
last.
"""
import ctypes

import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, dev_packed

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call(fn, x, q, s, z, N, G, y):
    """One C-ABI call on the current stream; returns the status code."""
    M, K = x.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return getattr(w4._lib, fn)(_ptr(x), _ptr(q), _ptr(s), _ptr(z), M, N, K, G, _ptr(y), stream)


def _problem(M, N, K, G, seed):
    w = wl.weight_f16(N, K, 0.02, seed)
    x = wl.activations_bf16(M, K, seed + 50)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    return x.cuda(), dev_packed(q, s, z), (wl.bits_u16(x), q, s, z)


def test_noalloc_matches_allocating_entry_point_on_two_calls():
    shapes = [(300, 264, 1024, 128, 11), (77, 520, 2048, 64, 12)]
    probs = [_problem(*sh) for sh in shapes]
    outs = []
    for (M, N, K, G, _), (x, dq, _) in zip(shapes, probs):           # two no-alloc calls in a row
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call("w4a16_linear_gemm_noalloc", x, *dq, N, G, y) == 0
        outs.append(y)
    torch.cuda.synchronize()
    for (M, N, K, G, _), (x, dq, host), y in zip(shapes, probs, outs):
        y_alloc = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert _call("w4a16_linear_gemm", x, *dq, N, G, y_alloc) == 0
        torch.cuda.synchronize()
        assert_close(y, y_alloc.double().cpu().numpy(), f"no-alloc vs allocating M={M} N={N} K={K} G={G}")
        assert_close(y, oracle.linear(*host, N, K, G), f"no-alloc vs oracle M={M} N={N} K={K} G={G}")
    assert w4.w4a16_device_status() == 0


def test_noalloc_refuses_problems_larger_than_its_array():
    N, K, G = 64, 4096, 128
    M = w4.NOALLOC_MAX_X_ELEMS // K + 1
    x = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    q, s, z = w4.empty_packed(N, K, G)
    y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    assert _call("w4a16_linear_gemm_noalloc", x, q, s, z, N, G, y) == 2        # W4A16_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)
