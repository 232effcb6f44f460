"""The kernels' bounded waits, made to run out without faulting, trapping or
hanging the GPU.

A test hook (w4a16_debug_withhold_copy) makes the next launch of one kernel
withhold one copy by construction: the decode kernel's first warp never
issues its first unit of weights, the tensor-core kernel's first block never
issues its first slice of codes.  Nothing is ever in flight against the
withheld barrier.  With the spin budget cut to ~0.1 ms (w4a16_debug_set_wait_limit),
the waiting warps give up, the kernel drains the copies it did issue and
returns; w4a16_device_status must then report W4A16_ERR_TIMEOUT with the
waiting role's bit (and no drain bit: every copy that was issued lands), and
the next call must be clean and correct.
"""
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, dev_packed

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu

TIMEOUT = 5
# tensor-core kernel: whichever of its roles (producer, MMA issuer, dequantisers,
# epilogue: bits 0..3) gives up first records its bit, the others follow the abort flag
BIT_GEMM_ROLES, BIT_GEMM_DRAIN = 0xF, 1 << 4
BIT_GEMV, BIT_GEMV_DRAIN = 1 << 8, 1 << 9
SHORT_WAIT = 200_000                 # SM cycles, ~0.1 ms at 2 GHz


def _problem(M, N, K, G, seed):
    w = wl.weight_f16(N, K, 0.02, seed)
    x = wl.activations_bf16(M, K, seed + 50)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    return x.cuda(), dev_packed(q, s, z), oracle.linear(wl.bits_u16(x), q, s, z, N, K, G)


@pytest.fixture
def short_waits():
    assert w4.device_status_word() == (0, 0)          # nothing pending from earlier tests
    w4._lib.w4a16_debug_set_wait_limit(SHORT_WAIT)
    yield
    w4._lib.w4a16_debug_withhold_copy(0)
    w4._lib.w4a16_debug_set_wait_limit(0)              # back to the default budget


@pytest.mark.parametrize("kernel,M,fn,bit,drain_bit", [
    (1, 1, "w4a16_linear_gemv", BIT_GEMV, BIT_GEMV_DRAIN),
    (1, 4, "w4a16_linear_gemv", BIT_GEMV, BIT_GEMV_DRAIN),
    (2, 64, "w4a16_linear_gemm", BIT_GEMM_ROLES, BIT_GEMM_DRAIN),
    (2, 300, "w4a16_linear_gemm", BIT_GEMM_ROLES, BIT_GEMM_DRAIN),
])
def test_withheld_copy_times_out_and_reports(short_waits, kernel, M, fn, bit, drain_bit):
    N, K, G = 1032, 4096, 128
    x, dq, y_ref = _problem(M, N, K, G, seed=900 + kernel + M)
    assert w4._lib.w4a16_debug_withhold_copy(kernel) == 0
    getattr(w4, fn)(x, *dq, G)                         # this launch gives up on its withheld copy
    st, word = w4.device_status_word()
    assert st == TIMEOUT, (st, hex(word))
    assert word & bit, hex(word)
    assert not word & ~(bit | drain_bit), hex(word)   # only the kernel that was armed gave up
    assert not word & drain_bit, hex(word)            # every copy it did issue landed
    assert w4.device_status_word() == (0, 0)          # the word was cleared
    y = getattr(w4, fn)(x, *dq, G)                     # the hook is one-shot: this call is clean
    st, word = w4.device_status_word()
    assert (st, word) == (0, 0)
    assert_close(y, y_ref, f"{fn} after a timeout")

