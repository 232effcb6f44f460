"""GPU parity of the tensor-core (prefill) path against the CPU oracle, through
the C ABI (via the binding).

  * w4a16_linear_gemm at sizes that span several 128-row weight tiles and
    several activation tiles, with ragged M, N and K tails, every group size;
  * w4a16_linear dispatches M > 16 to this path; the dual entry point runs it
    once per projection on one FP16 copy of x;
  * special cases with exact answers (one-hot x, power-of-two scaling);
  * guard regions around y stay untouched.

The tolerance is the one in helpers.py (relative L2 <= 2e-3 and the per-element
bound).  The kernel multiplies FP16 operands: x converted from BF16 (exact for
these inputs) and W_hat rounded once to FP16, so every product carries at
most one FP16 rounding of the weight.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, dev_packed, host_u16

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _case(M, N, K, G, seed, sigma=0.02, outliers=0.0):
    w = wl.weight_f16(N, K, sigma, seed, outliers)
    x = wl.activations_bf16(M, K, seed + 50)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    y_ref = oracle.linear(wl.bits_u16(x), q, s, z, N, K, G)
    return x, (q, s, z), y_ref


GEMM_SHAPES = [
    # (M, N, K, G): M tails (not a multiple of 32 / of the 256-row tile), N tails
    # (not a multiple of 128), K tails (not a multiple of the 256-k code slice)
    (17, 136, 256, 32), (32, 264, 640, 64), (100, 520, 1024, 128), (256, 128, 2048, 256),
    (300, 264, 1280, 128), (513, 392, 768, 64), (40, 8, 96, 32), (64, 1032, 4096, 128),
    (777, 136, 512, 256), (1, 264, 1024, 128), (16, 136, 5120, 32),
    # one activation tile wider than 128 rows (BN = 160, 256): the epilogue parks the first 128
    # columns' BF16 pairs in tensor memory
    (160, 264, 1024, 128), (230, 392, 768, 32),
    # 100 narrow tiles (more than half the SMs of a B300): each cut in four along K, 400 pieces
    (17, 12792, 2048, 64),
]


@pytest.mark.parametrize("M,N,K,G", GEMM_SHAPES)
def test_gemm_parity(M, N, K, G):
    x, (q, s, z), y_ref = _case(M, N, K, G, seed=M + 3 * N + K + G, outliers=0.002)
    y = w4.w4a16_linear_gemm(x.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    assert_close(y, y_ref, f"gemm M={M} N={N} K={K} G={G}")


@pytest.mark.parametrize("M", [17, 48, 600])
def test_linear_dispatches_to_gemm(M):
    N, K, G = 264, 1024, 128
    assert w4.w4a16_linear_path(M, N, K, G) == 2
    x, (q, s, z), y_ref = _case(M, N, K, G, seed=17 + M)
    y = w4.w4a16_linear(x.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    assert_close(y, y_ref, "linear (gemm)")


def test_gemm_and_gemv_agree_on_small_batches():
    """Both kernels run the same layer; at M <= 16 each is checked against the
    oracle and against the other within twice the output tolerance."""
    N, K, G, M = 520, 2048, 128, 9
    x, (q, s, z), y_ref = _case(M, N, K, G, seed=4242)
    dq = dev_packed(q, s, z)
    xd = x.cuda()
    ya = w4.w4a16_linear_gemm(xd, *dq, G)
    yb = w4.w4a16_linear_gemv(xd, *dq, G)
    torch.cuda.synchronize()
    assert_close(ya, y_ref, "gemm")
    assert_close(yb, y_ref, "gemv")


@pytest.mark.parametrize("M", [40, 200])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_gemm_one_hot_rows(G, M):
    """x rows = e_k: y[i, n] = bf16_rn(fp16_rn(W_hat[n, k_i])).  The kernel's
    weight operand is W_hat rounded once to FP16, and a single product by 1.0
    accumulates exactly in FP32.  M = 40 spans two 32-column chunks of the
    epilogue; M = 200 (BN = 224) its parked first half."""
    N, K = 264, 4 * G
    w = wl.weight_f16(N, K, 0.02, 99 + G)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    what = oracle.dequant(q, s, z, N, K, G)
    ks = [0, 1, 7, 8, G - 1, G, K - 33, K - 1]
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    for i in range(M):
        x[i, ks[i % len(ks)]] = 1.0
    y = w4.w4a16_linear_gemm(x.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    got = host_u16(y)
    for i in range(M):
        k = ks[i % len(ks)]
        w16 = what[:, k].astype(np.float16).astype(np.float64)      # RN to FP16 (numpy rounds to nearest even)
        expect = np.array([oracle.f64_to_bf16(float(v)) for v in w16], np.uint16)
        assert np.array_equal(got[i], expect), (i, k)


def test_gemm_power_of_two_scaling_is_exact():
    M, N, K, G = 70, 264, 1024, 64
    x, (q, s, z), _ = _case(M, N, K, G, seed=321)
    dq = dev_packed(q, s, z)
    y0 = w4.w4a16_linear_gemm(x.cuda(), *dq, G).float()
    for j in (-3, 2):
        xs = (x.float() * 2.0 ** j).to(torch.bfloat16)
        yj = w4.w4a16_linear_gemm(xs.cuda(), *dq, G).float()
        assert torch.equal(yj, y0 * 2.0 ** j)


@pytest.mark.parametrize("M", [17, 300])
def test_dual_uses_gemm_above_16_rows(M):
    N, K, G = 264, 1024, 128
    wg, wu = wl.weight_f16(N, K, 0.02, 5000 + M), wl.weight_f16(N, K, 0.02, 6000 + M)
    x = wl.activations_bf16(M, K, 7000 + M)
    pg, pu = oracle.pack(wl.bits_u16(wg), G), oracle.pack(wl.bits_u16(wu), G)
    xd = x.cuda()
    dg, du = dev_packed(*pg), dev_packed(*pu)
    yg, yu = w4.w4a16_linear_dual(xd, dg, du, G)
    torch.cuda.synchronize()
    xb = wl.bits_u16(x)
    assert_close(yg, oracle.linear(xb, *pg, N, K, G), "dual gate")
    assert_close(yu, oracle.linear(xb, *pu, N, K, G), "dual up")
    assert torch.equal(yg, w4.w4a16_linear_gemm(xd, *dg, G))
    assert torch.equal(yu, w4.w4a16_linear_gemm(xd, *du, G))


def test_gemm_leaves_guard_regions_untouched():
    M, N, K, G = 45, 136, 512, 128
    x, (q, s, z), y_ref = _case(M, N, K, G, seed=11)
    pad = 8192
    canary = torch.full((2 * pad + M * N,), -777.0, dtype=torch.bfloat16, device="cuda")
    y = canary[pad: pad + M * N].view(M, N)
    w4.w4a16_linear_gemm(x.cuda(), *dev_packed(q, s, z), G, out=y)
    torch.cuda.synchronize()
    assert torch.all(canary[:pad] == -777.0) and torch.all(canary[pad + M * N:] == -777.0)
    assert_close(y, y_ref, "guarded gemm")


def test_gemm_repeated_calls_are_identical():
    M, N, K, G = 260, 264, 2048, 128
    x, (q, s, z), _ = _case(M, N, K, G, seed=5)
    dq = dev_packed(q, s, z)
    xd = x.cuda()
    y0 = w4.w4a16_linear_gemm(xd, *dq, G)
    for _ in range(3):
        assert torch.equal(w4.w4a16_linear_gemm(xd, *dq, G), y0)


def _split_shape(case, sms):
    """(M, N, K, G, R) of a K-split case; R = the tiles cut in two."""
    if case == "tail":
        # M = 3000: 256-row activation tiles, 12 per weight tile, the last one ragged; N ragged.
        # Whole tiles fill the SMs once, then R tiles remain: those are split (K = 4096: 16 stages).
        ntiles = -(-(sms + 20) // 12)
        M, N, K, G = 3000, 128 * ntiles - 8, 4096, 128
        T = 12 * ntiles
        R = T % sms if T > sms else T
    else:
        # 160-row tiles (M = 150), 30 of them, the only wave: every tile is cut in three; K = 6208
        # (97 slices of 64, a ragged last stage: 25 stages) puts the range boundaries at slices 32
        # and 64
        M, N, K, G = 150, 128 * 30 - 40, 6208, 64
        R = 30
    return M, N, K, G, R


@pytest.mark.parametrize("case", ["tail", "all"])
def test_gemm_wide_tiles_split_along_k(case):
    """Wide tiles (BN > 64) of a last wave at most half full are cut along K (in
    two, or up to three when they are the only wave); y adds the ranges' FP32
    partials in a fixed order."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K, G, R = _split_shape(case, sms)
    assert 0 < 2 * R <= sms
    x, (q, s, z), y_ref = _case(M, N, K, G, seed=M + N, outliers=0.002)
    dq = dev_packed(q, s, z)
    xd = x.cuda()
    y = w4.w4a16_linear_gemm(xd, *dq, G)
    torch.cuda.synchronize()
    assert_close(y, y_ref, f"split gemm {case} M={M} N={N} K={K} G={G}")
    for _ in range(2):                               # the partials are added in a fixed order
        assert torch.equal(w4.w4a16_linear_gemm(xd, *dq, G), y)
    # FP32 outputs of the same call: unrounded sums, against the oracle's
    y32 = w4.w4a16_linear_f32(xd, *dq, G, path=2)
    torch.cuda.synchronize()
    assert torch.equal(y32.to(torch.bfloat16), y)
    assert_close(y32, y_ref, f"split gemm fp32 {case}")


def test_gemm_no_kernel_gave_up_waiting():
    assert w4.w4a16_device_status() == 0
