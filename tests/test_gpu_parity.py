"""GPU parity: the CUDA path against the CPU oracle on identical seeded inputs,
through the C ABI (via the binding).

  * pack and dequant: bit-exact, padding included;
  * GEMV / dual GEMV: within the output tolerance of tests/helpers.py, at
    sizes that span several CTAs, all group sizes, M = 1..16 and ragged N;
  * special cases with exact answers (one-hot x, power-of-two scaling);
  * guard regions around outputs stay untouched; bad arguments are refused.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, bf16_ulp, dev_packed, host_u16, host_u32

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _weights(N, K, seed, sigma=0.02, outliers=0.0):
    return wl.weight_f16(N, K, sigma, seed, outliers)


def _case(M, N, K, G, seed, sigma=0.02, outliers=0.0):
    w = _weights(N, K, seed, sigma, outliers)
    x = wl.activations_bf16(M, K, seed + 50)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    y_ref = oracle.linear(wl.bits_u16(x), q, s, z, N, K, G)
    return w, x, (q, s, z), y_ref


# --------------------------------------------------------------------------
# pack / dequant: bit-exact
# --------------------------------------------------------------------------

PACK_CASES = [(8, 32, 32), (24, 256, 64), (40, 640, 128), (136, 1024, 256), (64, 5120, 128),
              (16, 4096, 32), (72, 13824, 128), (32, 2560, 256)]


@pytest.mark.parametrize("N,K,G", PACK_CASES)
@pytest.mark.parametrize("kind", ["normal", "outliers", "special"])
def test_pack_bit_exact(N, K, G, kind):
    w = _weights(N, K, N * 7 + K, 0.02, 0.01 if kind == "outliers" else 0.0)
    if kind == "special":
        w[0].zero_()                                  # all-zero row: degenerate groups
        w[1, : K // 2] = 1e-7                         # scale underflows FP16
        w[2] = w[2].abs()                             # all non-negative
        w[3] = -w[3].abs()                            # all non-positive
        w[4, ::3] = 0.0
    qo, so, zo = oracle.pack(wl.bits_u16(w), G)
    q, s, z = w4.w4a16_pack(w.cuda(), G)
    torch.cuda.synchronize()
    assert np.array_equal(host_u32(q), qo)
    assert np.array_equal(host_u16(s), so)
    assert np.array_equal(host_u32(z), zo)


@pytest.mark.parametrize("N,K,G", PACK_CASES[:5])
def test_dequant_bit_exact(N, K, G):
    w = _weights(N, K, 11 * N + K, 0.02, 0.01)
    qo, so, zo = oracle.pack(wl.bits_u16(w), G)
    ref = oracle.dequant(qo, so, zo, N, K, G)
    out = w4.w4a16_dequant(*dev_packed(qo, so, zo), N, K, G)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------------------------
# GEMV parity
# --------------------------------------------------------------------------

GEMV_SHAPES = [
    # (N, K, G): several CTAs, ragged N (N % 16 == 8), K spanning several warps' groups
    (8, 256, 32), (24, 512, 64), (136, 1024, 128), (264, 2048, 256), (520, 640, 128),
    (1032, 4096, 128), (200, 3072, 32), (72, 5120, 64), (48, 1280, 256),
]


@pytest.mark.parametrize("N,K,G", GEMV_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 16])
def test_gemv_parity(M, N, K, G):
    w, x, (q, s, z), y_ref = _case(M, N, K, G, seed=M * 31 + N + K + G, outliers=0.002)
    y = w4.w4a16_linear_gemv(x.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    assert_close(y, y_ref, f"gemv M={M} N={N} K={K} G={G}")


@pytest.mark.parametrize("M,N,K", [(1, 264, 28672), (3, 264, 28672), (1, 520, 65536)])
def test_gemv_long_rows_with_streamed_scales(M, N, K):
    """Groups of 32 on long rows: the scales stream with the weight units (only the zero rows stay
    resident), so K = 65536 runs as a GEMV; several CTAs, ragged N, up to 2048 groups per row."""
    G = 32
    assert w4.w4a16_linear_path(M, N, K, G) == 1
    w, x, (q, s, z), y_ref = _case(M, N, K, G, seed=M * 17 + N + K, outliers=0.002)
    y = w4.w4a16_linear_gemv(x.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    assert_close(y, y_ref, f"gemv long rows M={M} N={N} K={K} G={G}")


# Long rows: x (M * K FP16) would leave the kernel a short weight ring or no room, so two CTAs of
# a cluster each stage and stream half of every row's chunks and add their partial sums through
# distributed shared memory.  Two column blocks (M = 9..16) and one with 1, 2 or 4 group parities
# (M <= 8); odd chunk counts (rank 1 streams one fewer), a last chunk cut short (K % 256 != 0),
# several CTA pairs, ragged N.
KSPLIT_SHAPES = [(16, 520, 8192, 128), (9, 136, 12288, 64), (12, 1032, 8192, 256), (11, 392, 10560, 64),
                 (16, 264, 6400, 128), (8, 264, 13824, 128), (3, 136, 28672, 128), (2, 72, 49152, 64),
                 (4, 392, 20480, 128), (6, 264, 13824, 256), (5, 520, 16384, 64), (7, 136, 16384, 64),
                 # groups of 32: the scales stream with the units, each CTA's from its own first chunk
                 (12, 264, 8192, 32), (4, 136, 28672, 32)]


def _gemv_plan(M, N, K, G):
    import ctypes
    plan = (ctypes.c_int32 * 6)()
    assert w4._lib.w4a16_debug_gemv_plan(M, N, K, G, 0, plan) == 0
    return list(plan)


@pytest.mark.parametrize("M,N,K,G", KSPLIT_SHAPES)
def test_gemv_k_split_across_a_cluster(M, N, K, G):
    assert _gemv_plan(M, N, K, G)[3] == 1                          # the planner takes the split
    w, x, (q, s, z), y_ref = _case(M, N, K, G, seed=M * 13 + N + K + G, outliers=0.002)
    dq = dev_packed(q, s, z)
    xd = x.cuda()
    y = w4.w4a16_linear_gemv(xd, *dq, G)
    torch.cuda.synchronize()
    assert_close(y, y_ref, f"gemv k-split M={M} N={N} K={K} G={G}")
    assert torch.equal(w4.w4a16_linear_gemv(xd, *dq, G), y)          # the two ranks add in a fixed order
    y32 = w4.w4a16_linear_f32(xd, *dq, G, path=1)
    torch.cuda.synchronize()
    assert torch.equal(y32.to(torch.bfloat16), y)
    assert w4.w4a16_device_status() == 0


@pytest.mark.parametrize("M", [1, 4, 8, 9, 16])
def test_linear_dispatches_to_gemv(M):
    N, K, G = 264, 1024, 128
    assert w4.w4a16_linear_path(M, N, K, G) == 1
    w, x, (q, s, z), y_ref = _case(M, N, K, G, seed=5 + M)
    y = w4.w4a16_linear(x.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    assert_close(y, y_ref, "linear")


@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_gemv_one_hot_is_exact(G):
    """x = e_k gives y[0,n] = bf16_rn(W_hat[n,k]) exactly: every product is exact."""
    N, K = 136, 4 * G
    w = _weights(N, K, 77 + G)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    what = oracle.dequant(q, s, z, N, K, G)
    dq = dev_packed(q, s, z)
    for k in (0, 1, 7, G - 1, G, K - 1):
        x = torch.zeros(1, K, dtype=torch.bfloat16)
        x[0, k] = 1.0
        y = w4.w4a16_linear_gemv(x.cuda(), *dq, G)
        expect = np.array([oracle.f64_to_bf16(float(v)) for v in what[:, k]], np.uint16)
        assert np.array_equal(host_u16(y)[0], expect), k


def test_gemv_power_of_two_scaling_is_exact():
    N, K, G, M = 264, 2048, 128, 3
    w, x, (q, s, z), _ = _case(M, N, K, G, seed=123)
    dq = dev_packed(q, s, z)
    y0 = w4.w4a16_linear_gemv(x.cuda(), *dq, G).float()
    for j in (-4, 3):
        xs = (x.float() * 2.0 ** j).to(torch.bfloat16)
        yj = w4.w4a16_linear_gemv(xs.cuda(), *dq, G).float()
        assert torch.equal(yj, y0 * 2.0 ** j)


def test_gemv_codes_equal_zero_give_near_zero():
    """q == z in every group: y is zero up to FP32 rounding of the zero-point
    correction.  The kernel forms, per group, s * (sum_k x_k (c_k + q_k) -
    sum_k c_k x_k - z sum_k x_k) with offsets c_k in {64, 1024}; the FP32
    rounding of those sums stays far inside 2^-14 * s * (128 + z) * sum|x|."""
    N, K, G, M = 64, 1024, 128, 2
    w = _weights(N, K, 9)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    zeros = oracle.unpack_zeros(z, K, G)
    qz = np.zeros_like(q)
    for k in range(K):
        qz[:, k // 8] |= zeros[:, k // G].astype(np.uint32) << np.uint32(4 * (k % 8))
    x = wl.activations_bf16(M, K, 3)
    y = w4.w4a16_linear_gemv(x.cuda(), *dev_packed(qz, s, z), G).float().cpu().numpy()
    sc = s[:, : K // G].view(np.float16).astype(np.float64)
    xa = np.abs(x.float().numpy()).reshape(M, K // G, G).sum(-1)                 # [M, groups]
    bound = 2.0 ** -14 * (xa @ (sc * (128 + zeros.astype(np.float64))).T)     # [M, N]
    assert np.all(np.abs(y) <= bound)


@pytest.mark.parametrize("M", [1, 4, 11])
@pytest.mark.parametrize("N,K,G", [(136, 1024, 128), (264, 5120, 128), (40, 512, 32)])
def test_dual_parity(M, N, K, G):
    wg, wu = _weights(N, K, 1000 + N), _weights(N, K, 2000 + N)
    x = wl.activations_bf16(M, K, 3000 + M)
    pg = oracle.pack(wl.bits_u16(wg), G)
    pu = oracle.pack(wl.bits_u16(wu), G)
    yg_ref = oracle.linear(wl.bits_u16(x), *pg, N, K, G)
    yu_ref = oracle.linear(wl.bits_u16(x), *pu, N, K, G)
    dg, du = dev_packed(*pg), dev_packed(*pu)
    xd = x.cuda()
    yg, yu = w4.w4a16_linear_dual(xd, dg, du, G)
    torch.cuda.synchronize()
    assert_close(yg, yg_ref, "dual gate")
    assert_close(yu, yu_ref, "dual up")
    # Against a single-matrix call of the kernel the dual call ran (the decode GEMV
    # up to M = 8; at M = 9..16 the GEMV where two matrices' x leaves it all its
    # warps, else the tensor-core GEMM): the dual GEMV splits the concatenated
    # tiles of both matrices over the SMs, so a tile's partial sums may be added
    # in a different order than in a single-matrix call, and the two agree to
    # within one BF16 ulp.
    def within_ulp(y2, y1):
        a, b = y2.double().cpu().numpy(), y1.double().cpu().numpy()
        return bool(np.all(np.abs(a - b) <= bf16_ulp(np.maximum(np.abs(a), np.abs(b)))))

    for y2, d in ((yg, dg), (yu, du)):
        if M <= 8:
            assert within_ulp(y2, w4.w4a16_linear_gemv(xd, *d, G))
        else:
            assert within_ulp(y2, w4.w4a16_linear_gemv(xd, *d, G)) or within_ulp(y2, w4.w4a16_linear_gemm(xd, *d, G))


# --------------------------------------------------------------------------
# guard regions, empty problems, refused arguments
# --------------------------------------------------------------------------

def test_outputs_leave_guard_regions_untouched():
    M, N, K, G = 3, 264, 1024, 64
    w, x, (q, s, z), y_ref = _case(M, N, K, G, seed=99)
    pad = 4096
    canary = torch.full((2 * pad + M * N,), -12345.0, dtype=torch.bfloat16, device="cuda")
    y = canary[pad: pad + M * N].view(M, N)
    w4.w4a16_linear_gemv(x.cuda(), *dev_packed(q, s, z), G, out=y)
    torch.cuda.synchronize()
    assert torch.all(canary[:pad] == -12345.0) and torch.all(canary[pad + M * N:] == -12345.0)
    assert_close(y, y_ref, "guarded")
    # packer guard regions
    wd = w.cuda()
    qs, ss, zs = w4.packed_shapes(N, K, G)
    big = torch.full((2 * pad + qs[0] * qs[1],), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    qv = big[pad: pad + qs[0] * qs[1]].view(qs)
    zbig = torch.full((2 * pad + zs[0] * zs[1],), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    zv = zbig[pad: pad + zs[0] * zs[1]].view(zs)
    sbig = torch.full((2 * pad + ss[0] * ss[1],), 7.0, dtype=torch.float16, device="cuda")
    sv = sbig[pad: pad + ss[0] * ss[1]].view(ss)
    w4.w4a16_pack(wd, G, out=(qv, sv, zv))
    torch.cuda.synchronize()
    assert torch.all(big[:pad] == 0x5A5A5A5A) and torch.all(big[pad + qs[0] * qs[1]:] == 0x5A5A5A5A)
    assert torch.all(zbig[:pad] == 0x5A5A5A5A) and torch.all(zbig[pad + zs[0] * zs[1]:] == 0x5A5A5A5A)
    assert torch.all(sbig[:pad] == 7.0) and torch.all(sbig[pad + ss[0] * ss[1]:] == 7.0)
    assert np.array_equal(host_u32(qv), q)


def test_empty_problem_launches_nothing():
    K, N, G = 256, 64, 128
    q, s, z = w4.empty_packed(N, K, G)
    x = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    y = w4.w4a16_linear(x, q, s, z, G)
    assert y.shape == (0, N)


def test_refused_arguments_raise():
    N, K, G = 64, 256, 128
    q, s, z = w4.empty_packed(N, K, G)
    x = torch.zeros(2, K + 8, dtype=torch.bfloat16, device="cuda")[:, 8:].contiguous()
    with pytest.raises(w4.W4A16Error, match="UNSUPPORTED"):
        w4.w4a16_linear(x, q, s, z, 96)
    xm = torch.zeros(2 * K + 8, dtype=torch.bfloat16, device="cuda")[4:4 + 2 * K].view(2, K)  # 8-byte offset
    with pytest.raises(w4.W4A16Error, match="MISALIGNED"):
        w4.w4a16_linear(xm, q, s, z, G)
    with pytest.raises(w4.W4A16Error, match="UNSUPPORTED"):
        w4.w4a16_linear_gemv(torch.zeros(17, K, dtype=torch.bfloat16, device="cuda"), q, s, z, G)


def test_no_kernel_gave_up_waiting():
    assert w4.w4a16_device_status() == 0
