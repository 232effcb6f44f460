"""GPU parity of the 8-bit variant in the word layout (four codes per 32-bit
word, one FP16 scale and one 8-bit zero point per group), through the C ABI:

  * the packer is bit-exact against oracle.pack8w, padding included;
  * the checking aids run the kernels' own 8-bit expansions (w8a16_dequant:
    the decode kernel's nibble halves; w8a16_dequant_f16: the tensor-core
    kernel's byte permutes, its FP16 operand) and are bit-exact against the
    oracle on packed weights and on arbitrary bits;
  * the layer on both kernels is within the output tolerance of helpers.py
    (M and N tails, every group size the kernel takes), at full 13B size on
    sampled outputs, and bit-exact for one-hot x.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, host_u16, host_u32

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _dev(q, s, z):
    return (torch.from_numpy(q.view(np.int32)).cuda(), torch.from_numpy(s.view(np.float16)).cuda(),
            torch.from_numpy(z.view(np.int32)).cuda())


PACK = [(8, 32, 32), (24, 256, 64), (40, 640, 128), (136, 1024, 256), (64, 5120, 128), (16, 4096, 32),
        (8, 96, 32), (72, 13824, 128)]


@pytest.mark.parametrize("N,K,G", PACK)
def test_pack8w_bit_exact(N, K, G):
    w = wl.weight_f16(N, K, 0.02, N * 3 + K, 0.01)
    w[0].zero_()
    w[1, : K // 2] = 1e-7
    w[2] = w[2].abs()
    w[3] = -w[3].abs()
    qo, so, zo = oracle.pack8w(wl.bits_u16(w), G)
    q, s, z = w4.w8a16_pack(w.cuda(), G)
    torch.cuda.synchronize()
    assert np.array_equal(host_u32(q), qo)
    assert np.array_equal(host_u16(s), so)
    assert np.array_equal(host_u32(z), zo)


@pytest.mark.parametrize("N,K,G", PACK[:6])
def test_dequant_aids_bit_exact_on_packed_weights(N, K, G):
    w = wl.weight_f16(N, K, 0.02, N * 5 + K, 0.01)
    q, s, z = oracle.pack8w(wl.bits_u16(w), G)
    ref = oracle.dequant8w(q, s, z, N, K, G)
    d = _dev(q, s, z)
    a = w4.w8a16_dequant(*d, N, K, G)
    b = w4.w8a16_dequant_f16(*d, N, K, G)
    torch.cuda.synchronize()
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(b.cpu().numpy().view(np.uint16), ref.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("N,K,G", [(8, 256, 32), (16, 512, 64), (24, 1024, 128), (8, 768, 256)])
def test_dequant_aids_bit_exact_on_arbitrary_bits(N, K, G):
    q = wl.random_u32((N, K // 4), N + K)
    s = wl.random_f16_bits((N, oracle.scales_ld(K, G)), N + K + 1, 0, 30, True)
    z = wl.random_u32((N, oracle.zeros8w_ld(K, G)), N + K + 2)
    with np.errstate(over="ignore"):
        ref = oracle.dequant8w(q, s, z, N, K, G)
        ref16 = ref.astype(np.float16)
    d = _dev(q, s, z)
    a = w4.w8a16_dequant(*d, N, K, G)
    b = w4.w8a16_dequant_f16(*d, N, K, G)
    torch.cuda.synchronize()
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(b.cpu().numpy().view(np.uint16), ref16.view(np.uint16))


LAYER = [
    # (M, N, K, G, fn): decode kernel (M <= 8, G <= 128) and tensor-core kernel, ragged N and M
    (1, 264, 1024, 128, "w8a16_linear_gemv"), (3, 520, 2048, 64, "w8a16_linear_gemv"),
    (8, 136, 5120, 32, "w8a16_linear_gemv"), (5, 1032, 4096, 128, "w8a16_linear_gemv"),
    (2, 72, 640, 32, "w8a16_linear_gemv"),
    (9, 264, 1024, 128, "w8a16_linear_gemm"), (17, 136, 256, 32, "w8a16_linear_gemm"),
    (100, 520, 1024, 256, "w8a16_linear_gemm"), (300, 264, 1280, 64, "w8a16_linear_gemm"),
    # 160-row tiles, 30 of them, K = 2048 (16 stages of 128 8-bit codes): each cut in two along K
    (150, 3800, 2048, 128, "w8a16_linear_gemm"),
    # 100 narrow tiles, each cut in four along K
    (17, 12792, 2048, 128, "w8a16_linear_gemm"),
    (1, 264, 1024, 256, "w8a16_linear"), (4, 264, 2048, 128, "w8a16_linear"), (40, 392, 768, 32, "w8a16_linear"),
]


@pytest.mark.parametrize("M,N,K,G,fn", LAYER)
def test_linear8w_against_oracle(M, N, K, G, fn):
    w = wl.weight_f16(N, K, 0.02, M + N + K + G, 0.002)
    x = wl.activations_bf16(M, K, M + N + K + G + 50)
    q, s, z = oracle.pack8w(wl.bits_u16(w), G)
    y = getattr(w4, fn)(x.cuda(), *_dev(q, s, z), G)
    torch.cuda.synchronize()
    assert_close(y, oracle.linear8w(wl.bits_u16(x), q, s, z, N, K, G), f"{fn} M={M} N={N} K={K} G={G}")


@pytest.mark.parametrize("fn,G", [("w8a16_linear_gemv", 32), ("w8a16_linear_gemv", 128),
                                  ("w8a16_linear_gemm", 64), ("w8a16_linear_gemm", 256)])
def test_linear8w_one_hot_rows(fn, G):
    """x = e_k: the decode kernel returns bf16_rn(W_hat) (its FP32 sums are exact
    here), the tensor-core kernel bf16_rn(fp16_rn(W_hat)) (its FP16 operand)."""
    N, K = 264, 4 * G
    w = wl.weight_f16(N, K, 0.02, 7 + G)
    q, s, z = oracle.pack8w(wl.bits_u16(w), G)
    what = oracle.dequant8w(q, s, z, N, K, G).astype(np.float64)
    ks = [0, 1, 2, 3, 5, G - 1, G, K - 1]
    M = 1 if fn.endswith("gemv") else len(ks)
    for i0 in range(0, len(ks), M):
        x = torch.zeros(M, K, dtype=torch.bfloat16)
        for i in range(M):
            x[i, ks[i0 + i]] = 1.0
        y = host_u16(getattr(w4, fn)(x.cuda(), *_dev(q, s, z), G))
        torch.cuda.synchronize()
        for i in range(M):
            col = what[:, ks[i0 + i]]
            if fn.endswith("gemm"):
                col = col.astype(np.float16).astype(np.float64)
            assert np.array_equal(y[i], np.array([oracle.f64_to_bf16(float(v)) for v in col], np.uint16))


@pytest.mark.parametrize("M,fn", [(1, "w8a16_linear"), (4, "w8a16_linear"), (32, "w8a16_linear")])
def test_linear8w_full_size_13b_up(M, fn):
    wk = wl.WORKLOADS["up13b_w8"]
    lin = wk.linears[0]
    G = 128
    w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, 0), wk.outlier_frac)
    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, 0))
    dq = w4.w8a16_pack(w.cuda(), G)
    y = getattr(w4, fn)(x.cuda(), *dq, G)
    torch.cuda.synchronize()
    q, s, z = (t.cpu().numpy() for t in dq)
    g = np.random.default_rng(31 + M)
    ms, ns = g.integers(0, M, 4096), g.integers(0, lin.N, 4096)
    ms[:2], ns[:2] = [0, M - 1], [0, lin.N - 1]
    y_ref = oracle.linear8w_sampled(wl.bits_u16(x), q.view(np.uint32), s.view(np.uint16), z.view(np.uint32), lin.K,
                                    G, ms, ns)
    assert_close(y.double().cpu().numpy()[ms, ns], y_ref, f"13B up W8 M={M}")
    assert w4.w4a16_device_status() == 0
