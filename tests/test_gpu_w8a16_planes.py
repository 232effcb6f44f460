"""The 8-bit variant (W8A16) through the C ABI on the GPU.

w8a16_planes_pack stores each 8-bit code as two 4-bit planes of a 2K-channel 4-bit
layer, and w8a16_planes_linear runs the 4-bit kernels on those planes over x repeated
twice.  Checked here: the packer bit for bit against the oracle (including
shapes where the two planes share a zero-point word), the layer against the
oracle's plain 8-bit definition on both kernels, bit-for-bit equality with the
4-bit call on the planes and an explicitly repeated x, and the full-size
workload.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, dev_packed, host_u16, host_u32

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu

# (N, K, G): K/G = 5, 4, 48, 40, 3 groups per row, so the lo plane's zeros often start
# inside the hi plane's last zero word
SHAPES = [(24, 640, 128), (136, 1024, 256), (40, 1536, 32), (264, 5120, 128), (16, 192, 64)]


def _weights(N, K, seed):
    return wl.weight_f16(N, K, 0.02, seed, 0.002)


@pytest.mark.parametrize("N,K,G", SHAPES)
def test_pack8_bit_exact(N, K, G):
    w = _weights(N, K, N + K + G)
    q, s, z = oracle.pack8(wl.bits_u16(w), G)
    dq, ds, dz = w4.w8a16_planes_pack(w.cuda(), G)
    torch.cuda.synchronize()
    assert np.array_equal(host_u32(dq), q)
    assert np.array_equal(host_u16(ds), s)
    assert np.array_equal(host_u32(dz), z)


@pytest.mark.parametrize("N,K,G", SHAPES)
@pytest.mark.parametrize("M", [1, 3, 8, 9, 40])
def test_linear8_parity(M, N, K, G):
    w = _weights(N, K, 7 * N + K + G)
    q, s, z = oracle.pack8(wl.bits_u16(w), G)
    x = wl.activations_bf16(M, K, N + M)
    y = w4.w8a16_planes_linear(x.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    if M <= 8 or M > 16:
        assert w4.w4a16_linear_path(M, N, 2 * K, G) == (1 if M <= 8 else 2)
    assert_close(y, oracle.linear8(wl.bits_u16(x), q, s, z, N, K, G), f"w8a16 M={M} N={N} K={K} G={G}")


@pytest.mark.parametrize("M", [1, 5, 24])
def test_linear8_is_the_4bit_layer_over_repeated_x_bitwise(M):
    N, K, G = 264, 2048, 128
    w = _weights(N, K, 33)
    packed = dev_packed(*oracle.pack8(wl.bits_u16(w), G))
    x = wl.activations_bf16(M, K, 44).cuda()
    y8 = w4.w8a16_planes_linear(x, *packed, G)
    y4 = w4.w4a16_linear(torch.cat([x, x], dim=1).contiguous(), *packed, G)
    torch.cuda.synchronize()
    assert torch.equal(y8, y4)


@pytest.mark.parametrize("M", [1, 4, 32])
def test_w8_workload(M):
    wk = wl.WORKLOADS["up13b_w8"]
    lin = wk.linears[0]
    G = wk.Gs[0]
    w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, 0), wk.outlier_frac)
    q, s, z = oracle.pack8(wl.bits_u16(w), G)
    dev = w4.w8a16_planes_pack(w.cuda(), G)
    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, 0))
    y = w4.w8a16_planes_linear(x.cuda(), *dev, G)
    torch.cuda.synchronize()
    assert np.array_equal(host_u32(dev[0]), q) and np.array_equal(host_u16(dev[1]), s) \
        and np.array_equal(host_u32(dev[2]), z), "8-bit packer not bit-exact at full size"
    assert_close(y, oracle.linear8(wl.bits_u16(x), q, s, z, lin.N, lin.K, G), f"up13b_w8 M={M}")
