"""The layer with a per-input-channel activation scale (the deployed form of
activation-aware weight quantisation), through the C ABI on the GPU.

w4a16_linear_act_scaled computes y = (x * x_scale) * W_hat^T: each input
channel k of x is multiplied by x_scale[k] in FP32 and rounded to FP16 once
before it meets the weights, on both kernels (the decode GEMV's x staging and
the tensor-core path's FP16 copy of x).  The oracle is oracle.linear_xs, the
plain FP64 definition; the tolerance is that of helpers.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, bf16_ulp, dev_packed

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _weights(N, K, seed):
    return wl.weight_f16(N, K, 0.02, seed, 0.002)


def _problem(M, N, K, G, seed, scale="salient"):
    if scale == "salient":                  # the deployed form: W * alpha packed, x_scale = 1 / alpha
        xs = wl.act_scale_f32(K, seed + 70)
        w = wl.awq_weight_f16(_weights(N, K, seed), xs)
    else:                                   # any factors (magnitudes 1/4..4, both signs, one zero), any W
        g = torch.Generator().manual_seed(seed + 71)
        xs = (0.25 * 16.0 ** torch.rand(K, generator=g)) * torch.where(torch.rand(K, generator=g) < 0.2, -1.0, 1.0)
        xs[K // 2] = 0.0
        w = _weights(N, K, seed)
    x = wl.activations_bf16(M, K, seed + 50)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    return x, xs, (q, s, z)


SHAPES = [(136, 1024, 128), (264, 5120, 128), (40, 512, 32), (72, 768, 64), (24, 2048, 256)]


@pytest.mark.parametrize("N,K,G", SHAPES)
@pytest.mark.parametrize("M", [1, 3, 8, 16, 48])
@pytest.mark.parametrize("scale", ["salient", "arbitrary"])
def test_act_scaled_parity(M, N, K, G, scale):
    x, xs, (q, s, z) = _problem(M, N, K, G, seed=N + K + G + M, scale=scale)
    y = w4.w4a16_linear_act_scaled(x.cuda(), xs.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    y_ref = oracle.linear_xs(wl.bits_u16(x), xs.numpy(), q, s, z, N, K, G)
    assert_close(y, y_ref, f"act-scaled M={M} N={N} K={K} G={G} ({scale})")


@pytest.mark.parametrize("M", [1, 5, 40])
def test_unit_scale_is_the_plain_layer_bitwise(M):
    N, K, G = 136, 1024, 128
    x, _, packed = _problem(M, N, K, G, seed=3)
    xd, dq = x.cuda(), dev_packed(*packed)
    y1 = w4.w4a16_linear_act_scaled(xd, torch.ones(K, device="cuda"), *dq, G)
    y0 = w4.w4a16_linear(xd, *dq, G)
    torch.cuda.synchronize()
    assert torch.equal(y1, y0)


@pytest.mark.parametrize("M", [1, 5, 40])
def test_power_of_two_scale_equals_prescaled_x_bitwise(M):
    # x_k * 2^j_k is exact in BF16 and in FP32, so the fused scale and a scaled input agree bit for bit
    N, K, G = 136, 1024, 128
    x, _, packed = _problem(M, N, K, G, seed=4)
    j = torch.randint(-3, 4, (K,), generator=torch.Generator().manual_seed(9)).float()
    pre = (x.float() * 2.0 ** j).to(torch.bfloat16)
    assert torch.equal(pre.float(), x.float() * 2.0 ** j)
    dq = dev_packed(*packed)
    y1 = w4.w4a16_linear_act_scaled(x.cuda(), (2.0 ** j).cuda(), *dq, G)
    y0 = w4.w4a16_linear(pre.cuda(), *dq, G)
    torch.cuda.synchronize()
    assert torch.equal(y1, y0)


def test_zero_scale_gives_zero():
    N, K, G = 40, 512, 32
    x, _, packed = _problem(3, N, K, G, seed=5)
    y = w4.w4a16_linear_act_scaled(x.cuda(), torch.zeros(K, device="cuda"), *dev_packed(*packed), G)
    torch.cuda.synchronize()
    assert torch.all(y == 0)


@pytest.mark.parametrize("M", [1, 4, 11])
def test_dual_act_scaled(M):
    N, K, G = 264, 5120, 128
    xs = wl.act_scale_f32(K, 77)
    wg = wl.awq_weight_f16(_weights(N, K, 1100), xs)
    wu = wl.awq_weight_f16(_weights(N, K, 2100), xs)
    pg, pu = oracle.pack(wl.bits_u16(wg), G), oracle.pack(wl.bits_u16(wu), G)
    x = wl.activations_bf16(M, K, 3100 + M)
    xd, xsd, dg, du = x.cuda(), xs.cuda(), dev_packed(*pg), dev_packed(*pu)
    yg, yu = w4.w4a16_linear_dual_act_scaled(xd, xsd, dg, du, G)
    torch.cuda.synchronize()
    xb = wl.bits_u16(x)
    assert_close(yg, oracle.linear_xs(xb, xs.numpy(), *pg, N, K, G), "dual act-scaled gate")
    assert_close(yu, oracle.linear_xs(xb, xs.numpy(), *pu, N, K, G), "dual act-scaled up")
    for y2, d in ((yg, dg), (yu, du)):      # against the single call that dispatches the same way
        y1 = w4.w4a16_linear_act_scaled(xd, xsd, *d, G)
        a, b = y2.double().cpu().numpy(), y1.double().cpu().numpy()
        assert np.all(np.abs(a - b) <= bf16_ulp(np.maximum(np.abs(a), np.abs(b))))


@pytest.mark.parametrize("j", [0, 1])
@pytest.mark.parametrize("M", [1, 4, 32])
def test_act_scaled_workload(j, M):
    """The 13B FFN workload with 1 % salient input channels at full size."""
    wk = wl.WORKLOADS["ffn13b_awq"]
    lin = wk.linears[j]
    G = wk.Gs[0]
    xs = wl.act_scale_f32(lin.K, wl.matrix_seed(wk, j) + 70)
    w = wl.awq_weight_f16(wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac), xs)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    dev = w4.w4a16_pack(w.cuda(), G)
    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j))
    y = w4.w4a16_linear_act_scaled(x.cuda(), xs.cuda(), *dev, G)
    torch.cuda.synchronize()
    y_ref = oracle.linear_xs(wl.bits_u16(x), xs.numpy(), q, s, z, lin.N, lin.K, G)
    assert_close(y, y_ref, f"ffn13b_awq/{lin.name} M={M}")


def test_scale_with_the_k_split():
    """M = 16 on 8192-long rows: the decode kernel splits K over a two-CTA cluster, each CTA
    staging (and scaling) its half of x."""
    N, K, G, M = 520, 8192, 128, 16
    x, xs, (q, s, z) = _problem(M, N, K, G, seed=77, scale="arbitrary")
    assert w4.w4a16_linear_path(M, N, K, G) == 1
    y = w4.w4a16_linear_act_scaled(x.cuda(), xs.cuda(), *dev_packed(q, s, z), G)
    torch.cuda.synchronize()
    assert_close(y, oracle.linear_xs(wl.bits_u16(x), xs.numpy(), q, s, z, N, K, G), "k-split scaled")


def test_both_kernels_take_the_scale():
    """The explicit-path entries are not scaled; run both kernels through the
    act-scaled entry at an M each one serves and compare with the oracle."""
    N, K, G = 264, 1024, 128
    for M in (8, 17):
        x, xs, (q, s, z) = _problem(M, N, K, G, seed=21 + M, scale="arbitrary")
        assert w4.w4a16_linear_path(M, N, K, G) == (1 if M <= 8 else 2)
        y = w4.w4a16_linear_act_scaled(x.cuda(), xs.cuda(), *dev_packed(q, s, z), G)
        torch.cuda.synchronize()
        assert_close(y, oracle.linear_xs(wl.bits_u16(x), xs.numpy(), q, s, z, N, K, G), f"M={M}")
