"""The layer kernels' own unpacking routines, pinned bit for bit, and their
FP32 sums checked against the literal output bound.

Dequantising checking aids (each runs one kernel's inline expansion routine
over every packed word; see include/w4a16.h):
  * w4a16_dequant     -- the decode kernel's shift + LOP3 expansion into FP16
                         1024 + q / 64 + q, its zero and scale extraction;
  * w4a16_dequant_f16 -- the tensor-core kernel's PRMT + LOP3 expansion and
                         packed FP16 subtract / multiply (its A operand);
  * q4k_dequant       -- the decode kernel's super-block record decoding.
Each is compared with the oracle's dequantised weights, bit for bit, on
arbitrary bit patterns (every code and zero value, scales across the whole
finite FP16 range including subnormals) as well as on packed weights.

FP32-output layer (w4a16_linear_f32, both kernels): the kernels' sums before
the BF16 output rounding must meet max |y - y_ref| <= 1e-2 * rms(y_ref)
literally, and relative L2 <= 2e-3 (the benchmark spec's tolerances, which a BF16
output can only meet with a half-ulp allowance per element).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import MAXABS_RMS, REL_L2, dev_packed, record_literal

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _random_packed(N, K, G, seed, exp_lo=0, exp_hi=30, sign=True):
    """Arbitrary packed bits in the 4-bit layout: random code words, random zero
    words, random finite FP16 scales (row padding included)."""
    q = wl.random_u32((N, oracle.qweight_ld(K)), seed)
    s = wl.random_f16_bits((N, oracle.scales_ld(K, G)), seed + 1, exp_lo, exp_hi, sign)
    z = wl.random_u32((N, oracle.zeros_ld(K, G)), seed + 2)
    return q, s, z


SHAPES = [(8, 256, 32), (16, 512, 64), (24, 1024, 128), (40, 2048, 256), (8, 96, 32), (16, 640, 128)]


@pytest.mark.parametrize("N,K,G", SHAPES)
def test_decode_expansion_is_exact_on_arbitrary_bits(N, K, G):
    q, s, z = _random_packed(N, K, G, seed=N * 31 + K + G)
    ref = oracle.dequant(q, s, z, N, K, G)
    got = w4.w4a16_dequant(*dev_packed(q, s, z), N, K, G)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("N,K,G", SHAPES)
def test_tensor_core_expansion_is_the_fp16_rounded_weight(N, K, G):
    """The GEMM's A operand is RN_fp16((q - z) * s): the oracle's exact FP32
    W_hat rounded once to FP16 (numpy rounds to nearest even, subnormals and
    overflow to infinity included)."""
    q, s, z = _random_packed(N, K, G, seed=N * 37 + K + G)
    with np.errstate(over="ignore"):
        ref = oracle.dequant(q, s, z, N, K, G).astype(np.float16)
    got = w4.w4a16_dequant_f16(*dev_packed(q, s, z), N, K, G)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint16), ref.view(np.uint16))


@pytest.mark.parametrize("N,K,G", [(64, 4096, 128), (72, 5120, 32), (40, 13824, 256)])
def test_both_expansions_on_packed_weights(N, K, G):
    w = wl.weight_f16(N, K, 0.02, N + K + G, 0.01)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    ref = oracle.dequant(q, s, z, N, K, G)
    dq = dev_packed(q, s, z)
    a = w4.w4a16_dequant(*dq, N, K, G)
    b = w4.w4a16_dequant_f16(*dq, N, K, G)
    torch.cuda.synchronize()
    assert np.array_equal(a.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(b.cpu().numpy().view(np.uint16), ref.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("N,K", [(8, 256), (16, 1024), (24, 2560)])
def test_super_block_decoding_is_exact_on_arbitrary_records(N, K):
    """Random codes and random 16-byte records (finite FP16 d and dmin of either
    sign, every 6-bit sc and m value) against the oracle's reading of the layout."""
    q = wl.random_u32((N, K // 8), seed=K + N)
    meta = wl.random_u32((N, K // 256 * 4), seed=K + N + 1)
    dd = wl.random_f16_bits((N, K // 256, 2), seed=K + N + 2, exp_lo=0, exp_hi=30, sign=True).astype(np.uint32)
    meta.reshape(N, K // 256, 4)[:, :, 0] = dd[:, :, 0] | (dd[:, :, 1] << 16)
    ref = oracle.q4k_dequant(q, meta, N, K)
    got = w4.q4k_dequant(torch.from_numpy(q.view(np.int32)).cuda(), torch.from_numpy(meta.view(np.int32)).cuda(), N, K)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_super_block_decoding_on_packed_weights():
    N, K = 48, 8192
    w = wl.weight_f16(N, K, 0.015, 77, 0.001)
    q, meta = oracle.q4k_pack(wl.bits_u16(w))
    ref = oracle.q4k_dequant(q, meta, N, K)
    got = w4.q4k_dequant(torch.from_numpy(q.view(np.int32)).cuda(), torch.from_numpy(meta.view(np.int32)).cuda(), N, K)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------------------------
# FP32 outputs against the literal bound
# --------------------------------------------------------------------------

def _check_literal(y32, y_ref, what):
    y = y32.double().cpu().numpy() if isinstance(y32, torch.Tensor) else np.asarray(y32, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    rms = np.sqrt(np.mean(y_ref ** 2))
    rel = np.linalg.norm(y - y_ref) / np.linalg.norm(y_ref)
    lit = np.abs(y - y_ref).max() / rms
    record_literal(what, rel, lit, fp32=True)
    assert rel <= REL_L2, f"{what}: relL2 {rel:.3e}"
    assert lit <= MAXABS_RMS, f"{what}: max|err| / rms {lit:.3e} > {MAXABS_RMS}"


F32_CASES = [
    # (M, N, K, G, path): path 1 = decode kernel, 2 = tensor-core kernel
    (1, 264, 1024, 128, 1), (3, 520, 2048, 64, 1), (8, 136, 5120, 32, 1), (16, 264, 1280, 256, 1),
    (1, 1032, 4096, 128, 1), (17, 136, 256, 32, 2), (100, 520, 1024, 128, 2), (300, 264, 1280, 64, 2),
    (513, 392, 768, 256, 2), (64, 1032, 4096, 128, 2),
]


@pytest.mark.parametrize("M,N,K,G,path", F32_CASES)
def test_fp32_output_meets_the_literal_bound(M, N, K, G, path):
    w = wl.weight_f16(N, K, 0.02, M + N + K + G, 0.002)
    x = wl.activations_bf16(M, K, M + N + K + G + 50)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    y_ref = oracle.linear(wl.bits_u16(x), q, s, z, N, K, G)
    y = w4.w4a16_linear_f32(x.cuda(), *dev_packed(q, s, z), G, path=path)
    torch.cuda.synchronize()
    _check_literal(y, y_ref, f"fp32 path={path} M={M} N={N} K={K} G={G}")


@pytest.mark.parametrize("name,j,M,path", [("ffn70b", 0, 1, 1), ("ffn70b", 1, 1, 1), ("ffn70b", 0, 2048, 2),
                                            ("ffn70b", 1, 2048, 2), ("single_4096", 0, 1, 1),
                                            ("layer13b_decode", 6, 1, 1)])
def test_fp32_output_literal_bound_at_full_size(name, j, M, path):
    """Full workload shapes: 4096 sampled outputs (every tile corner among them)
    against the oracle computed one by one."""
    wk = wl.WORKLOADS[name]
    lin = wk.linears[j]
    G = wk.Gs[0]
    w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac)
    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j) + (7 if M > 1 else 0))
    dq = w4.w4a16_pack(w.cuda(), G)
    y = w4.w4a16_linear_f32(x.cuda(), *dq, G, path=path)
    torch.cuda.synchronize()
    q, s, z = (t.cpu().numpy() for t in dq)
    g = np.random.default_rng(1234 + j)
    ms = g.integers(0, M, 4096)
    ns = g.integers(0, lin.N, 4096)
    ms[:4], ns[:4] = [0, 0, M - 1, M - 1], [0, lin.N - 1, 0, lin.N - 1]
    y_ref = oracle.linear_sampled(wl.bits_u16(x), q.view(np.uint32), s.view(np.uint16), z.view(np.uint32), lin.K, G,
                                  ms.astype(np.int64), ns.astype(np.int64))
    _check_literal(y.cpu().numpy()[ms, ns], y_ref, f"fp32 {name}/{lin.name} M={M} path={path}")
