"""The super-block (Q4_K-style) variant through the C ABI on the GPU.

q4k_pack quantises 256-channel super-blocks (8 sub-blocks of 32, 6-bit
sub-block scales and minima against FP16 factors) and q4k_linear runs the
decode kernel on the codes and the 16-byte records.  Checked here: the packer
bit for bit against the oracle, including zero super-blocks, rows without
negative weights and outlier channels; the layer against the oracle's plain
definition for every kernel geometry the shapes select (segments P = 1..8,
group parities H = 1..4, the M = 1 specialisation and the general kernel, row
blocks for M > 8); the paired gate/up call; and the full-size 70B FFN shapes
on sampled outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, host_u32

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu

# (N, K): K/256 = 1, 3, 4, 20, 9, 12 super-blocks per row, so M = 1 takes P = 1 (H = 4),
# 2 or 4 segments and the general kernel at P = 1; N leaves ragged CTA tile ranges
SHAPES = [(8, 256), (24, 768), (136, 1024), (264, 5120), (40, 2304), (1032, 3072)]


def _weights(N, K, seed):
    w = wl.weight_f16(N, K, 0.02, seed, 0.002)
    if N >= 16:
        w[1, :256] = 0                          # an all-zero super-block
        w[2, 256 % K:] = w[2, 256 % K:].abs()   # super-blocks without negative weights
        w[3, 32:64] = 0                         # a zero sub-block amid others
    return w


def _dev(q, meta):
    return torch.from_numpy(q.view(np.int32)).cuda(), torch.from_numpy(meta.view(np.int32)).cuda()


@pytest.mark.parametrize("N,K", SHAPES)
def test_q4k_pack_bit_exact(N, K):
    w = _weights(N, K, 3 * N + K)
    q, meta = oracle.q4k_pack(wl.bits_u16(w))
    dq, dm = w4.q4k_pack(w.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(host_u32(dq), q)
    assert np.array_equal(host_u32(dm), meta)


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 17])
def test_q4k_linear_parity(M, N, K):
    w = _weights(N, K, 5 * N + K)
    q, meta = oracle.q4k_pack(wl.bits_u16(w))
    x = wl.activations_bf16(M, K, N + M + K)
    y = w4.q4k_linear(x.cuda(), *_dev(q, meta))
    torch.cuda.synchronize()
    assert_close(y, oracle.q4k_linear(wl.bits_u16(x), q, meta, N, K), f"q4k M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 3, 8, 12])
def test_q4k_dual_parity(M):
    N, K = 264, 2048
    wg, wu = _weights(N, K, 71), _weights(N, K, 72)
    pg, pu = oracle.q4k_pack(wl.bits_u16(wg)), oracle.q4k_pack(wl.bits_u16(wu))
    x = wl.activations_bf16(M, K, 73)
    yg, yu = w4.q4k_linear_dual(x.cuda(), _dev(*pg), _dev(*pu))
    torch.cuda.synchronize()
    xb = wl.bits_u16(x)
    assert_close(yg, oracle.q4k_linear(xb, *pg, N, K), f"q4k dual gate M={M}")
    assert_close(yu, oracle.q4k_linear(xb, *pu, N, K), f"q4k dual up M={M}")


def test_q4k_empty_and_status():
    q, meta = w4.q4k_pack(torch.zeros(8, 256, dtype=torch.float16, device="cuda"))
    y = torch.full((0, 8), 7.0, dtype=torch.bfloat16, device="cuda")
    w4.q4k_linear(torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"), q, meta, out=y)
    y1 = w4.q4k_linear(torch.ones(1, 256, dtype=torch.bfloat16, device="cuda"), q, meta)
    torch.cuda.synchronize()
    assert not y1.float().any()                 # all-zero weights reconstruct as zeros
    assert w4.w4a16_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(3, 264, 28672), (5, 136, 16384), (2, 72, 49152)])
def test_q4k_linear_k_split(M, N, K):
    """Long rows: x of M rows leaves the kernel too little room, so two CTAs of a cluster each
    stream half of every row's super-blocks (records included) and add their partial sums."""
    w = _weights(N, K, 7 * N + K)
    q, meta = oracle.q4k_pack(wl.bits_u16(w))
    x = wl.activations_bf16(M, K, N + M + K)
    y = w4.q4k_linear(x.cuda(), *_dev(q, meta))
    torch.cuda.synchronize()
    assert_close(y, oracle.q4k_linear(wl.bits_u16(x), q, meta, N, K), f"q4k k-split M={M} N={N} K={K}")


@pytest.mark.parametrize("j", [0, 1])
@pytest.mark.parametrize("M", [1, 3])
def test_q4k_workload(j, M):
    """The 70B FFN gate and down in the super-block layout at full size: the packer bit for bit,
    and 512 sampled outputs of the layer against the oracle."""
    wk = wl.WORKLOADS["ffn70b_q4k"]
    lin = wk.linears[j]
    w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac)
    q, meta = oracle.q4k_pack(wl.bits_u16(w))
    dq, dm = w4.q4k_pack(w.cuda())
    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j))
    y = w4.q4k_linear(x.cuda(), dq, dm)
    torch.cuda.synchronize()
    assert np.array_equal(host_u32(dq), q) and np.array_equal(host_u32(dm), meta), \
        "super-block packer not bit-exact at full size"
    rng = np.random.default_rng(17 + j)
    ns = np.concatenate([[0, lin.N - 1], rng.integers(0, lin.N, 510)])
    ms = rng.integers(0, M, ns.size)
    ref = oracle.q4k_linear_sampled(wl.bits_u16(x), q, meta, lin.K, ms, ns)
    got = y.float().cpu().numpy()[ms, ns]
    assert_close(got, ref, f"ffn70b_q4k {lin.name} M={M} (sampled)")


def test_q4k_dual_workload_shape():
    """The pair at the 70B gate shape (8192 -> 28672): its records do not fit one CTA's shared memory
    together, so the call runs one launch per matrix; sampled outputs against the oracle."""
    wk = wl.WORKLOADS["ffn70b_q4k"]
    lin = wk.linears[0]
    ws = [wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac) for j in (0, 2)]
    packs = [oracle.q4k_pack(wl.bits_u16(w)) for w in ws]
    x = wl.activations_bf16(1, lin.K, wl.act_seed(wk, 0))
    yg, yu = w4.q4k_linear_dual(x.cuda(), _dev(*packs[0]), _dev(*packs[1]))
    torch.cuda.synchronize()
    rng = np.random.default_rng(23)
    ns = rng.integers(0, lin.N, 512)
    ms = np.zeros(ns.size, np.int64)
    for y, (q, meta), name in ((yg, packs[0], "gate"), (yu, packs[1], "up")):
        ref = oracle.q4k_linear_sampled(wl.bits_u16(x), q, meta, lin.K, ms, ns)
        assert_close(y.float().cpu().numpy()[ms, ns], ref, f"q4k dual {name} at 8192 -> 28672 (sampled)")


@pytest.mark.parametrize("M", [1, 2])
def test_q4k_row_slices(M):
    """N = 4752, K = 49152: the records of the rows a CTA would hold do not fit its shared memory even for
    one activation row, so the call cuts the weight rows into slices and runs one activation row per launch.
    Sampled outputs (every slice edge among them) against the oracle."""
    N, K = 4752, 49152
    w = wl.weight_f16(N, K, 0.01, 77)
    q, meta = oracle.q4k_pack(wl.bits_u16(w))
    x = wl.activations_bf16(M, K, 78 + M)
    y = w4.q4k_linear(x.cuda(), *_dev(q, meta))
    torch.cuda.synchronize()
    assert w4.w4a16_device_status() == 0
    rng = np.random.default_rng(79)
    edges = [0, 7, 8, 2375, 2376, 2383, N - 8, N - 1]
    ns = np.concatenate([np.tile(edges, M), rng.integers(0, N, 256 * M)])
    ms = np.concatenate([np.repeat(np.arange(M), len(edges)), rng.integers(0, M, 256 * M)])
    ref = oracle.q4k_linear_sampled(wl.bits_u16(x), q, meta, K, ms, ns)
    assert_close(y.float().cpu().numpy()[ms, ns], ref, f"q4k row slices M={M} (sampled)")
