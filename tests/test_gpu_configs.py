"""Parity at the full workload sizes, in the launch configuration the
benchmark times (the public entry points with their default dispatch).

Decode shapes (M <= 16) are compared element by element against the full FP64
oracle; prefill shapes against oracle outputs sampled one by one.  The packer
is bit-exact at every full size.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, dev_packed, host_u16, host_u32

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _decode_cases():
    cases = []
    for name, wk in wl.WORKLOADS.items():
        if wk.dual or wk.act_scaled or wk.bits != 4 or wk.q4k:        # those have their own tests
            continue
        for j, lin in enumerate(wk.linears):
            for G in wk.Gs:
                for M in wk.Ms:
                    if M <= 16:
                        cases.append(pytest.param(name, j, G, M, id=f"{name}-{lin.name}-G{G}-M{M}"))
    return cases


_packed_cache = {}


def _packed(name, j, G):
    key = (name, j, G)
    if key not in _packed_cache:
        _packed_cache.clear()
        wk = wl.WORKLOADS[name]
        lin = wk.linears[j]
        w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac)
        ref = oracle.pack(wl.bits_u16(w), G)
        dev = w4.w4a16_pack(w.cuda(), G)
        torch.cuda.synchronize()
        _packed_cache[key] = (ref, dev)
    return _packed_cache[key]


@pytest.mark.parametrize("name,j,G,M", _decode_cases())
def test_decode_workload(name, j, G, M):
    wk = wl.WORKLOADS[name]
    lin = wk.linears[j]
    (q, s, z), dev = _packed(name, j, G)
    assert np.array_equal(host_u32(dev[0]), q) and np.array_equal(host_u16(dev[1]), s) \
        and np.array_equal(host_u32(dev[2]), z), "packer not bit-exact at full size"
    x = wl.activations_bf16(M, lin.K, wl.act_seed(wk, j))
    y = w4.w4a16_linear(x.cuda(), *dev, G)
    torch.cuda.synchronize()
    y_ref = oracle.linear(wl.bits_u16(x), q, s, z, lin.N, lin.K, G)
    assert_close(y, y_ref, f"{name}/{lin.name} G={G} M={M}")


@pytest.mark.parametrize("M", [1, 4])
def test_dual_workload(M):
    wk = wl.WORKLOADS["gateup13b_dual"]
    G = wk.Gs[0]
    lg, lu = wk.linears
    wg = wl.weight_f16(lg.N, lg.K, wk.sigma, wl.matrix_seed(wk, 0), wk.outlier_frac)
    wu = wl.weight_f16(lu.N, lu.K, wk.sigma, wl.matrix_seed(wk, 1), wk.outlier_frac)
    pg, pu = oracle.pack(wl.bits_u16(wg), G), oracle.pack(wl.bits_u16(wu), G)
    x = wl.activations_bf16(M, lg.K, wl.act_seed(wk, 0))
    yg, yu = w4.w4a16_linear_dual(x.cuda(), dev_packed(*pg), dev_packed(*pu), G)
    torch.cuda.synchronize()
    xb = wl.bits_u16(x)
    assert_close(yg, oracle.linear(xb, *pg, lg.N, lg.K, G), "dual gate")
    assert_close(yu, oracle.linear(xb, *pu, lu.N, lu.K, G), "dual up")


def _prefill_cases():
    cases = []
    for name, wk in wl.WORKLOADS.items():
        if wk.dual or wk.act_scaled or wk.bits != 4 or wk.q4k:        # those have their own tests
            continue
        for j, lin in enumerate(wk.linears):
            for G in wk.Gs:
                for M in wk.Ms:
                    if M > 16:
                        cases.append(pytest.param(name, j, G, M, id=f"{name}-{lin.name}-G{G}-M{M}"))
    return cases


def _sample_positions(M, N, count, seed):
    """Seeded random (m, n) pairs plus every tile corner the kernel has."""
    rng = np.random.default_rng(seed)
    ms = list(rng.integers(0, M, count))
    ns = list(rng.integers(0, N, count))
    edge_m = sorted({0, 1, M - 1, M - 2} | {v for b in range(256, M, 256) for v in (b - 1, b)})
    edge_n = sorted({0, 1, N - 1, N - 2} | {v for b in range(128, N, 128 * 7) for v in (b - 1, b)})
    for m in edge_m:
        for n in edge_n:
            ms.append(m)
            ns.append(n)
    return np.array(ms, np.int64), np.array(ns, np.int64)


@pytest.mark.parametrize("name,j,G,M", _prefill_cases())
def test_prefill_workload(name, j, G, M):
    """Full workload sizes through w4a16_linear (the tensor-core path for M > 16).
    Small problems are compared in full; the M = 2048 ones on >= 4096 sampled
    outputs, each computed one by one by the oracle (relative L2 over the
    sample, per-element bound with rms(y_ref) over the sample)."""
    wk = wl.WORKLOADS[name]
    lin = wk.linears[j]
    (q, s, z), dev = _packed(name, j, G)
    seed = wl.act_seed(wk, j) + (7 if M == 2048 else 0)   # the benchmark's prefill activations
    x = wl.activations_bf16(M, lin.K, seed)
    assert w4.w4a16_linear_path(M, lin.N, lin.K, G) == 2
    y = w4.w4a16_linear(x.cuda(), *dev, G)
    torch.cuda.synchronize()
    xb = wl.bits_u16(x)
    if M * lin.N * lin.K <= 4e9:
        y_ref = oracle.linear(xb, q, s, z, lin.N, lin.K, G)
        assert_close(y, y_ref, f"{name}/{lin.name} G={G} M={M}")
        return
    ms, ns = _sample_positions(M, lin.N, 4096, seed=M + lin.N)
    y_ref = oracle.linear_sampled(xb, q, s, z, lin.K, G, ms, ns)
    got = y.float().cpu().numpy()[ms, ns].astype(np.float64)
    assert_close(got, y_ref, f"{name}/{lin.name} G={G} M={M} (sampled)")
    assert np.all(np.isfinite(y.float().cpu().numpy()))
