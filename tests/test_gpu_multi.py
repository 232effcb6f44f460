"""GPU parity of w4a16_linear_multi: up to four matrices sharing x, each with
its own output size, in one decode launch (M <= 8) or the tensor-core kernel
per matrix (larger M).  Each output is checked against its own oracle GEMV,
and against the single-matrix call of the same kernel (the multi launch does
the same arithmetic per row, so the two agree to within one BF16 ulp)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, bf16_ulp, dev_packed

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _mats(Ns, K, G, seed):
    out = []
    for i, N in enumerate(Ns):
        w = wl.weight_f16(N, K, 0.02, seed + 100 * i, 0.001)
        out.append(oracle.pack(wl.bits_u16(w), G))
    return out


CASES = [
    # (Ns, K, G, M): q/k/v of one width; grouped-query shapes (k, v narrower); ragged N; four matrices
    ((1024, 1024, 1024), 2048, 128, 1), ((2048, 256, 256), 2048, 64, 1), ((520, 136, 264), 1024, 32, 3),
    ((1032, 1032, 512, 256), 4096, 128, 1), ((264, 264), 640, 128, 8), ((136,), 256, 256, 2),
    ((1024, 256, 256), 5120, 128, 4), ((264, 520, 136), 1024, 128, 40),
]


@pytest.mark.parametrize("Ns,K,G,M", CASES)
def test_multi_against_oracle(Ns, K, G, M):
    mats = _mats(Ns, K, G, seed=sum(Ns) + K + G + M)
    x = wl.activations_bf16(M, K, 4321 + M)
    dmats = [dev_packed(*m) for m in mats]
    ys = w4.w4a16_linear_multi(x.cuda(), dmats, G)
    torch.cuda.synchronize()
    xb = wl.bits_u16(x)
    for i, (N, m, y) in enumerate(zip(Ns, mats, ys)):
        assert y.shape == (M, N)
        y_ref = oracle.linear(xb, *m, N, K, G)
        assert_close(y, y_ref, f"multi[{i}] N={N} K={K} G={G} M={M}")
        single = w4.w4a16_linear(x.cuda(), *dmats[i], G)
        diff = np.abs(y.double().cpu().numpy() - single.double().cpu().numpy())
        assert (diff <= bf16_ulp(single.double().cpu().numpy())).all(), f"multi[{i}] vs single"


def test_multi_qkv_13b_shape_at_decode():
    """The 13B attention projections (q, k, v: 5120 -> 5120, G = 128) in one launch."""
    wk = wl.WORKLOADS["layer13b_decode"]
    lins = wk.linears[:3]
    mats = []
    for j, lin in enumerate(lins):
        w = wl.weight_f16(lin.N, lin.K, wk.sigma, wl.matrix_seed(wk, j), wk.outlier_frac)
        mats.append(oracle.pack(wl.bits_u16(w), 128))
    x = wl.activations_bf16(1, 5120, wl.act_seed(wk, 0))
    ys = w4.w4a16_linear_multi(x.cuda(), [dev_packed(*m) for m in mats], 128)
    torch.cuda.synchronize()
    for j, (lin, m, y) in enumerate(zip(lins, mats, ys)):
        assert_close(y, oracle.linear(wl.bits_u16(x), *m, lin.N, lin.K, 128), f"qkv {lin.name}")


def test_multi_skips_empty_matrices_and_leaves_guards():
    K, G, M = 512, 128, 2
    mats = _mats((136, 8), K, G, seed=77)
    x = wl.activations_bf16(M, K, 78)
    dm = [dev_packed(*m) for m in mats]
    pad = 4096
    canary = torch.full((2 * pad + M * 136,), -5.0, dtype=torch.bfloat16, device="cuda")
    y0 = canary[pad:pad + M * 136].view(M, 136)
    y1 = torch.empty(M, 8, dtype=torch.bfloat16, device="cuda")
    w4.w4a16_linear_multi(x.cuda(), dm, G, out=[y0, y1])
    torch.cuda.synchronize()
    assert torch.all(canary[:pad] == -5.0) and torch.all(canary[pad + M * 136:] == -5.0)
    assert_close(y0, oracle.linear(wl.bits_u16(x), *mats[0], 136, K, G), "guarded multi")
    assert w4.w4a16_device_status() == 0
