"""Pins for the CPU oracle: what the pages and the mathematics fix, checked on
the CPU without any GPU code.

Each test ties the oracle to something other than itself:
  * library routines for the IEEE conversions (numpy float16, torch bfloat16);
  * hand-derived packing examples (tests/golden/pack_examples.json);
  * numbers the pages print (tests/golden/closed_forms.json);
  * closed forms (on-grid round trip, the rounding-error bound);
  * exact rational brute force of dequantise-then-multiply on tiny shapes;
  * special cases with exact answers (one-hot x, q == z, power-of-two x).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _h(s):
    return int(s, 16)


# --------------------------------------------------------------------------
# IEEE conversions against library routines
# --------------------------------------------------------------------------

def test_f16_to_f32_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f16_probe_values(rng):
    v = []
    # random magnitudes spanning subnormal .. overflow
    e = rng.uniform(-27, 17, 20000)
    v.append(np.sign(rng.standard_normal(20000)) * np.exp2(e))
    # exact midpoints between neighbouring FP16 values (ties), normal and subnormal
    b = rng.integers(0, 0x7BFF, 5000).astype(np.uint16)
    lo = b.view(np.float16).astype(np.float64)
    hi = (b + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    v.append((lo + hi) / 2)
    v.append(np.array([65504.0, 65519.0, 65519.996, 65520.0, 65536.0, 1e6, 2.0 ** -24, 2.0 ** -25,
                       2.0 ** -25 * 1.0001, 2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -12), 0.0, -0.0]))
    return np.concatenate(v).astype(np.float32)


def test_f32_to_f16_rne_matches_numpy():
    rng = np.random.default_rng(1)
    vals = _f16_probe_values(rng)
    with np.errstate(over="ignore"):                   # the probes include values that round to +-inf
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(float(x)) for x in vals], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_conversions_match_torch():
    rng = np.random.default_rng(2)
    e = rng.uniform(-140, 127, 20000)
    vals = (np.sign(rng.standard_normal(20000)) * np.exp2(e)).astype(np.float32)
    # ties: FP32 values exactly halfway between neighbouring BF16 values
    b = rng.integers(0, 0x7F7F, 5000).astype(np.uint32)
    ties = ((b << 16) | 0x8000).astype(np.uint32).view(np.float32)
    vals = np.concatenate([vals, ties, np.array([0.0, -0.0, 3.4e38, 1e-45], np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(x)) for x in vals], np.uint16)
    assert np.array_equal(got, ref)
    # widening is exact: every finite pattern round-trips
    pats = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    wide = oracle.bf16_bits_to_f32_array(pats)
    fin = np.isfinite(wide)
    back = torch.from_numpy(wide[fin]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(back, pats[fin])


# --------------------------------------------------------------------------
# Hand-derived packing examples
# --------------------------------------------------------------------------

@pytest.mark.parametrize("idx", range(4))
def test_golden_group(idx):
    g = _golden("pack_examples.json")["groups"][idx]
    w = np.array(g["w"], np.float32)
    sb, z, codes = oracle.quantize_group(w)
    assert sb == _h(g["scale_bits"]), g["name"]
    assert z == g["zero"], g["name"]
    assert codes.tolist() == g["codes"], g["name"]
    # the same group through the full packer (FP16 input, N = 1, K = G)
    q, s, zz = oracle.pack(w.astype(np.float16).reshape(1, -1), g["G"])
    assert [int(v) for v in q[0]] == [_h(v) for v in g["words"]]
    assert int(s[0, 0]) == _h(g["scale_bits"])
    assert int(zz[0, 0]) == g["zero"]
    # sum of the dequantised row (exact)
    what = oracle.dequant(q, s, zz, 1, w.shape[0], g["G"])
    assert float(what.astype(np.float64).sum()) == g["sum_w_hat"]


def test_golden_two_group_row():
    d = _golden("pack_examples.json")
    row = np.concatenate([np.array(d["groups"][0]["w"]), np.array(d["groups"][2]["w"])])
    w = row.astype(np.float16).reshape(1, 64)
    q, s, z = oracle.pack(w, 32)
    ex = d["two_group_row"]
    assert [int(v) for v in s[0]] == [_h(v) for v in ex["scales_row"]]
    assert [int(v) for v in z[0]] == [_h(v) for v in ex["zeros_row"]]
    x = np.full((1, 64), 0x3F80, np.uint16)          # BF16 1.0
    y = oracle.linear(x, q, s, z, 1, 64, 32)
    assert y[0, 0] == ex["y_all_ones"]


# --------------------------------------------------------------------------
# Numbers printed on the pages
# --------------------------------------------------------------------------

def _algorithmic_bytes(q, N, K, G):
    """Packed bytes per matrix: codes + one FP16 scale + one 4-bit zero per group (padding excluded)."""
    return q.nbytes + N * (K // G) * 2 + N * (K // G) // 2


def test_closed_form_bits_per_weight_and_model_sizes():
    cf = _golden("closed_forms.json")
    N, K, G = 8, 4096, 128
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    q, s, z = oracle.pack(w, G)
    bpw = _algorithmic_bytes(q, N, K, G) * 8 / (N * K)
    assert bpw == 4 + (16 + 4) / 128                        # 4.15625
    assert round(bpw, cf["bits_per_weight_g128"]["decimals"]) == cf["bits_per_weight_g128"]["value"]
    m = cf["model_13b_bytes"]
    fp16_gb = m["params"] * 16 / 8 / 1e9
    w4_gb = m["params"] * bpw / 8 / 1e9
    assert round(fp16_gb, 1) == m["fp16_gb"]
    assert round(w4_gb, 2) == m["w4_gb"]
    assert round(fp16_gb - w4_gb, 1) == m["saved_gb"]
    a = cf["activation_row_5120"]
    x = np.zeros((1, a["hidden"]), np.uint16)                # one BF16 activation row
    assert round(x.nbytes / 1000, 1) == a["bf16_kb"]
    assert round(x.nbytes / 2 / 1000, 1) == a["int8_kb"]
    b = cf["model_70b_bytes"]
    assert b["params"] * 2 / 1e9 == b["bf16_gb"]
    assert b["params"] * 4 / 8 / 1e9 == b["int4_gb"]


# --------------------------------------------------------------------------
# Closed forms: on-grid round trip and the error bound
# --------------------------------------------------------------------------

@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_on_grid_round_trip(G):
    """Weights already on a group's grid are recovered exactly: q, s and z."""
    rng = np.random.default_rng(G)
    N, K = 8, 2 * G
    ng = K // G
    mant = rng.integers(64, 128, (N, ng))                   # 7-bit significands
    expo = rng.integers(-18, -8, (N, ng))
    s = mant.astype(np.float64) * np.exp2(expo)
    z = rng.integers(0, 16, (N, ng))
    q = rng.integers(0, 16, (N, K))
    for n in range(N):
        for g in range(ng):
            pos = rng.choice(G, 2, replace=False)
            q[n, g * G + pos[0]] = 0
            q[n, g * G + pos[1]] = 15
    w = (q - np.repeat(z, G, axis=1)) * np.repeat(s, G, axis=1)
    w16 = w.astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w)          # on the FP16 grid
    qq, ss, zz = oracle.pack(w16, G)
    assert np.array_equal(oracle.unpack_codes(qq, K), q.astype(np.uint8))
    assert np.array_equal(oracle.unpack_zeros(zz, K, G), z.astype(np.uint8))
    assert np.array_equal(ss[:, :ng].view(np.float16).astype(np.float64), s)


@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_error_bound_and_extremes(G):
    """|w - W_hat| <= (1/2 + 16*2^-11) s for every weight, the group minimum maps
    to code 0 when it is negative, and codes are monotone in w within a group."""
    rng = np.random.default_rng(100 + G)
    N, K = 16, 4 * G
    w = rng.standard_normal((N, K)) * 0.02
    w[:, rng.choice(K, 3, replace=False)] *= 20.0             # outlier channels
    w16 = w.astype(np.float16)
    q, s, z = oracle.pack(w16, G)
    what = oracle.dequant(q, s, z, N, K, G).astype(np.float64)
    codes = oracle.unpack_codes(q, K)
    sc = np.repeat(s[:, : K // G].view(np.float16).astype(np.float64), G, axis=1)
    wf = w16.astype(np.float64)
    assert np.all(np.abs(wf - what) <= (0.5 + 16 * 2.0 ** -11) * sc)
    for n in range(N):
        for g in range(K // G):
            ww = wf[n, g * G:(g + 1) * G]
            cc = codes[n, g * G:(g + 1) * G].astype(int)
            if ww.min() < 0:
                assert cc[np.argmin(ww)] == 0
            order = np.argsort(ww, kind="stable")
            assert np.all(np.diff(cc[order]) >= 0)


def test_degenerate_groups():
    w = np.zeros((8, 64), np.float16)
    w[1, :32] = np.float16(1e-7)           # scale underflows FP16 -> degenerate
    w[2, 32:] = np.float16(-3e-8)
    q, s, z = oracle.pack(w, 32)
    assert np.all(q == 0)
    assert np.all(s[:, :2] == 0x3C00)
    assert np.all(z == 0)
    assert np.all(oracle.dequant(q, s, z, 8, 64, 32) == 0)


def test_pack_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.pack(np.zeros((8, 48), np.float16), 32)       # K % G != 0
    with pytest.raises(ValueError):
        oracle.pack(np.zeros((8, 512), np.float16), 512)     # G beyond 256


# --------------------------------------------------------------------------
# Exact rational brute force of dequantise-then-multiply
# --------------------------------------------------------------------------

def _frac_f16(bits):
    return Fraction(float(np.array([bits], np.uint16).view(np.float16)[0]))


def _frac_bf16(bits):
    return Fraction(float(oracle.bf16_bits_to_f32_array(np.array([bits], np.uint16))[0]))


@pytest.mark.parametrize("M,N,Kg,G", [(1, 8, 1, 32), (3, 16, 2, 32), (1, 16, 2, 64), (3, 8, 1, 128)])
def test_brute_force_rational(M, N, Kg, G):
    K = Kg * G
    rng = np.random.default_rng(M * 1000 + N * 10 + Kg)
    w16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    xb = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    x = xb.view(torch.int16).numpy().view(np.uint16)
    q, s, z = oracle.pack(w16, G)
    y = oracle.linear(x, q, s, z, N, K, G)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                code = (int(q[n, k // 8]) >> (4 * (k % 8))) & 0xF
                g = k // G
                zero = (int(z[n, g // 8]) >> (4 * (g % 8))) & 0xF
                acc += _frac_bf16(x[m, k]) * (code - zero) * _frac_f16(s[n, g])
            ref = float(acc)
            assert abs(y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref)), (m, n, y[m, n], ref)


# --------------------------------------------------------------------------
# Special cases with exact answers
# --------------------------------------------------------------------------

def _random_packed(N, K, G, seed):
    rng = np.random.default_rng(seed)
    w16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    return oracle.pack(w16, G)


def test_one_hot_selects_column_of_w_hat():
    N, K, G = 16, 256, 64
    q, s, z = _random_packed(N, K, G, 7)
    what = oracle.dequant(q, s, z, N, K, G)
    for k in (0, 5, 63, 64, 200, 255):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y = oracle.linear(x, q, s, z, N, K, G)
        assert np.array_equal(y[0], what[:, k].astype(np.float64))


def test_codes_equal_zero_give_zero():
    N, K, G = 8, 128, 32
    q, s, z = _random_packed(N, K, G, 8)
    zeros = oracle.unpack_zeros(z, K, G)
    qz = np.zeros_like(q)
    for k in range(K):
        qz[:, k // 8] |= (zeros[:, k // G].astype(np.uint32) << np.uint32(4 * (k % 8)))
    x = torch.randn(3, K, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    y = oracle.linear(x.view(torch.int16).numpy().view(np.uint16), qz, s, z, N, K, G)
    assert np.all(y == 0.0)


def test_power_of_two_scaling_of_x():
    N, K, G = 16, 256, 128
    q, s, z = _random_packed(N, K, G, 9)
    x = torch.randn(2, K, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    y0 = oracle.linear(x.view(torch.int16).numpy().view(np.uint16), q, s, z, N, K, G)
    for j in (-3, 4):
        xs = (x.float() * 2.0 ** j).to(torch.bfloat16)
        yj = oracle.linear(xs.view(torch.int16).numpy().view(np.uint16), q, s, z, N, K, G)
        assert np.array_equal(yj, y0 * 2.0 ** j)


# --------------------------------------------------------------------------
# Activation-scaled layer (x_scale per input channel)
# --------------------------------------------------------------------------

def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def test_act_scale_of_ones_is_the_plain_layer():
    N, K, G = 16, 512, 128
    q, s, z = _random_packed(N, K, G, 11)
    xb = _bits(torch.randn(3, K, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16))
    y = oracle.linear_xs(xb, np.ones(K, np.float32), q, s, z, N, K, G)
    assert np.array_equal(y, oracle.linear(xb, q, s, z, N, K, G))


def test_act_scale_by_powers_of_two_equals_prescaled_x():
    # x_k * 2^j_k is exact in BF16 for these values, so scaling inside the layer and
    # scaling the input beforehand must give the same FP64 sums bit for bit
    N, K, G = 16, 256, 64
    q, s, z = _random_packed(N, K, G, 12)
    x = torch.randn(2, K, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    j = torch.randint(-4, 5, (K,), generator=torch.Generator().manual_seed(5)).float()
    xs = (2.0 ** j).numpy().astype(np.float32)
    pre = (x.float() * 2.0 ** j).to(torch.bfloat16)
    assert torch.equal(pre.float(), x.float() * 2.0 ** j)
    y = oracle.linear_xs(_bits(x), xs, q, s, z, N, K, G)
    assert np.array_equal(y, oracle.linear(_bits(pre), q, s, z, N, K, G))


@pytest.mark.parametrize("M,N,Kg,G", [(1, 8, 1, 32), (2, 16, 2, 32), (3, 8, 1, 64)])
def test_act_scale_brute_force_rational(M, N, Kg, G):
    # arbitrary FP32 channel factors (not powers of two, some negative, one zero):
    # an index mix-up between channel k and column n or group g fails here
    K = Kg * G
    rng = np.random.default_rng(M * 7 + N + Kg)
    w16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    x = _bits(torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16))
    xs = (rng.uniform(0.2, 3.0, K) * rng.choice([-1.0, 1.0], K)).astype(np.float32)
    xs[K // 3] = 0.0
    q, s, z = oracle.pack(w16, G)
    y = oracle.linear_xs(x, xs, q, s, z, N, K, G)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                code = (int(q[n, k // 8]) >> (4 * (k % 8))) & 0xF
                g = k // G
                zero = (int(z[n, g // 8]) >> (4 * (g % 8))) & 0xF
                acc += _frac_bf16(x[m, k]) * Fraction(float(xs[k])) * (code - zero) * _frac_f16(s[n, g])
            ref = float(acc)
            assert abs(y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref)), (m, n, y[m, n], ref)


# --------------------------------------------------------------------------
# The 8-bit variant: codes kept as two 4-bit planes of a 2K-channel layer
# --------------------------------------------------------------------------

def _planes(q, s, z, K, G):
    """(q8 [N,K], z8 [N,K/G], s8 [N,K/G] as float, s_hi [N,K/G] as float) decoded here
    from the stored planes with the layout rules written out directly."""
    N, ng = q.shape[0], K // G
    codes = oracle.unpack_codes(q, 2 * K)
    zeros = oracle.unpack_zeros(z, 2 * K, G)
    sf = s[:, : 2 * ng].view(np.float16).astype(np.float64)
    q8 = 16 * codes[:, :K].astype(np.int64) + codes[:, K:]
    z8 = 16 * zeros[:, :ng].astype(np.int64) + zeros[:, ng:2 * ng]
    return q8, z8, sf[:, ng:], sf[:, :ng]


@pytest.mark.parametrize("G", [32, 128, 256])
def test_pack8_on_grid_round_trip(G):
    # w = (q8 - z8) * s8 with s8 of <= 3 significant bits is exact in FP16; with codes 0 and
    # 255 in every group, lo = -z8 s8 and hi = (255 - z8) s8, so (hi - lo) / 255 = s8 exactly
    # and the packer must return these codes, zeros and scales
    rng = np.random.default_rng(G)
    N, K = 6, 2 * G
    q8 = rng.integers(0, 256, (N, K))
    z8 = rng.integers(0, 256, (N, K // G))
    s8 = (rng.integers(4, 8, (N, K // G)) * 2.0 ** rng.integers(-14, -6, (N, K // G))).astype(np.float64)
    for n in range(N):
        for g in range(K // G):
            q8[n, g * G] = 0
            q8[n, g * G + 1] = 255
    w = ((q8 - np.repeat(z8, G, axis=1)) * np.repeat(s8, G, axis=1))
    w16 = w.astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w)
    q, s, z = oracle.pack8(w16, G)
    gq8, gz8, gs8, gshi = _planes(q, s, z, K, G)
    assert np.array_equal(gq8, q8) and np.array_equal(gz8, z8) and np.array_equal(gs8, s8)
    assert np.array_equal(gshi, 16.0 * s8)


@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_pack8_error_bound_and_planes(G):
    rng = np.random.default_rng(100 + G)
    N, K = 8, 4 * G
    w16 = (rng.standard_normal((N, K)) * 0.03).astype(np.float16)
    w16[:, 3] = 0.0
    q, s, z = oracle.pack8(w16, G)
    q8, z8, s8, shi = _planes(q, s, z, K, G)
    assert q8.min() >= 0 and q8.max() <= 255 and z8.min() >= 0 and z8.max() <= 255
    assert np.array_equal(shi, 16.0 * s8)                       # hi-plane scale is 16 * s8, exactly
    what = (q8 - np.repeat(z8, G, axis=1)) * np.repeat(s8, G, axis=1)
    err = np.abs(w16.astype(np.float64) - what)
    assert np.all(err <= (0.5 + 255 * 2.0 ** -11) * np.repeat(s8, G, axis=1))
    assert np.all(what[:, 3] == 0.0)                            # exact zeros stay exact
    assert np.array_equal(oracle.dequant8(q, s, z, N, K, G).astype(np.float64), what)
    # each stored plane is itself a valid 4-bit layer row (codes and zeros in 0..15)
    assert np.array_equal(oracle.dequant(q, s, z, N, 2 * K, G)[:, K:].astype(np.float64),
                          (q8 % 16 - np.repeat(z8 % 16, G, axis=1)) * np.repeat(s8, G, axis=1))


def test_pack8_degenerate_groups():
    G, K = 64, 128
    w16 = np.zeros((2, K), np.float16)
    w16[1, G:] = np.float16(2.0 ** -24)                          # range / 255 underflows FP16
    q, s, z = oracle.pack8(w16, G)
    q8, z8, s8, _ = _planes(q, s, z, K, G)
    assert np.all(q8 == 0) and np.all(z8 == 0) and np.all(s8 == 1.0)
    assert np.all(oracle.dequant8(q, s, z, 2, K, G) == 0.0)


@pytest.mark.parametrize("M,N,K,G", [(1, 16, 256, 128), (3, 8, 512, 64), (2, 24, 256, 32)])
def test_linear8_is_the_4bit_layer_over_both_planes(M, N, K, G):
    # the same result along the other route: the planes as a 4-bit layer with 2K input
    # channels, applied to x repeated twice (hi plane meets x, lo plane meets x again)
    rng = np.random.default_rng(M + N + K)
    w16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    x = _bits(torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16))
    q, s, z = oracle.pack8(w16, G)
    y8 = oracle.linear8(x, q, s, z, N, K, G)
    y4 = oracle.linear(np.concatenate([x, x], axis=1), q, s, z, N, 2 * K, G)
    assert np.all(np.abs(y8 - y4) <= 1e-12 * np.maximum(1.0, np.abs(y8)))


@pytest.mark.parametrize("M,N,Kg,G", [(1, 8, 1, 32), (2, 8, 2, 32), (1, 8, 1, 64)])
def test_linear8_brute_force_rational(M, N, Kg, G):
    K = Kg * G
    rng = np.random.default_rng(M * 11 + N + Kg)
    w16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    x = _bits(torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16))
    q, s, z = oracle.pack8(w16, G)
    y = oracle.linear8(x, q, s, z, N, K, G)
    ng = K // G
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                g = k // G
                hi = (int(q[n, k // 8]) >> (4 * (k % 8))) & 0xF
                lo = (int(q[n, (K + k) // 8]) >> (4 * ((K + k) % 8))) & 0xF
                zhi = (int(z[n, g // 8]) >> (4 * (g % 8))) & 0xF
                zlo = (int(z[n, (ng + g) // 8]) >> (4 * ((ng + g) % 8))) & 0xF
                acc += _frac_bf16(x[m, k]) * ((16 * hi + lo) - (16 * zhi + zlo)) * _frac_f16(s[n, ng + g])
            ref = float(acc)
            assert abs(y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref)), (m, n, y[m, n], ref)


# ---- the 8-bit variant in the word layout (four codes per 32-bit word) ----------

def _bytes_of(words, count):
    """Bytes of little-endian 32-bit words, row by row (numpy's own view, not a shift)."""
    return np.ascontiguousarray(words, dtype="<u4").view(np.uint8)[:, :count]


@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_pack8w_equals_the_two_plane_quantiser(G):
    # the same 255-step quantiser: W_hat is bit-identical to the (separately pinned) two-plane
    # storage, on random, outlier and special rows
    rng = np.random.default_rng(300 + G)
    N, K = 10, 4 * G
    w16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    w16[1, ::7] *= np.float16(20.0)
    w16[2] = 0.0
    w16[3] = np.abs(w16[3])
    w16[4] = -np.abs(w16[4])
    w16[5, :G] = np.float16(2.0 ** -24)
    q, s, z = oracle.pack8w(w16, G)
    q2, s2, z2 = oracle.pack8(w16, G)
    a = oracle.dequant8w(q, s, z, N, K, G)
    b = oracle.dequant8(q2, s2, z2, N, K, G)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # the codes, zeros and scales themselves, read through numpy's byte view of the words
    q8, z8, s8, _ = _planes(q2, s2, z2, K, G)
    assert np.array_equal(_bytes_of(q, K).astype(np.int64), q8)
    assert np.array_equal(_bytes_of(z, K // G).astype(np.int64), z8)
    assert np.array_equal(s[:, : K // G].view(np.float16).astype(np.float64), s8)
    assert np.all(s[:, K // G:] == 0) and np.all(_bytes_of(z, z.shape[1] * 4)[:, K // G:] == 0)    # padding


@pytest.mark.parametrize("G", [32, 128])
def test_pack8w_on_grid_round_trip(G):
    rng = np.random.default_rng(400 + G)
    N, K = 6, 2 * G
    q8 = rng.integers(0, 256, (N, K))
    z8 = rng.integers(0, 256, (N, K // G))
    s8 = (rng.integers(4, 8, (N, K // G)) * 2.0 ** rng.integers(-14, -6, (N, K // G))).astype(np.float64)
    q8[:, ::G] = 0
    q8[:, 1::G] = 255
    w = (q8 - np.repeat(z8, G, axis=1)) * np.repeat(s8, G, axis=1)
    w16 = w.astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w)
    q, s, z = oracle.pack8w(w16, G)
    assert np.array_equal(_bytes_of(q, K).astype(np.int64), q8)
    assert np.array_equal(_bytes_of(z, K // G).astype(np.int64), z8)
    assert np.array_equal(s[:, : K // G].view(np.float16).astype(np.float64), s8)


@pytest.mark.parametrize("M,N,Kg,G", [(1, 8, 1, 32), (2, 8, 2, 32), (1, 8, 1, 64)])
def test_linear8w_brute_force_rational(M, N, Kg, G):
    K = Kg * G
    rng = np.random.default_rng(M * 13 + N + Kg)
    w16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    x = _bits(torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16))
    q, s, z = oracle.pack8w(w16, G)
    y = oracle.linear8w(x, q, s, z, N, K, G)
    qb, zb = _bytes_of(q, K), _bytes_of(z, K // G)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                g = k // G
                acc += _frac_bf16(x[m, k]) * (int(qb[n, k]) - int(zb[n, g])) * _frac_f16(s[n, g])
            ref = float(acc)
            assert abs(y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref)), (m, n, y[m, n], ref)
    ms, ns = np.repeat(np.arange(M), N), np.tile(np.arange(N), M)
    assert np.array_equal(oracle.linear8w_sampled(x, q, s, z, K, G, ms, ns), y.reshape(-1))


def test_sampled_equals_full():
    N, K, G = 24, 512, 128
    q, s, z = _random_packed(N, K, G, 10)
    x = torch.randn(4, K, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    y = oracle.linear(xb, q, s, z, N, K, G)
    ms = np.array([0, 3, 1, 2, 3])
    ns = np.array([0, 23, 7, 11, 5])
    ys = oracle.linear_sampled(xb, q, s, z, K, G, ms, ns)
    assert np.array_equal(ys, y[ms, ns])


def test_bf16_output_rounding_is_rne():
    # the oracle's FP64 -> BF16 used by the one-hot exactness checks
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5e-3, 7.0e4, 3.0e38], np.float64)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)
    assert math.isclose(oracle.bf16_to_f32(0x3F80), 1.0)


# --------------------------------------------------------------------------
# The super-block (Q4_K-style) variant
# --------------------------------------------------------------------------

def _q4k_superblock_weights(d, dmin, sc, m, rng):
    """256 weights on the grid of (d, dmin, sc, m): sub-block j holds d*sc_j*q - dmin*m_j for q = 0..15
    (each code twice, in a random order), computed exactly in FP64."""
    w = np.zeros(256, np.float64)
    codes = np.zeros(256, np.int64)
    for j in range(8):
        q = rng.permutation(np.tile(np.arange(16), 2))
        codes[32 * j:32 * j + 32] = q
        w[32 * j:32 * j + 32] = d * sc[j] * q - dmin * m[j]
    return w, codes


def test_q4k_golden_record():
    """The packer writes the hand-derived record, and the record reads back to the same factors and codes."""
    gd = _golden("q4k_record.json")
    d, dmin = oracle.f16_to_f32(_h(gd["d_bits"])), oracle.f16_to_f32(_h(gd["dmin_bits"]))
    w, codes = _q4k_superblock_weights(d, dmin, gd["sc"], gd["m"], np.random.default_rng(5))
    w16 = w.astype(np.float16)
    assert np.array_equal(w16.astype(np.float64), w)          # the example is exact in FP16
    q, meta = oracle.q4k_pack(w16.reshape(1, 256))
    assert [int(v) for v in meta[0]] == [_h(s) for s in gd["words"]]
    assert np.array_equal(oracle.unpack_codes(q, 256)[0], codes)
    dd, dm, sc, m = oracle.q4k_record(meta, 256, 0, 0)
    assert (dd, dm) == (d, dmin)
    assert list(sc) == gd["sc"] and list(m) == gd["m"]
    assert np.array_equal(oracle.q4k_dequant(q, meta, 1, 256)[0].astype(np.float64), w)


@pytest.mark.parametrize("seed", range(6))
def test_q4k_on_grid_round_trip(seed):
    """Weights on a super-block's grid (any FP16 d, dmin; sc and m spanning 0..63 with 63 present, and
    15 d sc_j >= dmin m_j so each sub-block's range is [-dmin m_j, 15 d sc_j - dmin m_j]) come back exactly:
    factors, 6-bit codes and 4-bit codes."""
    rng = np.random.default_rng(100 + seed)
    d = float(np.float16(rng.uniform(1e-4, 1e-2)))
    dmin = float(np.float16(rng.uniform(1e-4, 1e-2)))
    sc = rng.integers(1, 64, 8)
    sc[rng.integers(8)] = 63
    m = np.array([min(63, int(rng.integers(0, 64))) for _ in range(8)])
    m[rng.integers(8)] = 63
    for j in range(8):                                          # keep 0 inside the sub-block's range
        while 15 * d * sc[j] < dmin * m[j]:
            sc[j] += 1
    sc = np.minimum(sc, 63)
    assert all(15 * d * sc[j] >= dmin * m[j] for j in range(8))
    w, codes = _q4k_superblock_weights(d, dmin, sc, m, rng)
    w32 = w.astype(np.float32)            # d*sc*q is exact in FP32; the subtraction may round
    db, dmb, sc_o, m_o, q_o = oracle.q4k_quantize_superblock(w32)
    assert oracle.f16_to_f32(db) == d and oracle.f16_to_f32(dmb) == dmin
    assert np.array_equal(sc_o, sc) and np.array_equal(m_o, m)
    assert np.array_equal(q_o.astype(np.int64), codes)


@pytest.mark.parametrize("seed", range(4))
def test_q4k_error_bounds(seed):
    """Hierarchical step: the stored sub-block scale and minimum are within d/2 and dmin/2 of the sub-block's
    own min-max values (6-bit codes of FP16 factors that are the maxima over 63).  Reconstruction: a weight
    inside the stored range [-b'_j, 15 a'_j - b'_j] is within a'_j / 2 of its reconstruction; one outside is
    clamped to the nearer end."""
    rng = np.random.default_rng(200 + seed)
    scale = [0.02, 1.0, 3e-3, 40.0][seed]
    w = (rng.standard_normal(256) * scale).astype(np.float16).astype(np.float32)
    w[rng.integers(256)] *= 6.0                                  # an outlier in one sub-block
    db, dmb, sc, m, q = oracle.q4k_quantize_superblock(w)
    d, dmin = oracle.f16_to_f32(db), oracle.f16_to_f32(dmb)
    for j in range(8):
        blk = w[32 * j:32 * j + 32].astype(np.float64)
        lo, hi = min(0.0, blk.min()), max(0.0, blk.max())
        a, b = (hi - lo) / 15, -lo
        ap, bp = d * sc[j], dmin * m[j]
        assert abs(ap - a) <= d / 2 * (1 + 1e-3) + 1e-7 * a, (j, ap, a, d)
        assert abs(bp - b) <= dmin / 2 * (1 + 1e-3) + 1e-7 * b, (j, bp, b, dmin)
        rec = ap * q[32 * j:32 * j + 32] - bp
        for v, r in zip(blk, rec):
            if -bp <= v <= 15 * ap - bp:
                assert abs(v - r) <= ap / 2 * (1 + 1e-5) + 1e-7 * abs(v), (j, v, r, ap)
            else:
                assert r == (-bp if v < -bp else 15 * ap - bp)


def test_q4k_degenerate_superblocks():
    """All-zero super-block: d = 1, dmin = 0, every code 0, W_hat = 0.  A zero sub-block amid others
    reconstructs as exact zeros.  A super-block without negative weights stores dmin = 0 and m = 0."""
    z = np.zeros(256, np.float32)
    db, dmb, sc, m, q = oracle.q4k_quantize_superblock(z)
    assert (db, dmb) == (0x3C00, 0) and not sc.any() and not m.any() and not q.any()
    rng = np.random.default_rng(7)
    w = (rng.standard_normal(256) * 0.02).astype(np.float16)
    w[64:96] = 0
    q, meta = oracle.q4k_pack(w.reshape(1, 256))
    wh = oracle.q4k_dequant(q, meta, 1, 256)[0]
    assert not wh[64:96].any()
    pos = np.abs(w).reshape(1, 256)
    q, meta = oracle.q4k_pack(pos)
    dd, dm, sc, m = oracle.q4k_record(meta, 256, 0, 0)
    assert dm == 0.0 and not m.any()
    # weights far from 0 on one side: the range widened to hold 0 keeps every weight within half a step
    # plus the 6-bit rounding of the sub-block scale (|d sc_j - a_j| <= d/2, over 15 steps)
    far = rng.uniform(0.5, 1.0, (1, 256)).astype(np.float16)
    q, meta = oracle.q4k_pack(far)
    dd, dm, sc, m = oracle.q4k_record(meta, 256, 0, 0)
    wh = oracle.q4k_dequant(q, meta, 1, 256)[0].astype(np.float64)
    err = np.abs(wh - far[0].astype(np.float64)).reshape(8, 32).max(axis=1)
    assert (err <= dd * sc / 2 + 15 * dd / 2 + 1e-6).all(), (err, dd, sc)
    with pytest.raises(ValueError):
        oracle.q4k_pack(np.zeros((2, 384), np.float16))


@pytest.mark.parametrize("M,N,K", [(1, 4, 256), (2, 3, 512)])
def test_q4k_brute_force_rational(M, N, K):
    """y = sum_k x * (d sc_j q - dmin m_j), the fields decoded here from the record definition and summed
    in exact rationals; the oracle's FP32 W_hat rounds once (relative 2^-24 per weight)."""
    rng = np.random.default_rng(M * 100 + N + K)
    w16 = (rng.standard_normal((N, K)) * 0.05).astype(np.float16)
    xb = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    x = xb.view(torch.int16).numpy().view(np.uint16)
    q, meta = oracle.q4k_pack(w16)
    y = oracle.q4k_linear(x, q, meta, N, K)
    for n in range(N):
        for mm in range(M):
            acc, mag = Fraction(0), 0.0
            for k in range(K):
                rec = [int(v) for v in meta[n, (k // 256) * 4:(k // 256) * 4 + 4]]
                j = (k % 256) // 32
                sc = ((rec[1] >> (4 * j)) & 15) | (((rec[3] >> (2 * j)) & 3) << 4)
                mj = ((rec[2] >> (4 * j)) & 15) | (((rec[3] >> (16 + 2 * j)) & 3) << 4)
                code = (int(q[n, k // 8]) >> (4 * (k % 8))) & 0xF
                wv = _frac_f16(rec[0] & 0xFFFF) * sc * code - _frac_f16(rec[0] >> 16) * mj
                acc += _frac_bf16(x[mm, k]) * wv
                mag += abs(float(_frac_bf16(x[mm, k]) * wv))
            ref = float(acc)
            assert abs(y[mm, n] - ref) <= 2 ** -23 * mag + 1e-12, (mm, n, y[mm, n], ref)


def test_q4k_linear_matches_dequant_then_matmul_and_sampling():
    rng = np.random.default_rng(11)
    N, K, M = 37, 768, 3
    w16 = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    xb = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    x = xb.view(torch.int16).numpy().view(np.uint16)
    q, meta = oracle.q4k_pack(w16)
    y = oracle.q4k_linear(x, q, meta, N, K)
    wh = oracle.q4k_dequant(q, meta, N, K).astype(np.float64)
    ref = xb.float().numpy().astype(np.float64) @ wh.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # one-hot x picks a column of W_hat
    e = np.zeros((1, K), np.uint16)
    e[0, 300] = 0x3F80                                           # BF16 1.0
    assert np.array_equal(oracle.q4k_linear(e, q, meta, N, K)[0], wh[:, 300])
    ms, ns = np.array([0, 2, 1, 2]), np.array([0, 36, 17, 5])
    assert np.array_equal(oracle.q4k_linear_sampled(x, q, meta, K, ms, ns), y[ms, ns])


def test_q4k_bits_per_weight_and_70b_size():
    """4 bits per code plus one 16-byte record per 256 weights: 4.5 bits per weight.  The pages put a 70B
    model at about 35 GB in an ideal 4-bit encoding and note that real Q4_K files are larger because block
    scales and minima take space (zhuai.tech, section 2 'Capacity comes first')."""
    cf = _golden("closed_forms.json")["model_70b_bytes"]
    N, K = 4, 1024
    q, meta = oracle.q4k_pack(np.zeros((N, K), np.float16))
    bpw = (q.nbytes + meta.nbytes) * 8 / (N * K)
    assert bpw == 4.5
    gb = cf["params"] * bpw / 8 / 1e9
    assert gb > cf["int4_gb"] and round(gb, 2) == 39.38


# property-based: any super-block on the grid of (d, dmin, sc, m) comes back exactly
from hypothesis import HealthCheck, given, settings, strategies as st  # noqa: E402


@st.composite
def _q4k_grid(draw):
    # FP16 factors across a wide exponent range; the d*sc*q - dmin*m grid kept inside FP16's normal range
    d = float(np.float16(draw(st.floats(2.0 ** -14, 2.0 ** -2, allow_nan=False, allow_infinity=False))))
    dmin = float(np.float16(draw(st.floats(2.0 ** -14, 2.0 ** -2, allow_nan=False, allow_infinity=False))))
    sc = draw(st.lists(st.integers(0, 63), min_size=8, max_size=8))
    m = draw(st.lists(st.integers(0, 63), min_size=8, max_size=8))
    sc[draw(st.integers(0, 7))] = 63
    m[draw(st.integers(0, 7))] = 63
    for j in range(8):                       # zero inside each sub-block's range, and a'_j > 0
        if sc[j] == 0 or 15 * d * sc[j] < dmin * m[j]:
            sc[j] = 63
            if 15 * d * 63 < dmin * m[j]:
                m[j] = int(15 * d * 63 // dmin)
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return d, dmin, np.array(sc), np.array(m), seed


@settings(max_examples=60, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(_q4k_grid())
def test_q4k_on_grid_round_trip_property(grid):
    d, dmin, sc, m, seed = grid
    if m.max() < 63 or 15 * d * 63 < dmin * 63:
        return                                # the clamp above removed the 63 that fixes dmin
    w, codes = _q4k_superblock_weights(d, dmin, sc, m, np.random.default_rng(seed))
    db, dmb, sc_o, m_o, q_o = oracle.q4k_quantize_superblock(w.astype(np.float32))
    assert oracle.f16_to_f32(db) == d and oracle.f16_to_f32(dmb) == dmin
    assert np.array_equal(sc_o, sc) and np.array_equal(m_o, m)
    assert np.array_equal(q_o.astype(np.int64), codes)


@st.composite
def _w4_grid(draw):
    G = draw(st.sampled_from([32, 64, 128, 256]))
    mant = draw(st.integers(64, 127))                     # 7-bit significand: (q - z) * s is exact in FP16
    expo = draw(st.integers(-18, -8))
    z = draw(st.integers(0, 15))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return G, mant * 2.0 ** expo, z, seed


@settings(max_examples=60, deadline=None)
@given(_w4_grid())
def test_on_grid_round_trip_property(grid):
    """One group on the grid of any (s, z), codes 0 and 15 both present: the packer gives back s, z and every
    code, including z = 0 (no negative weight) and z = 15 (no positive weight)."""
    G, s, z, seed = grid
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 16, G)
    pos = rng.choice(G, 2, replace=False)
    q[pos[0]], q[pos[1]] = 0, 15
    w = (q - z) * s
    w16 = w.astype(np.float16).reshape(1, G)
    assert np.array_equal(w16.astype(np.float64)[0], w)
    qq, ss, zz = oracle.pack(w16, G)
    assert np.array_equal(oracle.unpack_codes(qq, G)[0], q.astype(np.uint8))
    assert oracle.unpack_zeros(zz, G, G)[0, 0] == z
    assert ss[0, 0].view(np.float16).astype(np.float64) == s
