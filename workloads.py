"""Seeded synthetic inputs and the workload table for the W4A16 linear layer.

This module holds no quantisation or GEMM arithmetic.  It only draws the
random inputs (FP16 weights, BF16 activations) that both the CUDA path and the
CPU oracle consume, so the two sides see bit-identical data.

Input recipe (weights are never trained; no dataset is involved):
  * torch CPU generator, ``torch.Generator().manual_seed(seed)``;
  * W ~ N(0, sigma) drawn in FP32, optional outlier input channels multiplied
    by 20 in FP32, then round-to-nearest-even to FP16;
  * x ~ N(0, 1) drawn in FP32, then round-to-nearest-even to BF16;
  * the j-th matrix of a workload uses seed + 100*j, its activations seed +
    100*j + 50;
  * super-block (Q4_K-style) workloads draw W the same way and pack it into
    256-channel super-blocks (G is then the 32-channel sub-block);
  * activation-scaled workloads draw x_scale = 1/alpha with alpha = 1 except on a
    seeded 1 % of input channels, where alpha ~ U[2, 4) (seed + 100*j + 70), and
    pack W * alpha rounded to FP16.

The shapes follow the pages' examples: a 13B-class layer (hidden 5120, FFN
13824: multigrid.ai "Weight-Only Quantization Explained", section "The memory
arithmetic") and a 70B-class layer (hidden 8192, FFN 28672: zhuai.tech
"Quantization Is Not a Zip File", section 2 "Capacity comes first" sizes a 70B
model).  Group sizes are 32/64/128/256 (same page, section 3, "Block
locality").  Decode uses M=1..16 rows, prefill M=2048.
"""
from dataclasses import dataclass
from typing import Tuple

import torch


@dataclass(frozen=True)
class Linear:
    name: str
    K: int
    N: int


@dataclass(frozen=True)
class Workload:
    name: str
    linears: Tuple[Linear, ...]
    Ms: Tuple[int, ...]
    Gs: Tuple[int, ...]
    sigma: float
    outlier_frac: float
    seed: int
    dual: bool = False
    act_scaled: bool = False     # layer with a per-input-channel activation scale
    bits: int = 4                # weight code width: 4, or 8 (the W8A16 variant)
    q4k: bool = False            # super-block (Q4_K-style) layout instead of groups of G


WORKLOADS = {
    # single 4096x4096 decode GEMV
    "single_4096": Workload("single_4096", (Linear("linear", 4096, 4096),), (1,), (128,), 0.02, 0.0, 0),
    # 13B-shaped decoder-layer linears at decode
    "layer13b_decode": Workload(
        "layer13b_decode",
        (Linear("q", 5120, 5120), Linear("k", 5120, 5120), Linear("v", 5120, 5120), Linear("o", 5120, 5120),
         Linear("gate", 5120, 13824), Linear("up", 5120, 13824), Linear("down", 13824, 5120)),
        (1,), (128,), 0.02, 0.001, 1),
    # batch x group-size sweep on the 5120->13824 up-projection
    "up13b_sweep": Workload("up13b_sweep", (Linear("up", 5120, 13824),), (1, 2, 4, 8, 16, 32),
                            (32, 64, 128, 256), 0.02, 0.001, 2),
    # paired gate/up projections sharing one x
    "gateup13b_dual": Workload("gateup13b_dual", (Linear("gate", 5120, 13824), Linear("up", 5120, 13824)),
                               (1, 4), (128,), 0.02, 0.0, 3, dual=True),
    # 13B FFN with an activation scale fused into x staging (salient channels 1 %)
    "ffn13b_awq": Workload("ffn13b_awq", (Linear("gate", 5120, 13824), Linear("down", 13824, 5120)),
                           (1, 4, 32), (128,), 0.02, 0.0, 5, act_scaled=True),
    # the 8-bit variant on the 13B up-projection, decode and a small batch
    "up13b_w8": Workload("up13b_w8", (Linear("up", 5120, 13824),), (1, 4, 32), (128,), 0.02, 0.0, 6, bits=8),
    # the 70B FFN gate and down in the super-block (Q4_K-style) layout, decode
    "ffn70b_q4k": Workload("ffn70b_q4k", (Linear("gate", 8192, 28672), Linear("down", 28672, 8192)), (1, 3),
                           (32,), 0.015, 0.0, 7, q4k=True),
    # 70B-shaped FFN gate and down, decode (M=1) and prefill (M=2048)
    "ffn70b": Workload("ffn70b", (Linear("gate", 8192, 28672), Linear("down", 28672, 8192)), (1, 2048),
                       (128,), 0.015, 0.0, 4),
}


def weight_f16(N: int, K: int, sigma: float, seed: int, outlier_frac: float = 0.0) -> torch.Tensor:
    """FP16 [N,K] weight: N(0, sigma) in FP32, outlier channels x20, RNE to FP16."""
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(N, K, generator=g, dtype=torch.float32) * sigma
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        cols = torch.randperm(K, generator=g)[:n_out]
        w[:, cols] *= 20.0
    return w.to(torch.float16)


def activations_bf16(M: int, K: int, seed: int) -> torch.Tensor:
    """BF16 [M,K] activations: N(0,1) in FP32, RNE to BF16."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)


def act_scale_f32(K: int, seed: int, salient_frac: float = 0.01) -> torch.Tensor:
    """FP32 [K] activation scale of the activation-scaled layer, x_scale = 1 / alpha:
    alpha = 1 on most input channels and alpha ~ U[2, 4) in FP32 on a seeded
    `salient_frac` of them (the channels whose weights activation-aware
    quantisation scales up before packing and whose activations it scales down)."""
    g = torch.Generator().manual_seed(seed)
    alpha = torch.ones(K, dtype=torch.float32)
    n_sal = max(1, int(round(salient_frac * K)))
    cols = torch.randperm(K, generator=g)[:n_sal]
    alpha[cols] = 2.0 + 2.0 * torch.rand(n_sal, generator=g, dtype=torch.float32)
    return 1.0 / alpha


def awq_weight_f16(w: torch.Tensor, x_scale: torch.Tensor) -> torch.Tensor:
    """FP16 [N,K] weight to pack for the activation-scaled layer: W * alpha per input
    channel (alpha = 1 / x_scale), formed in FP32 and rounded to FP16."""
    return (w.float() / x_scale.float()).to(torch.float16)


def matrix_seed(workload: Workload, j: int) -> int:
    return workload.seed + 100 * j


def act_seed(workload: Workload, j: int) -> int:
    return workload.seed + 100 * j + 50


def bits_u16(t: torch.Tensor):
    """FP16/BF16 tensor -> numpy uint16 bit patterns (for the oracle)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def random_u32(shape, seed: int):
    """numpy uint32 array of uniformly random words (every nibble and byte value
    occurs): raw packed codes, zero-point words or record fields for the checks
    that feed arbitrary bit patterns through the unpacking routines."""
    import numpy as np
    g = torch.Generator().manual_seed(seed)
    lo = torch.randint(0, 1 << 16, tuple(shape), generator=g, dtype=torch.int64)
    hi = torch.randint(0, 1 << 16, tuple(shape), generator=g, dtype=torch.int64)
    return ((hi << 16) | lo).numpy().astype(np.uint32)


def random_f16_bits(shape, seed: int, exp_lo: int = 1, exp_hi: int = 30, sign: bool = False):
    """numpy uint16 array of FP16 bit patterns with a uniformly random biased
    exponent in [exp_lo, exp_hi] (0 = subnormal, 30 = largest finite) and
    mantissa, positive unless `sign`: arbitrary finite scale values."""
    import numpy as np
    g = torch.Generator().manual_seed(seed)
    e = torch.randint(exp_lo, exp_hi + 1, tuple(shape), generator=g, dtype=torch.int64)
    m = torch.randint(0, 1 << 10, tuple(shape), generator=g, dtype=torch.int64)
    s = torch.randint(0, 2, tuple(shape), generator=g, dtype=torch.int64) if sign else torch.zeros_like(e)
    return ((s << 15) | (e << 10) | m).numpy().astype(np.uint16)
