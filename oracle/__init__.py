"""CPU oracle for the W4A16 weight-only linear layer -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the `cpu_baseline` / reference
leg of `bench.py` may import this package.  The product path (the CUDA
library and its Python binding) never imports it and shares no code with it.

This module is a thin ctypes wrapper around `w4a16_oracle.c` (plain C99,
FP64 accumulation); every function's arithmetic lives in that file and is
documented there with the page and section it follows.  Arrays are numpy:
FP16 and BF16 values travel as their uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        u16 = ctypes.c_uint16
        p = ctypes.c_void_p
        lib.oracle_f16_to_f32.argtypes, lib.oracle_f16_to_f32.restype = [u16], f32
        lib.oracle_bf16_to_f32.argtypes, lib.oracle_bf16_to_f32.restype = [u16], f32
        lib.oracle_f32_to_f16.argtypes, lib.oracle_f32_to_f16.restype = [f32], u16
        lib.oracle_f32_to_bf16.argtypes, lib.oracle_f32_to_bf16.restype = [f32], u16
        lib.oracle_f64_to_bf16.argtypes, lib.oracle_f64_to_bf16.restype = [f64], u16
        lib.oracle_qweight_ld.argtypes, lib.oracle_qweight_ld.restype = [i64], i64
        lib.oracle_scales_ld.argtypes, lib.oracle_scales_ld.restype = [i64, i64], i64
        lib.oracle_zeros_ld.argtypes, lib.oracle_zeros_ld.restype = [i64, i64], i64
        lib.oracle_quantize_group.argtypes = [p, i64, p, p, p]
        lib.oracle_quantize_group.restype = None
        lib.oracle_pack.argtypes = [p, i64, i64, i64, p, p, p, i32]
        lib.oracle_pack.restype = i32
        lib.oracle_dequant.argtypes = [p, p, p, i64, i64, i64, p, i32]
        lib.oracle_dequant.restype = None
        lib.oracle_linear.argtypes = [p, p, p, p, i64, i64, i64, i64, p, i32]
        lib.oracle_linear.restype = None
        lib.oracle_linear_sampled.argtypes = [p, p, p, p, i64, i64, p, p, i64, p, i32]
        lib.oracle_linear_sampled.restype = None
        lib.oracle_pack8.argtypes = [p, i64, i64, i64, p, p, p, i32]
        lib.oracle_pack8.restype = i32
        lib.oracle_dequant8.argtypes = [p, p, p, i64, i64, i64, p, i32]
        lib.oracle_dequant8.restype = None
        lib.oracle_linear8.argtypes = [p, p, p, p, i64, i64, i64, i64, p, i32]
        lib.oracle_linear8.restype = None
        lib.oracle_zeros8w_ld.argtypes, lib.oracle_zeros8w_ld.restype = [i64, i64], i64
        lib.oracle_pack8w.argtypes = [p, i64, i64, i64, p, p, p, i32]
        lib.oracle_pack8w.restype = i32
        lib.oracle_dequant8w.argtypes = [p, p, p, i64, i64, i64, p, i32]
        lib.oracle_dequant8w.restype = None
        lib.oracle_linear8w.argtypes = [p, p, p, p, i64, i64, i64, i64, p, i32]
        lib.oracle_linear8w.restype = None
        lib.oracle_linear8w_sampled.argtypes = [p, p, p, p, i64, i64, p, p, i64, p, i32]
        lib.oracle_linear8w_sampled.restype = None
        lib.oracle_linear_xs.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, i32]
        lib.oracle_linear_xs.restype = None
        lib.oracle_q4k_meta_ld.argtypes, lib.oracle_q4k_meta_ld.restype = [i64], i64
        lib.oracle_q4k_quantize_superblock.argtypes = [p, p, p, p, p, p]
        lib.oracle_q4k_quantize_superblock.restype = None
        lib.oracle_q4k_pack.argtypes = [p, i64, i64, p, p, i32]
        lib.oracle_q4k_pack.restype = i32
        lib.oracle_q4k_record.argtypes = [p, i64, i64, i64, p, p, p, p]
        lib.oracle_q4k_record.restype = None
        lib.oracle_q4k_dequant.argtypes = [p, p, i64, i64, p, i32]
        lib.oracle_q4k_dequant.restype = None
        lib.oracle_q4k_linear.argtypes = [p, p, p, i64, i64, i64, p, i32]
        lib.oracle_q4k_linear.restype = None
        lib.oracle_q4k_linear_sampled.argtypes = [p, p, p, i64, p, p, i64, p, i32]
        lib.oracle_q4k_linear_sampled.restype = None
        lib.oracle_max_threads.argtypes, lib.oracle_max_threads.restype = [], i32
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, f"expected FP16/BF16 bit patterns as uint16, got {a.dtype}"
    return a


# ---- scalar conversions (IEEE definitions) ---------------------------------

def f16_to_f32(h: int) -> float:
    return _load().oracle_f16_to_f32(int(h))


def bf16_to_f32(b: int) -> float:
    return _load().oracle_bf16_to_f32(int(b))


def f32_to_f16(f: float) -> int:
    return _load().oracle_f32_to_f16(float(np.float32(f)))


def f32_to_bf16(f: float) -> int:
    return _load().oracle_f32_to_bf16(float(np.float32(f)))


def f64_to_bf16(d: float) -> int:
    return _load().oracle_f64_to_bf16(float(d))


def bf16_bits_to_f32_array(b: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns (the top half of a binary32)."""
    b = _u16(b)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---- layout -----------------------------------------------------------------

def qweight_ld(K: int) -> int:
    return _load().oracle_qweight_ld(K)


def scales_ld(K: int, G: int) -> int:
    return _load().oracle_scales_ld(K, G)


def zeros_ld(K: int, G: int) -> int:
    return _load().oracle_zeros_ld(K, G)


# ---- quantiser / packer -----------------------------------------------------

def quantize_group(w: np.ndarray):
    """One group: returns (scale_bits: int, zero: int, codes: uint8[G])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    G = w.shape[0]
    sb = np.zeros(1, np.uint16)
    z = np.zeros(1, np.int32)
    codes = np.zeros(G, np.uint8)
    _load().oracle_quantize_group(_ptr(w), G, _ptr(sb), _ptr(z), _ptr(codes))
    return int(sb[0]), int(z[0]), codes


def pack(w_f16: np.ndarray, G: int, nthreads: int = 0):
    """FP16 W [N,K] -> (qweight u32 [N,K/8], scales u16 [N,ldS], zeros u32 [N,ldZ])."""
    w = _u16(w_f16)
    N, K = w.shape
    q = np.zeros((N, qweight_ld(K)), np.uint32)
    s = np.zeros((N, scales_ld(K, G)), np.uint16)
    z = np.zeros((N, zeros_ld(K, G)), np.uint32)
    rc = _load().oracle_pack(_ptr(w), N, K, G, _ptr(q), _ptr(s), _ptr(z), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_pack rejected N={N} K={K} G={G}")
    return q, s, z


# ---- unpack / dequant ---------------------------------------------------------

def unpack_codes(q: np.ndarray, K: int) -> np.ndarray:
    """Codes [N,K] (uint8), nibble k%8 of word k/8, low nibble first."""
    q = np.ascontiguousarray(q, dtype=np.uint32)
    N = q.shape[0]
    out = np.zeros((N, K), np.uint8)
    for j in range(8):
        out[:, j::8] = ((q[:, : K // 8] >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.uint8)
    return out


def unpack_zeros(z: np.ndarray, K: int, G: int) -> np.ndarray:
    """Zero points [N, K/G] (uint8)."""
    z = np.ascontiguousarray(z, dtype=np.uint32)
    ng = K // G
    N = z.shape[0]
    out = np.zeros((N, ng), np.uint8)
    for g in range(ng):
        out[:, g] = ((z[:, g // 8] >> np.uint32(4 * (g % 8))) & np.uint32(0xF)).astype(np.uint8)
    return out


def dequant(q, s, z, N: int, K: int, G: int, nthreads: int = 0) -> np.ndarray:
    """W_hat [N,K] FP32, (q - z) * s per element."""
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    out = np.zeros((N, K), np.float32)
    _load().oracle_dequant(_ptr(q), _ptr(s), _ptr(z), N, K, G, _ptr(out), nthreads)
    return out


# ---- the layer ------------------------------------------------------------------

def linear(x_bf16: np.ndarray, q, s, z, N: int, K: int, G: int, nthreads: int = 0) -> np.ndarray:
    """y_ref [M,N] FP64 = x * W_hat^T, unrounded."""
    x = _u16(x_bf16)
    M = x.shape[0]
    assert x.shape[1] == K
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    y = np.zeros((M, N), np.float64)
    _load().oracle_linear(_ptr(x), _ptr(q), _ptr(s), _ptr(z), M, N, K, G, _ptr(y), nthreads)
    return y


def linear_sampled(x_bf16: np.ndarray, q, s, z, K: int, G: int, ms, ns, nthreads: int = 0) -> np.ndarray:
    """y_ref at the listed (m, n) positions only, FP64."""
    x = _u16(x_bf16)
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    assert ms.shape == ns.shape
    y = np.zeros(ms.shape[0], np.float64)
    _load().oracle_linear_sampled(_ptr(x), _ptr(q), _ptr(s), _ptr(z), K, G, _ptr(ms), _ptr(ns),
                                  ms.shape[0], _ptr(y), nthreads)
    return y


def linear_xs(x_bf16: np.ndarray, x_scale: np.ndarray, q, s, z, N: int, K: int, G: int,
              nthreads: int = 0) -> np.ndarray:
    """y_ref [M,N] FP64 = (x * x_scale) * W_hat^T, unrounded; x_scale FP32 [K]
    multiplies input channel k (the activation-scaled layer)."""
    x = _u16(x_bf16)
    M = x.shape[0]
    assert x.shape[1] == K
    xs = np.ascontiguousarray(x_scale, dtype=np.float32)
    assert xs.shape == (K,)
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    y = np.zeros((M, N), np.float64)
    _load().oracle_linear_xs(_ptr(x), _ptr(xs), _ptr(q), _ptr(s), _ptr(z), M, N, K, G, _ptr(y), nthreads)
    return y


# ---- the 8-bit variant ---------------------------------------------------------

def pack8(w_f16: np.ndarray, G: int, nthreads: int = 0):
    """FP16 [N,K] -> (qweight u32 [N, K/4], scales u16 [N, scales_ld(2K, G)],
    zeros u32 [N, zeros_ld(2K, G)]): 8-bit codes kept as two 4-bit planes of a
    2K-channel 4-bit layer (hi nibbles, then lo nibbles; scales 16*s8 then s8;
    zeros z8 >> 4 then z8 & 15)."""
    w = _u16(w_f16)
    N, K = w.shape
    q = np.zeros((N, qweight_ld(2 * K)), np.uint32)
    s = np.zeros((N, scales_ld(2 * K, G)), np.uint16)
    z = np.zeros((N, zeros_ld(2 * K, G)), np.uint32)
    rc = _load().oracle_pack8(_ptr(w), N, K, G, _ptr(q), _ptr(s), _ptr(z), nthreads)
    if rc != 0:
        raise ValueError("oracle_pack8: bad shape")
    return q, s, z


def dequant8(q, s, z, N: int, K: int, G: int, nthreads: int = 0) -> np.ndarray:
    """W_hat8 [N,K] FP32 = (q8 - z8) * s8 read back from the planes."""
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    out = np.zeros((N, K), np.float32)
    _load().oracle_dequant8(_ptr(q), _ptr(s), _ptr(z), N, K, G, _ptr(out), nthreads)
    return out


def linear8(x_bf16: np.ndarray, q, s, z, N: int, K: int, G: int, nthreads: int = 0) -> np.ndarray:
    """y_ref [M,N] FP64 = x * W_hat8^T, unrounded."""
    x = _u16(x_bf16)
    M = x.shape[0]
    assert x.shape[1] == K
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    y = np.zeros((M, N), np.float64)
    _load().oracle_linear8(_ptr(x), _ptr(q), _ptr(s), _ptr(z), M, N, K, G, _ptr(y), nthreads)
    return y


# ---- the 8-bit variant in the word layout (four codes per 32-bit word) -----------

def zeros8w_ld(K: int, G: int) -> int:
    """uint32 words per zeros row of the word layout (four 8-bit zero points per word)."""
    return _load().oracle_zeros8w_ld(K, G)


def pack8w(w_f16: np.ndarray, G: int, nthreads: int = 0):
    """FP16 [N,K] -> (qweight u32 [N, K/4], scales u16 [N, scales_ld(K, G)],
    zeros u32 [N, zeros8w_ld(K, G)]): 8-bit codes four per word, low byte
    first; one FP16 scale and one 8-bit zero point per group."""
    w = _u16(w_f16)
    N, K = w.shape
    q = np.zeros((N, K // 4), np.uint32)
    s = np.zeros((N, scales_ld(K, G)), np.uint16)
    z = np.zeros((N, zeros8w_ld(K, G)), np.uint32)
    rc = _load().oracle_pack8w(_ptr(w), N, K, G, _ptr(q), _ptr(s), _ptr(z), nthreads)
    if rc != 0:
        raise ValueError("oracle_pack8w: bad shape")
    return q, s, z


def dequant8w(q, s, z, N: int, K: int, G: int, nthreads: int = 0) -> np.ndarray:
    """W_hat [N,K] FP32 = (q - z) * s of the word layout."""
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    out = np.zeros((N, K), np.float32)
    _load().oracle_dequant8w(_ptr(q), _ptr(s), _ptr(z), N, K, G, _ptr(out), nthreads)
    return out


def linear8w(x_bf16: np.ndarray, q, s, z, N: int, K: int, G: int, nthreads: int = 0) -> np.ndarray:
    """y_ref [M,N] FP64 = x * W_hat^T of the word layout, unrounded."""
    x = _u16(x_bf16)
    M = x.shape[0]
    assert x.shape[1] == K
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    y = np.zeros((M, N), np.float64)
    _load().oracle_linear8w(_ptr(x), _ptr(q), _ptr(s), _ptr(z), M, N, K, G, _ptr(y), nthreads)
    return y


def linear8w_sampled(x_bf16: np.ndarray, q, s, z, K: int, G: int, ms, ns, nthreads: int = 0) -> np.ndarray:
    """y_ref of the word layout at the listed (m, n) positions only, FP64."""
    x = _u16(x_bf16)
    q = np.ascontiguousarray(q, dtype=np.uint32)
    s = _u16(s)
    z = np.ascontiguousarray(z, dtype=np.uint32)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.zeros(ms.shape[0], np.float64)
    _load().oracle_linear8w_sampled(_ptr(x), _ptr(q), _ptr(s), _ptr(z), K, G, _ptr(ms), _ptr(ns), ms.shape[0],
                                    _ptr(y), nthreads)
    return y


# ---- the super-block (Q4_K-style) variant ----------------------------------------

def q4k_meta_ld(K: int) -> int:
    """uint32 words per row of the super-block records (4 per 256 channels)."""
    return _load().oracle_q4k_meta_ld(K)


def q4k_quantize_superblock(w: np.ndarray):
    """256 FP32 weights -> (d bits, dmin bits, sc[8], m[8], q[256])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    assert w.shape == (256,)
    db, dmb = np.zeros(1, np.uint16), np.zeros(1, np.uint16)
    sc, m = np.zeros(8, np.int32), np.zeros(8, np.int32)
    q = np.zeros(256, np.uint8)
    _load().oracle_q4k_quantize_superblock(_ptr(w), _ptr(db), _ptr(dmb), _ptr(sc), _ptr(m), _ptr(q))
    return int(db[0]), int(dmb[0]), sc, m, q


def q4k_pack(w_f16: np.ndarray, nthreads: int = 0):
    """FP16 [N,K] -> (qweight u32 [N, K/8], meta u32 [N, K/256*4])."""
    w = _u16(w_f16)
    N, K = w.shape
    q = np.zeros((N, qweight_ld(K)), np.uint32)
    meta = np.zeros((N, max(q4k_meta_ld(K), 1)), np.uint32)
    rc = _load().oracle_q4k_pack(_ptr(w), N, K, _ptr(q), _ptr(meta), nthreads)
    if rc != 0:
        raise ValueError("oracle_q4k_pack: K must be a positive multiple of 256")
    return q, meta


def q4k_record(meta, K: int, n: int, sb: int):
    """(d, dmin, sc[8], m[8]) of super-block sb of row n, read back from its record."""
    meta = np.ascontiguousarray(meta, dtype=np.uint32)
    d, dmin = ctypes.c_float(), ctypes.c_float()
    sc, m = np.zeros(8, np.int32), np.zeros(8, np.int32)
    _load().oracle_q4k_record(_ptr(meta), K, n, sb, ctypes.byref(d), ctypes.byref(dmin), _ptr(sc), _ptr(m))
    return d.value, dmin.value, sc, m


def q4k_dequant(q, meta, N: int, K: int, nthreads: int = 0) -> np.ndarray:
    """W_hat [N,K] FP32 = d*sc_j*q - dmin*m_j."""
    q = np.ascontiguousarray(q, dtype=np.uint32)
    meta = np.ascontiguousarray(meta, dtype=np.uint32)
    out = np.zeros((N, K), np.float32)
    _load().oracle_q4k_dequant(_ptr(q), _ptr(meta), N, K, _ptr(out), nthreads)
    return out


def q4k_linear(x_bf16: np.ndarray, q, meta, N: int, K: int, nthreads: int = 0) -> np.ndarray:
    """y_ref [M,N] FP64 = x * W_hat^T, unrounded."""
    x = _u16(x_bf16)
    M = x.shape[0]
    assert x.shape[1] == K
    q = np.ascontiguousarray(q, dtype=np.uint32)
    meta = np.ascontiguousarray(meta, dtype=np.uint32)
    y = np.zeros((M, N), np.float64)
    _load().oracle_q4k_linear(_ptr(x), _ptr(q), _ptr(meta), M, N, K, _ptr(y), nthreads)
    return y


def q4k_linear_sampled(x_bf16: np.ndarray, q, meta, K: int, ms, ns, nthreads: int = 0) -> np.ndarray:
    """y_ref[ms[i], ns[i]] (FP64) for a list of outputs."""
    x = _u16(x_bf16)
    q = np.ascontiguousarray(q, dtype=np.uint32)
    meta = np.ascontiguousarray(meta, dtype=np.uint32)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.zeros(len(ms), np.float64)
    _load().oracle_q4k_linear_sampled(_ptr(x), _ptr(q), _ptr(meta), K, _ptr(ms), _ptr(ns), len(ms), _ptr(y),
                                      nthreads)
    return y


def max_threads() -> int:
    return _load().oracle_max_threads()
