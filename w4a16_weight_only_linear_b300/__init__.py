"""B300 (sm_103a) W4A16 weight-only linear layer -- Python binding.

A thin ctypes binding of ``libw4a16.so`` (declared in ``include/w4a16.h``).
Every function here only marshals arguments: checks dtypes, devices and
shapes of torch tensors, allocates outputs with torch when the caller does
not pass them, and forwards raw device pointers plus the current CUDA stream
to the C entry point of the same name.  All arithmetic runs in the library's
CUDA kernels; there is no fallback path.  Importing this module fails loudly
if the library has not been built (``python w4a16_weight_only_linear_b300/build.py``).

Packed format (see the header): qweight uint32 [N, K/8], scales FP16
[N, ldS], zeros uint32 [N, ldZ]; W_hat = (q - z) * s; y = x * W_hat^T.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libw4a16.so")

STATUS_NAMES = {
    0: "W4A16_OK", 1: "W4A16_ERR_INVALID_ARG", 2: "W4A16_ERR_UNSUPPORTED", 3: "W4A16_ERR_MISALIGNED",
    4: "W4A16_ERR_CUDA", 5: "W4A16_ERR_TIMEOUT", 6: "W4A16_ERR_NO_DEVICE",
}

# Entry points of the C ABI, with their ctypes signatures.
_vp, _i64, _i32, _u32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
EXPORTS = {
    "w4a16_status_string": ([_i32], ctypes.c_char_p),
    "w4a16_qweight_ld": ([_i64], _i64),
    "w4a16_scales_ld": ([_i64, _i32], _i64),
    "w4a16_zeros_ld": ([_i64, _i32], _i64),
    "w4a16_pack": ([_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp], _i32),
    "w4a16_dequant": ([_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_dequant_debug": ([_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_dequant_f16": ([_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_linear_f32": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _vp, _vp], _i32),
    "q4k_dequant": ([_vp, _vp, _i64, _i64, _vp, _vp], _i32),
    "w4a16_linear": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_linear_dual": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp], _i32),
    "w4a16_linear_multi": ([_vp, _i32, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_linear_gemv": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_linear_gemm": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_linear_gemm_noalloc": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_linear_act_scaled": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w8a16_qweight_ld": ([_i64], _i64),
    "w8a16_scales_ld": ([_i64, _i32], _i64),
    "w8a16_zeros_ld": ([_i64, _i32], _i64),
    "w8a16_pack": ([_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp], _i32),
    "w8a16_linear": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w8a16_linear_gemv": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w8a16_linear_gemm": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w8a16_dequant": ([_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp], _i32),
    "w8a16_dequant_f16": ([_vp, _vp, _vp, _i64, _i64, _i32, _vp, _vp], _i32),
    "w8a16_planes_qweight_ld": ([_i64], _i64),
    "w8a16_planes_scales_ld": ([_i64, _i32], _i64),
    "w8a16_planes_zeros_ld": ([_i64, _i32], _i64),
    "w8a16_planes_pack": ([_vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp], _i32),
    "w8a16_planes_linear": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp], _i32),
    "w4a16_linear_dual_act_scaled": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, _vp,
                                      _vp], _i32),
    "q4k_meta_ld": ([_i64], _i64),
    "q4k_pack": ([_vp, _i64, _i64, _vp, _vp, _vp], _i32),
    "q4k_linear": ([_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp], _i32),
    "q4k_linear_dual": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp], _i32),
    "w4a16_linear_path": ([_i64, _i64, _i64, _i32], _i32),
    "w4a16_device_status": ([_vp], _i32),
    "w4a16_debug_set_wait_limit": ([_i64], None),
    "w4a16_debug_withhold_copy": ([_i32], _i32),
    "w4a16_debug_gemv_plan": ([_i64, _i64, _i64, _i32, _i32, _vp], _i32),
}


class W4A16Error(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}")


def _load_library():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python w4a16_weight_only_linear_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in EXPORTS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load_library()


def _check(fn, status):
    if status != 0:
        raise W4A16Error(fn, status)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


# ---- layout helpers ------------------------------------------------------------

def w4a16_qweight_ld(K):
    return _lib.w4a16_qweight_ld(K)


def w4a16_scales_ld(K, G):
    return _lib.w4a16_scales_ld(K, G)


def w4a16_zeros_ld(K, G):
    return _lib.w4a16_zeros_ld(K, G)


def w4a16_status_string(status):
    return _lib.w4a16_status_string(status).decode()


def packed_shapes(N, K, G):
    """Shapes of (qweight, scales, zeros) for an [N,K] weight."""
    return (N, w4a16_qweight_ld(K)), (N, w4a16_scales_ld(K, G)), (N, w4a16_zeros_ld(K, G))


def empty_packed(N, K, G, device="cuda"):
    qs, ss, zs = packed_shapes(N, K, G)
    return (torch.empty(qs, dtype=torch.int32, device=device), torch.empty(ss, dtype=torch.float16, device=device),
            torch.empty(zs, dtype=torch.int32, device=device))


# ---- entry points -----------------------------------------------------------------

def w4a16_pack(w, G, out=None, stream=None):
    """FP16 W [N,K] (CUDA) -> (qweight int32 [N,K/8], scales fp16 [N,ldS], zeros int32 [N,ldZ]).

    The uint32 words travel as int32 tensors (torch has no uint32 arithmetic);
    the bits are identical."""
    N, K = w.shape
    q, s, z = out if out is not None else empty_packed(N, K, G, w.device)
    _check("w4a16_pack", _lib.w4a16_pack(_dev(w, torch.float16, "w"), N, K, G, _dev(q, torch.int32, "qweight"),
                                         _dev(s, torch.float16, "scales"), _dev(z, torch.int32, "zeros"),
                                         _stream(stream)))
    return q, s, z


def w4a16_dequant(q, s, z, N, K, G, out=None, stream=None):
    """W_hat FP32 [N,K] = (q - z) * s, through the decode kernel's own expansion
    routine (checking aid)."""
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=q.device)
    _check("w4a16_dequant", _lib.w4a16_dequant(_dev(q, torch.int32, "qweight"), _dev(s, torch.float16, "scales"),
                                               _dev(z, torch.int32, "zeros"), N, K, G,
                                               _dev(out, torch.float32, "out"), _stream(stream)))
    return out


def w4a16_dequant_f16(q, s, z, N, K, G, out=None, stream=None):
    """RN_fp16(W_hat) FP16 [N,K], through the tensor-core kernel's own expansion
    routine (the operand it writes into tensor memory; checking aid)."""
    if out is None:
        out = torch.empty((N, K), dtype=torch.float16, device=q.device)
    _check("w4a16_dequant_f16", _lib.w4a16_dequant_f16(
        _dev(q, torch.int32, "qweight"), _dev(s, torch.float16, "scales"), _dev(z, torch.int32, "zeros"), N, K, G,
        _dev(out, torch.float16, "out"), _stream(stream)))
    return out


def w4a16_linear_f32(x, q, s, z, G, path=0, out=None, stream=None):
    """y FP32 [M,N] = x * W_hat^T without the BF16 output rounding.  path: 0 =
    the kernel w4a16_linear would choose, 1 = decode kernel, 2 = tensor-core kernel."""
    M, K = x.shape
    N = q.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check("w4a16_linear_f32", _lib.w4a16_linear_f32(
        _dev(x, torch.bfloat16, "x"), _dev(q, torch.int32, "qweight"), _dev(s, torch.float16, "scales"),
        _dev(z, torch.int32, "zeros"), M, N, K, G, path, _dev(out, torch.float32, "y"), _stream(stream)))
    return out


def _linear(fn, x, q, s, z, N, G, out, stream):
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(fn, getattr(_lib, fn)(_dev(x, torch.bfloat16, "x"), _dev(q, torch.int32, "qweight"),
                                 _dev(s, torch.float16, "scales"), _dev(z, torch.int32, "zeros"), M, N, K, G,
                                 _dev(out, torch.bfloat16, "y"), _stream(stream)))
    return out


def w4a16_linear(x, q, s, z, G, out=None, stream=None):
    """y BF16 [M,N] = x BF16 [M,K] * W_hat^T (N taken from qweight's rows)."""
    return _linear("w4a16_linear", x, q, s, z, q.shape[0], G, out, stream)


def w4a16_linear_gemv(x, q, s, z, G, out=None, stream=None):
    """Decode kernel only (M <= 16)."""
    return _linear("w4a16_linear_gemv", x, q, s, z, q.shape[0], G, out, stream)


def w4a16_linear_gemm(x, q, s, z, G, out=None, stream=None):
    """Tensor-core kernel only (any M)."""
    return _linear("w4a16_linear_gemm", x, q, s, z, q.shape[0], G, out, stream)


def w4a16_linear_gemm_noalloc(x, q, s, z, G, out=None, stream=None):
    """Tensor-core kernel only, with its FP16 copy of x in the library's fixed
    device array instead of an allocation (M * K <= NOALLOC_MAX_X_ELEMS).  The
    C call allocates nothing; pass `out` to keep this wrapper from allocating
    y with torch."""
    return _linear("w4a16_linear_gemm_noalloc", x, q, s, z, q.shape[0], G, out, stream)


NOALLOC_MAX_X_ELEMS = 8 * 1024 * 1024


def w4a16_linear_dual(x, gate, up, G, out=None, stream=None):
    """(y_gate, y_up) = (x * W_hat_gate^T, x * W_hat_up^T); gate/up = (qweight, scales, zeros)."""
    M, K = x.shape
    N = gate[0].shape[0]
    if out is None:
        out = (torch.empty((M, N), dtype=torch.bfloat16, device=x.device),
               torch.empty((M, N), dtype=torch.bfloat16, device=x.device))
    yg, yu = out
    _check("w4a16_linear_dual", _lib.w4a16_linear_dual(
        _dev(x, torch.bfloat16, "x"),
        _dev(gate[0], torch.int32, "qweight_gate"), _dev(gate[1], torch.float16, "scales_gate"),
        _dev(gate[2], torch.int32, "zeros_gate"),
        _dev(up[0], torch.int32, "qweight_up"), _dev(up[1], torch.float16, "scales_up"),
        _dev(up[2], torch.int32, "zeros_up"),
        M, N, K, G, _dev(yg, torch.bfloat16, "y_gate"), _dev(yu, torch.bfloat16, "y_up"), _stream(stream)))
    return yg, yu


def w4a16_linear_multi(x, mats, G, out=None, stream=None):
    """[x * W_hat_i^T for each (qweight, scales, zeros) in mats] (1..4 matrices
    sharing x, each with its own output size), in one decode launch at M <= 8
    (and M <= 16 where that launch runs with all its warps)."""
    M, K = x.shape
    n = len(mats)
    if not 1 <= n <= 4:
        raise ValueError("w4a16_linear_multi takes 1 to 4 matrices")
    Ns = [m[0].shape[0] for m in mats]
    if out is None:
        out = [torch.empty((M, Ni), dtype=torch.bfloat16, device=x.device) for Ni in Ns]
    arr = ctypes.c_void_p * n
    qs = arr(*[_dev(m[0], torch.int32, "qweight") for m in mats])
    ss = arr(*[_dev(m[1], torch.float16, "scales") for m in mats])
    zs = arr(*[_dev(m[2], torch.int32, "zeros") for m in mats])
    ys = arr(*[_dev(o, torch.bfloat16, "y") for o in out])
    ns = (ctypes.c_int64 * n)(*Ns)
    _check("w4a16_linear_multi", _lib.w4a16_linear_multi(_dev(x, torch.bfloat16, "x"), n, qs, ss, zs, ns, M, K, G,
                                                         ys, _stream(stream)))
    return out


def w4a16_linear_act_scaled(x, x_scale, q, s, z, G, out=None, stream=None):
    """y BF16 [M,N] = (x * x_scale) * W_hat^T: x_scale FP32 [K] multiplies each
    input channel of x before it is rounded to FP16 (the deployed form of
    activation-aware quantisation, with W packed from W * diag(1 / x_scale))."""
    M, K = x.shape
    N = q.shape[0]
    if x_scale.shape != (K,):
        raise ValueError(f"x_scale must have shape ({K},), got {tuple(x_scale.shape)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check("w4a16_linear_act_scaled", _lib.w4a16_linear_act_scaled(
        _dev(x, torch.bfloat16, "x"), _dev(x_scale, torch.float32, "x_scale"), _dev(q, torch.int32, "qweight"),
        _dev(s, torch.float16, "scales"), _dev(z, torch.int32, "zeros"), M, N, K, G,
        _dev(out, torch.bfloat16, "y"), _stream(stream)))
    return out


def w4a16_linear_dual_act_scaled(x, x_scale, gate, up, G, out=None, stream=None):
    """w4a16_linear_dual with the activation scale x_scale FP32 [K] applied to the shared x."""
    M, K = x.shape
    N = gate[0].shape[0]
    if x_scale.shape != (K,):
        raise ValueError(f"x_scale must have shape ({K},), got {tuple(x_scale.shape)}")
    if out is None:
        out = (torch.empty((M, N), dtype=torch.bfloat16, device=x.device),
               torch.empty((M, N), dtype=torch.bfloat16, device=x.device))
    yg, yu = out
    _check("w4a16_linear_dual_act_scaled", _lib.w4a16_linear_dual_act_scaled(
        _dev(x, torch.bfloat16, "x"), _dev(x_scale, torch.float32, "x_scale"),
        _dev(gate[0], torch.int32, "qweight_gate"), _dev(gate[1], torch.float16, "scales_gate"),
        _dev(gate[2], torch.int32, "zeros_gate"),
        _dev(up[0], torch.int32, "qweight_up"), _dev(up[1], torch.float16, "scales_up"),
        _dev(up[2], torch.int32, "zeros_up"),
        M, N, K, G, _dev(yg, torch.bfloat16, "y_gate"), _dev(yu, torch.bfloat16, "y_up"), _stream(stream)))
    return yg, yu


# ---- the 8-bit variant ---------------------------------------------------------

def w8a16_packed_shapes(N, K, G):
    """Shapes of (qweight int32, scales FP16, zeros int32) of the 8-bit word layout."""
    return (N, _lib.w8a16_qweight_ld(K)), (N, _lib.w8a16_scales_ld(K, G)), (N, _lib.w8a16_zeros_ld(K, G))


def w8a16_pack(w, G, out=None, stream=None):
    """FP16 W [N,K] -> (qweight, scales, zeros) of the 8-bit word layout (four codes
    per word, one FP16 scale and one 8-bit zero point per group)."""
    N, K = w.shape
    if out is None:
        sq, ss, sz = w8a16_packed_shapes(N, K, G)
        out = (torch.empty(sq, dtype=torch.int32, device=w.device), torch.empty(ss, dtype=torch.float16, device=w.device),
               torch.empty(sz, dtype=torch.int32, device=w.device))
    q, s, z = out
    _check("w8a16_pack", _lib.w8a16_pack(_dev(w, torch.float16, "w"), N, K, G, _dev(q, torch.int32, "qweight"),
                                         _dev(s, torch.float16, "scales"), _dev(z, torch.int32, "zeros"),
                                         _stream(stream)))
    return q, s, z


def w8a16_linear(x, q, s, z, G, out=None, stream=None):
    """y BF16 [M,N] = x BF16 [M,K] * W_hat8^T, 8-bit word layout."""
    return _linear("w8a16_linear", x, q, s, z, q.shape[0], G, out, stream)


def w8a16_linear_gemv(x, q, s, z, G, out=None, stream=None):
    """8-bit word layout, decode kernel only (M <= 8, G <= 128)."""
    return _linear("w8a16_linear_gemv", x, q, s, z, q.shape[0], G, out, stream)


def w8a16_linear_gemm(x, q, s, z, G, out=None, stream=None):
    """8-bit word layout, tensor-core kernel only (any M)."""
    return _linear("w8a16_linear_gemm", x, q, s, z, q.shape[0], G, out, stream)


def w8a16_dequant(q, s, z, N, K, G, out=None, stream=None):
    """W_hat FP32 [N,K] of the 8-bit word layout through the decode kernel's own
    8-bit expansion (checking aid)."""
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=q.device)
    _check("w8a16_dequant", _lib.w8a16_dequant(_dev(q, torch.int32, "qweight"), _dev(s, torch.float16, "scales"),
                                               _dev(z, torch.int32, "zeros"), N, K, G, _dev(out, torch.float32, "out"),
                                               _stream(stream)))
    return out


def w8a16_dequant_f16(q, s, z, N, K, G, out=None, stream=None):
    """RN_fp16(W_hat) FP16 [N,K] of the 8-bit word layout through the tensor-core
    kernel's own 8-bit expansion (checking aid)."""
    if out is None:
        out = torch.empty((N, K), dtype=torch.float16, device=q.device)
    _check("w8a16_dequant_f16", _lib.w8a16_dequant_f16(
        _dev(q, torch.int32, "qweight"), _dev(s, torch.float16, "scales"), _dev(z, torch.int32, "zeros"), N, K, G,
        _dev(out, torch.float16, "out"), _stream(stream)))
    return out


def w8a16_planes_packed_shapes(N, K, G):
    """Shapes of (qweight int32, scales FP16, zeros int32) of an 8-bit layer."""
    return (N, _lib.w8a16_planes_qweight_ld(K)), (N, _lib.w8a16_planes_scales_ld(K, G)), (N, _lib.w8a16_planes_zeros_ld(K, G))


def w8a16_planes_pack(w, G, out=None, stream=None):
    """FP16 W [N,K] -> (qweight, scales, zeros) of the 8-bit layer (codes as two
    4-bit planes; see the header)."""
    N, K = w.shape
    if out is None:
        sq, ss, sz = w8a16_planes_packed_shapes(N, K, G)
        out = (torch.empty(sq, dtype=torch.int32, device=w.device), torch.empty(ss, dtype=torch.float16, device=w.device),
               torch.empty(sz, dtype=torch.int32, device=w.device))
    q, s, z = out
    _check("w8a16_planes_pack", _lib.w8a16_planes_pack(_dev(w, torch.float16, "w"), N, K, G, _dev(q, torch.int32, "qweight"),
                                         _dev(s, torch.float16, "scales"), _dev(z, torch.int32, "zeros"),
                                         _stream(stream)))
    return q, s, z


def w8a16_planes_linear(x, q, s, z, G, out=None, stream=None):
    """y BF16 [M,N] = x BF16 [M,K] * W_hat8^T."""
    return _linear("w8a16_planes_linear", x, q, s, z, q.shape[0], G, out, stream)


def q4k_packed_shapes(N, K):
    """Shapes of (qweight int32, meta int32) of a super-block (Q4_K-style) layer."""
    return (N, _lib.w4a16_qweight_ld(K)), (N, _lib.q4k_meta_ld(K))


def q4k_pack(w, out=None, stream=None):
    """FP16 W [N,K] (K a multiple of 256) -> (qweight, meta) of the super-block layout."""
    N, K = w.shape
    if out is None:
        sq, sm = q4k_packed_shapes(N, K)
        out = (torch.empty(sq, dtype=torch.int32, device=w.device), torch.empty(sm, dtype=torch.int32, device=w.device))
    q, meta = out
    _check("q4k_pack", _lib.q4k_pack(_dev(w, torch.float16, "w"), N, K, _dev(q, torch.int32, "qweight"),
                                     _dev(meta, torch.int32, "meta"), _stream(stream)))
    return q, meta


def q4k_dequant(q, meta, N, K, out=None, stream=None):
    """W_hat FP32 [N,K] of the super-block layout, through the decode kernel's own
    code expansion and record decoding (checking aid)."""
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=q.device)
    _check("q4k_dequant", _lib.q4k_dequant(_dev(q, torch.int32, "qweight"), _dev(meta, torch.int32, "meta"), N, K,
                                           _dev(out, torch.float32, "out"), _stream(stream)))
    return out


def q4k_linear(x, q, meta, out=None, stream=None):
    """y BF16 [M,N] = x BF16 [M,K] * W_hat^T for the super-block layout (N from qweight's rows)."""
    M, K = x.shape
    N = q.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check("q4k_linear", _lib.q4k_linear(_dev(x, torch.bfloat16, "x"), _dev(q, torch.int32, "qweight"),
                                         _dev(meta, torch.int32, "meta"), M, N, K, _dev(out, torch.bfloat16, "y"),
                                         _stream(stream)))
    return out


def q4k_linear_dual(x, gate, up, out=None, stream=None):
    """(y_gate, y_up) for two super-block matrices sharing x; gate/up = (qweight, meta)."""
    M, K = x.shape
    N = gate[0].shape[0]
    if out is None:
        out = (torch.empty((M, N), dtype=torch.bfloat16, device=x.device),
               torch.empty((M, N), dtype=torch.bfloat16, device=x.device))
    yg, yu = out
    _check("q4k_linear_dual", _lib.q4k_linear_dual(
        _dev(x, torch.bfloat16, "x"), _dev(gate[0], torch.int32, "qweight_gate"), _dev(gate[1], torch.int32, "meta_gate"),
        _dev(up[0], torch.int32, "qweight_up"), _dev(up[1], torch.int32, "meta_up"), M, N, K,
        _dev(yg, torch.bfloat16, "y_gate"), _dev(yu, torch.bfloat16, "y_up"), _stream(stream)))
    return yg, yu


def w4a16_linear_path(M, N, K, G):
    """1 = decode GEMV, 2 = tensor-core GEMM, 0 = rejected."""
    return _lib.w4a16_linear_path(M, N, K, G)


def w4a16_device_status():
    """Synchronise; raise if a kernel's bounded wait gave up since the last call."""
    word = ctypes.c_uint32(0)
    _check("w4a16_device_status", _lib.w4a16_device_status(ctypes.byref(word)))
    return word.value


def device_status_word():
    """Synchronise; (status, raw word) of w4a16_device_status without raising:
    W4A16_ERR_TIMEOUT (5) with the give-up bits, or 0."""
    word = ctypes.c_uint32(0)
    st = _lib.w4a16_device_status(ctypes.byref(word))
    return st, word.value
