// capi.cu -- the extern "C" boundary declared in include/w4a16.h.
//
// Every entry point validates its arguments on the host and returns a status
// before anything is launched; kernels are enqueued on the caller's stream.
// The runtime chooses a kernel by problem shape, the way a backend picks a
// direct kernel for a packed format (zhuai.tech "Quantization Is Not a Zip
// File", section 1: the backend selects a kernel by format and device).
#include <cuda_runtime.h>

#include "../../include/w4a16.h"
#include "common.cuh"
#include "kernels.h"

namespace {

using w4a16::GemvMat;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool group_ok(int G) { return G == 32 || G == 64 || G == 128 || G == 256; }

// Largest element count an index may reach (kernels use 64-bit row offsets,
// 32-bit group and step counters).
constexpr int64_t kMaxDim = int64_t(1) << 30;

w4a16_status check_weight_shape(int64_t N, int64_t K, int G) {
    if (!group_ok(G)) return W4A16_ERR_UNSUPPORTED;
    if (N < 0 || K <= 0 || N > kMaxDim || K > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (K % G != 0 || N % 8 != 0) return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

w4a16_status check_weights(const uint32_t* q, const void* s, const uint32_t* z) {
    if (!q || !s || !z) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(s) || !aligned16(z)) return W4A16_ERR_MISALIGNED;
    return W4A16_OK;
}

w4a16_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return W4A16_OK;
    if (e == cudaErrorNotSupported) return W4A16_ERR_UNSUPPORTED;
    return W4A16_ERR_CUDA;
}

// Path for a shape whose arguments are valid: 1 = GEMV, 2 = GEMM.
// Automatic dispatch: the decode GEMV up to 8 activation rows wherever it fits, and up to 16
// where it runs with all its warps (two MMA column blocks per tile; x of long rows split
// along K over a two-CTA cluster) and also takes M = 8, so that a shape leaves the GEMV at
// one batch size for good.  Measured on one B300 at M = 9-16: 5120 -> 13824 (G = 128)
// 20.1-24.9 us against the tensor-core call's 29.1-32 us, 5120 -> 5120 at M = 16 17.5
// against 21-26 us.  Where x crowds out the GEMV's weight rings it loses (43.8 against 35 us at
// M = 16 before the K split), hence the full-warp condition.
constexpr int64_t kGemvDispatchMaxM = 16;
constexpr int64_t kGemvAnyFitMaxM = 8;

bool gemv_dispatch(int64_t M, const int64_t* Ns, int nmat, int64_t K, int G) {
    if (M <= kGemvAnyFitMaxM) return w4a16::gemv_fits(M, Ns, nmat, K, G);
    return M <= kGemvDispatchMaxM && w4a16::gemv_fits(kGemvAnyFitMaxM, Ns, nmat, K, G) &&
           w4a16::gemv_runs_full(M, Ns, nmat, K, G);
}

int choose_path(int64_t M, int64_t N, int64_t K, int G, int nmat) {
    int64_t Ns[w4a16::kMaxMat];
    for (int i = 0; i < w4a16::kMaxMat; ++i) Ns[i] = N;
    return gemv_dispatch(M, Ns, nmat, K, G) ? 1 : 2;
}

w4a16_status linear_common(const void* x, const uint32_t* q, const void* s, const uint32_t* z, int64_t M,
                           int64_t N, int64_t K, int G, void* y, w4a16_stream_t stream, int force,
                           const float* xsc = nullptr, int64_t kx = 0) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (M < 0 || M > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A16_OK;
    if ((st = check_weights(q, s, z)) != W4A16_OK) return st;
    if (!x || !y) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return W4A16_ERR_MISALIGNED;
    int path = force ? force : choose_path(M, N, K, G, 1);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    GemvMat mat{q, s, z, y};
    if (path == 1) {
        if (M > 16 || !w4a16::gemv_fits(M, N, K, G, 1)) return W4A16_ERR_UNSUPPORTED;
        return from_cuda(w4a16::launch_gemv(x, &mat, 1, M, N, K, G, cs, xsc, kx));
    }
    return from_cuda(w4a16::launch_gemm(x, &mat, 1, M, N, K, G, cs, xsc, kx));
}

w4a16_status dual_common(const void* x_bf16, const uint32_t* qweight_gate, const void* scales_gate,
                         const uint32_t* zeros_gate, const uint32_t* qweight_up, const void* scales_up,
                         const uint32_t* zeros_up, int64_t M, int64_t N, int64_t K, int G, void* y_gate_bf16,
                         void* y_up_bf16, w4a16_stream_t stream, const float* xsc) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (M < 0 || M > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A16_OK;
    if ((st = check_weights(qweight_gate, scales_gate, zeros_gate)) != W4A16_OK) return st;
    if ((st = check_weights(qweight_up, scales_up, zeros_up)) != W4A16_OK) return st;
    if (!x_bf16 || !y_gate_bf16 || !y_up_bf16) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(y_gate_bf16) || !aligned16(y_up_bf16)) return W4A16_ERR_MISALIGNED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const GemvMat mats[2] = {{qweight_gate, scales_gate, zeros_gate, y_gate_bf16},
                             {qweight_up, scales_up, zeros_up, y_up_bf16}};
    if (choose_path(M, N, K, G, 2) == 1)
        return from_cuda(w4a16::launch_gemv(x_bf16, mats, 2, M, N, K, G, cs, xsc));
    return from_cuda(w4a16::launch_gemm(x_bf16, mats, 2, M, N, K, G, cs, xsc));
}

// Up to four matrices of their own output sizes sharing x (w4a16_linear_multi).
w4a16_status multi_common(const void* x, int nmat, const uint32_t* const* q, const void* const* s,
                          const uint32_t* const* z, const int64_t* Ns, int64_t M, int64_t K, int G, void* const* y,
                          w4a16_stream_t stream) {
    if (nmat < 1 || nmat > w4a16::kMaxMat || !q || !s || !z || !Ns || !y) return W4A16_ERR_INVALID_ARG;
    w4a16_status st;
    for (int i = 0; i < nmat; ++i)
        if ((st = check_weight_shape(Ns[i], K, G)) != W4A16_OK) return st;
    if (M < 0 || M > kMaxDim) return W4A16_ERR_INVALID_ARG;
    GemvMat mats[w4a16::kMaxMat];
    int64_t Nl[w4a16::kMaxMat];
    int n = 0;
    for (int i = 0; i < nmat; ++i) {
        if (Ns[i] == 0) continue;                     // an empty matrix: nothing to compute
        if ((st = check_weights(q[i], s[i], z[i])) != W4A16_OK) return st;
        if (!y[i]) return W4A16_ERR_INVALID_ARG;
        if (!aligned16(y[i])) return W4A16_ERR_MISALIGNED;
        mats[n] = GemvMat{q[i], s[i], z[i], y[i], Ns[i]};
        Nl[n++] = Ns[i];
    }
    if (M == 0 || n == 0) return W4A16_OK;
    if (!x) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x)) return W4A16_ERR_MISALIGNED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (gemv_dispatch(M, Nl, n, K, G)) return from_cuda(w4a16::launch_gemv(x, mats, n, M, 0, K, G, cs));
    return from_cuda(w4a16::launch_gemm(x, mats, n, M, 0, K, G, cs));
}

// The activation-scale vector of the *_act_scaled entry points: present and 16-byte aligned.
w4a16_status check_act_scale(const float* x_scale) {
    if (!x_scale) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x_scale)) return W4A16_ERR_MISALIGNED;
    return W4A16_OK;
}

// The super-block layout: K a positive multiple of 256, N a multiple of 8.
w4a16_status check_q4k_shape(int64_t N, int64_t K) {
    if (N < 0 || K <= 0 || N > kMaxDim || K > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (K % 256 != 0 || N % 8 != 0) return W4A16_ERR_INVALID_ARG;
    return W4A16_OK;
}

w4a16_status check_q4k_weights(const uint32_t* q, const uint32_t* meta) {
    if (!q || !meta) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(meta)) return W4A16_ERR_MISALIGNED;
    return W4A16_OK;
}

// The super-block layer for nmat matrices sharing x: the decode kernel over row blocks of
// up to 8 activation rows (as many as its shared memory holds at this K).
w4a16_status q4k_common(const void* x, const uint32_t* const* q, const uint32_t* const* meta, void* const* y,
                        int nmat, int64_t M, int64_t N, int64_t K, w4a16_stream_t stream) {
    w4a16_status st = check_q4k_shape(N, K);
    if (st != W4A16_OK) return st;
    if (M < 0 || M > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A16_OK;
    for (int i = 0; i < nmat; ++i) {
        if ((st = check_q4k_weights(q[i], meta[i])) != W4A16_OK) return st;
        if (!y[i]) return W4A16_ERR_INVALID_ARG;
        if (!aligned16(y[i])) return W4A16_ERR_MISALIGNED;
    }
    if (!x) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x)) return W4A16_ERR_MISALIGNED;
    int64_t mb = M < 8 ? M : 8;
    while (mb >= 1 && !w4a16::gemv_fits(mb, N, K, 32, nmat, true)) --mb;
    if (mb < 1 && nmat == 2) {
        // a pair holds twice the rows per CTA; where their records do not fit, one launch per matrix
        for (int i = 0; i < 2; ++i)
            if ((st = q4k_common(x, q + i, meta + i, y + i, 1, M, N, K, stream)) != W4A16_OK) return st;
        return W4A16_OK;
    }
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const auto* xb = static_cast<const uint16_t*>(x);
    if (mb < 1) {
        // too many weight rows per CTA for their records: cut the rows into the largest slices
        // (multiples of 8) that fit and run one activation row per launch, since a slice of
        // y's row m is contiguous
        int64_t nc = N;
        while (nc > 8 && !w4a16::gemv_fits(1, nc, K, 32, 1, true)) nc = (nc / 2 + 7) / 8 * 8;
        if (!w4a16::gemv_fits(1, nc, K, 32, 1, true)) return W4A16_ERR_UNSUPPORTED;
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n0 = 0; n0 < N; n0 += nc) {
                const int64_t nr = N - n0 < nc ? N - n0 : nc;
                const GemvMat mat{q[0] + n0 * (K / 8), meta[0] + n0 * (K / 256 * 4), nullptr,
                                  static_cast<uint16_t*>(y[0]) + m * N + n0};
                const cudaError_t e = w4a16::launch_gemv(xb + m * K, &mat, 1, 1, nr, K, 32, cs, nullptr, 0, true);
                if (e != cudaSuccess) return from_cuda(e);
            }
        return W4A16_OK;
    }
    for (int64_t m0 = 0; m0 < M; m0 += mb) {
        const int64_t mr = M - m0 < mb ? M - m0 : mb;
        GemvMat mats[2];
        for (int i = 0; i < nmat; ++i) mats[i] = {q[i], meta[i], nullptr, static_cast<uint16_t*>(y[i]) + m0 * N};
        const cudaError_t e = w4a16::launch_gemv(xb + m0 * K, mats, nmat, mr, N, K, 32, cs, nullptr, 0, true);
        if (e != cudaSuccess) return from_cuda(e);
    }
    return W4A16_OK;
}

}  // namespace

extern "C" {

const char* w4a16_status_string(w4a16_status status) {
    switch (status) {
        case W4A16_OK: return "W4A16_OK";
        case W4A16_ERR_INVALID_ARG: return "W4A16_ERR_INVALID_ARG";
        case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED";
        case W4A16_ERR_MISALIGNED: return "W4A16_ERR_MISALIGNED";
        case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA";
        case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT";
        case W4A16_ERR_NO_DEVICE: return "W4A16_ERR_NO_DEVICE";
    }
    return "W4A16_ERR_UNKNOWN";
}

int64_t w4a16_qweight_ld(int64_t K) { return w4a16::qweight_ld(K); }
int64_t w4a16_scales_ld(int64_t K, int G) { return G > 0 ? w4a16::scales_ld(K, G) : 0; }
int64_t w4a16_zeros_ld(int64_t K, int G) { return G > 0 ? w4a16::zeros_ld(K, G) : 0; }

int64_t w8a16_qweight_ld(int64_t K) { return K / 4; }
int64_t w8a16_scales_ld(int64_t K, int G) { return G > 0 ? w4a16::scales_ld(K, G) : 0; }
int64_t w8a16_zeros_ld(int64_t K, int G) { return G > 0 ? w4a16::zeros8_ld(K, G) : 0; }

w4a16_status w8a16_pack(const void* w_f16, int64_t N, int64_t K, int G, uint32_t* qweight, void* scales_f16,
                        uint32_t* zeros, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!w_f16) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_f16)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_pack8w(w_f16, N, K, G, qweight, scales_f16, zeros,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w8a16_dequant(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros, int64_t N,
                           int64_t K, int G, float* w_out, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!w_out) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_out)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_dequant8w(qweight, scales_f16, zeros, N, K, G, w_out,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w8a16_dequant_f16(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros, int64_t N,
                               int64_t K, int G, void* w_out_f16, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!w_out_f16) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_out_f16)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_dequant8w_f16(qweight, scales_f16, zeros, N, K, G, w_out_f16,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

// path: 0 = automatic (the decode kernel for M <= 8 and G <= 128 where it fits, else the
// tensor-core kernel), 1 = decode kernel, 2 = tensor-core kernel.
static w4a16_status w8_common(const void* x, const uint32_t* q, const void* s, const uint32_t* z, int64_t M,
                              int64_t N, int64_t K, int G, void* y, w4a16_stream_t stream, int path) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (M < 0 || M > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A16_OK;
    if ((st = check_weights(q, s, z)) != W4A16_OK) return st;
    if (!x || !y) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return W4A16_ERR_MISALIGNED;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    GemvMat mat{q, s, z, y};
    const int64_t Ns[1] = {N};
    const bool gemv_ok = M <= 8 && G <= 128 && w4a16::gemv_fits(M, Ns, 1, K, G, false, true);
    if (path == 0) path = M <= kGemvDispatchMaxM && gemv_ok ? 1 : 2;
    if (path == 1) {
        if (!gemv_ok) return W4A16_ERR_UNSUPPORTED;
        return from_cuda(w4a16::launch_gemv(x, &mat, 1, M, N, K, G, cs, nullptr, 0, false, false, true));
    }
    return from_cuda(w4a16::launch_gemm(x, &mat, 1, M, N, K, G, cs, nullptr, 0, false, true));
}

w4a16_status w8a16_linear(const void* x_bf16, const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros,
                          int64_t M, int64_t N, int64_t K, int G, void* y_bf16, w4a16_stream_t stream) {
    return w8_common(x_bf16, qweight, scales_f16, zeros, M, N, K, G, y_bf16, stream, 0);
}

w4a16_status w8a16_linear_gemv(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                               const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G, void* y_bf16,
                               w4a16_stream_t stream) {
    return w8_common(x_bf16, qweight, scales_f16, zeros, M, N, K, G, y_bf16, stream, 1);
}

w4a16_status w8a16_linear_gemm(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                               const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G, void* y_bf16,
                               w4a16_stream_t stream) {
    return w8_common(x_bf16, qweight, scales_f16, zeros, M, N, K, G, y_bf16, stream, 2);
}

int64_t w8a16_planes_qweight_ld(int64_t K) { return w4a16::qweight_ld(2 * K); }
int64_t w8a16_planes_scales_ld(int64_t K, int G) { return G > 0 ? w4a16::scales_ld(2 * K, G) : 0; }
int64_t w8a16_planes_zeros_ld(int64_t K, int G) { return G > 0 ? w4a16::zeros_ld(2 * K, G) : 0; }

w4a16_status w8a16_planes_pack(const void* w_f16, int64_t N, int64_t K, int G, uint32_t* qweight, void* scales_f16,
                        uint32_t* zeros, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (2 * K > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!w_f16) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_f16)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_pack8(w_f16, N, K, G, qweight, scales_f16, zeros,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w8a16_planes_linear(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                          const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G, void* y_bf16,
                          w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (2 * K > kMaxDim) return W4A16_ERR_INVALID_ARG;
    // the two planes are a 4-bit layer of 2K input channels over x repeated twice
    return linear_common(x_bf16, qweight, scales_f16, zeros, M, N, 2 * K, G, y_bf16, stream, 0, nullptr, K);
}

w4a16_status w4a16_pack(const void* w_f16, int64_t N, int64_t K, int G, uint32_t* qweight, void* scales_f16,
                        uint32_t* zeros, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!w_f16) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_f16)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_pack(w_f16, N, K, G, qweight, scales_f16, zeros,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_dequant(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros, int64_t N,
                           int64_t K, int G, float* w_out, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!w_out) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_out)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_dequant(qweight, scales_f16, zeros, N, K, G, w_out,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_dequant_debug(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros,
                                 int64_t N, int64_t K, int G, float* w_out, w4a16_stream_t stream) {
    return w4a16_dequant(qweight, scales_f16, zeros, N, K, G, w_out, stream);
}

w4a16_status w4a16_dequant_f16(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros, int64_t N,
                               int64_t K, int G, void* w_out_f16, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!w_out_f16) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_out_f16)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_dequant_f16(qweight, scales_f16, zeros, N, K, G, w_out_f16,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_linear_f32(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                              const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G, int path, float* y_f32,
                              w4a16_stream_t stream) {
    if (path < 0 || path > 2) return W4A16_ERR_INVALID_ARG;
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (M < 0 || M > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!x_bf16 || !y_f32) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(y_f32)) return W4A16_ERR_MISALIGNED;
    if (path == 0) path = choose_path(M, N, K, G, 1);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    GemvMat mat{qweight, scales_f16, zeros, y_f32};
    if (path == 1) {
        if (M > 16 || !w4a16::gemv_fits(M, N, K, G, 1)) return W4A16_ERR_UNSUPPORTED;
        return from_cuda(w4a16::launch_gemv(x_bf16, &mat, 1, M, N, K, G, cs, nullptr, 0, false, true));
    }
    return from_cuda(w4a16::launch_gemm(x_bf16, &mat, 1, M, N, K, G, cs, nullptr, 0, true));
}

w4a16_status w4a16_linear(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                          const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G, void* y_bf16,
                          w4a16_stream_t stream) {
    return linear_common(x_bf16, qweight, scales_f16, zeros, M, N, K, G, y_bf16, stream, 0);
}

w4a16_status w4a16_linear_gemv(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                               const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G, void* y_bf16,
                               w4a16_stream_t stream) {
    return linear_common(x_bf16, qweight, scales_f16, zeros, M, N, K, G, y_bf16, stream, 1);
}

w4a16_status w4a16_linear_gemm(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                               const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G, void* y_bf16,
                               w4a16_stream_t stream) {
    return linear_common(x_bf16, qweight, scales_f16, zeros, M, N, K, G, y_bf16, stream, 2);
}

w4a16_status w4a16_linear_dual(const void* x_bf16, const uint32_t* qweight_gate, const void* scales_gate,
                               const uint32_t* zeros_gate, const uint32_t* qweight_up, const void* scales_up,
                               const uint32_t* zeros_up, int64_t M, int64_t N, int64_t K, int G,
                               void* y_gate_bf16, void* y_up_bf16, w4a16_stream_t stream) {
    return dual_common(x_bf16, qweight_gate, scales_gate, zeros_gate, qweight_up, scales_up, zeros_up, M, N, K, G,
                       y_gate_bf16, y_up_bf16, stream, nullptr);
}

w4a16_status w4a16_linear_multi(const void* x_bf16, int nmat, const uint32_t* const* qweight,
                                const void* const* scales_f16, const uint32_t* const* zeros, const int64_t* N,
                                int64_t M, int64_t K, int G, void* const* y_bf16, w4a16_stream_t stream) {
    return multi_common(x_bf16, nmat, qweight, scales_f16, zeros, N, M, K, G, y_bf16, stream);
}

w4a16_status w4a16_linear_act_scaled(const void* x_bf16, const float* x_scale, const uint32_t* qweight,
                                     const void* scales_f16, const uint32_t* zeros, int64_t M, int64_t N, int64_t K,
                                     int G, void* y_bf16, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if ((st = check_act_scale(x_scale)) != W4A16_OK) return st;
    return linear_common(x_bf16, qweight, scales_f16, zeros, M, N, K, G, y_bf16, stream, 0, x_scale);
}

w4a16_status w4a16_linear_dual_act_scaled(const void* x_bf16, const float* x_scale, const uint32_t* qweight_gate,
                                          const void* scales_gate, const uint32_t* zeros_gate,
                                          const uint32_t* qweight_up, const void* scales_up,
                                          const uint32_t* zeros_up, int64_t M, int64_t N, int64_t K, int G,
                                          void* y_gate_bf16, void* y_up_bf16, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if ((st = check_act_scale(x_scale)) != W4A16_OK) return st;
    return dual_common(x_bf16, qweight_gate, scales_gate, zeros_gate, qweight_up, scales_up, zeros_up, M, N, K, G,
                       y_gate_bf16, y_up_bf16, stream, x_scale);
}

w4a16_status w4a16_linear_gemm_noalloc(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                                       const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G,
                                       void* y_bf16, w4a16_stream_t stream) {
    w4a16_status st = check_weight_shape(N, K, G);
    if (st != W4A16_OK) return st;
    if (M < 0 || M > kMaxDim) return W4A16_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4A16_OK;
    if ((st = check_weights(qweight, scales_f16, zeros)) != W4A16_OK) return st;
    if (!x_bf16 || !y_bf16) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(y_bf16)) return W4A16_ERR_MISALIGNED;
    if (M * K > (int64_t)W4A16_NOALLOC_MAX_X_ELEMS) return W4A16_ERR_UNSUPPORTED;
    const GemvMat mat{qweight, scales_f16, zeros, y_bf16};
    return from_cuda(w4a16::launch_gemm_noalloc(x_bf16, mat, M, N, K, G, reinterpret_cast<cudaStream_t>(stream)));
}

int64_t q4k_meta_ld(int64_t K) { return K > 0 && K % 256 == 0 ? K / 256 * 4 : 0; }

w4a16_status q4k_dequant(const uint32_t* qweight, const uint32_t* meta, int64_t N, int64_t K, float* w_out,
                         w4a16_stream_t stream) {
    w4a16_status st = check_q4k_shape(N, K);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if ((st = check_q4k_weights(qweight, meta)) != W4A16_OK) return st;
    if (!w_out) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_out)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_dequant_q4k(qweight, meta, N, K, w_out, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status q4k_pack(const void* w_f16, int64_t N, int64_t K, uint32_t* qweight, uint32_t* meta,
                      w4a16_stream_t stream) {
    w4a16_status st = check_q4k_shape(N, K);
    if (st != W4A16_OK) return st;
    if (N == 0) return W4A16_OK;
    if ((st = check_q4k_weights(qweight, meta)) != W4A16_OK) return st;
    if (!w_f16) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(w_f16)) return W4A16_ERR_MISALIGNED;
    return from_cuda(w4a16::launch_pack_q4k(w_f16, N, K, qweight, meta, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status q4k_linear(const void* x_bf16, const uint32_t* qweight, const uint32_t* meta, int64_t M, int64_t N,
                        int64_t K, void* y_bf16, w4a16_stream_t stream) {
    return q4k_common(x_bf16, &qweight, &meta, &y_bf16, 1, M, N, K, stream);
}

w4a16_status q4k_linear_dual(const void* x_bf16, const uint32_t* qweight_gate, const uint32_t* meta_gate,
                             const uint32_t* qweight_up, const uint32_t* meta_up, int64_t M, int64_t N, int64_t K,
                             void* y_gate_bf16, void* y_up_bf16, w4a16_stream_t stream) {
    const uint32_t* q[2] = {qweight_gate, qweight_up};
    const uint32_t* meta[2] = {meta_gate, meta_up};
    void* y[2] = {y_gate_bf16, y_up_bf16};
    return q4k_common(x_bf16, q, meta, y, 2, M, N, K, stream);
}

int w4a16_linear_path(int64_t M, int64_t N, int64_t K, int G) {
    if (check_weight_shape(N, K, G) != W4A16_OK || M < 0) return 0;
    return choose_path(M, N, K, G, 1);
}

void w4a16_debug_set_wait_limit(int64_t cycles) { w4a16::set_wait_limit(cycles); }

w4a16_status w4a16_debug_gemv_plan(int64_t M, int64_t N, int64_t K, int G, int mode, int32_t* plan) {
    if (!plan || mode < 0 || mode > 2 || M < 1 || M > 16 || check_weight_shape(N, K, G) != W4A16_OK)
        return W4A16_ERR_INVALID_ARG;
    return w4a16::gemv_describe(M, N, K, G, mode, plan) ? W4A16_OK : W4A16_ERR_UNSUPPORTED;
}

w4a16_status w4a16_debug_withhold_copy(int kernel) {
    if (kernel < 0 || kernel > 2) return W4A16_ERR_INVALID_ARG;
    w4a16::arm_withhold(kernel);
    return W4A16_OK;
}

w4a16_status w4a16_device_status(uint32_t* detail) {
    uint32_t word = 0;
    cudaError_t e = w4a16::read_and_clear_status(&word);
    if (detail) *detail = word;
    if (e != cudaSuccess) return W4A16_ERR_CUDA;
    return word ? W4A16_ERR_TIMEOUT : W4A16_OK;
}

}  // extern "C"
