// gemv.cu -- decode path of the W4A16 linear layer (M <= 16 activation rows).
//
// Decode rereads every weight for each generated token with little work per
// weight, so this kernel is bound by HBM bandwidth on the packed weights
// (klaylearn.com glossary "Weight-Only Quantisation", FAQ "Why is it
// especially useful for decode?"; zhuai.tech "Quantization Is Not a Zip
// File", section 2 "Moving fewer bytes can make decode faster": packed
// weights decoded block by block straight into the accumulation).
//
// Structure (one CTA = 16*R weight rows x all of K, 8 warps splitting K):
//   1. every thread issues 128-bit loads for its first D k-steps of packed
//      codes before anything else, so HBM latency overlaps the staging;
//   2. x [M,K] is staged once per CTA in shared memory, already permuted
//      into the MMA B-fragment order, with FP32 per-group sums sum_k x;
//      the CTA's scales/zeros become per-(row, group) pairs {s, -(128+z)*s};
//   3. the codes become exact BF16 integers 128+q by LOP3 (no conversion
//      instruction) and meet x in warp MMA m16n8k16 with FP32 accumulation;
//      per group: acc += s * P - (128+z) * s * sum_k x, which equals
//      s * sum_k x_k (q_k - z) with every product exact;
//   4. the 8 warps' partial sums are reduced through shared memory in a fixed
//      order and rounded to BF16 once per output.
// The warp MMA is used as a wide exact dot-product instruction: one MMA
// consumes 256 codes, which keeps the instruction count per weight near one
// and the kernel on the memory bound rather than the issue bound.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct GemvParams {
    const __nv_bfloat16* x;
    GemvMat mat[2];
    int64_t N, K;
    int M, G;
    int dual;   // 1: tile r of a CTA reads matrix r (same rows); 0: tiles are consecutive rows of matrix 0
};

// Vector load of V consecutive words.
template <int V>
__device__ __forceinline__ void load_words(const uint32_t* p, uint32_t (&w)[V]) {
    if constexpr (V == 4) {
        uint4 u = ldg_stream_v4(p);
        w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else if constexpr (V == 2) {
        uint2 u = ldg_stream_v2(p);
        w[0] = u.x; w[1] = u.y;
    } else {
        w[0] = ldg_stream_v1(p);
    }
}

// MT: column tiles of 8 activation rows (1: M <= 8, 2: M <= 16).
// V: packed words per thread per k-step (4 for G >= 128, 2 for G = 64, 1 for G = 32),
//    so that one k-step of the 4-thread quad (32*V codes) lies inside one group.
// SPG: k-steps per group (2 for G = 256, else 1).  R: row tiles of 16 per CTA.
// D: k-steps of codes kept in flight per thread.
template <int MT, int V, int SPG, int R, int D>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int M = p.M;
    const int G = p.G;
    const int64_t K = p.K, N = p.N;
    const int ngroups = (int)(K / G);
    const int nsteps = (int)(K / (32 * V));
    constexpr int MP = 8 * MT;

    uint4* xs = reinterpret_cast<uint4*>(smem_raw);                      // [nsteps][V][M][4]
    float* sx = reinterpret_cast<float*>(xs + (size_t)nsteps * V * M * 4);  // [ngroups][MP]
    float4* tab = reinterpret_cast<float4*>(sx + (size_t)ngroups * MP);     // [R][ngroups][8]
    float* red = reinterpret_cast<float*>(tab + (size_t)R * ngroups * 8);   // [kWarps][R][16][MP]

    // Row tiles of this CTA.
    const uint32_t* qrow[R][2];
    bool valid[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t rbase = p.dual ? (int64_t)blockIdx.x * 16 : ((int64_t)blockIdx.x * R + r) * 16;
        const uint32_t* qm = (p.dual && r == 1) ? p.mat[1].q : p.mat[0].q;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t row = rbase + g + 8 * h;
            valid[r][h] = row < N;
            qrow[r][h] = qm + (valid[r][h] ? row : 0) * qweight_ld(K) + t * V;
        }
    }

    // This warp's share of the groups (contiguous, balanced to within one).
    const int gpw = ngroups / kWarps, grem = ngroups % kWarps;
    const int gbeg = warp * gpw + min(warp, grem);
    const int gend = gbeg + gpw + (warp < grem ? 1 : 0);
    const int sbeg = gbeg * SPG, send = gend * SPG;

    uint32_t wbuf[D][R][2][V];
    auto load_step = [&](int s, uint32_t (&dst)[R][2][V]) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (valid[r][h]) {
                    load_words<V>(qrow[r][h] + (int64_t)s * 4 * V, dst[r][h]);
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v) dst[r][h][v] = 0u;
                }
            }
    };

    // (1) first loads in flight before any staging.
#pragma unroll
    for (int i = 0; i < D; ++i)
        if (sbeg + i < send) load_step(sbeg + i, wbuf[i]);

    // (2a) x -> B-fragment order + per-group sums.  Item = (m, word w8 of 8 k).
    {
        const int64_t wpr = K / 8;                   // 8-k words per activation row
        const int64_t total = (int64_t)M * wpr;
        const int gw = G / 8;                        // words per group (4..32), divides 32
        for (int64_t base = (int64_t)warp * 32; base < total; base += kThreads) {
            const int64_t item = base + lane;
            const bool ok = item < total;
            const int64_t m = ok ? item / wpr : 0;
            const int64_t w8 = ok ? item % wpr : 0;
            uint4 xv = make_uint4(0u, 0u, 0u, 0u);
            if (ok) xv = *reinterpret_cast<const uint4*>(p.x + m * K + w8 * 8);
            float f = bf16lo_to_f32(xv.x) + bf16hi_to_f32(xv.x) + bf16lo_to_f32(xv.y) + bf16hi_to_f32(xv.y) +
                      bf16lo_to_f32(xv.z) + bf16hi_to_f32(xv.z) + bf16lo_to_f32(xv.w) + bf16hi_to_f32(xv.w);
            for (int off = 1; off < gw; off <<= 1) f += __shfl_xor_sync(0xFFFFFFFFu, f, off);
            if (ok) {
                const int64_t s = w8 / (4 * V);
                const int tt = (int)((w8 % (4 * V)) / V);
                const int v = (int)(w8 % V);
                xs[((s * V + v) * M + m) * 4 + tt] =
                    make_uint4(__byte_perm(xv.x, xv.z, 0x5410), __byte_perm(xv.x, xv.z, 0x7632),
                               __byte_perm(xv.y, xv.w, 0x5410), __byte_perm(xv.y, xv.w, 0x7632));
                if (w8 % gw == 0) sx[(w8 / gw) * MP + m] = f;
            }
        }
        for (int i = tid; i < ngroups * (MP - M); i += kThreads) {
            const int grp = i / (MP - M), m = M + i % (MP - M);
            sx[grp * MP + m] = 0.0f;
        }
    }

    // (2b) per-(row, group) {s, -(128+z)*s}; both products are exact in FP32.
    {
        const int64_t lds = scales_ld(K, G), ldz = zeros_ld(K, G);
        float* tf = reinterpret_cast<float*>(tab);
        for (int e = tid; e < R * 16 * ngroups; e += kThreads) {
            const int r = e / (16 * ngroups);
            const int rr = (e / ngroups) % 16;
            const int grp = e % ngroups;
            const int64_t row = (p.dual ? (int64_t)blockIdx.x * 16 : ((int64_t)blockIdx.x * R + r) * 16) + rr;
            float s = 0.0f, c = 0.0f;
            if (row < N) {
                const bool second = p.dual && r == 1;
                const __half* sp = static_cast<const __half*>(second ? p.mat[1].s : p.mat[0].s);
                const uint32_t* zp = second ? p.mat[1].z : p.mat[0].z;
                s = __half2float(sp[row * lds + grp]);
                const uint32_t zw = zp[row * ldz + grp / 8];
                c = -(128.0f + (float)nibble(zw, grp & 7)) * s;
            }
            float* dst = tf + ((size_t)(r * ngroups + grp) * 8 + (rr & 7)) * 4 + (rr >= 8 ? 2 : 0);
            dst[0] = s;
            dst[1] = c;
        }
    }
    __syncthreads();

    // (3) main loop over this warp's k-steps.
    float acc[R][MT][4];
    float part[R][MT][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int ct = 0; ct < MT; ++ct)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][ct][e] = part[r][ct][e] = 0.0f;

    bool colv[MT];
#pragma unroll
    for (int ct = 0; ct < MT; ++ct) colv[ct] = (g + 8 * ct) < M;

    for (int s0 = sbeg; s0 < send; s0 += D) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            const int s = s0 + i;
            if (s < send) {
                uint4 bfr[MT][V];
#pragma unroll
                for (int ct = 0; ct < MT; ++ct)
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        bfr[ct][v] = colv[ct] ? xs[(((int64_t)s * V + v) * M + g + 8 * ct) * 4 + t]
                                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        uint32_t plo[4], phi[4];
                        codes_to_bf16x2(wbuf[i][r][0][v], plo);
                        codes_to_bf16x2(wbuf[i][r][1][v], phi);
                        const uint32_t a0[4] = {plo[0], phi[0], plo[1], phi[1]};
                        const uint32_t a1[4] = {plo[2], phi[2], plo[3], phi[3]};
#pragma unroll
                        for (int ct = 0; ct < MT; ++ct) {
                            mma_bf16_16816(part[r][ct], a0, bfr[ct][v].x, bfr[ct][v].y);
                            mma_bf16_16816(part[r][ct], a1, bfr[ct][v].z, bfr[ct][v].w);
                        }
                    }
                if (s + D < send) load_step(s + D, wbuf[i]);
                if ((s + 1) % SPG == 0) {
                    const int grp = s / SPG;
#pragma unroll
                    for (int ct = 0; ct < MT; ++ct) {
                        const float2 sxv = *reinterpret_cast<const float2*>(sx + grp * MP + 8 * ct + 2 * t);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const float4 tv = tab[(size_t)(r * ngroups + grp) * 8 + g];
                            acc[r][ct][0] = fmaf(tv.y, sxv.x, fmaf(tv.x, part[r][ct][0], acc[r][ct][0]));
                            acc[r][ct][1] = fmaf(tv.y, sxv.y, fmaf(tv.x, part[r][ct][1], acc[r][ct][1]));
                            acc[r][ct][2] = fmaf(tv.w, sxv.x, fmaf(tv.z, part[r][ct][2], acc[r][ct][2]));
                            acc[r][ct][3] = fmaf(tv.w, sxv.y, fmaf(tv.z, part[r][ct][3], acc[r][ct][3]));
#pragma unroll
                            for (int e = 0; e < 4; ++e) part[r][ct][e] = 0.0f;
                        }
                    }
                }
            }
        }
    }

    // (4) split-K reduction across the 8 warps, fixed order, one rounding.
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int ct = 0; ct < MT; ++ct) {
            float* d = red + ((size_t)(warp * R + r) * 16) * MP + 8 * ct + 2 * t;
            d[g * MP] = acc[r][ct][0];
            d[g * MP + 1] = acc[r][ct][1];
            d[(g + 8) * MP] = acc[r][ct][2];
            d[(g + 8) * MP + 1] = acc[r][ct][3];
        }
    __syncthreads();
    for (int e = tid; e < R * 16 * M; e += kThreads) {
        const int r = e / (16 * M);
        const int m = (e / 16) % M;
        const int rr = e % 16;
        const int64_t row = (p.dual ? (int64_t)blockIdx.x * 16 : ((int64_t)blockIdx.x * R + r) * 16) + rr;
        if (row >= N) continue;
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += red[((size_t)(w * R + r) * 16 + rr) * MP + m];
        __nv_bfloat16* y = static_cast<__nv_bfloat16*>((p.dual && r == 1) ? p.mat[1].y : p.mat[0].y);
        y[(int64_t)m * N + row] = __float2bfloat16_rn(sum);
    }
}

template <int MT, int V, int SPG, int R, int D>
cudaError_t launch_one(const GemvParams& p, size_t smem, int64_t ctas, cudaStream_t stream) {
    auto kern = gemv_kernel<MT, V, SPG, R, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)ctas), dim3(kThreads), smem, stream>>>(p);
    return cudaGetLastError();
}

// Loads in flight per thread: ~128 bytes of codes (D * R * 2 rows * V words * 4 B).
template <int MT, int V, int SPG, int R>
cudaError_t launch_d(const GemvParams& p, size_t smem, int64_t ctas, cudaStream_t stream) {
    constexpr int D = (16 / (R * V)) < 1 ? 1 : (16 / (R * V));
    return launch_one<MT, V, SPG, R, D>(p, smem, ctas, stream);
}

template <int MT, int R>
cudaError_t launch_g(const GemvParams& p, size_t smem, int64_t ctas, cudaStream_t stream) {
    switch (p.G) {
        case 32: return launch_d<MT, 1, 1, R>(p, smem, ctas, stream);
        case 64: return launch_d<MT, 2, 1, R>(p, smem, ctas, stream);
        case 128: return launch_d<MT, 4, 1, R>(p, smem, ctas, stream);
        case 256: return launch_d<MT, 4, 2, R>(p, smem, ctas, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t gemv_smem_bytes(int64_t M, int64_t K, int G, int ntiles) {
    if (M < 1 || M > 16) return 0;
    const int64_t MP = M <= 8 ? 8 : 16;
    const int64_t ngroups = K / G;
    const int64_t xs = M * K * 2;
    const int64_t sx = ngroups * MP * 4;
    const int64_t tab = (int64_t)ntiles * ngroups * 8 * 16;
    const int64_t red = (int64_t)kWarps * ntiles * 16 * MP * 4;
    return (size_t)(xs + sx + tab + red);
}

size_t device_smem_optin() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    return (size_t)v;
}

cudaError_t launch_gemv(const void* x, const GemvMat* mats, int nmat, int64_t M, int64_t N, int64_t K, int G,
                        cudaStream_t stream) {
    GemvParams p;
    p.x = static_cast<const __nv_bfloat16*>(x);
    p.mat[0] = mats[0];
    p.mat[1] = nmat == 2 ? mats[1] : mats[0];
    p.N = N;
    p.K = K;
    p.M = (int)M;
    p.G = G;
    p.dual = nmat == 2 ? 1 : 0;
    const int R = nmat == 2 ? 2 : 1;
    const size_t smem = gemv_smem_bytes(M, K, G, R);
    const int64_t ctas = nmat == 2 ? (N + 15) / 16 : (N + 16 * R - 1) / (16 * R);
    if (smem == 0) return cudaErrorInvalidValue;
    if (M <= 8) return R == 2 ? launch_g<1, 2>(p, smem, ctas, stream) : launch_g<1, 1>(p, smem, ctas, stream);
    return R == 2 ? launch_g<2, 2>(p, smem, ctas, stream) : launch_g<2, 1>(p, smem, ctas, stream);
}

}  // namespace w4a16
