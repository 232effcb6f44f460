// gemv.cu -- decode path of the W4A16 linear layer (M <= 16 activation rows).
//
// Decode rereads every weight for each generated token with little work per
// weight, so this kernel is bound by HBM bandwidth on the packed weights
// (klaylearn.com glossary "Weight-Only Quantisation", FAQ "Why is it
// especially useful for decode?"; zhuai.tech "Quantization Is Not a Zip
// File", section 2 "Moving fewer bytes can make decode faster": packed
// weights decoded block by block straight into the accumulation).
//
// Structure.  Work is cut into tiles of 16 weight rows x all of K.  A CTA of
// 8 warps handles T = 8/S tiles at a time, S warps splitting each tile's
// groups; the grid is sized so every CTA gets the same number of such
// iterations (a contiguous run of tiles), with at most two CTAs per SM.
//   1. every thread first issues 128-bit loads for its next D k-steps of
//      packed codes (and the scale / zero of their groups), so HBM latency
//      overlaps everything else; the ring of loads runs across tile
//      boundaries, so the stream of codes never drains between tiles;
//   2. x [M,K] is staged once per CTA in shared memory, permuted into the
//      warp-MMA B-fragment order, with FP32 per-group sums sum_k x;
//   3. codes become exact BF16 integers 128+q with one LOP3 per pair (no
//      conversion instruction) and meet x in warp MMA m16n8k16 with FP32
//      accumulation; per group acc += s*P - (128+z)*s*sum_k x, which equals
//      s * sum_k x_k (q_k - z) with every product exact;
//   4. with S > 1, the S partial sums of a tile are added through shared
//      memory in a fixed order; every output is rounded to BF16 once.
// The warp MMA serves as a wide exact dot-product instruction: one MMA
// consumes 256 codes, keeping the instruction count near one per weight so
// the kernel stays on the memory bound, not the issue bound.
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
    int tiles_per_mat;   // ceil(N / 16)
    int total_tiles;     // tiles_per_mat * number of matrices
    int tile_groups;     // ceil(total_tiles / T); CTA b takes groups [b*tg/grid, (b+1)*tg/grid)
};

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

// 16-bit load straight into a 32-bit register (the load zero-extends), so no
// instruction consumes the value before it is needed.
__device__ __forceinline__ uint32_t ldg_u16(const unsigned short* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// MT: column tiles of 8 activation rows (1: M <= 8, 2: M <= 16).
// V: packed words per thread per k-step (4 for G >= 128, 2 for G = 64, 1 for
//    G = 32), so the 4-thread quad's 32*V codes of a k-step lie in one group.
// SPG: k-steps per group (2 for G = 256, else 1).
// S: warps splitting one tile's groups (1, 2, 4, 8).  D: k-steps in flight.
template <int MT, int V, int SPG, int S, int D>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvParams p) {
    constexpr int T = kWarps / S;
    constexpr int MP = 8 * MT;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int ti = warp / S, si = warp % S;
    const int M = p.M;
    const int G = p.G;
    const int64_t K = p.K, N = p.N;
    const int ngroups = (int)(K / G);
    const int nsteps = (int)(K / (32 * V));
    const int spt = (ngroups / S) * SPG;          // k-steps per tile for this warp
    const int step0 = si * spt;                   // its first k-step
    const int64_t ldq = qweight_ld(K), lds = scales_ld(K, G), ldz = zeros_ld(K, G);

    uint4* xs = reinterpret_cast<uint4*>(smem_raw);                        // [nsteps][V][M][4]
    float* sx = reinterpret_cast<float*>(xs + (size_t)nsteps * V * M * 4);    // [ngroups][MP]
    float* red = sx + (size_t)ngroups * MP;                                   // [2][T][S][16][MP]

    // This CTA's contiguous, balanced run of tile groups (uniform in the CTA).
    const int tg = p.tile_groups;
    const int g0 = (int)(((int64_t)blockIdx.x * tg) / gridDim.x);
    const int iters = (int)(((int64_t)(blockIdx.x + 1) * tg) / gridDim.x) - g0;

    // ---- register ring: codes, scales and zero words of D k-steps --------
    uint32_t wbuf[D][2][V];
    uint32_t sbuf[D][2];
    uint32_t zbuf[D][2];

    // Load cursor: pointers advance by a constant per k-step; 64-bit address
    // arithmetic happens only when the cursor moves to the next tile.
    int itl = 0, sl = 0, lgrp = 0;
    bool lv0 = false, lv1 = false;
    const uint32_t* lq0 = nullptr;
    const uint32_t* lq1 = nullptr;
    const unsigned short* ls0 = nullptr;
    const unsigned short* ls1 = nullptr;
    const uint32_t* lz0 = nullptr;
    const uint32_t* lz1 = nullptr;
    auto set_load_tile = [&]() {
        const int tau = (g0 + itl) * T + ti;
        const bool ok = itl < iters && tau < p.total_tiles;
        const int second = tau >= p.tiles_per_mat;
        const int tile = second ? tau - p.tiles_per_mat : tau;
        const int64_t row = (int64_t)tile * 16 + g;
        lv0 = ok && row < N;
        lv1 = ok && row + 8 < N;
        const int64_t r = lv0 ? row : 0;          // pointers of an absent row stay in the matrix
        const uint32_t* qm = second ? p.mat[1].q : p.mat[0].q;
        const unsigned short* sm = static_cast<const unsigned short*>(second ? p.mat[1].s : p.mat[0].s);
        const uint32_t* zm = second ? p.mat[1].z : p.mat[0].z;
        lgrp = step0 / SPG;
        lq0 = qm + r * ldq + step0 * 4 * V + t * V;
        lq1 = lq0 + (lv1 ? 8 * ldq : 0);
        ls0 = sm + r * lds + lgrp;
        ls1 = ls0 + (lv1 ? 8 * lds : 0);
        lz0 = zm + r * ldz;
        lz1 = lz0 + (lv1 ? 8 * ldz : 0);
    };
    auto load_slot = [&](uint32_t (&w)[2][V], uint32_t (&sv)[2], uint32_t (&zv)[2]) {
        if (lv0) {
            load_words<V>(lq0, w[0]);
            sv[0] = ldg_u16(ls0);
            zv[0] = ldg_u32(lz0 + (lgrp >> 3));
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v) w[0][v] = 0u;
            sv[0] = 0u;          // scale 0: an absent row contributes nothing
            zv[0] = 0u;
        }
        if (lv1) {
            load_words<V>(lq1, w[1]);
            sv[1] = ldg_u16(ls1);
            zv[1] = ldg_u32(lz1 + (lgrp >> 3));
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v) w[1][v] = 0u;
            sv[1] = 0u;
            zv[1] = 0u;
        }
        lq0 += 4 * V;
        lq1 += 4 * V;
        if (SPG == 1 || (sl & 1)) {
            ++ls0;
            ++ls1;
            ++lgrp;
        }
        if (++sl == spt) {
            sl = 0;
            ++itl;
            set_load_tile();
        }
    };

    // (1) first loads in flight before any staging.
    set_load_tile();
#pragma unroll
    for (int i = 0; i < D; ++i) load_slot(wbuf[i], sbuf[i], zbuf[i]);

    // (2) x -> B-fragment order + per-group sums; item = (m, 8-k word w8).
    {
        // x fits in shared memory, so every index here fits in 32 bits
        const int wpr = (int)(K / 8);
        const int total = M * wpr;
        const int gw = G / 8;                     // words per group, a power of two dividing 32
        const int gshift = __ffs(gw) - 1;
        constexpr int U = 4;
        for (int base0 = warp * 32; base0 < total; base0 += U * kThreads) {
            uint4 xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int item = base0 + u * kThreads + lane;
                xv[u] = make_uint4(0u, 0u, 0u, 0u);
                if (item < total) xv[u] = *reinterpret_cast<const uint4*>(p.x + (int64_t)item * 8);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int item = base0 + u * kThreads + lane;
                float f = bf16lo_to_f32(xv[u].x) + bf16hi_to_f32(xv[u].x) + bf16lo_to_f32(xv[u].y) +
                          bf16hi_to_f32(xv[u].y) + bf16lo_to_f32(xv[u].z) + bf16hi_to_f32(xv[u].z) +
                          bf16lo_to_f32(xv[u].w) + bf16hi_to_f32(xv[u].w);
                for (int off = 1; off < gw; off <<= 1) f += __shfl_xor_sync(0xFFFFFFFFu, f, off);
                if (item < total) {
                    const int m = item / wpr, w8 = item - m * wpr;
                    const int s = w8 / (4 * V);
                    const int tt = (w8 % (4 * V)) / V;
                    const int v = w8 % V;
                    xs[((s * V + v) * M + m) * 4 + tt] =
                        make_uint4(__byte_perm(xv[u].x, xv[u].z, 0x5410), __byte_perm(xv[u].x, xv[u].z, 0x7632),
                                   __byte_perm(xv[u].y, xv[u].w, 0x5410), __byte_perm(xv[u].y, xv[u].w, 0x7632));
                    if ((w8 & (gw - 1)) == 0) sx[(w8 >> gshift) * MP + m] = f;
                }
            }
        }
        for (int i = tid; i < ngroups * (MP - M); i += kThreads) {
            const int grp = i / (MP - M), m = M + i % (MP - M);
            sx[grp * MP + m] = 0.0f;
        }
    }
    __syncthreads();

    // (3) stream the warp's k-steps, tile after tile.
    float acc[MT][4];
    float part[MT][4];
#pragma unroll
    for (int ct = 0; ct < MT; ++ct)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[ct][e] = part[ct][e] = 0.0f;
    bool colv[MT];
#pragma unroll
    for (int ct = 0; ct < MT; ++ct) colv[ct] = (g + 8 * ct) < M;

    const int xstep = V * M * 4;                  // uint4 per k-step of staged x
    const int xlane = g * 4 + t;
    int itc = 0, sc = 0;                          // compute cursor
    int xoff = step0 * xstep;
    int cgrp = step0 / SPG;
    const int total_steps = iters * spt;
    for (int j0 = 0; j0 < total_steps; j0 += D) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            if (j0 + i < total_steps) {
                uint4 bfr[MT][V];
#pragma unroll
                for (int ct = 0; ct < MT; ++ct)
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        bfr[ct][v] = colv[ct] ? xs[xoff + v * M * 4 + xlane + 32 * ct] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    uint32_t plo[4], phi[4];
                    codes_to_bf16x2(wbuf[i][0][v], plo);
                    codes_to_bf16x2(wbuf[i][1][v], phi);
                    const uint32_t a0[4] = {plo[0], phi[0], plo[1], phi[1]};
                    const uint32_t a1[4] = {plo[2], phi[2], plo[3], phi[3]};
#pragma unroll
                    for (int ct = 0; ct < MT; ++ct) {
                        mma_bf16_16816(part[ct], a0, bfr[ct][v].x, bfr[ct][v].y);
                        mma_bf16_16816(part[ct], a1, bfr[ct][v].z, bfr[ct][v].w);
                    }
                }
                if (SPG == 1 || (sc & 1)) {           // group complete: scale and zero correction
                    float s_[2], c_[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        s_[h] = __half2float(__ushort_as_half((unsigned short)sbuf[i][h]));
                        // 128 + z exactly: 2^23 + 128 + z has ulp 1, minus 2^23
                        c_[h] = __uint_as_float(0x4B000080u + nibble(zbuf[i][h], cgrp & 7)) - 8388608.0f;
                    }
#pragma unroll
                    for (int ct = 0; ct < MT; ++ct) {
                        const float2 sxv = *reinterpret_cast<const float2*>(sx + cgrp * MP + 8 * ct + 2 * t);
                        acc[ct][0] = fmaf(s_[0], fmaf(-c_[0], sxv.x, part[ct][0]), acc[ct][0]);
                        acc[ct][1] = fmaf(s_[0], fmaf(-c_[0], sxv.y, part[ct][1]), acc[ct][1]);
                        acc[ct][2] = fmaf(s_[1], fmaf(-c_[1], sxv.x, part[ct][2]), acc[ct][2]);
                        acc[ct][3] = fmaf(s_[1], fmaf(-c_[1], sxv.y, part[ct][3]), acc[ct][3]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) part[ct][e] = 0.0f;
                    }
                    ++cgrp;
                }
                load_slot(wbuf[i], sbuf[i], zbuf[i]);  // refill this slot D steps ahead
                xoff += xstep;
                if (++sc == spt) {                     // tile complete (same step for every warp)
                    if constexpr (S == 1) {
                        const int tau = (g0 + itc) * T + ti;
                        if (tau < p.total_tiles) {
                            const int second = tau >= p.tiles_per_mat;
                            const int tile = second ? tau - p.tiles_per_mat : tau;
                            __nv_bfloat16* y = static_cast<__nv_bfloat16*>(second ? p.mat[1].y : p.mat[0].y);
#pragma unroll
                            for (int ct = 0; ct < MT; ++ct)
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int m = 8 * ct + 2 * t + (e & 1);
                                    const int64_t row = (int64_t)tile * 16 + g + 8 * (e >> 1);
                                    if (m < M && row < N) y[(int64_t)m * N + row] = __float2bfloat16_rn(acc[ct][e]);
                                }
                        }
                    } else {
                        float* rb = red + ((size_t)((itc & 1) * T + ti) * S + si) * 16 * MP;
#pragma unroll
                        for (int ct = 0; ct < MT; ++ct) {
                            rb[g * MP + 8 * ct + 2 * t] = acc[ct][0];
                            rb[g * MP + 8 * ct + 2 * t + 1] = acc[ct][1];
                            rb[(g + 8) * MP + 8 * ct + 2 * t] = acc[ct][2];
                            rb[(g + 8) * MP + 8 * ct + 2 * t + 1] = acc[ct][3];
                        }
                        __syncthreads();
                        const float* rbuf = red + (size_t)(itc & 1) * T * S * 16 * MP;
                        for (int e = tid; e < T * 16 * M; e += kThreads) {
                            const int tj = e / (16 * M);
                            const int m = (e / 16) % M;
                            const int rr = e % 16;
                            const int tau2 = (g0 + itc) * T + tj;
                            if (tau2 >= p.total_tiles) continue;
                            const int second = tau2 >= p.tiles_per_mat;
                            const int tile = second ? tau2 - p.tiles_per_mat : tau2;
                            const int64_t row = (int64_t)tile * 16 + rr;
                            if (row >= N) continue;
                            float sum = 0.0f;
#pragma unroll
                            for (int q = 0; q < S; ++q) sum += rbuf[((tj * S + q) * 16 + rr) * MP + m];
                            __nv_bfloat16* y = static_cast<__nv_bfloat16*>(second ? p.mat[1].y : p.mat[0].y);
                            y[(int64_t)m * N + row] = __float2bfloat16_rn(sum);
                        }
                    }
#pragma unroll
                    for (int ct = 0; ct < MT; ++ct)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[ct][e] = 0.0f;
                    sc = 0;
                    ++itc;
                    xoff = step0 * xstep;
                    cgrp = step0 / SPG;
                }
            }
        }
    }
}

struct Plan {
    int S, iters, grid;
};

template <int MT, int V, int SPG, int S>
cudaError_t launch_s(const GemvParams& p0, size_t smem, int sms, cudaStream_t stream);

// Per kernel instance and device: raise the dynamic shared memory limit once, as needed.
constexpr int kMaxDevices = 64;
template <typename Kern>
cudaError_t ensure_smem(Kern kern, size_t smem, int (&cached)[kMaxDevices]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && (int)smem <= cached[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) cached[dev] = (int)smem;
    return e;
}

template <int MT, int V, int SPG, int S>
cudaError_t launch_s(const GemvParams& p0, size_t smem, int sms, cudaStream_t stream) {
    // k-steps in flight per thread: as deep as the 128-register budget allows without spilling
    constexpr int D = MT == 1 ? (V == 4 ? 6 : (V == 2 ? 8 : 10)) : (V == 4 ? 4 : (V == 2 ? 6 : 8));
    auto kern = gemv_kernel<MT, V, SPG, S, D>;
    static int cached[kMaxDevices] = {};
    cudaError_t e = ensure_smem(kern, smem, cached);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    per_sm = per_sm > 2 ? 2 : per_sm;
    GemvParams p = p0;
    constexpr int T = kWarps / S;
    p.tile_groups = (p.total_tiles + T - 1) / T;
    const int grid = p.tile_groups < sms * per_sm ? p.tile_groups : sms * per_sm;
    kern<<<dim3((unsigned)grid), dim3(kThreads), smem, stream>>>(p);
    return cudaGetLastError();
}

// Splitting S: among the splits that divide the group count, the one whose
// balanced partition leaves the busiest SM with the least work.  CTA b is
// assumed to land on SM b % sms; an SM's work is the warp k-steps of its
// CTAs; the score is the mean useful work per SM over the busiest SM's work.
// Ties go to the smallest S (fewest cross-warp reductions).
int choose_split(int total_tiles, int ngroups, int sms, int per_sm) {
    int best = 0;
    double best_score = -1.0;
    for (int S : {1, 2, 4, 8}) {
        if (ngroups % S) continue;
        const int T = kWarps / S;
        const int tg = (total_tiles + T - 1) / T;
        const int grid = tg < sms * per_sm ? tg : sms * per_sm;
        const int64_t spt = ngroups / S;
        int64_t busiest = 0;
        for (int sm = 0; sm < sms && sm < grid; ++sm) {
            int64_t w = 0;
            for (int b = sm; b < grid; b += sms) {
                const int64_t it = ((int64_t)(b + 1) * tg) / grid - ((int64_t)b * tg) / grid;
                w += it * kWarps * spt;
            }
            if (w > busiest) busiest = w;
        }
        const double useful = (double)total_tiles * ngroups / sms;
        const double score = busiest > 0 ? useful / (double)busiest : 0.0;
        if (score > best_score + 1e-9) {
            best_score = score;
            best = S;
        }
    }
    return best;
}

template <int MT, int V, int SPG>
cudaError_t launch_v(const GemvParams& p, size_t smem, int sms, cudaStream_t stream) {
    const int per_sm = smem <= 100 * 1024 ? 2 : 1;
    switch (choose_split(p.total_tiles, (int)(p.K / p.G), sms, per_sm)) {
        case 1: return launch_s<MT, V, SPG, 1>(p, smem, sms, stream);
        case 2: return launch_s<MT, V, SPG, 2>(p, smem, sms, stream);
        case 4: return launch_s<MT, V, SPG, 4>(p, smem, sms, stream);
        case 8: return launch_s<MT, V, SPG, 8>(p, smem, sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int MT>
cudaError_t launch_g(const GemvParams& p, size_t smem, int sms, cudaStream_t stream) {
    switch (p.G) {
        case 32: return launch_v<MT, 1, 1>(p, smem, sms, stream);
        case 64: return launch_v<MT, 2, 1>(p, smem, sms, stream);
        case 128: return launch_v<MT, 4, 1>(p, smem, sms, stream);
        case 256: return launch_v<MT, 4, 2>(p, smem, sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t gemv_smem_bytes(int64_t M, int64_t K, int G, int /*ntiles*/) {
    if (M < 1 || M > 16) return 0;
    const int64_t MP = M <= 8 ? 8 : 16;
    const int64_t ngroups = K / G;
    const int64_t xs = M * K * 2;
    const int64_t sx = ngroups * MP * 4;
    const int64_t red = 2 * (int64_t)kWarps * 16 * MP * 4;
    return (size_t)(xs + sx + red);
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
    p.tiles_per_mat = (int)((N + 15) / 16);
    p.total_tiles = p.tiles_per_mat * nmat;
    p.tile_groups = 0;
    const size_t smem = gemv_smem_bytes(M, K, G, nmat);
    if (smem == 0) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    return M <= 8 ? launch_g<1>(p, smem, sms, stream) : launch_g<2>(p, smem, sms, stream);
}

}  // namespace w4a16
