// pack.cu -- FP16 weight -> packed 4-bit codes + FP16 scales + 4-bit zeros
// (and the 8-bit and super-block variants), and the dequantising checking aids
// that run the layer kernels' own expansion routines.
//
// Quantiser: group-wise asymmetric min-max over G consecutive input channels
// of one output column (klaylearn.com glossary "Weight-Only Quantisation",
// main body: small integers plus scale and zero-point per group; instagit
// "Comparison of Quantization Methods", section "Practical Code Examples":
// asymmetric codes reconstruct as (q - zero_point) * scale; zhuai.tech
// "Quantization Is Not a Zip File", section 3: groups of 32..256).
//   lo = min(0, min w), hi = max(0, max w)
//   s  = RNE_fp16((hi - lo) / 15) in IEEE binary32; s == 0 -> s = 1, z = 0
//   z  = clamp(rne(-lo / s), 0, 15),  q = clamp(rne(w / s) + z, 0, 15)
// All divisions are correctly rounded binary32 (the library is built without
// fast-math), so the codes are bit-identical to any IEEE implementation.
#include "common.cuh"
#include "kernels.h"
#include "unpack.cuh"

namespace w4a16 {

// The PER consecutive FP16 weights at src (PER = 1, 2, 4 or 8; src aligned to
// PER halves) as floats.
template <int PER>
__device__ __forceinline__ void load_weights(const __half* src, float (&v)[PER]) {
    if constexpr (PER == 8) {
        uint4 u = *reinterpret_cast<const uint4*>(src);
        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __half2float(__ushort_as_half((unsigned short)(uw[i] & 0xFFFF)));
            v[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(uw[i] >> 16)));
        }
    } else if constexpr (PER == 4) {
        uint2 u = *reinterpret_cast<const uint2*>(src);
        v[0] = __half2float(__ushort_as_half((unsigned short)(u.x & 0xFFFF)));
        v[1] = __half2float(__ushort_as_half((unsigned short)(u.x >> 16)));
        v[2] = __half2float(__ushort_as_half((unsigned short)(u.y & 0xFFFF)));
        v[3] = __half2float(__ushort_as_half((unsigned short)(u.y >> 16)));
    } else if constexpr (PER == 2) {
        uint32_t u = *reinterpret_cast<const uint32_t*>(src);
        v[0] = __half2float(__ushort_as_half((unsigned short)(u & 0xFFFF)));
        v[1] = __half2float(__ushort_as_half((unsigned short)(u >> 16)));
    } else {
        v[0] = __half2float(src[0]);
    }
}

// Range of a group over the warp: lo = min(0, min w), hi = max(0, max w).
template <int PER>
__device__ __forceinline__ void group_range(const float (&v)[PER], float& lo, float& hi) {
    lo = 0.0f;
    hi = 0.0f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        lo = fminf(lo, v[i]);
        hi = fmaxf(hi, v[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
        hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
    }
}

// One warp per weight row; the row's groups are processed in order.  Lane l
// holds the G/32 consecutive weights l*G/32 .. of the current group.
template <int G>
__global__ void __launch_bounds__(256) pack_kernel(const __half* __restrict__ w, int64_t N, int64_t K,
                                                   uint32_t* __restrict__ qw, __half* __restrict__ sc,
                                                   uint32_t* __restrict__ zr) {
    constexpr int PER = G / 32;              // weights per lane: 1, 2, 4, 8
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (row >= N) return;                    // uniform per warp
    const int64_t ngroups = K / G;
    const int64_t ldq = qweight_ld(K), lds = scales_ld(K, G), ldz = zeros_ld(K, G);
    const __half* wrow = w + row * K;
    uint32_t* qrow = qw + row * ldq;
    __half* srow = sc + row * lds;
    uint32_t* zrow = zr + row * ldz;

    uint32_t zword = 0;
    for (int64_t g = 0; g < ngroups; ++g) {
        float v[PER];
        load_weights<PER>(wrow + g * G + lane * PER, v);
        float lo, hi;
        group_range<PER>(v, lo, hi);
        const float range = __fsub_rn(hi, lo);
        __half sh = __float2half_rn(__fdiv_rn(range, 15.0f));
        float s = __half2float(sh);
        int zp = 0;
        if (s == 0.0f) {                     // all-zero (or underflowing) group
            sh = __float2half_rn(1.0f);
            s = 1.0f;
        } else {
            zp = min(max(__float2int_rn(__fdiv_rn(-lo, s)), 0), 15);
        }
        uint32_t bits = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int c = min(max(__float2int_rn(__fdiv_rn(v[i], s)) + zp, 0), 15);
            bits |= (uint32_t)c << (4 * ((lane * PER + i) & 7));
        }
        if constexpr (PER < 8) {             // lanes sharing one word OR their nibbles
#pragma unroll
            for (int off = 1; off < 8 / PER; off <<= 1) bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, off);
        }
        if (((lane * PER) & 7) == 0) qrow[(g * G + lane * PER) / 8] = bits;
        if (lane == 0) srow[g] = sh;
        zword |= (uint32_t)zp << (4 * (g & 7));
        if ((g & 7) == 7 || g == ngroups - 1) {
            if (lane == 0) zrow[g / 8] = zword;
            zword = 0;
        }
    }
    for (int64_t i = ngroups + lane; i < lds; i += 32) srow[i] = __ushort_as_half((unsigned short)0);
    for (int64_t i = (ngroups + 7) / 8 + lane; i < ldz; i += 32) zrow[i] = 0u;
}

// The 8-bit variant: 255 steps, s8 = RNE_fp16((hi - lo) / 255), z8 and codes in
// 0..255.  Each 8-bit code is stored as two 4-bit planes of a 4-bit layer with
// 2K input channels: the row's K high nibbles (channels 0..K-1), then its K low
// nibbles (channels K..2K-1); scales 16*s8 (hi plane groups) then s8 (lo plane
// groups); zeros z8 >> 4 then z8 & 15.  The 4-bit kernels then compute the
// 8-bit layer exactly: 16 s8 (q_hi - z_hi) + s8 (q_lo - z_lo) = s8 (q8 - z8).
template <int G>
__global__ void __launch_bounds__(256) pack8_kernel(const __half* __restrict__ w, int64_t N, int64_t K,
                                                    uint32_t* __restrict__ qw, __half* __restrict__ sc,
                                                    uint32_t* __restrict__ zr) {
    constexpr int PER = G / 32;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (row >= N) return;                    // uniform per warp
    const int64_t ngroups = K / G, K2 = 2 * K;
    const int64_t ldq = qweight_ld(K2), lds = scales_ld(K2, G), ldz = zeros_ld(K2, G);
    const __half* wrow = w + row * K;
    uint32_t* qrow = qw + row * ldq;
    __half* srow = sc + row * lds;
    uint32_t* zrow = zr + row * ldz;
    // zero words may hold nibbles of both planes (when K/G is not a multiple of 8): lane 0
    // clears the row's words, then ORs each group's two nibbles in
    if (lane == 0)
        for (int64_t i = 0; i < ldz; ++i) zrow[i] = 0u;
    for (int64_t g = 0; g < ngroups; ++g) {
        float v[PER];
        load_weights<PER>(wrow + g * G + lane * PER, v);
        float lo, hi;
        group_range<PER>(v, lo, hi);
        const float range = __fsub_rn(hi, lo);
        __half sh = __float2half_rn(__fdiv_rn(range, 255.0f));
        float s = __half2float(sh);
        int zp = 0;
        if (s == 0.0f) {
            sh = __float2half_rn(1.0f);
            s = 1.0f;
        } else {
            zp = min(max(__float2int_rn(__fdiv_rn(-lo, s)), 0), 255);
        }
        uint32_t bh = 0, bl = 0;               // this lane's hi and lo nibbles, at their word positions
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int c = min(max(__float2int_rn(__fdiv_rn(v[i], s)) + zp, 0), 255);
            const int sh4 = 4 * ((lane * PER + i) & 7);
            bh |= (uint32_t)(c >> 4) << sh4;
            bl |= (uint32_t)(c & 15) << sh4;
        }
        if constexpr (PER < 8) {
#pragma unroll
            for (int off = 1; off < 8 / PER; off <<= 1) {
                bh |= __shfl_xor_sync(0xFFFFFFFFu, bh, off);
                bl |= __shfl_xor_sync(0xFFFFFFFFu, bl, off);
            }
        }
        if (((lane * PER) & 7) == 0) {
            const int64_t k = g * G + lane * PER;                 // K and G are multiples of 8
            qrow[k / 8] = bh;
            qrow[(K + k) / 8] = bl;
        }
        if (lane == 0) {
            srow[g] = __float2half_rn(16.0f * s);                 // exact: a power-of-two scaling
            srow[ngroups + g] = sh;
            atomicOr(zrow + g / 8, (uint32_t)(zp >> 4) << (4 * (g & 7)));
            atomicOr(zrow + (ngroups + g) / 8, (uint32_t)(zp & 15) << (4 * ((ngroups + g) & 7)));
        }
    }
    for (int64_t i = 2 * ngroups + lane; i < lds; i += 32) srow[i] = __ushort_as_half((unsigned short)0);
}

// The 8-bit quantiser of pack8_kernel in the word layout: four codes per 32-bit
// word (code of k in byte k % 4 of word k / 4), one FP16 scale per group as the
// 4-bit layout, one 8-bit zero point per group four to a word (byte g % 4 of
// word g / 4, ldZ8 = zeros8_ld).  One warp per weight row walks its groups.
template <int G>
__global__ void __launch_bounds__(256) pack8w_kernel(const __half* __restrict__ w, int64_t N, int64_t K,
                                                     uint32_t* __restrict__ qw, __half* __restrict__ sc,
                                                     uint32_t* __restrict__ zr) {
    constexpr int PER = G / 32;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (row >= N) return;                    // uniform per warp
    const int64_t ngroups = K / G;
    const int64_t ldq = K / 4, lds = scales_ld(K, G), ldz = zeros8_ld(K, G);
    const __half* wrow = w + row * K;
    uint32_t* qrow = qw + row * ldq;
    __half* srow = sc + row * lds;
    uint32_t* zrow = zr + row * ldz;
    uint32_t zacc = 0;                       // lane 0: the zero word being filled
    for (int64_t g = 0; g < ngroups; ++g) {
        float v[PER];
        load_weights<PER>(wrow + g * G + lane * PER, v);
        float lo, hi;
        group_range<PER>(v, lo, hi);
        const float range = __fsub_rn(hi, lo);
        __half sh = __float2half_rn(__fdiv_rn(range, 255.0f));
        float s = __half2float(sh);
        int zp = 0;
        if (s == 0.0f) {
            sh = __float2half_rn(1.0f);
            s = 1.0f;
        } else {
            zp = min(max(__float2int_rn(__fdiv_rn(-lo, s)), 0), 255);
        }
        // this lane's codes at their byte positions, words shared by 4 / PER lanes merged
        uint32_t wv[PER >= 4 ? PER / 4 : 1] = {};
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int c = min(max(__float2int_rn(__fdiv_rn(v[i], s)) + zp, 0), 255);
            wv[i / 4] |= (uint32_t)c << (8 * ((lane * PER + i) & 3));
        }
        const int64_t k0 = g * G + lane * PER;
        if constexpr (PER >= 4) {
#pragma unroll
            for (int j = 0; j < PER / 4; ++j) qrow[k0 / 4 + j] = wv[j];
        } else {
#pragma unroll
            for (int off = 1; off < 4 / PER; off <<= 1) wv[0] |= __shfl_xor_sync(0xFFFFFFFFu, wv[0], off);
            if ((k0 & 3) == 0) qrow[k0 / 4] = wv[0];
        }
        if (lane == 0) {
            srow[g] = sh;
            zacc |= (uint32_t)zp << (8 * (g & 3));
            if ((g & 3) == 3 || g == ngroups - 1) {
                zrow[g / 4] = zacc;
                zacc = 0;
            }
        }
    }
    for (int64_t i = ngroups + lane; i < lds; i += 32) srow[i] = __ushort_as_half((unsigned short)0);
    for (int64_t i = (ngroups + 3) / 4 + lane; i < ldz; i += 32) zrow[i] = 0u;
}

// ---- dequantising checking aids ------------------------------------------------------
// Each runs one layer kernel's own expansion routine (unpack.cuh) over every
// packed word, so their bit-exact checks against the oracle pin that routine.
// One thread per packed word (8 outputs).

// W_hat = (q - z) * s in FP32 through the decode kernel's expansion: the
// word's codes as the FP16 values 1024 + q / 64 + q it multiplies, the zero
// point and the scale as it extracts them; q - z and the product are exact.
__global__ void __launch_bounds__(256) dequant_kernel(const uint32_t* __restrict__ qw, const __half* __restrict__ sc,
                                                      const uint32_t* __restrict__ zr, int64_t N, int64_t K, int G,
                                                      float* __restrict__ out) {
    const int64_t words = K / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= N * words) return;
    const int64_t n = idx / words, w8 = idx % words;
    const int64_t g = (w8 * 8) / G;
    const uint32_t word = qw[n * qweight_ld(K) + w8];
    const float s = __half2float(sc[n * scales_ld(K, G) + g]);
    const float z = meta_zero(zr[n * zeros_ld(K, G) + g / 8] >> (4 * (g & 7)), 0);
    uint32_t e[4];
    expand_codes_f16(word, e[0], e[1], e[2], e[3]);
    float o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {          // pair i holds codes i (low half) and i + 4 (high half)
        o[i] = __fmul_rn(__fsub_rn(__fsub_rn(half_lo(e[i]), expand_offset(i)), z), s);
        o[i + 4] = __fmul_rn(__fsub_rn(__fsub_rn(half_hi(e[i]), expand_offset(i)), z), s);
    }
    float4* dst = reinterpret_cast<float4*>(out + n * K + w8 * 8);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
}

// RN_fp16((q - z) * s) through the tensor-core kernel's expansion: the same
// 128-bit scale chunk and zero word, group constants and packed FP16
// subtract/multiply it writes into tensor memory as the MMA's A operand.
__global__ void __launch_bounds__(256) dequant_f16_kernel(const uint32_t* __restrict__ qw,
                                                          const unsigned short* __restrict__ sc,
                                                          const uint32_t* __restrict__ zr, int64_t N, int64_t K,
                                                          int G, uint32_t* __restrict__ out) {
    const int64_t words = K / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= N * words) return;
    const int64_t n = idx / words, w8 = idx % words;
    const int64_t g = (w8 * 8) / G;
    const uint4 sv = *reinterpret_cast<const uint4*>(sc + n * scales_ld(K, G) + (g >> 3) * 8);
    const uint32_t zw = zr[n * zeros_ld(K, G) + (g >> 3)];
    uint32_t s2, zz;
    group_consts(sv, zw, (int)(g & 7), true, s2, zz);
    uint32_t o[4];
    dequant_word(qw[n * qweight_ld(K) + w8], s2, zz, o);
    *reinterpret_cast<uint4*>(out + (n * K + w8 * 8) / 2) = make_uint4(o[0], o[1], o[2], o[3]);
}

// 8-bit word layout, W_hat = (q - z) * s in FP32 through the decode kernel's
// 8-bit expansion (each code as its two nibble halves 1024 + l and 1024 + 16 h,
// added back) and its 8-bit zero extraction.  One thread per word (4 outputs).
__global__ void __launch_bounds__(256) dequant8w_kernel(const uint32_t* __restrict__ qw, const __half* __restrict__ sc,
                                                        const uint32_t* __restrict__ zr, int64_t N, int64_t K, int G,
                                                        float* __restrict__ out) {
    const int64_t words = K / 4;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= N * words) return;
    const int64_t n = idx / words, w4 = idx % words;
    const int64_t g = (w4 * 4) / G;
    const float s = __half2float(sc[n * scales_ld(K, G) + g]);
    const float z = meta_zero8(zr[n * zeros8_ld(K, G) + g / 4] >> (8 * (g & 3)), 0);
    uint32_t e0, e1, e2, e3;
    expand_codes8_f16(qw[n * (K / 4) + w4], e0, e1, e2, e3);
    // codes 0 and 2 from e0 (low nibbles) and e1 (high nibbles), codes 1 and 3 from e2 and e3
    const float c0 = __fadd_rn(__fsub_rn(half_lo(e0), 1024.0f), __fsub_rn(half_lo(e1), 1024.0f));
    const float c2 = __fadd_rn(__fsub_rn(half_hi(e0), 1024.0f), __fsub_rn(half_hi(e1), 1024.0f));
    const float c1 = __fadd_rn(__fsub_rn(half_lo(e2), 1024.0f), __fsub_rn(half_lo(e3), 1024.0f));
    const float c3 = __fadd_rn(__fsub_rn(half_hi(e2), 1024.0f), __fsub_rn(half_hi(e3), 1024.0f));
    *reinterpret_cast<float4*>(out + n * K + w4 * 4) =
        make_float4(__fmul_rn(__fsub_rn(c0, z), s), __fmul_rn(__fsub_rn(c1, z), s), __fmul_rn(__fsub_rn(c2, z), s),
                    __fmul_rn(__fsub_rn(c3, z), s));
}

// 8-bit word layout, RN_fp16((q - z) * s) through the tensor-core kernel's
// 8-bit expansion and group constants (its FP16 A operand).
__global__ void __launch_bounds__(256) dequant8w_f16_kernel(const uint32_t* __restrict__ qw,
                                                            const unsigned short* __restrict__ sc,
                                                            const uint32_t* __restrict__ zr, int64_t N, int64_t K,
                                                            int G, uint32_t* __restrict__ out) {
    const int64_t words = K / 4;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= N * words) return;
    const int64_t n = idx / words, w4 = idx % words;
    const int64_t g = (w4 * 4) / G;
    const uint4 sv = *reinterpret_cast<const uint4*>(sc + n * scales_ld(K, G) + (g >> 3) * 8);
    const uint32_t zw = zr[n * zeros8_ld(K, G) + g / 4];
    uint32_t s2, zz, o[2];
    group_consts8(sv, zw, (int)(g & 7), (int)(g & 3), true, s2, zz);
    dequant_word8(qw[n * (K / 4) + w4], s2, zz, o);
    *reinterpret_cast<uint2*>(out + (n * K + w4 * 4) / 2) = make_uint2(o[0], o[1]);
}

// Super-block layout: W_hat = d*sc_j*q - dmin*m_j in FP32 through the decode
// kernel's super-block mode: codes from its expansion, the record's FP16
// factors and 6-bit codes as it decodes them, s = d*sc_j and mn = dmin*m_j
// (both exact), then s*q (exact) minus mn, rounded once.
__global__ void __launch_bounds__(256) dequant_q4k_kernel(const uint32_t* __restrict__ qw,
                                                          const uint32_t* __restrict__ meta, int64_t N, int64_t K,
                                                          float* __restrict__ out) {
    const int64_t words = K / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= N * words) return;
    const int64_t n = idx / words, w8 = idx % words;
    const int64_t sb = w8 / 32;
    const int j = (int)((w8 % 32) / 4);                 // sub-block of 32 channels
    const uint4 rec = *reinterpret_cast<const uint4*>(meta + n * (K / 256 * 4) + sb * 4);
    const float s = half_lo(rec.x) * kq_code(rec.y, rec.w, j, 0);
    const float mn = half_hi(rec.x) * kq_code(rec.z, rec.w, j, 16);
    uint32_t e[4];
    expand_codes_f16(qw[n * qweight_ld(K) + w8], e[0], e[1], e[2], e[3]);
    float o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[i] = __fsub_rn(__fmul_rn(s, __fsub_rn(half_lo(e[i]), expand_offset(i))), mn);
        o[i + 4] = __fsub_rn(__fmul_rn(s, __fsub_rn(half_hi(e[i]), expand_offset(i))), mn);
    }
    float4* dst = reinterpret_cast<float4*>(out + n * K + w8 * 8);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
}

// Super-block (Q4_K-style) quantiser: 256 consecutive input channels of one
// output row form a super-block of 8 sub-blocks of 32, each with its own scale
// and minimum, and those are quantised against two FP16 factors per
// super-block (zhuai.tech "Quantization Is Not a Zip File", section 3, table
// "How to read common GGUF quantization names": K-quants keep sub-block
// scales and minima inside 256-weight super-blocks, hierarchically).
//   sub-block j:  lo = min(0, min w), hi = max(0, max w), a_j = (hi - lo) / 15, b_j = -lo
//   d = RNE_fp16(max a_j / 63) (0 -> 1),  dmin = RNE_fp16(max b_j / 63)
//   sc_j = clamp(rne(a_j / d), 0, 63),  m_j = dmin == 0 ? 0 : clamp(rne(b_j / dmin), 0, 63)
//   q = d*sc_j > 0 ? clamp(rne((w + dmin*m_j) / (d*sc_j)), 0, 15) : 0
// W_hat = d*sc_j*q - dmin*m_j.  Codes go to the 4-bit layout; each
// super-block gets a 16-byte record: d | dmin << 16; sc_j & 15 at bits 4j;
// m_j & 15 at bits 4j; sc_j >> 4 at bits 2j and m_j >> 4 at bits 16 + 2j.
// One warp per super-block: lane l holds channels 8l..8l+7 (one code word),
// so lanes 4j..4j+3 hold sub-block j.
__global__ void __launch_bounds__(256) pack_q4k_kernel(const __half* __restrict__ w, int64_t N, int64_t K,
                                                       uint32_t* __restrict__ qw, uint32_t* __restrict__ meta) {
    const int lane = threadIdx.x & 31;
    const int64_t nsb = K / 256;
    const int64_t sbg = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;   // super-block, row-major
    if (sbg >= N * nsb) return;                                                     // warp-uniform
    const int64_t n = sbg / nsb, sb = sbg - n * nsb;
    float v[8];
    load_weights<8>(w + n * K + sb * 256 + lane * 8, v);
    float lo = 0.0f, hi = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        lo = fminf(lo, v[i]);
        hi = fmaxf(hi, v[i]);
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
        hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
    }
    // b = 0 - lo rather than -lo: a sub-block without negative weights has minimum +0, so
    // dmin of a super-block of them is stored as +0
    const float a = __fdiv_rn(__fsub_rn(hi, lo), 15.0f), b = __fsub_rn(0.0f, lo);
    float amax = a, bmax = b;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
        bmax = fmaxf(bmax, __shfl_xor_sync(0xFFFFFFFFu, bmax, off));
    }
    __half dh = __float2half_rn(__fdiv_rn(amax, 63.0f));
    const __half mh = __float2half_rn(__fdiv_rn(bmax, 63.0f));
    float d = __half2float(dh);
    const float dmin = __half2float(mh);
    if (d == 0.0f) {
        dh = __ushort_as_half((unsigned short)0x3C00);
        d = 1.0f;
    }
    const int sc = min(max(__float2int_rn(__fdiv_rn(a, d)), 0), 63);
    const int m = dmin == 0.0f ? 0 : min(max(__float2int_rn(__fdiv_rn(b, dmin)), 0), 63);
    const float ap = __fmul_rn(d, (float)sc), bp = __fmul_rn(dmin, (float)m);    // exact products
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = ap > 0.0f ? min(max(__float2int_rn(__fdiv_rn(__fadd_rn(v[i], bp), ap)), 0), 15) : 0;
        word |= (uint32_t)q << (4 * i);
    }
    qw[n * qweight_ld(K) + sb * 32 + lane] = word;
    // the record: every lane gathers the 8 sub-blocks' codes, lane 0 stores it
    uint32_t w1 = 0, w2 = 0, w3 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int scj = __shfl_sync(0xFFFFFFFFu, sc, 4 * j), mj = __shfl_sync(0xFFFFFFFFu, m, 4 * j);
        w1 |= (uint32_t)(scj & 15) << (4 * j);
        w2 |= (uint32_t)(mj & 15) << (4 * j);
        w3 |= ((uint32_t)(scj >> 4) << (2 * j)) | ((uint32_t)(mj >> 4) << (16 + 2 * j));
    }
    if (lane == 0) {
        const uint32_t w0 = (uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(mh) << 16);
        *reinterpret_cast<uint4*>(meta + n * (nsb * 4) + sb * 4) = make_uint4(w0, w1, w2, w3);
    }
}

cudaError_t launch_pack_q4k(const void* w, int64_t N, int64_t K, uint32_t* qw, uint32_t* meta, cudaStream_t stream) {
    const int warps = 8;
    const int64_t total = N * (K / 256);
    if ((total + warps - 1) / warps > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((total + warps - 1) / warps));
    pack_q4k_kernel<<<grid, dim3(32 * warps), 0, stream>>>(static_cast<const __half*>(w), N, K, qw, meta);
    return cudaGetLastError();
}

cudaError_t launch_pack(const void* w, int64_t N, int64_t K, int G, uint32_t* qw, void* sc, uint32_t* zr,
                        cudaStream_t stream) {
    const int warps = 8;
    const dim3 block(32 * warps);
    const dim3 grid((unsigned)((N + warps - 1) / warps));
    const __half* wp = static_cast<const __half*>(w);
    __half* sp = static_cast<__half*>(sc);
    switch (G) {
        case 32: pack_kernel<32><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 64: pack_kernel<64><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 128: pack_kernel<128><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 256: pack_kernel<256><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_pack8(const void* w, int64_t N, int64_t K, int G, uint32_t* qw, void* sc, uint32_t* zr,
                         cudaStream_t stream) {
    const int warps = 8;
    const dim3 block(32 * warps);
    const dim3 grid((unsigned)((N + warps - 1) / warps));
    const __half* wp = static_cast<const __half*>(w);
    __half* sp = static_cast<__half*>(sc);
    switch (G) {
        case 32: pack8_kernel<32><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 64: pack8_kernel<64><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 128: pack8_kernel<128><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 256: pack8_kernel<256><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_pack8w(const void* w, int64_t N, int64_t K, int G, uint32_t* qw, void* sc, uint32_t* zr,
                          cudaStream_t stream) {
    const int warps = 8;
    const dim3 block(32 * warps);
    const dim3 grid((unsigned)((N + warps - 1) / warps));
    const __half* wp = static_cast<const __half*>(w);
    __half* sp = static_cast<__half*>(sc);
    switch (G) {
        case 32: pack8w_kernel<32><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 64: pack8w_kernel<64><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 128: pack8w_kernel<128><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        case 256: pack8w_kernel<256><<<grid, block, 0, stream>>>(wp, N, K, qw, sp, zr); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// Grid for one thread per packed word of N x K codes (false when it does not fit one launch).
static bool word_grid(int64_t N, int64_t K, dim3& grid) {
    const int64_t blocks = (N * (K / 8) + 255) / 256;
    if (blocks > 0x7FFFFFFF) return false;
    grid = dim3((unsigned)blocks);
    return true;
}

cudaError_t launch_dequant(const uint32_t* qw, const void* sc, const uint32_t* zr, int64_t N, int64_t K, int G,
                           float* out, cudaStream_t stream) {
    dim3 grid;
    if (!word_grid(N, K, grid)) return cudaErrorInvalidValue;
    dequant_kernel<<<grid, 256, 0, stream>>>(qw, static_cast<const __half*>(sc), zr, N, K, G, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant_f16(const uint32_t* qw, const void* sc, const uint32_t* zr, int64_t N, int64_t K, int G,
                               void* out, cudaStream_t stream) {
    dim3 grid;
    if (!word_grid(N, K, grid)) return cudaErrorInvalidValue;
    dequant_f16_kernel<<<grid, 256, 0, stream>>>(qw, static_cast<const unsigned short*>(sc), zr, N, K, G,
                                                 static_cast<uint32_t*>(out));
    return cudaGetLastError();
}

cudaError_t launch_dequant8w(const uint32_t* qw, const void* sc, const uint32_t* zr, int64_t N, int64_t K, int G,
                             float* out, cudaStream_t stream) {
    const int64_t blocks = (N * (K / 4) + 255) / 256;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    dequant8w_kernel<<<(unsigned)blocks, 256, 0, stream>>>(qw, static_cast<const __half*>(sc), zr, N, K, G, out);
    return cudaGetLastError();
}

cudaError_t launch_dequant8w_f16(const uint32_t* qw, const void* sc, const uint32_t* zr, int64_t N, int64_t K, int G,
                                 void* out, cudaStream_t stream) {
    const int64_t blocks = (N * (K / 4) + 255) / 256;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    dequant8w_f16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(qw, static_cast<const unsigned short*>(sc), zr, N, K,
                                                               G, static_cast<uint32_t*>(out));
    return cudaGetLastError();
}

cudaError_t launch_dequant_q4k(const uint32_t* qw, const uint32_t* meta, int64_t N, int64_t K, float* out,
                               cudaStream_t stream) {
    dim3 grid;
    if (!word_grid(N, K, grid)) return cudaErrorInvalidValue;
    dequant_q4k_kernel<<<grid, 256, 0, stream>>>(qw, meta, N, K, out);
    return cudaGetLastError();
}

}  // namespace w4a16
