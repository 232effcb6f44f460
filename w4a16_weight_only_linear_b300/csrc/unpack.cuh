// unpack.cuh -- the in-register expansions of packed codes and group metadata
// that the layer kernels run.
//
// The decode kernel (gemv.cu), the tensor-core kernel (gemm_tc.cu) and the
// dequantising checking aids (pack.cu) all call these inline functions, so a
// bit-exact check of an aid's output against the oracle's dequantised weights
// pins the very instructions the layer runs: which nibble lands in which
// half, the offsets, the zero-point and scale extraction, the super-block
// record decoding.  Reconstruction is the asymmetric rule (q - zero_point) *
// scale (instagit.com "Comparison of Quantization Methods: INT8 vs GPTQ vs AWQ
// vs GGUF", section "Practical Code Examples"); the super-block form
// d*sc_j*q - dmin*m_j follows zhuai.tech "Quantization Is Not a Zip File",
// section 3, K-quants row of the GGUF names table.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "common.cuh"

namespace w4a16 {

// ---- decode kernel -----------------------------------------------------------------
//
// One packed word of eight codes c0..c7 (c0 in bits 0..3) -> four FP16 pairs,
// one shift and four LOP3s.  The FP16 exponent of 1024 has ulp 1, so a nibble
// in bits 0..3 of a half reads as exactly 1024 + c; the exponent of 64 has ulp
// 1/16, so a nibble in bits 4..7 reads as exactly 64 + c.
//   e0 = (1024 + c0 | 1024 + c4 << 16)    e1 = (64 + c1 | 64 + c5 << 16)
//   e2 = (1024 + c2 | 1024 + c6 << 16)    e3 = (64 + c3 | 64 + c7 << 16)
// The decode kernel stages x in the same pairing ((x0,x4), (x1,x5), ...) and
// subtracts the offsets' share once per block of groups.
__device__ __forceinline__ void expand_codes_f16(uint32_t w, uint32_t& e0, uint32_t& e1, uint32_t& e2,
                                                 uint32_t& e3) {
    const uint32_t w8 = w >> 8;
    e0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
    e1 = lop3_and_or(w, 0x00F000F0u, 0x54005400u);
    e2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
    e3 = lop3_and_or(w8, 0x00F000F0u, 0x54005400u);
}

// Offset carried by pair i of expand_codes_f16 (both halves).
__host__ __device__ constexpr float expand_offset(int i) { return (i & 1) ? 64.0f : 1024.0f; }

// Decode kernel, 8-bit codes: one word of four codes b0..b3 (b0 in bits 0..7,
// b = 16 h + l) -> four FP16 pairs, the same shift and four LOP3s with the
// exponent of 1024 (ulp 1) on both nibble positions, so a high nibble in bits
// 4..7 reads as exactly 1024 + 16 h:
//   e0 = (1024 + l0 | 1024 + l2 << 16)        e1 = (1024 + 16 h0 | 1024 + 16 h2 << 16)
//   e2 = (1024 + l1 | 1024 + l3 << 16)        e3 = (1024 + 16 h1 | 1024 + 16 h3 << 16)
// The kernel meets e0 and e1 with the same x pair (x0, x2), e2 and e3 with
// (x1, x3), so the two halves of a code add up to x (2048 + b).
__device__ __forceinline__ void expand_codes8_f16(uint32_t w, uint32_t& e0, uint32_t& e1, uint32_t& e2,
                                                  uint32_t& e3) {
    const uint32_t w8 = w >> 8;
    e0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
    e1 = lop3_and_or(w, 0x00F000F0u, 0x64006400u);
    e2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
    e3 = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);
}

// Zero point in nibble j of a (shifted) zero word, as a float (2^23 + z has ulp 1).
__device__ __forceinline__ float meta_zero(uint32_t zshifted, int j) {
    return __uint_as_float(0x4B000000u | ((zshifted >> (4 * j)) & 0xFu)) - 8388608.0f;
}

// 8-bit zero point in byte j of a (shifted) zero word, as a float.
__device__ __forceinline__ float meta_zero8(uint32_t zshifted, int j) {
    return __uint_as_float(0x4B000000u | ((zshifted >> (8 * j)) & 0xFFu)) - 8388608.0f;
}

// 6-bit code j of a super-block record as a float: low 4 bits at bit 4j of
// `lo`, high 2 bits at bit 2j + hs of `hi` (hs = 0 for sc, 16 for m).
__device__ __forceinline__ float kq_code(uint32_t lo, uint32_t hi, int j, int hs) {
    const uint32_t v = ((lo >> (4 * j)) & 0xFu) | (((hi >> (2 * j + hs)) & 3u) << 4);
    return __uint_as_float(0x4B000000u | v) - 8388608.0f;
}

// The FP16 halves of a 32-bit word as floats (scales; a record's d and dmin).
__device__ __forceinline__ float half_lo(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// ---- tensor-core kernel --------------------------------------------------------------

__device__ __forceinline__ uint32_t hsub2_rn(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Eight codes (one packed word, k = 8j .. 8j+7) -> four FP16 pairs
// (k = 8j+2i in the low half, 8j+2i+1 in the high half) of RN_fp16((q - z) * s).
// Byte i of the word holds codes 2i (low nibble) and 2i+1 (high nibble);
// PRMT copies it into both halves, one LOP3 keeps the low nibble in the low
// half and the high nibble at bits 4..7 of the high half and ORs in the
// FP16 exponents of 1024 (ulp 1) and 64 (ulp 1/16), giving 1024 + q and
// 64 + q exactly.  zz holds 1024 + z and 64 + z, so the packed subtraction
// is the exact code difference, and one packed multiply rounds it times s.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s2, uint32_t zz, uint32_t* out) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t r = __byte_perm(w, 0u, 0x4040u + 0x0101u * i);
        const uint32_t t = lop3_and_or(r, 0x00F0000Fu, 0x54006400u);
        out[i] = hmul2_rn(hsub2_rn(t, zz), s2);
    }
}

// 8-bit codes: one word of four codes (k = 4j .. 4j+3) -> two FP16 pairs (k =
// 4j+2i in the low half, 4j+2i+1 in the high half) of RN_fp16((q - z) * s).
// PRMT places each code byte under the byte 0x64, the FP16 exponent of 1024
// (ulp 1), giving 1024 + q exactly; zz holds 1024 + z in both halves.
__device__ __forceinline__ void dequant_word8(uint32_t w, uint32_t s2, uint32_t zz, uint32_t* out) {
    out[0] = hmul2_rn(hsub2_rn(__byte_perm(w, 0x64646464u, 0x4140u), zz), s2);
    out[1] = hmul2_rn(hsub2_rn(__byte_perm(w, 0x64646464u, 0x4342u), zz), s2);
}

// Scale (both halves) and the 8-bit zero offsets of group h of an 8-group chunk
// (sv: the chunk's eight FP16 scales; zw: a word of four 8-bit zero points, the
// group's in byte hz).
__device__ __forceinline__ void group_consts8(const uint4& sv, uint32_t zw, int h, int hz, bool valid, uint32_t& s2,
                                              uint32_t& zz) {
    const uint32_t word = (h & 4) ? ((h & 2) ? sv.w : sv.z) : ((h & 2) ? sv.y : sv.x);
    uint32_t sb = (h & 1) ? (word >> 16) : (word & 0xFFFFu);
    sb = valid ? sb : 0u;
    const uint32_t z = (zw >> (8 * hz)) & 0xFFu;
    s2 = sb | (sb << 16);
    zz = (0x6400u | z) * 0x10001u;
}

// Scale (both halves) and zero offsets of group h of an 8-group chunk: sv holds
// the chunk's eight FP16 scales, zw its eight zero nibbles.  An invalid group
// (past the row end) gets scale 0.
__device__ __forceinline__ void group_consts(const uint4& sv, uint32_t zw, int h, bool valid, uint32_t& s2,
                                             uint32_t& zz) {
    const uint32_t word = (h & 4) ? ((h & 2) ? sv.w : sv.z) : ((h & 2) ? sv.y : sv.x);
    uint32_t sb = (h & 1) ? (word >> 16) : (word & 0xFFFFu);
    sb = valid ? sb : 0u;
    const uint32_t z = (zw >> (4 * h)) & 0xFu;
    s2 = sb | (sb << 16);
    zz = ((0x5400u | (z << 4)) << 16) | (0x6400u | z);
}

}  // namespace w4a16
