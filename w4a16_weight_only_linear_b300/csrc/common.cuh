// common.cuh -- device helpers shared by the W4A16 kernels (sm_103a).
//
// Packed format (the library's ABI, see include/w4a16.h):
//   qweight[n][k/8] : code of (n,k) in bits 4*(k%8).., low nibble first
//   scales[n][g]    : FP16 scale of group g = k/G, row pitch ldS halves
//   zeros[n][g/8]   : 4-bit zero point of group g in bits 4*(g%8)..
//   W_hat[n][k]     = (q - z) * s
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace w4a16 {

// Row pitches of the packed format (elements).
__host__ __device__ inline int64_t qweight_ld(int64_t K) { return K / 8; }
__host__ __device__ inline int64_t scales_ld(int64_t K, int G) { return ((K / G) + 7) / 8 * 8; }
__host__ __device__ inline int64_t zeros_ld(int64_t K, int G) { return (((K / G) + 7) / 8 + 3) / 4 * 4; }
// 8-bit word layout: uint32 words per zeros row, four 8-bit zero points per word,
// rounded up to 16 bytes.
__host__ __device__ inline int64_t zeros8_ld(int64_t K, int G) { return (((K / G) + 3) / 4 + 3) / 4 * 4; }

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Exact widening of the BF16 halves of a 32-bit register.
__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

}  // namespace w4a16
