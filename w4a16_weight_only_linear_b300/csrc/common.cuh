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

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Nibble -> BF16 without a conversion instruction.  BF16 0x4300 is 128.0 and
// its 7 fraction bits weigh 1 each, so OR-ing a 4-bit code c into the low
// fraction bits gives exactly 128 + c.  One LOP3 builds two such values (the
// low and high halves of a 32-bit register).  For a word holding codes
// c0..c7 (c0 in bits 0..3) the four results are
//   p[0] = (128+c0 | 128+c4<<16), p[1] = (128+c1 | 128+c5<<16),
//   p[2] = (128+c2 | 128+c6<<16), p[3] = (128+c3 | 128+c7<<16).
// Consumers pair them with activations staged in the same order.
__device__ __forceinline__ void codes_to_bf16x2(uint32_t w, uint32_t (&p)[4]) {
    constexpr uint32_t kMask = 0x000F000Fu;
    constexpr uint32_t kMagic = 0x43004300u;   // BF16 128.0 in both halves
    p[0] = lop3_and_or(w, kMask, kMagic);
    p[1] = lop3_and_or(w >> 4, kMask, kMagic);
    p[2] = lop3_and_or(w >> 8, kMask, kMagic);
    p[3] = lop3_and_or(w >> 12, kMask, kMagic);
}

// Exact widening of the BF16 halves of a 32-bit register.
__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// 4-bit field i of a word.
__device__ __forceinline__ uint32_t nibble(uint32_t w, int i) { return (w >> (4 * i)) & 0xFu; }

// Warp MMA m16n8k16, BF16 inputs, FP32 accumulate (D = A*B + C).
// A fragment: a0 = A[g][2t..2t+1], a1 = A[g+8][2t..], a2 = A[g][2t+8..],
// a3 = A[g+8][2t+8..]; B fragment: b0 = B[2t..2t+1][g], b1 = B[2t+8..][g];
// C/D: d0 = C[g][2t], d1 = C[g][2t+1], d2 = C[g+8][2t], d3 = C[g+8][2t+1]
// with g = lane/4, t = lane%4; the lower half of a register is the lower k.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Read-only global loads that do not allocate in L1 (weights are streamed once).
__device__ __forceinline__ uint4 ldg_stream_v4(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream_v2(const uint32_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream_v1(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

}  // namespace w4a16
