// gemm_tc.cu -- prefill path of the W4A16 linear layer on the tcgen05 tensor
// cores (any M; the library routes M > 16 here, M = 9..16 where the decode
// kernel would not run with all its warps, and decode shapes whose x the
// decode kernel cannot stage).
//
// At prefill many activation rows share each weight, so the layer is a dense
// contraction bound by tensor-core throughput; the dequantisation is extra
// CUDA-core work on the critical path (klaylearn.com glossary "Weight-Only
// Quantisation", FAQ on prefill; multigrid.ai "Weight-Only Quantization
// Explained", section "Where it stops being the right answer").
//
// Formulation.  The kernel computes the transposed product
//     D[n, m] = sum_k W_hat[n, k] * x[m, k]      (y[m, n] = D[n, m])
// so that the dequantised weights are the MMA's A operand, which tcgen05 can
// read straight from tensor memory: expanded weights are written by CUDA
// cores into TMEM and never touch shared memory or HBM.  x is the B operand,
// brought into shared memory by TMA.
//
// Precision.  Operands are FP16: A = RN_fp16((q - z) * s) (the code difference
// is exact in FP16, one rounding for the product), B = x converted from BF16
// to FP16 once per call (exact for normal-range values), FP32 accumulation in
// TMEM, one BF16 rounding per output (or none: FP32 outputs).  A BF16 A
// operand would round W_hat to 8 significant bits, which alone costs more
// relative error than the output tolerance leaves after the BF16 output
// rounding; FP16 keeps 11.
//
// Structure: a persistent kernel, one 320-thread CTA per SM, warp-specialised.
//   warp 0      TMA producer: 128-k slices of x (two 64-k boxes of BN rows,
//               128-byte swizzle) and code stages of 128 rows x 128 bytes
//               (256 4-bit or 128 8-bit codes per row, swizzled)
//   warp 1      tensor-memory owner and MMA issuer (one thread): per 128-k
//               slice, eight 128 x BN x 16 MMAs and one commit, A from TMEM,
//               B from smem
//   warps 2..5  dequantisers: thread = weight row = TMEM lane; codes from
//               smem -> FP16 pairs with PRMT/LOP3 (no conversion
//               instruction), code difference and scale in packed FP16 ->
//               tcgen05.st into a ring of 128-k A slices in TMEM
//   warps 6..9  epilogue: tcgen05.ld of the FP32 accumulator, BF16 rounding,
//               stores to y
// Tiles are 128 weight rows x BN activation rows (BN <= 256), ordered with the
// activation tile fastest so consecutive CTAs share a weight tile in L2.  When
// narrow tiles (BN <= 64) fill at most half the SMs, each is cut along K; when
// the last wave of wider tiles is at most half full, its tiles are cut in two
// along K.  The pieces' FP32 partials are added in a fixed order (see
// GemmParams).
// Every wait is bounded: on expiry the kernel records a code in the status
// word, waits (bounded) for its own copies and MMAs in flight, frees its
// tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/w4a16.h"
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "unpack.cuh"

namespace w4a16 {

// Per-device word that kernels set when a bounded wait gives up.
__device__ uint32_t g_status_word = 0;

namespace {

constexpr int kThreads = 320;              // 10 warps
constexpr int kBM = 128;                   // weight rows per tile (MMA M)
constexpr int kMaxS = 4;                   // slice ring: x (smem) and A (TMEM) slices of 128 k
constexpr int kMaxCS = 3;                  // code ring: stages of 128 bytes of codes per row
constexpr uint32_t kCodeStageBytes = 128u * 128u;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = 256;           // D uses columns [0, BN), A slices (64 columns each) [256, 512)
constexpr uint32_t kParkCol = 448;         // BN = 256 (three A slices): the epilogue parks BF16 pairs here
constexpr int kNumBars = 3 * kMaxS + 2 * kMaxCS + 2;

// Status codes (bit fields) recorded when a wait gives up.
constexpr uint32_t kStatusProducer = 1u << 0;
constexpr uint32_t kStatusMma = 1u << 1;
constexpr uint32_t kStatusDequant = 1u << 2;
constexpr uint32_t kStatusEpilogue = 1u << 3;
constexpr uint32_t kStatusDrain = 1u << 4;

// Work units.  A tile is 128 weight rows x BN activation rows; units [0, full)
// are whole tiles (tile = unit).  The last `split` tiles (all of them when
// narrow tiles are few for the SMs; the last, partial wave of wider tiles) are
// each cut along K into `parts` ranges of code stages, unit full + j * split
// + i being range j of tile full + i.  A range's FP32 partial goes to a workspace, and the last of a
// tile's ranges to finish adds them in a fixed order (so results do not
// depend on arrival order) and writes y.
struct GemmParams {
    const unsigned short* s;   // FP16 scales [N, lds]
    const uint32_t* z;         // packed zeros [N, ldz] (4-bit: 8 per word; 8-bit: 4 per word)
    void* y;                   // [M, N], BF16 (or FP32 when yf32)
    float* ws;                 // K-split partials [split * parts][BN / 4][128][4]
    uint32_t* cnt;             // arrivals per K-split tile (zero at launch)
    int yf32;                  // 1: FP32 outputs (no BF16 rounding)
    int M, N, K, BN;
    int lds, ldz, ngroups;
    int mtiles, tiles;
    int nk64;
    int subs, nstage;          // 64-k slices per code stage (4: 4-bit codes, 2: 8-bit), code stages
    int full, split, parts, units;
    long long spin_limit;      // cycles a bounded wait spins before it gives up
    int withhold;              // test hook: CTA 0 never issues its first code copy
};

struct Unit {
    int tile;                  // tile index (n-tile * mtiles + m-tile)
    int kb0, kb1;              // its 64-k slices [kb0, kb1) (kb0 on a code-stage boundary)
    int part;                  // K range of a split tile: its partial's slot; else -1
    int stile;                 // split tile index (counter slot), or -1
};

__device__ __forceinline__ Unit unit_of(const GemmParams& p, int u) {
    Unit U;
    if (u < p.full) {
        U.tile = u;
        U.kb0 = 0;
        U.kb1 = p.nk64;
        U.part = -1;
        U.stile = -1;
        return U;
    }
    const int v = u - p.full;
    const int j = v / p.split, i = v - j * p.split;
    U.tile = p.full + i;
    U.kb0 = p.subs * ((j * p.nstage) / p.parts);
    U.kb1 = min(p.subs * (((j + 1) * p.nstage) / p.parts), p.nk64);
    U.part = i * p.parts + j;
    U.stile = i;
    return U;
}

// Ring depths for BN activation rows.  A slice is 128 k: two 64-k x boxes (BN
// rows of 128 bytes each) and 64 tensor-memory columns of A.  Four slices up
// to BN = 128 (x slots of at most 32 KB, three code stages); at BN = 256 three
// (192 KB of x, the most that leaves room for two code stages).  x slices come
// from L2 with a latency of several slice times, so the x ring is as deep as
// shared memory allows.
__host__ __device__ constexpr int slice_slots(int BN) { return BN <= 128 ? 4 : 3; }
__host__ __device__ constexpr int code_stages(int BN) { return BN <= 128 ? 3 : 2; }

// Dynamic shared memory per CTA.  Never less than 120 KB, so at most one CTA
// is resident per SM and the 512 tensor-memory columns it allocates are free.
size_t gemm_smem_bytes(int BN) {
    const size_t need = 1024 + (size_t)slice_slots(BN) * BN * 256 + (size_t)code_stages(BN) * kCodeStageBytes +
                        kNumBars * 8 + 16;
    return need < 120 * 1024 ? 120 * 1024 : need;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 ldg128_nc(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg32_nc(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

struct Smem {
    uint8_t* x;       // slice_slots(BN) slices of 2 x BN * 128 bytes
    uint8_t* c;       // code_stages(BN) stages of 16 KB
    uint64_t* bar;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    volatile int* last_flag;   // epilogue: this CTA completes the split tile
    // slice slot i: x_full (its x copy landed), a_full (its A slice written), s_empty (the MMAs
    // that read both completed: one commit frees the x slot and the A slot)
    __device__ uint32_t x_full(int i) const { return tc::smem_u32(bar + i); }
    __device__ uint32_t a_full(int i) const { return tc::smem_u32(bar + kMaxS + i); }
    __device__ uint32_t s_empty(int i) const { return tc::smem_u32(bar + 2 * kMaxS + i); }
    __device__ uint32_t c_full(int i) const { return tc::smem_u32(bar + 3 * kMaxS + i); }
    __device__ uint32_t c_empty(int i) const { return tc::smem_u32(bar + 3 * kMaxS + kMaxCS + i); }
    __device__ uint32_t d_full() const { return tc::smem_u32(bar + 3 * kMaxS + 2 * kMaxCS); }
    __device__ uint32_t d_empty() const { return tc::smem_u32(bar + 3 * kMaxS + 2 * kMaxCS + 1); }
};

// Bounded wait for a barrier phase; gives up (recording `site`) after `limit`
// cycles, or at once when another role has given up.  The first poll is
// inline; the spin loop is a call, taken only when the phase is not complete.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t site,
                                             long long limit) {
    const long long t0 = clock64();
    while (true) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            atomicOr(&g_status_word, site);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, uint32_t site,
                                           long long limit) {
    return tc::mbar_try_wait(bar, parity) || wait_phase_slow(bar, parity, abort_flag, site, limit);
}

// Bounded wait used while shutting down after a give-up: ignores the abort flag.
__device__ void drain_phase(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            atomicOr(&g_status_word, kStatusDrain);
            return;
        }
    }
}

// Named barrier of the four epilogue warps, and the same barrier as a vote: true
// on every epilogue thread when `v` is true on all of them (so the four warps
// always take the same branch around the barriers below).
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epilogue_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Epilogue of one K range of a split tile (the four epilogue warps, thread r =
// weight row r of the tile).  A range's FP32 partial goes to the workspace in
// quads of activation rows, [part][m / 4][r][m % 4], so that thread r moves 16
// bytes per access and a warp 512 contiguous bytes; the last of the tile's
// ranges to finish adds every range's partial in range order and
// writes y.  A range that finds the others all done before it writes skips
// its own write, and a range that is its CTA's last unit (hold) keeps its
// accumulator in tensor memory until its sum is done; when the summing range
// still holds its accumulator it reads its own partial from there, the same
// FP32 values, so the result does not depend on which range sums.
__device__ __forceinline__ void release_accumulator(const Smem& sm, int lane) {
    tc::tc_fence_before();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(sm.d_empty());
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* a) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

__device__ __forceinline__ void epilogue_partial(const GemmParams& p, const Smem& sm, const Unit& U, int n, int m0,
                                                 uint32_t d_lane, int lane, int r, bool hold) {
    const uint32_t others = (uint32_t)(p.parts - 1);
    if (threadIdx.x == 6 * 32) *sm.last_flag = ld_acquire_u32(p.cnt + U.stile) == others;
    epilogue_sync();
    bool last = *sm.last_flag != 0;
    epilogue_sync();                                  // every thread has read the flag
    bool own_tmem = last;                             // this range's partial is still in tensor memory
    if (!last) {
        float4* wp = reinterpret_cast<float4*>(p.ws + (size_t)U.part * p.BN * kBM) + r;
#pragma unroll 1
        for (int c = 0; c < p.BN; c += 16) {
            uint32_t v[16];
            tc::tmem_ld16_wait(d_lane + (uint32_t)c, v);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                __stcg(wp + (size_t)(c / 4 + q) * kBM,
                       make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
        }
        if (!hold) release_accumulator(sm, lane);
        __threadfence();
        epilogue_sync();
        if (threadIdx.x == 6 * 32) *sm.last_flag = atomicAdd(p.cnt + U.stile, 1u) == others;
        epilogue_sync();
        last = *sm.last_flag != 0;
        epilogue_sync();
        if (!last) {
            if (hold) release_accumulator(sm, lane);
            return;
        }
        own_tmem = hold;
    }
    __threadfence();
    const int lim = min(p.BN, p.M - m0);              // activation rows of the tile
    const int own = U.part - U.stile * p.parts;       // this unit's range
    const float4* wt = reinterpret_cast<const float4*>(p.ws + (size_t)U.stile * p.parts * p.BN * kBM) + r;
#pragma unroll 1
    for (int h = 0; h < lim; h += 32) {
        float acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
#pragma unroll 1
        for (int j = 0; j < p.parts; ++j) {           // ranges in order; 32 values of one in flight
            float v[32];
            if (j == own && own_tmem) {
                uint32_t b[32];
                tc::tmem_ld32_wait(d_lane + (uint32_t)h, b);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(b[i]);
            } else {
                const float4* wj = wt + ((size_t)j * p.BN + h) / 4 * kBM;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 f = __ldcg(wj + (size_t)q * kBM);
                    v[4 * q] = f.x;
                    v[4 * q + 1] = f.y;
                    v[4 * q + 2] = f.z;
                    v[4 * q + 3] = f.w;
                }
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] += v[i];
        }
        if (n < p.N) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (h + i < lim) {
                    const int64_t o = (int64_t)(m0 + h + i) * p.N + n;
                    if (p.yf32)
                        static_cast<float*>(p.y)[o] = acc[i];
                    else
                        static_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(acc[i]);
                }
            }
        }
    }
    if (own_tmem) release_accumulator(sm, lane);
}

// One 64-k slice of A from 8-bit codes (the word layout): the slice's 64 codes
// are four 16-byte words of the swizzled stage (a stage holds 128 codes per
// row); sv holds the 8-group scale chunk and zv the four zero words (16
// groups) of the stage's groups.
template <int G>
__device__ __forceinline__ void dequant_slice8(uint32_t rowp, int r, int sub, int ks, const uint4& sv,
                                               const uint4& zv, int ngroups, uint32_t (&a)[32]) {
    uint4 w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = lds128(rowp + ((uint32_t)((4 * sub + i) ^ (r & 7)) << 4));
    const int ga = (ks * 128 + sub * 64) / G;        // group of the slice's first code
    const int gc = (ks * 128 / G) & ~7;              // first group of the scale chunk
    const int gz = (ks * 128 / G) & ~15;             // first group of the zero words
    const uint32_t zs[4] = {zv.x, zv.y, zv.z, zv.w};
    uint32_t s2a, zza, s2b, zzb;
    group_consts8(sv, zs[((ga - gz) >> 2) & 3], ga - gc, ga & 3, ga < ngroups, s2a, zza);
    if constexpr (G == 32) {
        group_consts8(sv, zs[((ga + 1 - gz) >> 2) & 3], ga + 1 - gc, (ga + 1) & 3, ga + 1 < ngroups, s2b, zzb);
    } else {
        s2b = s2a;
        zzb = zza;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t s2 = i < 2 ? s2a : s2b, zz = i < 2 ? zza : zzb;
        dequant_word8(w[i].x, s2, zz, a + 8 * i + 0);
        dequant_word8(w[i].y, s2, zz, a + 8 * i + 2);
        dequant_word8(w[i].z, s2, zz, a + 8 * i + 4);
        dequant_word8(w[i].w, s2, zz, a + 8 * i + 6);
    }
}

template <int G, bool W8>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_q,
                const GemmParams p) {
    // 64-k slices per code stage (a stage is 128 bytes of codes per row: 256 4-bit codes, or
    // 128 8-bit codes)
    constexpr int kSubs = W8 ? 2 : 4;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t xhalf = (uint32_t)p.BN * 128u;      // one 64-k box of x
    const uint32_t xbytes = 2u * xhalf;                 // a slice slot
    Smem sm;
    sm.x = base;
    const int NS = slice_slots(p.BN), NC = code_stages(p.BN);
    sm.c = base + NS * xbytes;
    sm.bar = reinterpret_cast<uint64_t*>(sm.c + NC * kCodeStageBytes);
    sm.tmem_slot = reinterpret_cast<uint32_t*>(sm.bar + kNumBars);
    sm.abort_flag = reinterpret_cast<volatile int*>(sm.tmem_slot + 1);
    sm.last_flag = reinterpret_cast<volatile int*>(sm.tmem_slot + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // launched with programmatic stream serialisation: this grid touches no global memory
    // before the previous grid on the stream has completed (the wait below), so the barriers,
    // tensor memory and descriptor prefetches of the prologue overlap that grid's tail.  It
    // does not let the next launch in early: blocks of a next grid resident beside this one,
    // waiting, cost the contraction 2 % at M = 2048.
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            tc::mbar_init(sm.x_full(i), 1);
            tc::mbar_init(sm.a_full(i), 4);
            tc::mbar_init(sm.s_empty(i), 1);
        }
        for (int i = 0; i < NC; ++i) {
            tc::mbar_init(sm.c_full(i), 1);
            tc::mbar_init(sm.c_empty(i), 4);
        }
        tc::mbar_init(sm.d_full(), 1);
        tc::mbar_init(sm.d_empty(), 4);
        *sm.abort_flag = 0;
        *sm.last_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tm_x);
        tc::tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(sm.tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot;
    tc::griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int xi = 0, ci = 0;
            uint32_t xph = 0, cph = 0;
            long long x_issued = 0, c_issued = 0;
            bool ok = true;
            // test hook: CTA 0 skips its first code copy (slot 0, never refilled since its
            // consumers never release it), so the dequantisers' wait on it runs out
            const bool withhold = p.withhold && blockIdx.x == 0;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                const Unit U = unit_of(p, u);
                const int n0 = (U.tile / p.mtiles) * kBM, m0 = (U.tile % p.mtiles) * p.BN;
                for (int kb = U.kb0; kb < U.kb1; kb += 2) {      // slices of 128 k: 64-k boxes kb, kb+1
                    if ((kb & (kSubs - 1)) == 0) {
                        if (!(ok = wait_phase(sm.c_empty(ci), cph ^ 1u, sm.abort_flag, kStatusProducer, p.spin_limit))) break;
                        if (!(withhold && c_issued == 0)) {
                            tc::mbar_arrive_expect_tx(sm.c_full(ci), kCodeStageBytes);
                            tc::tma_load_2d(tc::smem_u32(sm.c + ci * kCodeStageBytes), &tm_q, (kb / kSubs) * 32, n0,
                                            sm.c_full(ci));
                        }
                        ++c_issued;
                        if (++ci == NC) { ci = 0; cph ^= 1u; }
                    }
                    if (!(ok = wait_phase(sm.s_empty(xi), xph ^ 1u, sm.abort_flag, kStatusProducer, p.spin_limit))) break;
                    const bool two = kb + 1 < U.kb1;
                    tc::mbar_arrive_expect_tx(sm.x_full(xi), two ? xbytes : xhalf);
                    tc::tma_load_2d(tc::smem_u32(sm.x + xi * xbytes), &tm_x, kb * 64, m0, sm.x_full(xi));
                    if (two)
                        tc::tma_load_2d(tc::smem_u32(sm.x + xi * xbytes + xhalf), &tm_x, kb * 64 + 64, m0, sm.x_full(xi));
                    ++x_issued;
                    if (++xi == NS) { xi = 0; xph ^= 1u; }
                }
            }
            if (!ok) {   // wait for the copies this thread started
                for (int s = 0; s < NS; ++s)
                    if (x_issued > s) drain_phase(sm.x_full(s), s < xi ? xph : (xph ^ 1u), p.spin_limit);
                for (int s = 0; s < NC; ++s)
                    if (c_issued > s && !(withhold && s == 0 && c_issued <= NC)) drain_phase(sm.c_full(s), s < ci ? cph : (cph ^ 1u), p.spin_limit);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16_f32(kBM, p.BN);
            int si = 0;
            uint32_t sph = 0, dph = 0, d_commits = 0;
            bool ok = true;
            bool issued = false;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                const Unit U = unit_of(p, u);
                if (!(ok = wait_phase(sm.d_empty(), dph ^ 1u, sm.abort_flag, kStatusMma, p.spin_limit))) break;
                dph ^= 1u;
                tc::tc_fence_after();
                for (int kb = U.kb0; kb < U.kb1; kb += 2) {
                    if (!(ok = wait_phase(sm.x_full(si), sph, sm.abort_flag, kStatusMma, p.spin_limit))) break;
                    if (!(ok = wait_phase(sm.a_full(si), sph, sm.abort_flag, kStatusMma, p.spin_limit))) break;
                    tc::tc_fence_after();
                    const uint64_t bdesc0 = tc::smem_desc_k_sw128(tc::smem_u32(sm.x + si * xbytes));
                    const uint64_t bdesc1 = tc::smem_desc_k_sw128(tc::smem_u32(sm.x + si * xbytes + xhalf));
                    const uint32_t a_t = tmem + kACol0 + (uint32_t)si * 64u;
                    const int nkk = kb + 1 < U.kb1 ? 8 : 4;       // K = 16 per MMA
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        if (kk < nkk)
                            tc::mma_f16_ts(tmem, a_t + 8u * kk,
                                           (kk < 4 ? bdesc0 : bdesc1) + (uint64_t)(2 * (kk & 3)), idesc,
                                           (kb != U.kb0 || kk != 0) ? 1u : 0u);
                    issued = true;
                    tc::mma_commit(sm.s_empty(si));
                    if (++si == NS) { si = 0; sph ^= 1u; }
                }
                if (!ok) break;
                tc::mma_commit(sm.d_full());
                ++d_commits;
            }
            if (!ok && issued) {   // wait for the MMAs this thread issued
                tc::mma_commit(sm.d_full());
                drain_phase(sm.d_full(), d_commits & 1u, p.spin_limit);
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ dequantisers
        const int qd = warp & 3;
        const int r = qd * 32 + lane;                       // weight row in the tile = TMEM lane
        const uint32_t a_lane = tmem + ((uint32_t)(qd * 32) << 16) + kACol0;
        int ci = 0, ai = 0;                                   // ai: slice slot
        uint32_t cph = 0, aph = 0;
        bool ok = true;
        // this row's scale chunk (8 groups) and zero points of code stage ks of unit uu (4-bit:
        // the chunk's zero word; 8-bit: the 4-word block of 16 groups holding them); zeros for a
        // row past N
        auto load_meta = [&](int uu, int ks, uint4& sv, uint4& zv, uint32_t& zw) {
            const int nn = (unit_of(p, uu).tile / p.mtiles) * kBM + r;
            sv = make_uint4(0u, 0u, 0u, 0u);
            zv = make_uint4(0u, 0u, 0u, 0u);
            zw = 0u;
            if (nn < p.N) {
                const int g0 = ks * (kSubs * 64) / G;
                sv = ldg128_nc(p.s + (int64_t)nn * p.lds + (g0 & ~7));
                if constexpr (W8) zv = ldg128_nc(p.z + (int64_t)nn * p.ldz + ((g0 >> 2) & ~3));
                else zw = ldg32_nc(p.z + (int64_t)nn * p.ldz + (g0 >> 3));
            }
        };
        // the metadata is requested one code stage ahead of its use (the next unit's first
        // stage during a unit's last), so its latency hides behind a stage of expansion
        uint4 sv, zv;
        uint32_t zw;
        if (blockIdx.x < p.units) load_meta(blockIdx.x, unit_of(p, blockIdx.x).kb0 / kSubs, sv, zv, zw);
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            const Unit U = unit_of(p, u);
            const int ks_end = (U.kb1 + kSubs - 1) / kSubs;
            for (int ks = U.kb0 / kSubs; ks < ks_end && ok; ++ks) {
                uint4 svn = sv, zvn = zv;
                uint32_t zwn = zw;
                if (ks + 1 < ks_end) load_meta(u, ks + 1, svn, zvn, zwn);
                else if (u + (int)gridDim.x < p.units)
                    load_meta(u + gridDim.x, unit_of(p, u + gridDim.x).kb0 / kSubs, svn, zvn, zwn);
                ok = wait_phase(sm.c_full(ci), cph, sm.abort_flag, kStatusDequant, p.spin_limit);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                const uint32_t rowp = tc::smem_u32(sm.c + ci * kCodeStageBytes) + (uint32_t)r * 128u;
                const int nsub = min(kSubs, p.nk64 - ks * kSubs);
                // 64-k sub-slice `sub` of the stage -> 32 FP16 pairs
                auto expand = [&](int sub, uint32_t (&a)[32]) {
                    if constexpr (W8) {
                        dequant_slice8<G>(rowp, r, sub, ks, sv, zv, p.ngroups, a);
                    } else {
                        const uint4 w0 = lds128(rowp + ((uint32_t)((2 * sub) ^ (r & 7)) << 4));
                        const uint4 w1 = lds128(rowp + ((uint32_t)((2 * sub + 1) ^ (r & 7)) << 4));
                        const int ga = (ks * 256 + sub * 64) / G;        // group of the sub-slice's first code
                        uint32_t s2a, zza, s2b, zzb;
                        group_consts(sv, zw, ga & 7, ga < p.ngroups, s2a, zza);
                        if constexpr (G == 32) {
                            group_consts(sv, zw, (ga + 1) & 7, ga + 1 < p.ngroups, s2b, zzb);
                        } else {
                            s2b = s2a;
                            zzb = zza;
                        }
                        dequant_word(w0.x, s2a, zza, a + 0);
                        dequant_word(w0.y, s2a, zza, a + 4);
                        dequant_word(w0.z, s2a, zza, a + 8);
                        dequant_word(w0.w, s2a, zza, a + 12);
                        dequant_word(w1.x, s2b, zzb, a + 16);
                        dequant_word(w1.y, s2b, zzb, a + 20);
                        dequant_word(w1.z, s2b, zzb, a + 24);
                        dequant_word(w1.w, s2b, zzb, a + 28);
                    }
                };
                for (int sub = 0; sub < nsub; sub += 2) {          // one 128-k slice: sub, sub + 1
                    ok = wait_phase(sm.s_empty(ai), aph ^ 1u, sm.abort_flag, kStatusDequant, p.spin_limit);
                    if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                    tc::tc_fence_after();
                    uint32_t a0[32], a1[32];
                    expand(sub, a0);
                    tc::tmem_st32(a_lane + (uint32_t)ai * 64u, a0);
                    if (sub + 1 < nsub) {
                        expand(sub + 1, a1);
                        tc::tmem_st32(a_lane + (uint32_t)ai * 64u + 32u, a1);
                    }
                    tc::tmem_wait_st();
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(sm.a_full(ai));
                    if (++ai == NS) { ai = 0; aph ^= 1u; }
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(sm.c_empty(ci));
                if (++ci == NC) { ci = 0; cph ^= 1u; }
                sv = svn;
                zv = zvn;
                zw = zwn;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int qd = warp & 3;
        const int r = qd * 32 + lane;
        const uint32_t d_lane = tmem + ((uint32_t)(qd * 32) << 16);
        uint32_t dph = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            const Unit U = unit_of(p, u);
            const int n = (U.tile / p.mtiles) * kBM + r, m0 = (U.tile % p.mtiles) * p.BN;
            ok = wait_phase(sm.d_full(), dph, sm.abort_flag, kStatusEpilogue, p.spin_limit);
            if (!epilogue_all(ok)) {
                ok = false;
                break;
            }
            dph ^= 1u;
            tc::tc_fence_after();
            if (U.part >= 0) {
                epilogue_partial(p, sm, U, n, m0, d_lane, lane, r, u + (int)gridDim.x >= p.units);
                continue;
            }
            if (p.yf32) {
                // FP32 output (no BF16 rounding): each 32-column chunk is stored as loaded, and the
                // accumulator is released after the last one
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    if (ch * 32 < p.BN) {
                        uint32_t v[32];
                        tc::tmem_ld32_wait(d_lane + (uint32_t)ch * 32u, v);
                        if (n < p.N) {
                            float* yc = static_cast<float*>(p.y) + n;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const int m = m0 + ch * 32 + j;
                                if (m < p.M) yc[(int64_t)m * p.N] = __uint_as_float(v[j]);
                            }
                        }
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(sm.d_empty());
                continue;
            }
            // BF16 output: the row's columns are rounded into packed pairs and the accumulator is
            // released before the stores, so the next unit's MMAs overlap them.  At BN = 256 the
            // first 128 columns' pairs are parked in the 64 tensor-memory columns past the A ring
            // (the ring then holds three slices, columns 256..447), so at most 64 packed registers
            // are live and the epilogue does not spill.
            const bool wide = p.BN > 128;
            uint32_t packed[64];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                if (ch * 32 < p.BN) {
                    uint32_t v[32];
                    tc::tmem_ld32_wait(d_lane + (uint32_t)ch * 32u, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const __nv_bfloat162 b =
                            __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                        packed[ch * 16 + j] = *reinterpret_cast<const uint32_t*>(&b);
                    }
                }
            }
            if (wide) {
                uint32_t h0[32], h1[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    h0[j] = packed[j];
                    h1[j] = packed[32 + j];
                }
                tc::tmem_st32(d_lane + kParkCol, h0);
                tc::tmem_st32(d_lane + kParkCol + 32u, h1);
                tc::tmem_wait_st();
#pragma unroll
                for (int ch = 4; ch < 8; ++ch) {
                    uint32_t v[32];
                    tc::tmem_ld32_wait(d_lane + (uint32_t)ch * 32u, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const __nv_bfloat162 b =
                            __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                        packed[(ch - 4) * 16 + j] = *reinterpret_cast<const uint32_t*>(&b);
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(sm.d_empty());
            // packed holds columns [c0, c0 + 128): the second half when wide, else the only one
            unsigned short* yc = reinterpret_cast<unsigned short*>(p.y) + n;
            auto store_pairs = [&](const uint32_t* pr, int c0, int npairs) {
                if (n >= p.N) return;
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    if (q < npairs) {
                        const int m = m0 + c0 + 2 * q;
                        if (m < p.M) yc[(int64_t)m * p.N] = (unsigned short)(pr[q] & 0xFFFFu);
                        if (m + 1 < p.M) yc[(int64_t)(m + 1) * p.N] = (unsigned short)(pr[q] >> 16);
                    }
                }
            };
            const int c0 = wide ? 128 : 0;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (c0 + h * 64 < p.BN) store_pairs(packed + 32 * h, c0 + h * 64, 32);
            if (wide) {   // the parked first half (every lane loads: the tensor-memory load is warp-wide)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[32];
                    tc::tmem_ld32_wait(d_lane + kParkCol + 32u * (uint32_t)h, v);
                    store_pairs(v, h * 64, 32);
                }
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// BF16 -> FP16, round to nearest even (exact for normal-range values).  With a
// per-input-channel multiplier xsc [K] (null: none), x_k * xsc_k is formed in
// FP32 and rounded to FP16 once.  The output has kvec = K / 8 vectors per row;
// the input rows have kxvec = kx / 8, and output channel k reads input channel
// k mod kx (kx = K, or K / 2 for a layer over x repeated twice).  Block 0 also
// clears ncnt arrival counters (the launch is stream-ordered before the
// layer kernels that count on them).
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* __restrict__ x, uint4* __restrict__ out,
                                                          int64_t nvec, const float4* __restrict__ xsc,
                                                          int64_t kvec, int64_t kxvec, uint32_t* __restrict__ cnt,
                                                          int ncnt) {
    // programmatic stream serialisation: the layer kernel may be scheduled at once (its prologue
    // touches no global memory); this grid reads and writes nothing before the previous grid on
    // the stream has completed
    tc::griddep_launch_dependents();
    tc::griddep_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (blockIdx.x == 0)   // the K-split arrival counters of the call's layer launches start at zero
        for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0u;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        int64_t src = i, kv = 0;                 // input vector; its channel vector (when needed)
        if (kxvec != kvec || xsc != nullptr) {
            const int64_t m = i / kvec;
            kv = i - m * kvec;
            kv -= kv >= kxvec ? kxvec : 0;
            src = m * kxvec + kv;
        }
        const uint4 v = x[src];
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = bf16lo_to_f32(in[j]);
            f[2 * j + 1] = bf16hi_to_f32(in[j]);
        }
        if (xsc != nullptr) {
            const float4 s0 = xsc[2 * kv], s1 = xsc[2 * kv + 1];
            f[0] *= s0.x; f[1] *= s0.y; f[2] *= s0.z; f[3] *= s0.w;
            f[4] *= s1.x; f[5] *= s1.y; f[6] *= s1.z; f[7] *= s1.w;
        }
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 h = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
            o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        out[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ---- host side -----------------------------------------------------------------

template <int G, bool W8>
cudaError_t launch_g(const CUtensorMap& tmx, const CUtensorMap& tmq, const GemmParams& p, int grid, size_t smem,
                     int dev, cudaStream_t stream) {
    // largest dynamic shared memory this instance is already allowed per device (a raise may
    // race with another thread's: both set the attribute, the larger value stays)
    static std::atomic<int> cached[kMaxDevices];
    int have = cached[dev].load(std::memory_order_relaxed);
    if ((int)smem > have) {
        const cudaError_t e =
            cudaFuncSetAttribute(gemm_kernel<G, W8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        while (have < (int)smem && !cached[dev].compare_exchange_weak(have, (int)smem)) {
        }
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<G, W8>, tmx, tmq, p);
}

// Converts x (BF16 [M, kx]) into the FP16 B operand x16 [M, K] and clears the
// call's ncnt arrival counters (see bf16_to_f16_kernel).
cudaError_t convert_x(const void* x, void* x16, int64_t M, int64_t K, int64_t kx, const float* xsc, int sms,
                      uint32_t* cnt, int ncnt, cudaStream_t stream) {
    const int64_t nvec = M * K / 8;
    int64_t blocks = (nvec + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256u);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, bf16_to_f16_kernel, static_cast<const uint4*>(x), static_cast<uint4*>(x16), nvec,
                              reinterpret_cast<const float4*>(xsc), (int64_t)(K / 8), (int64_t)(kx / 8), cnt, ncnt);
}

// K split.  Narrow tiles (BN <= 64: small M, where a tile's time is its
// weight streaming and expansion) are each cut along K into s ranges of the
// nst code stages, s chosen to minimise an estimate in stage times: the waves
// of pieces times their length, plus about 0.1 stage per piece for its
// partial and the final reduction.  Among estimates within 1 % of the best the
// smallest s wins.  Tiles that fill at most half the SMs always split; up to
// four waves of them split when the estimate gains at least 10 % (a partial
// wave evened out: 108 tiles in 4 ranges fill 148 SMs about three times).
// Wider tiles run whole, except the R tiles of a last wave that is at most
// half full (2R <= SMs) when K spans at least 16 code stages: those are cut in
// two, so that wave takes about half a tile plus the partials' write and
// reduction (a 128 x BN FP32 partial per piece) instead of a whole tile; when
// they are the only wave, in up to three (at least 8 stages each) as the SMs
// allow.
void choose_split(int T, int nst, int BN, int sms, GemmParams& p) {
    p.full = T;
    p.split = 0;
    p.parts = 1;
    if (BN > 64) {
        const int R = T % sms;
        if (R == 0 || 2 * R > sms || nst < 16) return;
        p.full = T - R;
        p.split = R;
        p.parts = T < sms ? std::max(2, std::min(std::min(sms / T, 3), nst / 8)) : 2;
        return;
    }
    if (T > 4 * sms || nst < 2) return;
    auto cost = [&](int c) {
        const int waves = (T * c + sms - 1) / sms;
        return waves * ((double)((nst + c - 1) / c) + 0.1) + (c > 1 ? 0.1 * c : 0.0);
    };
    const int smax = std::min(std::min(nst, 16), std::max(1, 6 * sms / T));   // at most 6 pieces per SM
    double best = cost(1);
    for (int c = 2; c <= smax; ++c) best = std::min(best, cost(c));
    int s = 1;
    for (int c = 1; c <= smax; ++c)
        if (cost(c) <= best * 1.01) {
            s = c;
            break;
        }
    if (s > 1 && (2 * T <= sms || cost(s) <= 0.9 * cost(1))) {
        p.full = 0;
        p.split = T;
        p.parts = s;
    }
}

// Everything about one matrix's launch but its pointers.
struct GemmPlan {
    GemmParams p;
    int grid;
    size_t smem;
    size_t ws_bytes;    // K-split partials (0: no split)
};

bool plan_gemm(int64_t M, int64_t N, int64_t K, int G, bool w8, const DeviceInfo& di, bool allow_split,
               GemmPlan& pl) {
    GemmParams& p = pl.p;
    p = GemmParams{};
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.BN = gemm_tile_n(M);
    p.lds = (int)scales_ld(K, G);
    p.ldz = (int)(w8 ? zeros8_ld(K, G) : zeros_ld(K, G));
    p.ngroups = (int)(K / G);
    p.mtiles = (int)((M + p.BN - 1) / p.BN);
    const int64_t tiles = ((N + kBM - 1) / kBM) * p.mtiles;
    if (tiles > (1 << 24)) return false;
    p.tiles = (int)tiles;
    p.nk64 = (int)((K + 63) / 64);
    p.subs = w8 ? 2 : 4;
    p.nstage = (p.nk64 + p.subs - 1) / p.subs;
    if (allow_split) choose_split(p.tiles, p.nstage, p.BN, di.sms, p);
    else choose_split(p.tiles, 1, p.BN, di.sms, p);           // whole tiles only
    p.units = p.full + p.split * p.parts;
    pl.grid = p.units < di.sms ? p.units : di.sms;
    pl.smem = gemm_smem_bytes(p.BN);
    pl.ws_bytes = p.split ? (size_t)p.split * p.parts * p.BN * kBM * 4 : 0;
    p.spin_limit = wait_limit();
    return pl.smem <= di.smem_optin;
}

// Launches one matrix: the map of its codes, then the kernel.  ws: the call's
// K-split partials; cnt: this matrix's arrival counters (cleared by the conversion).
cudaError_t launch_one(const CUtensorMap& tmx, const GemvMat& mat, const GemmPlan& pl, int G, bool w8, void* ws,
                       uint32_t* cnt, int dev, cudaStream_t stream) {
    const uint64_t ldq = (uint64_t)(w8 ? pl.p.K / 4 : pl.p.K / 8);
    CUtensorMap tmq;
    if (!encode_tmap_2d(&tmq, CU_TENSOR_MAP_DATA_TYPE_UINT32, mat.q, ldq, (uint64_t)pl.p.N, ldq * 4, 32, kBM, dev))
        return cudaErrorInvalidValue;
    GemmParams p = pl.p;
    p.withhold = take_withhold(2) ? 1 : 0;
    p.s = static_cast<const unsigned short*>(mat.s);
    p.z = mat.z;
    p.y = mat.y;
    p.ws = static_cast<float*>(ws);
    p.cnt = cnt;
    if (w8) {
        switch (G) {
            case 32: return launch_g<32, true>(tmx, tmq, p, pl.grid, pl.smem, dev, stream);
            case 64: return launch_g<64, true>(tmx, tmq, p, pl.grid, pl.smem, dev, stream);
            case 128: return launch_g<128, true>(tmx, tmq, p, pl.grid, pl.smem, dev, stream);
            case 256: return launch_g<256, true>(tmx, tmq, p, pl.grid, pl.smem, dev, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (G) {
        case 32: return launch_g<32, false>(tmx, tmq, p, pl.grid, pl.smem, dev, stream);
        case 64: return launch_g<64, false>(tmx, tmq, p, pl.grid, pl.smem, dev, stream);
        case 128: return launch_g<128, false>(tmx, tmq, p, pl.grid, pl.smem, dev, stream);
        case 256: return launch_g<256, false>(tmx, tmq, p, pl.grid, pl.smem, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

bool encode_x_map(CUtensorMap* tmx, const void* x16, int64_t M, int64_t K, int BN, int dev) {
    return encode_tmap_2d(tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64,
                          (uint32_t)BN, dev);
}

}  // namespace

int gemm_tile_n(int64_t M) { return M >= 256 ? 256 : (int)((M + 31) / 32 * 32); }

// The FP16 copy of x, the K-split partials and the arrival counters are taken
// from the device's current memory pool with one stream-ordered allocation and
// freed on the stream after the call's kernels.  The library keeps no pool or
// cache of device memory of its own: what stays reserved between calls is
// that pool's policy (its release threshold), which belongs to the
// application.
cudaError_t launch_gemm(const void* x, const GemvMat* mats, int nmat, int64_t M, int64_t N, int64_t K, int G,
                        cudaStream_t stream, const float* xsc, int64_t kx, bool yf32, bool w8) {
    if (kx == 0) kx = K;
    if (kx != K && (kx * 2 != K || kx % 8 != 0)) return cudaErrorInvalidValue;
    if (nmat < 1 || nmat > kMaxMat) return cudaErrorInvalidValue;
    if (M < 1 || K < 1) return cudaSuccess;
    if (M > INT32_MAX || K > INT32_MAX || K % 32 != 0) return cudaErrorInvalidValue;
    if (!tmap_encoder_available()) return cudaErrorNotSupported;
    DeviceInfo di;
    cudaError_t e = current_device(di);
    if (e != cudaSuccess) return e;
    GemmPlan pl[kMaxMat];
    size_t ws_bytes = 0;
    int ncnt = 0, cnt0[kMaxMat];
    for (int i = 0; i < nmat; ++i) {
        const int64_t Ni = mats[i].n > 0 ? mats[i].n : N;     // every matrix's rows: its own n, else N
        if (Ni < 1 || Ni > INT32_MAX || !plan_gemm(M, Ni, K, G, w8, di, true, pl[i])) return cudaErrorInvalidValue;
        pl[i].p.yf32 = yf32 ? 1 : 0;
        ws_bytes = std::max(ws_bytes, pl[i].ws_bytes);        // the launches run one after another
        cnt0[i] = ncnt;
        ncnt += pl[i].p.split;
    }
    const size_t xbytes = ((size_t)M * (size_t)K * 2 + 255) / 256 * 256;
    const size_t wbytes = (ws_bytes + 255) / 256 * 256;
    void* buf = nullptr;
    if ((e = cudaMallocAsync(&buf, xbytes + wbytes + (size_t)ncnt * 4, stream)) != cudaSuccess) return e;
    uint8_t* ws = static_cast<uint8_t*>(buf) + xbytes;
    uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + wbytes);
    CUtensorMap tmx;
    if (!encode_x_map(&tmx, buf, M, K, pl[0].p.BN, di.dev)) e = cudaErrorInvalidValue;
    if (e == cudaSuccess) e = convert_x(x, buf, M, K, kx, xsc, di.sms, cnt, ncnt, stream);
    for (int i = 0; i < nmat && e == cudaSuccess; ++i)
        e = launch_one(tmx, mats[i], pl[i], G, w8, ws, cnt + cnt0[i], di.dev, stream);
    const cudaError_t ef = cudaFreeAsync(buf, stream);
    return e != cudaSuccess ? e : ef;
}


// ---- tensor-core path without any allocation ----------------------------------
//
// Some callers cannot allocate device memory while they run the layer: an
// engine that reserves its whole memory budget at start-up and forbids any
// later allocation, so that a running model never fails half-way on an
// out-of-memory error.  For them the FP16 copy of x lives in one file-scope
// device array of fixed size instead of a stream-ordered allocation, and the
// work is never split along K (a split needs a workspace).  Every GPU that
// loads the library holds this array until the process exits.  All
// calls share it, so two calls whose kernels overlap on the GPU (different
// streams, no ordering between them) race on its contents.
constexpr size_t kNoAllocScratchBytes = (size_t)W4A16_NOALLOC_MAX_X_ELEMS * 2;
static __device__ __align__(256) uint8_t g_noalloc_x16[kNoAllocScratchBytes];

// Device address of the array, looked up once per device with that device
// current (in host code the symbol itself is only a host-side stand-in).
cudaError_t noalloc_scratch(int dev, void** ptr) {
    static void* addr[kMaxDevices] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_x16);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_gemm_noalloc(const void* x, const GemvMat& mat, int64_t M, int64_t N, int64_t K, int G,
                                cudaStream_t stream) {
    if (M < 1 || N < 1 || K < 1) return cudaSuccess;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX || K % 32 != 0) return cudaErrorInvalidValue;
    if (M * K > (int64_t)W4A16_NOALLOC_MAX_X_ELEMS) return cudaErrorNotSupported;
    if (!tmap_encoder_available()) return cudaErrorNotSupported;
    DeviceInfo di;
    cudaError_t e = current_device(di);
    if (e != cudaSuccess) return e;
    void* x16 = nullptr;
    if ((e = noalloc_scratch(di.dev, &x16)) != cudaSuccess) return e;
    GemmPlan pl;
    CUtensorMap tmx;
    if (!plan_gemm(M, N, K, G, false, di, false, pl) || !encode_x_map(&tmx, x16, M, K, pl.p.BN, di.dev))
        return cudaErrorInvalidValue;
    // every element of the array this call reads is written first by the conversion
    if ((e = convert_x(x, x16, M, K, K, nullptr, di.sms, nullptr, 0, stream)) != cudaSuccess) return e;
    return launch_one(tmx, mat, pl, G, false, nullptr, nullptr, di.dev, stream);
}

cudaError_t read_and_clear_status(uint32_t* word) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_status_word, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0;
    if ((e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(uint32_t))) != cudaSuccess) return e;
    uint32_t gw = 0;
    e = gemv_take_status(&gw);
    *word |= gw;
    return e;
}

}  // namespace w4a16
