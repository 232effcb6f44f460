// gemv.cu -- decode path of the W4A16 linear layer (up to 16 activation rows;
// the library dispatches M <= 8 here, and M <= 16 where the kernel runs with
// all its warps).
//
// Decode rereads every weight for each generated token with little work per
// weight, so this kernel is bound by HBM bandwidth on the packed weights
// (klaylearn.com glossary "Weight-Only Quantisation", FAQ "Why is it
// especially useful for decode?"; zhuai.tech "Quantization Is Not a Zip
// File", section 2 "Moving fewer bytes can make decode faster": packed
// weights decoded block by block straight into the accumulation).
//
// Geometry.  Each weight row's K codes are cut into P equal segments, and a
// virtual row is one (row, segment) pair: the packed matrix [N, K/8] words is
// read as [N*P, K/(8P)].  A tile is 16 virtual rows = R = 16/P weight rows;
// the 16 rows of a warp MMA m16n8k16 are the tile's virtual rows, and the MMA's
// B columns hold (segment, group parity, activation row) triples of x (at most
// 8 per column block; two blocks for M > 8).  So one MMA advances all segments
// of R rows at once, and only the diagonal (segment of the row == segment of
// the column) of D is kept.  H group parities let one column collect every
// H-th group, so the scale/zero correction runs once per block of H groups.
// At M = 1 the columns are (parity, segment) pairs, P is a template constant,
// and each lane corrects only the one value per row it holds.
//
// Data path.  One CTA per SM (16 warps, or 12 when registers or shared memory
// are short; two CTAs of 8 warps for small layers) takes a balanced contiguous
// range of tiles; its warps take
// contiguous runs of 256-code chunks, balanced to the chunk.  Each warp
// streams its run with TMA (16 virtual rows x 128 bytes per chunk, 128-byte
// swizzle) into a private ring of shared-memory slots; a slot holds a unit of
// two chunks of one tile under one barrier (one chunk where a tile or a run
// ends).  Per word of 8 codes the lane makes four FP16 pairs with one shift
// and four LOP3s: the FP16 exponents of 1024 (ulp 1) and 64 (ulp 1/16) turn a
// nibble at bits 0..3 or 4..7 of a half into the exact values 1024 + q and
// 64 + q.  These meet x (converted to FP16 once per CTA and staged in shared
// memory in fragment order) in the warp MMA with FP32 accumulation.  At the end
// of each block the lane subtracts the staged sum of (1024 or 64) * x plus
// z * sum x, scales by s and accumulates; at the end of a tile the diagonal is
// reduced over segments and parities.  Warps that share a tile leave partial
// sums in fixed slots, added in a fixed order at the end, so results are
// deterministic.  Every output is rounded to BF16 once.
//
// Super-block mode (KQ).  Weights in the Q4_K-style layout (256-channel
// super-blocks of 8 sub-blocks of 32; sub-block j reconstructs as
// d*sc_j*q - dmin*m_j with 6-bit sc_j, m_j and FP16 d, dmin: zhuai.tech
// "Quantization Is Not a Zip File", section 3, K-quants row of the GGUF names
// table) run through the same path with G = 32: a 256-code chunk of a virtual
// row is exactly one super-block, whose 16-byte record takes the place of the
// scale and zero rows.  The block-end correction becomes
// acc += s*(D - E) - mn*X with s = d*sc_j and mn = dmin*m_j, both exact in FP32.
//
// 8-bit mode (W8).  Codes four per word with 8-bit zero points run as a 4-bit
// layer of 2K virtual channels and groups of 2G: both nibbles of a code are
// expanded against the exponent of 1024 and x is staged twice (see
// expand_codes8_f16), so the MMA sums x (2048 + b) exactly.
//
// Metadata.  At G >= 64 the CTA's scale and zero rows stay in shared memory for
// the whole launch.  At G = 32 (and for super-blocks) each ring unit also
// brings the scales (records) of its two chunks for the tile's 16 virtual rows
// by one more TMA box, and only the zero rows stay resident: long rows of fine
// groups would otherwise leave room for one unit per warp.
//
// Prologue.  The launch uses programmatic stream serialisation: a CTA lets the
// next launch be scheduled on entry and waits for the previous grid before it
// reads global memory.  One thread then bulk-copies the CTA's resident
// metadata rows while every warp loads its first x items; the weight ring
// starts once the rows have landed (copies issued together complete in no
// particular order), and x is staged while the first units are in flight.
// Small layers run an 8-warp instance that leaves room for a second CTA per
// SM; its CTAs ask L2 for their rows before the grid-dependency wait.
//
// K split.  On long rows the staged x (M * K FP16) would leave the weight
// rings too little shared memory (M >= 2); a cluster of two CTAs on two SMs
// then takes each tile range, each CTA streaming and staging half of every
// row's chunks, and the two add their partial sums through distributed shared
// memory (see gemv_kernel's KS).
//
// Instances cover one matrix, a pair (the dual call) or up to four sharing x.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "unpack.cuh"

namespace w4a16 {

// Per-device word the decode kernel sets when a bounded wait gives up (read
// and cleared together with the tensor-core path's word).
__device__ uint32_t g_gemv_status = 0;

namespace {

// Warps per CTA: 16 where the kernel instance fits 128 registers per thread
// (one activation-row block, G >= 64), else 12.
__host__ __device__ constexpr int cta_warps(int NB, int G) { return NB == 1 && G >= 64 ? 16 : 12; }
constexpr int kBoxBytes = 2048;           // one TMA box: 16 virtual rows x 128 bytes (256 codes)
constexpr int kUnitBytes = 2 * kBoxBytes;  // a ring slot: a unit of up to two consecutive chunks of a tile
constexpr int kSlots = 4;                 // partial-sum slots per output (warps sharing a tile)
constexpr int kMetaBytes = 512;           // streamed metadata of a unit: 16 virtual rows x 16 halves
// Small layers (a few tens of KB of weights per SM) are latency bound: a launch spends about
// 4 us in its prologue and on its first units' latency against 1-2 us of streaming.  Their
// instance runs 8 warps with at most half the shared memory, so two CTAs fit on an SM: the
// next launch's CTAs can become resident while this one runs (programmatic stream
// serialisation) and ask L2 for their weights before their grid-dependency wait.
constexpr int kDuoWarps = 8;
constexpr size_t kDuoSmem = 110 * 1024;
// Weight formats the decode kernel reads.  kFmt8: 8-bit codes four per word
// with 8-bit zero points; the kernel runs them as a 4-bit layer of 2K virtual
// channels and groups of 2G (each 8-bit code is two nibbles), expanding both
// nibbles against the exponent of 1024 and staging every x value twice (see
// expand_codes8_f16), so the MMA sums x (2048 + b) exactly.
constexpr int kFmt4 = 0, kFmtQ4K = 1, kFmt8 = 2;
constexpr uint32_t kStatusGemv = 1u << 8;
constexpr uint32_t kStatusGemvDrain = 1u << 9;

// MMA row i (< 8) of a warp reads virtual row sigma(i) = i/2 + 4*(i%2) of the
// tile (and row i + 8 reads sigma(i) + 8): lanes that share a shared-memory
// phase then hit swizzle patterns that differ in bit 2, so 128-bit code loads
// are free of bank conflicts.
__device__ __forceinline__ int sigma8(int i) { return (i >> 1) + ((i & 1) << 2); }

struct GemvParams {
    const __nv_bfloat16* x;                // [M, K]
    const float* xsc;                      // per-input-channel multiplier of x [K], or null
    int kx;                                // row length of x: channel k reads x[k mod kx] (kx = K or K/2)
    // per matrix (up to kMaxMat sharing x): FP16 scales [n, lds] (KQ: super-block records, 8
    // halves each), zeros [n, ldz] (KQ: unused, ldz = 0), output [M, n] BF16 (or FP32 when yf32)
    const uint32_t* q[kMaxMat];            // packed codes (read through the tensor maps; the small-layer
                                           // instance also asks L2 for them ahead of time)
    const unsigned short* s[kMaxMat];
    const uint32_t* z[kMaxMat];
    void* y[kMaxMat];
    int n[kMaxMat];                        // rows (outputs) of each matrix
    int tstart[kMaxMat + 1];               // first tile of each matrix; total_tiles from nmat on
    int yf32;                              // 1: FP32 outputs (no BF16 rounding)
    int M, K, G;
    int P, R, cols, xcols;                 // segments, weight rows per tile, B columns used (P*H*M),
                                           // staged x columns (P*M)
    int Ks, C, ngs, ng;                    // codes per segment padded to whole chunks (C of 256), groups
                                           // per padded segment, groups per row
    int lds, ldz;
    int total_tiles;
    int nw;                                // warps in the CTA
    int warps;                             // warps that take units (<= nw)
    int nst;                               // unit slots per warp ring (power of two)
    int pf;                                // chunks ahead of the ring each warp asks L2 for (0: none)
    int mstream;                           // 1: scales (super-block records) stream with the units
    int duo;                               // 1: the small-layer instance (two CTAs per SM, see kDuoWarps)
    int rows_cap;                          // weight rows per CTA the partial buffer holds
    long long spin_limit;                  // cycles a bounded wait spins before it gives up
    int withhold;                          // test hook: warp 0 of CTA 0 never issues its first unit
    int ks;                                // 1: K split across the two CTAs of a cluster (see gemv_kernel)
    int Ct, kc1;                           // KS: chunks per row; rank 0 streams chunks [0, kc1) of each
                                           // tile, rank 1 [kc1, Ct); C = kc1 sizes the staged x
    int nslot;                             // KS: partial-sum slots per output (<= kSlots; the most warps
                                           // sharing a tile), which sizes the partial buffer
};

struct Layout {
    uint32_t ring, mring, xs, zero, exs, ms, mz, part, red, bars;
    uint32_t total;
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// M = 1 with P >= 2 segments: the specialised kernel (its B columns are (parity, segment)
// pairs and it keeps one useful value per row; see gemv_kernel).
__host__ __device__ inline bool m1_kernel(const GemvParams& p) { return p.M == 1 && p.P >= 2; }

__host__ __device__ inline Layout make_layout(const GemvParams& p, int nb, int H) {
    const bool m1 = m1_kernel(p);
    Layout L;
    uint32_t off = 0;
    L.ring = off;
    off += (uint32_t)(p.nw * p.nst * kUnitBytes);
    L.mring = off;                                        // streamed metadata, one area per ring slot
    off += p.mstream ? (uint32_t)(p.nw * p.nst * kMetaBytes) : 0u;
    L.xs = off;
    off += align_up((uint32_t)p.xcols * (uint32_t)p.Ks * 2u, 16);        // xcols x Ks FP16 (whole chunks)
    L.zero = off;                                         // zeros read by idle B columns: one 16-byte
    off += m1 ? 8u * (uint32_t)p.xcols * 64u : 16u;        // block, or (M = 1) a chunk's 8 word steps of x
    L.exs = off;
    off += align_up((uint32_t)(p.ngs / H) * 8u * (uint32_t)nb * 8u, 16);
    L.ms = off;                                           // resident scale rows (or records) unless streamed
    off += p.mstream ? 0u : align_up((uint32_t)p.rows_cap * (uint32_t)p.lds * 2u, 16);
    L.mz = off;
    off += align_up((uint32_t)p.rows_cap * (uint32_t)p.ldz * 4u, 16);
    L.part = off;
    off += align_up((uint32_t)p.rows_cap * (uint32_t)p.M * (uint32_t)(p.ks ? p.nslot : kSlots) * 4u, 16);
    L.red = off;
    off += (uint32_t)p.nw * 16u * (m1 ? (uint32_t)H : 8u * (uint32_t)nb) * 4u;
    L.bars = off;
    off += (uint32_t)p.nw * (uint32_t)p.nst * 8u + 8u;    // ring barriers, then the prologue copies' barrier
    L.total = off;
    return L;
}

// Warp MMA m16n8k16, FP16 inputs, FP32 accumulate (D = A*B + C).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with C = 0 (starts a fresh accumulation).
__device__ __forceinline__ void mma_f16_c0(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// Matrix that tile tau belongs to (tiles are numbered matrix after matrix; an
// instance takes up to NM matrices).
template <int NM>
__device__ __forceinline__ int mat_of(const GemvParams& p, int tau) {
    int m = 0;
#pragma unroll
    for (int i = 1; i < NM; ++i) m += tau >= p.tstart[i];
    return m;
}

// The code maps of up to NM matrices, one kernel parameter; with MS also the
// maps of their scale rows (or super-block records) viewed per virtual row.
template <int NM, bool MS>
struct CodeMaps {
    CUtensorMap m[NM];
    CUtensorMap s[NM];
};
template <int NM>
struct CodeMaps<NM, false> {
    CUtensorMap m[NM];
};

// Instances whose scale rows (or super-block records) stream with the weight units instead of
// staying resident: groups of 32, where a row's metadata is long (0.0625-0.078 bytes per code,
// 100 KB per CTA at K = 28672) and would crowd the weight ring out of shared memory.
__host__ __device__ constexpr bool meta_streamed(int G) { return G == 32; }

// Thread-block cluster helpers (the K split): this CTA's rank in its cluster,
// a barrier of all threads of the cluster (release / acquire, so shared-memory
// writes before it are visible to the peer after it), the peer's address of a
// shared-memory location, and a load from there.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Bounded wait on a barrier phase (gives up after `limit` cycles); the thread
// sleeps between polls.
__device__ __forceinline__ bool gemv_wait(uint32_t bar, uint32_t parity, long long limit) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!tc::mbar_try_wait_sleep(bar, parity, 100000u)) {
        if (clock64() - t0 > limit) {
            atomicOr(&g_gemv_status, kStatusGemv);
            return false;
        }
    }
    return true;
}

// M1: one activation row with P >= 2 segments.  The B columns are then
// (parity, segment) pairs and each lane holds at most one useful D value per
// row, so the block-end correction is done once per row on that value only.
// NM: matrices the instance takes (1, 2, or 4 for three or four).
// KS: the K split.  Where M * K of x would crowd out the weight ring (long
// rows, M >= 2), each tile range is taken by a cluster of two
// CTAs on two SMs: rank r streams and stages only its half of the chunks of
// every row, and at the end the two CTAs add both ranks' partial sums, read
// through distributed shared memory, in a fixed order.
template <int NB, int G, int H, bool M1, int PT, int FMT, int NM, bool DUO = false, bool KS = false>
__global__ void __launch_bounds__(DUO ? kDuoWarps * 32 : cta_warps(NB, G) * 32, DUO ? 2 : 1)
    gemv_kernel(const __grid_constant__ CodeMaps<NM, meta_streamed(G)> tm, const GemvParams p) {
    constexpr int V = G >= 128 ? 4 : G / 32;      // words per lane per code load
    constexpr int GPC = 256 / G;                  // groups per chunk (H divides it)
    constexpr int WSG = G / 32;                   // word steps per group
    const int kWarps = p.nw;                      // warps launched (at most the launch bound)
    const int P = PT > 0 ? PT : p.P;            // segments per row (a template constant at M = 1)
    const int R = 16 / P;                         // weight rows per tile
    const int kThreads = kWarps * 32;
    static_assert(GPC % H == 0, "a block of H groups lies inside one chunk");
    constexpr bool KQ = FMT == kFmtQ4K;          // super-block records in place of scales and zeros
    constexpr bool W8 = FMT == kFmt8;            // 8-bit codes, four per word (a virtual 4-bit layer of 2K)
    static_assert(!KQ || G == 32, "a super-block is one chunk of 8 sub-blocks of 32");
    // MS: each unit also brings the scales (super-block records) of its two chunks for the tile's
    // 16 virtual rows, 32 bytes per row (kMetaBytes), into a per-slot area; only the zero rows
    // (4-bit) stay resident
    constexpr bool MS = meta_streamed(G);
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base; derived by pointer arithmetic on the shared array so
    // the compiler keeps every access below in the shared address space
    uint8_t* base = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    const Layout L = make_layout(p, NB, H);
    const uint32_t sbase = tc::smem_u32(base);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;

    // ---- this CTA's tiles and this warp's run of chunks -------------------------
    const int T = p.total_tiles;
    uint32_t crank = 0, cid = blockIdx.x, ncl = gridDim.x;    // KS: rank in the cluster, cluster, clusters
    if constexpr (KS) {
        crank = cluster_ctarank();
        cid = blockIdx.x >> 1;
        ncl = gridDim.x >> 1;
    }
    const int Cw = KS ? (crank == 0 ? p.kc1 : p.Ct - p.kc1) : p.C;   // chunks per tile this CTA streams
    const int kc0 = KS ? (int)crank * p.kc1 : 0;                      // the first of them in the row
    const int NSL = KS ? p.nslot : kSlots;                            // partial-sum slots per output
    const int tile0 = (int)((cid * (uint32_t)T) / ncl);        // T * grid < 2^32 (host check)
    const int tile1 = (int)(((cid + 1) * (uint32_t)T) / ncl);
    const int tc_ = tile1 - tile0;
    const int chunks = tc_ * Cw;                  // < 2^26 (host check), so products below fit 32 bits
    const bool active = warp < p.warps;
    const int ch0 = active ? (warp * chunks) / p.warps : 0;        // this warp's chunks [ch0, ch1)
    const int ch1 = active ? ((warp + 1) * chunks) / p.warps : 0;
    const int nsl = p.nst;                        // unit slots in this warp's ring (power of two)
    const uint32_t ring = sbase + L.ring + (uint32_t)(warp * nsl * kUnitBytes);
    const uint32_t mring = sbase + L.mring + (uint32_t)(warp * nsl * kMetaBytes);   // MS only
    const uint32_t bar0 = sbase + L.bars + (uint32_t)(warp * nsl * 8);

    // ---- stream: lane 0 of each warp keeps its ring of units filled -----------
    // A unit is two consecutive chunks of one tile under one barrier, or one chunk where the
    // tile or the run ends; producer and consumer walk the same sequence.
    int it_n = 0, it_ch = ch0, it_tl = 0, it_c = 0;   // units issued; next chunk, its tile and chunk in it
    if (active) {
        it_tl = ch0 / Cw;
        it_c = ch0 - it_tl * Cw;
    }
    // test hook: warp 0 of CTA 0 never issues its first unit, so its wait on it runs out
    const bool withhold = p.withhold && blockIdx.x == 0 && warp == 0;
    // copy = false (the test hook only) advances past a unit without issuing its copies
    // With a ring of one unit per warp (shared memory taken by long metadata rows) the copies in
    // flight do not cover the memory latency; each warp then also asks L2 for its next p.pf chunks
    // (boxes not yet in the ring, inside the warp's run) so that the ring's copies hit L2.  Only
    // groups of 32 (and super-blocks) have rows that long; the other instances leave the code
    // out, as its mere presence in the refill path costs them 1-2 %.
    constexpr bool kPf = G == 32;
    int pf_ch = it_ch, pf_tl = it_tl, pf_c = it_c;     // next chunk to prefetch
    auto prefetch_upto = [&](int lim) {
        lim = min(lim, ch1);
        for (; pf_ch < lim; ++pf_ch) {
            if (pf_ch >= it_ch) {
                const int tau = tile0 + pf_tl;
                const int mat = mat_of<NM>(p, tau);
                const void* map = &tm.m[0];
#pragma unroll
                for (int i = 1; i < NM; ++i)
                    if (mat == i) map = &tm.m[i];
                tc::tma_prefetch_2d(map, (kc0 + pf_c) * 32, (tau - p.tstart[mat]) * 16);
            }
            if (++pf_c == Cw) {
                pf_c = 0;
                ++pf_tl;
            }
        }
    };
    auto issue_next = [&](bool copy) {
        const int tau = tile0 + it_tl;
        const int mat = mat_of<NM>(p, tau);
        const int tile = tau - p.tstart[mat];
        const uint32_t slot = (uint32_t)(it_n & (nsl - 1));
        const uint32_t bar = bar0 + 8u * slot;
        const bool two = it_c + 1 < Cw && it_ch + 1 < ch1;
        if (copy) {
            tc::mbar_arrive_expect_tx(bar, (uint32_t)(two ? 2 * kBoxBytes : kBoxBytes) + (MS ? kMetaBytes : 0u));
            const void* map = &tm.m[0];
#pragma unroll
            for (int i = 1; i < NM; ++i)
                if (mat == i) map = &tm.m[i];
            tc::tma_load_2d(ring + slot * (uint32_t)kUnitBytes, map, (kc0 + it_c) * 32, tile * 16, bar);
            if (two)
                tc::tma_load_2d(ring + slot * (uint32_t)kUnitBytes + kBoxBytes, map, (kc0 + it_c + 1) * 32, tile * 16,
                                bar);
            if constexpr (MS) {   // the scales of chunks it_c, it_c + 1 (a box of 16 halves per virtual row)
                const void* smap = &tm.s[0];
#pragma unroll
                for (int i = 1; i < NM; ++i)
                    if (mat == i) smap = &tm.s[i];
                tc::tma_load_2d(mring + slot * (uint32_t)kMetaBytes, smap, (kc0 + it_c) * 8, tile * 16, bar);
            }
        }
        const int n = two ? 2 : 1;
        ++it_n;
        it_ch += n;
        it_c += n;
        if (it_c == Cw) {
            it_c = 0;
            ++it_tl;
        }
        if constexpr (kPf) {
            if (p.pf && copy) prefetch_upto(it_ch + p.pf);
        }
    };

    // ---- prologue ---------------------------------------------------------------------
    // One thread bulk-copies this CTA's scale and zero rows (contiguous in each matrix);
    // meanwhile every warp requests its first x items.  Once the rows have landed the
    // weight ring starts, and x is staged while its first units are in flight (copies
    // issued together complete in no particular order, so starting the ring earlier would
    // hold the small inputs behind its bytes).
    // Launched with programmatic stream serialisation: the next launch on the stream may be
    // scheduled at once (its CTAs take SMs as this grid's CTAs exit), and this grid reads no
    // global memory before the previous grid on the stream has completed.
    tc::griddep_launch_dependents();
    if constexpr (DUO) {
        if (tid == 0) {
            // the CTA's code, scale and zero rows into L2 now, while the previous grid may still be
            // running: a prefetch returns nothing to the program and L2 is the point of coherence, so
            // this reads nothing before the grid-dependency wait below
#pragma unroll 1
            for (int i = 0; i < NM; ++i) {
                const int a = max(tile0, p.tstart[i]), b = min(tile1, p.tstart[i + 1]);
                if (b <= a) continue;
                const int64_t r0 = (int64_t)(a - p.tstart[i]) * R;
                const int64_t rows = min((int64_t)(b - a) * R, (int64_t)p.n[i] - r0);
                if (rows <= 0) continue;
                const uint8_t* cq = reinterpret_cast<const uint8_t*>(p.q[i]) + r0 * (p.K / 2);
                for (int64_t off = 0, tot = rows * (p.K / 2); off < tot; off += 1 << 16)
                    tc::prefetch_l2(cq + off, (uint32_t)(tot - off < (1 << 16) ? tot - off : (1 << 16)));
                tc::prefetch_l2(p.s[i] + r0 * p.lds, (uint32_t)(rows * p.lds * 2));
                tc::prefetch_l2(p.z[i] + r0 * p.ldz, (uint32_t)(rows * p.ldz * 4));
            }
        }
    }
    const uint32_t pbar = sbase + L.bars + 8u * (uint32_t)(kWarps * nsl);
    bool pro_ok = true;                           // the prologue's copies landed (warp-uniform)
    if (tid == 0) {
        for (int i = 0; i < kWarps * nsl; ++i) tc::mbar_init(sbase + L.bars + 8u * i, 1);
        tc::mbar_init(pbar, 1);
        tc::fence_barrier_init();
    }
    tc::griddep_wait();
    __syncthreads();
    {
        // local rows follow the CTA's tiles: the part of matrix i is the tiles [a_i, b_i) of the
        // CTA's range, local rows [(a_i - tile0) R, (b_i - tile0) R); its rows below the matrix's
        // n are bulk-copied (they are contiguous in the matrix), the rest zero-filled below
        const uint32_t sbytes = MS ? 0u : (uint32_t)p.lds * 2u, zbytes = (uint32_t)p.ldz * 4u;   // per row
        const uint32_t ms = sbase + L.ms, mz = sbase + L.mz;
        int cl[NM], cc[NM];                            // local first row and rows copied, per matrix
        int gs[NM + 1], gn[NM + 1];                    // rows left to zero-fill: first, count
        int copied = 0, gaps = 0;
#pragma unroll
        for (int i = 0; i < NM; ++i) {
            const int a = max(tile0, p.tstart[i]), b = min(tile1, p.tstart[i + 1]);
            cl[i] = (a - tile0) * R;
            cc[i] = b > a ? max(0, min((b - a) * R, p.n[i] - (a - p.tstart[i]) * R)) : 0;
            gs[i] = cl[i] + cc[i];
            gn[i] = b > a ? (b - a) * R - cc[i] : 0;      // rows of the part past the matrix's n
            copied += cc[i];
            gaps += gn[i];
        }
        gs[NM] = tc_ * R;                                // rows past the CTA's tiles
        gn[NM] = p.rows_cap - tc_ * R;
        gaps += gn[NM];
        if (tid == 0) {
            tc::mbar_arrive_expect_tx(pbar, (uint32_t)copied * (sbytes + zbytes));
#pragma unroll
            for (int i = 0; i < NM; ++i) {
                if (cc[i] <= 0) continue;
                const int64_t r0 = (int64_t)(max(tile0, p.tstart[i]) - p.tstart[i]) * R;    // first row
                if (!MS) tc::bulk_load(ms + (uint32_t)cl[i] * sbytes, p.s[i] + r0 * p.lds, (uint32_t)cc[i] * sbytes, pbar);
                if (!KQ) tc::bulk_load(mz + (uint32_t)cl[i] * zbytes, p.z[i] + r0 * p.ldz, (uint32_t)cc[i] * zbytes, pbar);
            }
        }

        // x: work item of a warp = 32 consecutive words (one per lane) of one staged column
        // xc = (segment pseg, activation row m) and 32-word block c; the warp's items are
        // it = warp + k * kWarps, k = 0, 1, ..., stepped through without division.  Words of one
        // group sit in consecutive lanes, so the group sums are warp shuffles.  A batch of XB
        // items' loads is in flight before any is used.
        const int xcols = p.xcols, M = p.M, C = p.C;
        uint4* xs = reinterpret_cast<uint4*>(base + L.xs);
        float2* exs = reinterpret_cast<float2*>(base + L.exs);
        const int kseg = p.K / P;                        // real codes per segment
        const int kbase = kc0 * 256;                    // KS: first channel of this CTA's window
        constexpr int GW = G / 8;                          // words per group
        constexpr int XB = 8;                              // items per batch
        const int dxc = kWarps / C, dc = kWarps - dxc * C;                 // item step as (column, block)
        const uint32_t minv = (65536u + (uint32_t)M - 1u) / (uint32_t)M;  // xc / M = (xc * minv) >> 16 (xc < 2^12)
        int xc_n = warp / C, c_n = warp - (warp / C) * C;  // next item of this warp
        int bxc[XB], bc[XB];                               // the batch's items
        uint4 vv[XB];
        auto x_load = [&]() {                              // next batch: positions, then loads
#pragma unroll
            for (int j = 0; j < XB; ++j) {
                bxc[j] = xc_n;
                bc[j] = c_n;
                c_n += dc;
                xc_n += dxc;
                if (c_n >= C) {
                    c_n -= C;
                    ++xc_n;
                }
            }
#pragma unroll
            for (int j = 0; j < XB; ++j) {
                vv[j] = make_uint4(0u, 0u, 0u, 0u);
                const int pseg = (int)(((uint32_t)bxc[j] * minv) >> 16), m = bxc[j] - pseg * M;
                const int wseg = bc[j] * 32 + lane;
                if (bxc[j] < xcols && kbase + wseg * 8 < kseg) {
                    int kk = pseg * kseg + kbase + wseg * 8;       // channel of the layer (< 2 kx)
                    if constexpr (W8) {                    // the word's four real channels
                        const uint2 h = *reinterpret_cast<const uint2*>(p.x + (int64_t)m * p.kx + kk / 2);
                        vv[j] = make_uint4(h.x, h.y, 0u, 0u);
                    } else {
                        kk -= kk >= p.kx ? p.kx : 0;
                        vv[j] = *reinterpret_cast<const uint4*>(p.x + (int64_t)m * p.kx + kk);
                    }
                }
            }
        };
        auto x_stage = [&]() {
            const int bq = lane / (4 * V), rem = lane % (4 * V);
            const int tt = rem / V, ii = rem % V;
#pragma unroll
            for (int j = 0; j < XB; ++j) {
                if (bxc[j] >= xcols) break;                // warp-uniform
                const int xc = bxc[j], c = bc[j];
                const int pseg = (int)(((uint32_t)xc * minv) >> 16), m = xc - pseg * M;
                const int wseg = c * 32 + lane;            // word in the padded segment
                // FP16 pairs (x0,x4), (x1,x5), (x2,x6), (x3,x7) of the word's 8 values, and the
                // FP16-rounded values as floats for the sums
                const uint32_t in[4] = {vv[j].x, vv[j].y, vv[j].z, vv[j].w};
                float f[8];
                if constexpr (W8) {
                    // pairs (x0, x2), (x0, x2), (x1, x3), (x1, x3): both nibbles of a code meet its x
                    f[0] = f[1] = bf16lo_to_f32(in[0]);
                    f[2] = f[3] = bf16hi_to_f32(in[0]);
                    f[4] = f[5] = bf16lo_to_f32(in[1]);
                    f[6] = f[7] = bf16hi_to_f32(in[1]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        f[2 * q] = bf16lo_to_f32(in[q]);
                        f[2 * q + 1] = bf16hi_to_f32(in[q]);
                    }
                }
                if (p.xsc != nullptr && kbase + wseg * 8 < kseg) {  // activation scale: x_k * xsc_k in FP32
                    int kk = pseg * kseg + kbase + wseg * 8;
                    kk -= kk >= p.kx ? p.kx : 0;
                    const float4* sp = reinterpret_cast<const float4*>(p.xsc + kk);
                    const float4 s0 = sp[0], s1 = sp[1];
                    f[0] *= s0.x; f[1] *= s0.y; f[2] *= s0.z; f[3] *= s0.w;
                    f[4] *= s1.x; f[5] *= s1.y; f[6] *= s1.z; f[7] *= s1.w;
                }
                __half2 hp[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    hp[q] = __floats2half2_rn(f[q], f[q + 4]);
                    f[q] = __low2float(hp[q]);
                    f[q + 4] = __high2float(hp[q]);
                }
                // 1024 * (x0 + x2 + x4 + x6) + 64 * (x1 + x3 + x5 + x7), and sum x (8-bit: both
                // halves carry 1024 and every x appears twice, so 2048 * sum x and sum x)
                const float se = (f[0] + f[2]) + (f[4] + f[6]), so = (f[1] + f[3]) + (f[5] + f[7]);
                float e = W8 ? 2048.0f * se : fmaf(1024.0f, se, 64.0f * so);
                float xsum = W8 ? se : se + so;
#pragma unroll
                for (int off = 1; off < GW; off <<= 1) {
                    e += __shfl_xor_sync(0xFFFFFFFFu, e, off);
                    xsum += __shfl_xor_sync(0xFFFFFFFFu, xsum, off);
                }
                const int stp = c * 8 + bq * V + ii;
                xs[(stp * xcols + xc) * 4 + tt] =
                    make_uint4(*reinterpret_cast<const uint32_t*>(&hp[0]), *reinterpret_cast<const uint32_t*>(&hp[1]),
                               *reinterpret_cast<const uint32_t*>(&hp[2]), *reinterpret_cast<const uint32_t*>(&hp[3]));
                if ((lane & (GW - 1)) == 0) {
                    const int gam = wseg / GW;                 // group in the segment
                    const int col = M1 ? (gam % H) * P + pseg : ((pseg * H) + (gam % H)) * M + m;
                    exs[(gam / H) * (8 * NB) + col] = make_float2(e, xsum);
                }
            }
        };
        x_load();

        // zero fills: table rows not copied, E/X columns no (segment, parity, row) uses, the
        // zero block, the partial sums
        {
            const int sv = MS ? 0 : p.lds / 8, per = sv + p.ldz / 4;              // uint4 per row
            for (int i = tid; i < gaps * per; i += kThreads) {
                int k = i / per, lr = 0;
                const int col = i - k * per;
#pragma unroll
                for (int j = 0; j <= NM; ++j) {            // the k-th row of the gap ranges
                    if (k >= 0 && k < gn[j]) lr = gs[j] + k;
                    k -= gn[j];
                }
                const uint32_t dst = col < sv ? ms + (uint32_t)lr * sbytes + (uint32_t)col * 16u
                                              : mz + (uint32_t)lr * zbytes + (uint32_t)(col - sv) * 16u;
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(0u), "r"(0u), "r"(0u), "r"(0u)
                             : "memory");
            }
        }
        const int nblk = p.ngs / H;
        for (int i = tid; i < nblk * (8 * NB - p.cols); i += kThreads) {
            const int b = i / (8 * NB - p.cols), col = p.cols + i % (8 * NB - p.cols);
            exs[b * (8 * NB) + col] = make_float2(0.0f, 0.0f);
        }
        for (uint32_t i = tid; i < (M1 ? 8u * (uint32_t)P * 64u : 16u) / 16u; i += kThreads)
            reinterpret_cast<uint4*>(base + L.zero)[i] = make_uint4(0u, 0u, 0u, 0u);
        float* part = reinterpret_cast<float*>(base + L.part);
        for (int i = tid; i < p.rows_cap * p.M * NSL; i += kThreads) part[i] = 0.0f;

        // the scale/zero rows have landed: lane 0 of each warp starts its ring of units and keeps
        // it filled from here on
        pro_ok = __all_sync(0xFFFFFFFFu, gemv_wait(pbar, 0, p.spin_limit));
        if (pro_ok && active && lane == 0) {
            for (int i = 0; i < nsl && it_ch < ch1; ++i) issue_next(!(withhold && i == 0));
        }
        for (;;) {
            x_stage();
            if (xc_n >= xcols) break;                      // warp-uniform
            x_load();
        }
    }
    __syncthreads();

    // ---- compute -------------------------------------------------------------------
    bool ok = pro_ok;
    if (active) {
        const int va = sigma8(g), vb = va + 8, v7 = va & 7;
        const int rho_a = va / P, pa = va - rho_a * P;
        const int rho_b = vb / P, pb = vb - rho_b * P;
        float* red = reinterpret_cast<float*>(base + L.red) + warp * 16 * (M1 ? H : 8 * NB);
        float* part = reinterpret_cast<float*>(base + L.part);
        uint32_t coff[8 / V];                              // byte offset of this lane's words in a 128-byte row
#pragma unroll
        for (int bq = 0; bq < 8 / V; ++bq) {
            const int wf = bq * 4 * V + t * V;
            coff[bq] = ((uint32_t)((wf >> 2) ^ v7) << 4) + (uint32_t)(wf & 3) * 4u;
        }
        // B column of this lane per column block: (segment, group parity, activation row)
        const uint32_t xstep = (uint32_t)(M1 ? P : p.xcols) * 64u;   // bytes of staged x per word step
        const uint32_t zaddr = sbase + L.zero;
        uint32_t xl[NB];                                    // lane's staged column (bytes, without the step)
        int lh[NB];                                         // its group parity; -1 = idle column
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int j = nb * 8 + g;
            if (j < p.cols) {
                int m, hh, ps;
                if constexpr (M1) {
                    m = 0;
                    hh = j / P;
                    ps = j - hh * P;
                } else {
                    m = j % p.M;
                    const int ph = j / p.M;
                    hh = ph % H;
                    ps = ph / H;
                }
                xl[nb] = sbase + L.xs + (uint32_t)(((ps * p.M + m) * 4 + t) * 16);
                lh[nb] = hh;
            } else {
                xl[nb] = zaddr;
                lh[nb] = -1;
            }
        }
        // group parity of the lane's two D columns (2t, 2t+1) in each column block
        int hc[NB][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = nb * 8 + 2 * t + e;
                hc[nb][e] = j < p.cols ? (j / p.M) % H : 0;
            }
        const uint32_t exlane = sbase + L.exs + (uint32_t)(2 * t * 8);
        // M1: this lane's D columns 2t, 2t+1 are segments p0, p0+1 of parity h_use; it holds the
        // useful value of its rows (segment pa) when pa is one of them, in column e_use
        const int p0 = (2 * t) % P, h_use = (2 * t) / P;
        const int e_use = pa - p0;
        const bool useful = M1 && (unsigned)e_use < 2u && 2 * t < p.cols;   // columns past P*H are idle
        const uint32_t ex_m1 = sbase + L.exs + (uint32_t)((h_use * P + pa) * 8);

        // slot of the first tile of the run: warps before this one that hold chunks of it
        int first_slot = 0;
        {
            const int fch = (ch0 / Cw) * Cw;                // the tile's first chunk
            if (fch < ch0) {
                int fw = warp;
                while (fw > 0 && (fw * chunks) / p.warps > fch) --fw;
                first_slot = warp - fw;
            }
        }

        // this lane's rows (local to the CTA) for the scale/zero tables
        const unsigned short* smtab = reinterpret_cast<const unsigned short*>(base + L.ms);
        const uint32_t* zmtab = reinterpret_cast<const uint32_t*>(base + L.mz);

        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nb][e] = 0.0f;
        float acc_a = 0.0f, acc_b = 0.0f;                  // M1: this lane's useful sums
        int tl = ch0 / Cw, cu = ch0 - (ch0 / Cw) * Cw, ch = ch0;   // unit's tile, chunk in it, chunk in run
        const int lg = 31 - __clz(nsl);
        for (int k = 0; ch < ch1 && ok; ++k) {
            const uint32_t slot = (uint32_t)(k & (nsl - 1));
            ok = gemv_wait(bar0 + 8u * slot, (uint32_t)((k >> lg) & 1), p.spin_limit);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (ok) {
                const bool two = cu + 1 < Cw && ch + 1 < ch1;    // as in issue_next
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                  if (cc == 1 && !two) break;                 // one-chunk unit (uniform)
                  const int c = cu + cc;                      // chunk in the tile
                  const int rla = tl * R + rho_a, rlb = tl * R + rho_b;   // local rows
                  // scales of the chunk's groups: the resident row, or (MS) the unit's streamed box,
                  // 16 halves per virtual row, chunk cc at half 8 cc
                  const unsigned short* msu = reinterpret_cast<const unsigned short*>(
                      base + (mring - sbase) + slot * (uint32_t)kMetaBytes);
                  const unsigned short* sra =
                      MS ? msu + va * 16 + cc * 8 : smtab + rla * p.lds + pa * p.ngs + (kc0 + c) * GPC;
                  const unsigned short* srb =
                      MS ? msu + vb * 16 + cc * 8 : smtab + rlb * p.lds + pb * p.ngs + (kc0 + c) * GPC;
                  const uint32_t* zra = zmtab + rla * p.ldz;
                  const uint32_t* zrb = zmtab + rlb * p.ldz;
                  const int gia = pa * p.ngs + (kc0 + c) * GPC, gib = pb * p.ngs + (kc0 + c) * GPC;   // its first group
                  // M1: scales of the lane's parity; zero words shifted to the lane's first group
                  const unsigned short* sra1 = sra + h_use;
                  const unsigned short* srb1 = srb + h_use;
                  uint32_t zwa1 = 0u, zwb1 = 0u;
                  if constexpr (M1 && W8) {                   // 8-bit zero points, four per word
                      zwa1 = zra[gia >> 2] >> (8 * ((gia & 3) + h_use));
                      zwb1 = zrb[gib >> 2] >> (8 * ((gib & 3) + h_use));
                  } else if constexpr (M1 && !KQ) {
                      zwa1 = zra[gia >> 3] >> (4 * ((gia & 7) + h_use));
                      zwb1 = zrb[gib >> 3] >> (4 * ((gib & 7) + h_use));
                  }
                  // KQ: the super-block records of the lane's rows (segment pa/pb, chunk c); at M = 1 the
                  // code words are shifted to the lane's group parity
                  uint4 kra = make_uint4(0u, 0u, 0u, 0u), krb = kra;
                  float kda = 0.0f, kma = 0.0f, kdb = 0.0f, kmb = 0.0f;
                  if constexpr (KQ) {
                      kra = *reinterpret_cast<const uint4*>(sra);       // the record is 8 halves at the
                      krb = *reinterpret_cast<const uint4*>(srb);       // chunk's first group
                      kda = half_lo(kra.x);
                      kma = half_hi(kra.x);
                      kdb = half_lo(krb.x);
                      kmb = half_hi(krb.x);
                      if constexpr (M1) {
                          kra.y >>= 4 * h_use; kra.z >>= 4 * h_use; kra.w >>= 2 * h_use;
                          krb.y >>= 4 * h_use; krb.z >>= 4 * h_use; krb.w >>= 2 * h_use;
                      }
                  }
                  const uint32_t unit = ring + slot * (uint32_t)kUnitBytes + (uint32_t)cc * kBoxBytes;
                  const uint32_t row_a = unit + (uint32_t)va * 128u, row_b = row_a + 8u * 128u;
                  const uint32_t xu = (uint32_t)(c * 8) * xstep;
                  // per group parity: x base and step of this lane (idle lanes read zeros; at M = 1
                  // from a zero area as long as a chunk's x, so every lane steps by the same
                  // compile-time stride and the loads below take immediate offsets)
                  uint32_t xb[NB][H], xsp[NB][H];
#pragma unroll
                  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                      for (int hh = 0; hh < H; ++hh) {
                          const bool on = lh[nb] == hh;
                          xb[nb][hh] = on ? xl[nb] + xu : zaddr;
                          xsp[nb][hh] = (M1 || on) ? xstep : 0u;
                      }
                  float da[NB][4], db[NB][4];
#pragma unroll
                  for (int bq = 0; bq < 8 / V; ++bq) {
                      uint32_t wa[V], wb[V];
                      if constexpr (V == 4) {
                          const uint4 x0 = lds128(row_a + coff[bq]);
                          const uint4 x1 = lds128(row_b + coff[bq]);
                          wa[0] = x0.x; wa[1] = x0.y; wa[2] = x0.z; wa[3] = x0.w;
                          wb[0] = x1.x; wb[1] = x1.y; wb[2] = x1.z; wb[3] = x1.w;
                      } else if constexpr (V == 2) {
                          const uint2 x0 = lds64(row_a + coff[bq]);
                          const uint2 x1 = lds64(row_b + coff[bq]);
                          wa[0] = x0.x; wa[1] = x0.y;
                          wb[0] = x1.x; wb[1] = x1.y;
                      } else {
                          wa[0] = lds32(row_a + coff[bq]);
                          wb[0] = lds32(row_b + coff[bq]);
                      }
#pragma unroll
                      for (int i = 0; i < V; ++i) {
                          const int ws = bq * V + i;                   // word step in the chunk
                          const int jg = ws / WSG;                     // group in the chunk
                          const int hcur = jg % H;                     // its parity (c * GPC is a multiple of H)
                          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                          if constexpr (W8) {
                              expand_codes8_f16(wa[i], a0, a1, a2, a3);
                              expand_codes8_f16(wb[i], b0, b1, b2, b3);
                          } else {
                              expand_codes_f16(wa[i], a0, a1, a2, a3);
                              expand_codes_f16(wb[i], b0, b1, b2, b3);
                          }
#pragma unroll
                          for (int nb = 0; nb < NB; ++nb) {
                              const uint4 xv = lds128(xb[nb][hcur] + (uint32_t)ws * xsp[nb][hcur]);
                              if (ws % (WSG * H) == 0) {              // first step of a block
                                  mma_f16_c0(da[nb], a0, b0, a1, b1, xv.x, xv.y);
                                  mma_f16_c0(db[nb], a2, b2, a3, b3, xv.z, xv.w);
                              } else {
                                  mma_f16(da[nb], a0, b0, a1, b1, xv.x, xv.y);
                                  mma_f16(db[nb], a2, b2, a3, b3, xv.z, xv.w);
                              }
                          }
                          if ((ws + 1) % (WSG * H) == 0) {            // block of H groups complete
                              const int jg0 = jg - (H - 1);           // first group of the block in the chunk
                              const int blk = (c * GPC + jg0) / H;    // block in the segment
                              if constexpr (M1) {
                                  // one useful value per row: segment pa, parity h_use, column e_use
                                  const float va_ = e_use ? da[0][1] + db[0][1] : da[0][0] + db[0][0];
                                  const float vb_ = e_use ? da[0][3] + db[0][3] : da[0][2] + db[0][2];
                                  const float2 ex = *reinterpret_cast<const float2*>(
                                      base + (ex_m1 - sbase) + (uint32_t)(blk * 8 * 8));
                                  if constexpr (KQ) {
                                      // sub-block jg0 + h_use: s = d*sc, mn = dmin*m
                                      const float s_a = kda * kq_code(kra.y, kra.w, jg0, 0);
                                      const float s_b = kdb * kq_code(krb.y, krb.w, jg0, 0);
                                      const float n_a = kma * kq_code(kra.z, kra.w, jg0, 16);
                                      const float n_b = kmb * kq_code(krb.z, krb.w, jg0, 16);
                                      acc_a = fmaf(s_a, va_ - ex.x, fmaf(-n_a, ex.y, acc_a));
                                      acc_b = fmaf(s_b, vb_ - ex.x, fmaf(-n_b, ex.y, acc_b));
                                  } else {
                                      const float s_a = __half2float(__ushort_as_half(sra1[jg0]));
                                      const float s_b = __half2float(__ushort_as_half(srb1[jg0]));
                                      const float z_a = W8 ? meta_zero8(zwa1, jg0) : meta_zero(zwa1, jg0);
                                      const float z_b = W8 ? meta_zero8(zwb1, jg0) : meta_zero(zwb1, jg0);
                                      acc_a = fmaf(s_a, va_ - fmaf(z_a, ex.y, ex.x), acc_a);
                                      acc_b = fmaf(s_b, vb_ - fmaf(z_b, ex.y, ex.x), acc_b);
                                  }
                              } else {
                                  // scales of the block's H groups (consecutive halves) and their zero
                                  // points; groups past the row end (last, partial chunk of one
                                  // segment) get scale 0
                                  // KQ: za/zb hold the sub-blocks' minima dmin*m (a super-block is a
                                  // whole chunk, so no group lies past the row end)
                                  float sa[H], sb[H], za[H], zb[H];
                                  if constexpr (KQ) {
#pragma unroll
                                      for (int hh = 0; hh < H; ++hh) {
                                          sa[hh] = kda * kq_code(kra.y, kra.w, jg0 + hh, 0);
                                          sb[hh] = kdb * kq_code(krb.y, krb.w, jg0 + hh, 0);
                                          za[hh] = kma * kq_code(kra.z, kra.w, jg0 + hh, 16);
                                          zb[hh] = kmb * kq_code(krb.z, krb.w, jg0 + hh, 16);
                                      }
                                  } else {
                                      const uint32_t zwa = W8 ? zra[(gia + jg0) >> 2] >> (8 * ((gia + jg0) & 3))
                                                              : zra[(gia + jg0) >> 3] >> (4 * ((gia + jg0) & 7));
                                      const uint32_t zwb = W8 ? zrb[(gib + jg0) >> 2] >> (8 * ((gib + jg0) & 3))
                                                              : zrb[(gib + jg0) >> 3] >> (4 * ((gib + jg0) & 7));
#pragma unroll
                                      for (int hh = 0; hh < H; ++hh) {
                                          const bool va_ = gia + jg0 + hh < p.ng, vb_ = gib + jg0 + hh < p.ng;
                                          sa[hh] = va_ ? __half2float(__ushort_as_half(sra[jg0 + hh])) : 0.0f;
                                          sb[hh] = vb_ ? __half2float(__ushort_as_half(srb[jg0 + hh])) : 0.0f;
                                          za[hh] = W8 ? meta_zero8(zwa, hh) : meta_zero(zwa, hh);
                                          zb[hh] = W8 ? meta_zero8(zwb, hh) : meta_zero(zwb, hh);
                                      }
                                  }
#pragma unroll
                                  for (int nb = 0; nb < NB; ++nb) {
                                      const float4 ex = lds_f4(exlane + (uint32_t)((blk * 8 * NB + nb * 8) * 8));
#pragma unroll
                                      for (int e = 0; e < 2; ++e) {
                                          float s_a = sa[0], s_b = sb[0], z_a = za[0], z_b = zb[0];
#pragma unroll
                                          for (int hh = 1; hh < H; ++hh)
                                              if (hc[nb][e] == hh) {
                                                  s_a = sa[hh]; s_b = sb[hh]; z_a = za[hh]; z_b = zb[hh];
                                              }
                                          const float E = e ? ex.z : ex.x, X = e ? ex.w : ex.y;
                                          if constexpr (KQ) {
                                              acc[nb][e] = fmaf(s_a, (da[nb][e] + db[nb][e]) - E,
                                                                fmaf(-z_a, X, acc[nb][e]));
                                              acc[nb][2 + e] = fmaf(s_b, (da[nb][2 + e] + db[nb][2 + e]) - E,
                                                                    fmaf(-z_b, X, acc[nb][2 + e]));
                                          } else {
                                              acc[nb][e] = fmaf(s_a, (da[nb][e] + db[nb][e]) - fmaf(z_a, X, E),
                                                                acc[nb][e]);
                                              acc[nb][2 + e] = fmaf(s_b, (da[nb][2 + e] + db[nb][2 + e]) -
                                                                             fmaf(z_b, X, E), acc[nb][2 + e]);
                                          }
                                      }
                                  }
                              }
                          }
                      }
                  }
                }
                // tile finished in this warp's run: reduce the diagonal over segments and parities
                const int n = two ? 2 : 1;
                if (cu + n == Cw || ch + n == ch1) {
                    if constexpr (M1) {
                        // red[vrow][parity]: written by the one lane holding each useful sum
                        if (useful) {
                            red[va * H + h_use] = acc_a;
                            red[vb * H + h_use] = acc_b;
                        }
                        acc_a = acc_b = 0.0f;
                        __syncwarp();
                        const int slotp = (tl * Cw < ch0) ? first_slot : 0;
                        if (lane < R) {
                            float sum = 0.0f;
                            for (int q = 0; q < P; ++q)
#pragma unroll
                                for (int hh = 0; hh < H; ++hh) sum += red[(lane * P + q) * H + hh];
                            part[(tl * R + lane) * NSL + slotp] = sum;
                        }
                        __syncwarp();
                    } else {
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb) {
                            red[va * 8 * NB + nb * 8 + 2 * t] = acc[nb][0];
                            red[va * 8 * NB + nb * 8 + 2 * t + 1] = acc[nb][1];
                            red[vb * 8 * NB + nb * 8 + 2 * t] = acc[nb][2];
                            red[vb * 8 * NB + nb * 8 + 2 * t + 1] = acc[nb][3];
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[nb][e] = 0.0f;
                        }
                        __syncwarp();
                        const int slotp = (tl * Cw < ch0) ? first_slot : 0;
                        for (int o = lane; o < R * p.M; o += 32) {   // R*M reaches 256
                            const int rho = o / p.M, m = o - rho * p.M;
                            float sum = 0.0f;
                            for (int q = 0; q < P; ++q)
#pragma unroll
                                for (int hh = 0; hh < H; ++hh)
                                    sum += red[(rho * P + q) * 8 * NB + (q * H + hh) * p.M + m];
                            part[((tl * R + rho) * p.M + m) * NSL + slotp] = sum;
                        }
                        __syncwarp();
                    }
                }
                // this slot is read: refill it with the unit nsl ahead
                __syncwarp();
                if (lane == 0 && it_ch < ch1) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue_next(true);
                }
                ch += n;
                cu += n;
                if (cu == Cw) {
                    cu = 0;
                    ++tl;
                }
            }
        }
        if (!ok && lane == 0) {   // wait for this warp's ring copies still in flight
            for (int kk = it_n - nsl; kk < it_n; ++kk) {
                if (kk < 0 || (withhold && kk == 0)) continue;     // never issued
                const uint32_t bar = bar0 + 8u * (uint32_t)(kk & (nsl - 1));
                const long long t0 = clock64();
                while (!tc::mbar_try_wait(bar, (uint32_t)((kk >> lg) & 1))) {
                    if (clock64() - t0 > p.spin_limit) {
                        atomicOr(&g_gemv_status, kStatusGemvDrain);
                        break;
                    }
                }
            }
        }
    }
    if (!pro_ok && tid == 0) {    // the prologue's copies timed out: wait for them once more
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(pbar, 0)) {
            if (clock64() - t0 > p.spin_limit) {
                atomicOr(&g_gemv_status, kStatusGemvDrain);
                break;
            }
        }
    }
    __syncthreads();

    // ---- combine the slots in a fixed order and store ------------------------------
    // KS: both CTAs' partial sums are complete once the cluster barrier is passed; each CTA
    // then stores every other output, adding rank 0's slots and then rank 1's, read through
    // distributed shared memory, and the second barrier keeps both alive until the peer has
    // read.
    if constexpr (KS) cluster_sync();
    {
        const float* part = reinterpret_cast<const float*>(base + L.part);
        const int nout = tc_ * R * p.M;
        const int i0 = KS ? 2 * tid + (int)crank : tid, di = KS ? 2 * kThreads : kThreads;
        for (int i = i0; i < nout; i += di) {
            const int rl = i / p.M, m = i - rl * p.M;
            const int tl2 = rl / R, rho = rl - tl2 * R;
            const int tau = tile0 + tl2;
            const int mat = mat_of<NM>(p, tau);
            const int row = (tau - p.tstart[mat]) * R + rho;
            if (row >= p.n[mat]) continue;
            float sum = 0.0f;
            if constexpr (KS) {
                const uint32_t a = tc::smem_u32(part + i * NSL);
#pragma unroll
                for (uint32_t rk = 0; rk < 2; ++rk) {
                    const uint32_t ra = cluster_map(a, rk);
                    float v[kSlots];                     // the slots' loads in flight together
#pragma unroll
                    for (int q = 0; q < kSlots; ++q) v[q] = q < NSL ? ld_cluster_f32(ra + 4u * (uint32_t)q) : 0.0f;
#pragma unroll
                    for (int q = 0; q < kSlots; ++q)
                        if (q < NSL) sum += v[q];
                }
            } else {
#pragma unroll
                for (int q = 0; q < kSlots; ++q) sum += part[i * kSlots + q];
            }
            if (p.yf32)
                static_cast<float*>(p.y[mat])[(int64_t)m * p.n[mat] + row] = sum;
            else
                static_cast<__nv_bfloat16*>(p.y[mat])[(int64_t)m * p.n[mat] + row] = __float2bfloat16_rn(sum);
        }
    }
    if constexpr (KS) cluster_sync();
}

// ---- host side -------------------------------------------------------------------

// Packed codes viewed as [N*P virtual rows][K/(8P) words], boxes of 32 words x 16 rows.
bool make_code_map(CUtensorMap* map, const uint32_t* q, int64_t N, int64_t K, int P, int dev) {
    const uint64_t words = (uint64_t)(K / 8 / P);
    return encode_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, q, words, (uint64_t)(N * P), words * 4, 32, 16, dev);
}

// Scale rows (or super-block records) [N][lds halves] viewed per virtual row as [N*P][lds/P],
// unswizzled boxes of 16 halves (two chunks' groups of 32, or two records) x 16 rows.  A row's
// segments are consecutive (lds = P * the groups of a segment when a row's groups fill whole
// chunks, which make_plan checks), so virtual row n*P + seg is segment seg of row n.
bool make_meta_map(CUtensorMap* map, const void* s, int64_t N, int lds, int P, int dev) {
    const uint64_t halves = (uint64_t)(lds / P);
    return encode_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, s, halves, (uint64_t)(N * P), halves * 2, 16, 16, dev,
                          false);
}

// Segments P and group parities H per row for M activation rows: the B
// operand's columns are (segment, parity, row) triples, P*H*M <= 8 (one
// column block; M > 8 uses two blocks with P = H = 1).  Preferred: few weight
// rows per tile (P large, for an even split over the SMs) and H > 1 (the
// scale/zero correction runs once per H groups).  P > 1 needs each segment to
// be whole 256-code chunks; H must divide the groups of a chunk.  (2, 4) comes
// before (4, 2): at M = 1 every lane then holds a useful D value and the
// block-end corrections per chunk halve, which makes groups of 32 (and
// super-blocks) 3-14 % faster; groups of 128 or more cannot take H = 4.
void choose_segments(int64_t M, int64_t K, int G, bool kq, int& P, int& H) {
    P = 1;
    H = 1;
    if (M > 8) return;
    const int gpc = 256 / G;
    static const int pref[][2] = {{2, 4}, {4, 2}, {8, 1}, {4, 1}, {2, 2}, {1, 4}, {2, 1}, {1, 2}, {1, 1}};
    // 4-bit groups of 32 at M >= 2: group parities before segments, since a correction every group
    // (every word step) costs more than the extra rows per tile (5120 -> 13824: M = 2 17.9 -> 16.3 us,
    // M = 4 17.4 -> 17.0 us; the same order was 1-3 % slower at G = 128, and 4-11 % slower for
    // super-blocks at M = 3, whose correction is per record rather than per group)
    static const int pref_fine[][2] = {{2, 2}, {1, 4}, {1, 2}, {4, 1}, {2, 1}, {1, 1}, {1, 1}, {1, 1}, {1, 1}};
    for (const auto& c : (M >= 2 && G == 32 && !kq ? pref_fine : pref)) {
        const int p = c[0], h = c[1];
        if (p * h * M > 8 || h > gpc || gpc % h) continue;
        if (p > 1 && K % (256 * p)) continue;
        P = p;
        H = h;
        return;
    }
}

struct Plan {
    GemvParams p;
    int nb, grid, H;
    size_t smem;
};

// nmat matrices of Ns[i] rows sharing x (tiles numbered matrix after matrix).
// kq: the super-block layout (G = 32, K a multiple of 256, M <= 8): one 16-byte
// record per 256 codes in place of the scale row, no zero row.
// w8: the 8-bit word layout, planned as the 4-bit layer of K' = 2K channels and
// groups of G' = 2G it is run as (so K and G here are K' and G'; M <= 8, G' <= 256).
// One plan: the plain kernel (ks_ncl = 0) or the K split over ks_ncl two-CTA clusters, whose
// geometry is one segment per row (P = 1) with as many group parities as one column block of
// M <= 8 rows holds.
bool plan_one(int64_t M, const int64_t* Ns, int nmat, int64_t K, int G, int sms, size_t smem_cap, Plan& pl,
              bool kq, bool w8, int ks_ncl) {
    if (M < 1 || M > 16 || nmat < 1 || nmat > kMaxMat || K < 32 || K % 32 || K % G) return false;
    if (kq && (G != 32 || K % 256 || M > 8)) return false;
    if (w8 && (kq || M > 8 || G < 64 || G > 256 || K % 64)) return false;
    if (K > (int64_t)1 << 20) return false;                          // keeps tile/unit indices small
    for (int i = 0; i < nmat; ++i)
        if (Ns[i] < 1 || Ns[i] > (int64_t)1 << 24) return false;
    GemvParams& p = pl.p;
    p.M = (int)M;
    p.K = (int)K;
    p.G = G;
    if (ks_ncl > 0) {
        p.P = 1;
        pl.H = 1;
        for (int h = 4; h >= 2; h >>= 1)
            if (M <= 8 && h * M <= 8 && (256 / G) % h == 0) {
                pl.H = h;
                break;
            }
    } else {
        choose_segments(M, K, G, kq, p.P, pl.H);
    }
    p.R = 16 / p.P;
    p.cols = p.P * pl.H * p.M;
    p.xcols = p.P * p.M;
    pl.nb = M > 8 ? 2 : 1;
    p.C = (int)((K / p.P + 255) / 256);
    p.ks = ks_ncl > 0 ? 1 : 0;
    p.Ct = p.C;
    p.kc1 = p.ks ? (p.C + 1) / 2 : p.C;         // K split: rank 0 streams chunks [0, kc1), rank 1 the rest
    if (p.ks && (p.C < 2 || nmat != 1 || w8)) return false;
    p.C = p.kc1;                                // chunks this CTA stages x for (the K split: rank 0's)
    p.Ks = p.C * 256;                           // equals K / P whenever P > 1 (and no K split)
    p.ng = (int)(K / G);
    p.ngs = p.Ks / G;
    p.lds = kq ? (int)(K / 256 * 8) : (int)scales_ld(K, G);
    p.mstream = meta_streamed(G) ? 1 : 0;
    // streamed metadata needs each segment's groups (records) to be whole chunks laid out back to back
    if (p.mstream && (p.lds % p.P != 0 || p.lds / p.P != p.Ct * (256 / G) || (p.lds / p.P) % 8 != 0)) return false;
    p.ldz = kq ? 0 : w8 ? (int)zeros8_ld(K / 2, G / 2) : (int)zeros_ld(K, G);
    int64_t t = 0;
    for (int i = 0; i < kMaxMat; ++i) {
        p.tstart[i] = (int)t;
        p.n[i] = i < nmat ? (int)Ns[i] : 0;
        if (i < nmat) t += (Ns[i] + p.R - 1) / p.R;
    }
    if (t > (int64_t)1 << 26) return false;
    p.tstart[kMaxMat] = (int)t;
    for (int i = nmat; i < kMaxMat; ++i) p.tstart[i] = (int)t;
    p.total_tiles = (int)t;
    // CTAs (the K split: clusters of two) and the tiles each takes
    const int units = p.ks ? (p.total_tiles < ks_ncl ? p.total_tiles : ks_ncl)
                           : (p.total_tiles < sms ? p.total_tiles : sms);
    pl.grid = p.ks ? 2 * units : units;
    const int tmin = p.total_tiles / units, tmax = (p.total_tiles + units - 1) / units;
    if ((long long)tmax * p.C >= (1ll << 26)) return false;
    if ((long long)p.total_tiles * pl.grid >= (1ll << 32)) return false;
    p.rows_cap = tmax * p.R;
    // CTA warps (the instance's launch bound, or fewer when shared memory is short), then the
    // deepest per-warp ring of units that fits
    // warps taking units: as many as keep every tile within kSlots consecutive warps
    // (tiles per CTA at least tn, each of cn chunks: the K split's rank 1 streams the fewer)
    auto set_warps = [&](int nw, int tn, int cn) {
        p.nw = nw;
        p.warps = 1;
        p.nslot = kSlots;
        for (int w = nw; w >= 1; --w) {
            const long long chunks = (long long)tn * cn;
            const long long per = chunks / w;
            if (per < 1) continue;
            const long long span = (p.C + per - 1) / per + 1;
            if (span <= kSlots) {
                p.warps = w;
                p.nslot = (int)span;       // the most warps whose runs meet one tile
                break;
            }
        }
    };
    // the small-layer instance: M = 1 at G = 128 with the 70B/13B geometry (P = 4, H = 2), one or
    // three-four matrices, at most kDuoMaxBytes of weights per CTA, and a layout that leaves room
    // for a second CTA on the SM.  Measured against the 16-warp instance: 4096^2 5.45 -> 5.26 us,
    // 5120^2 6.85 -> 6.51 us; at 240 KB per CTA (5120 -> 13824) 11.6 -> 13.7 us, where 8 warps
    // no longer keep up with the stream, hence the bound.
    constexpr int64_t kDuoMaxBytes = 128 * 1024;
    int64_t wbytes = 0;
    for (int i = 0; i < nmat; ++i) wbytes += Ns[i] * (K / 2);
    p.duo = 0;
    if (M == 1 && G == 128 && !kq && !w8 && p.P == 4 && pl.H == 2 && nmat != 2 &&
        wbytes / pl.grid <= kDuoMaxBytes) {
        set_warps(kDuoWarps, tmin, p.C);
        for (int nst = 4; nst >= 1; nst >>= 1) {
            p.nst = nst;
            p.pf = 0;
            pl.smem = make_layout(p, pl.nb, pl.H).total + 1024;
            if (pl.smem <= kDuoSmem) {
                p.duo = 1;
                return true;
            }
        }
    }
    // the CTA's warps (the instance's launch bound, or fewer when shared memory is short), then
    // the deepest ring that fits
    auto fit = [&](int tn, int cn) {
        for (int nw = cta_warps(pl.nb, G); nw >= 4; nw -= 4) {
            set_warps(nw, tn, cn);
            for (int nst = 4; nst >= 1; nst >>= 1) {
                p.nst = nst;
                p.pf = nst == 1 && G == 32 ? 4 : 0;   // measured: 4 chunks ahead helps a one-unit ring at G = 32
                pl.smem = make_layout(p, pl.nb, pl.H).total + 1024;
                if (pl.smem <= smem_cap) return true;
            }
        }
        return false;
    };
    return fit(tmin, p.ks ? p.Ct - p.kc1 : p.C);
}

// The plan of a launch.  The K split (one matrix of 4-bit codes with resident metadata, M >= 2;
// ks_clusters: two-CTA clusters the device runs at once, 0 = never) is taken
//   * when x leaves the plain kernel fewer warps than its launch bound, or no room at all,
//     and the split has more;
//   * with all warps either way, when it evens out the work: the busiest CTA's weight rows
//     times the share of K it streams at least 10 % below the plain kernel's (5120 -> 5120 at
//     M = 8: 320 tiles on 148 CTAs, 3 against 2.5 tiles' work, 15.6 -> 12.6 us), or on rows of
//     8192 or more codes when the plain kernel has one ring unit per warp and the split two
//     (13824 -> 5120 at M = 4: 20.2 -> 17.6 us).  Measured where neither holds (5120 -> 13824
//     at M = 2..12, 8192 -> 28672 at M = 2 and 4, 5120 -> 5120 at M = 4), the split was 2-25 %
//     slower.
bool make_plan(int64_t M, const int64_t* Ns, int nmat, int64_t K, int G, int sms, size_t smem_cap, Plan& pl,
               bool kq = false, bool w8 = false, int ks_clusters = 0) {
    const bool plain_ok = plan_one(M, Ns, nmat, K, G, sms, smem_cap, pl, kq, w8, 0);
    const bool ks_able = ks_clusters >= 1 && M >= 2 && nmat == 1 && !w8;
    if (!ks_able) return plain_ok;
    Plan kp;
    if (!plan_one(M, Ns, nmat, K, G, sms, smem_cap, kp, kq, w8, ks_clusters)) return plain_ok;
    bool take;
    if (!plain_ok) {
        take = true;
    } else if (pl.p.nw < cta_warps(pl.nb, G)) {
        take = kp.p.nw > pl.p.nw;
    } else {
        // the busiest CTA's work in weight rows x half rows of K: plain ceil(T / grid) tiles of R rows
        // over all of K, split ceil(T' / clusters) tiles of 16 rows over half of it
        const long long wp = (long long)((pl.p.total_tiles + pl.grid - 1) / pl.grid) * pl.p.R * 2;
        const int ncl = kp.grid / 2;
        const long long wk = (long long)((kp.p.total_tiles + ncl - 1) / ncl) * kp.p.R;
        take = kp.p.nw >= pl.p.nw && (10 * wk <= 9 * wp || (K >= 8192 && pl.p.nst == 1 && kp.p.nst >= 2));
    }
    if (take) pl = kp;
    return plain_ok || take;
}

template <int NB, int G, int H, bool M1, int PT, int FMT, int NM, bool DUO = false, bool KS = false>
cudaError_t launch_m(const CUtensorMap* tm, const Plan& pl, int dev, cudaStream_t stream) {
    // largest dynamic shared memory this instance is already allowed per device (a raise may
    // race with another thread's: both set the attribute, the larger value stays)
    static std::atomic<int> cached[kMaxDevices];
    int have = cached[dev].load(std::memory_order_relaxed);
    if ((int)pl.smem > have) {
        cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB, G, H, M1, PT, FMT, NM, DUO, KS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (e == cudaSuccess && DUO)   // the shared-memory carveout that lets two CTAs share an SM
            e = cudaFuncSetAttribute(gemv_kernel<NB, G, H, M1, PT, FMT, NM, DUO, KS>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        while (have < (int)pl.smem && !cached[dev].compare_exchange_weak(have, (int)pl.smem)) {
        }
    }
    // programmatic stream serialisation: set-up overlaps the tail of the previous launch
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;     // KS: clusters of two CTAs
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3((unsigned)(pl.p.nw * 32));
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = KS ? 2 : 1;
    // tm[0, kMaxMat): code maps; tm[kMaxMat, 2 kMaxMat): streamed-metadata maps (MS instances)
    CodeMaps<NM, meta_streamed(G)> maps;
    for (int i = 0; i < NM; ++i) maps.m[i] = tm[i];
    if constexpr (meta_streamed(G))
        for (int i = 0; i < NM; ++i) maps.s[i] = tm[kMaxMat + i];
    return cudaLaunchKernelEx(&cfg, gemv_kernel<NB, G, H, M1, PT, FMT, NM, DUO, KS>, maps, pl.p);
}

template <int NB, int G, int H, int FMT, int NM>
cudaError_t launch_t(const CUtensorMap* tm, const Plan& pl, int dev, cudaStream_t stream) {
    if constexpr (NB == 1) {
        if (m1_kernel(pl.p)) {                       // M = 1: the segment count is a template constant
            switch (pl.p.P) {
                case 2: return launch_m<NB, G, H, true, 2, FMT, NM>(tm, pl, dev, stream);
                case 4: return launch_m<NB, G, H, true, 4, FMT, NM>(tm, pl, dev, stream);
                case 8: return launch_m<NB, G, H, true, 8, FMT, NM>(tm, pl, dev, stream);
            }
            return cudaErrorInvalidValue;
        }
    }
    return launch_m<NB, G, H, false, 0, FMT, NM>(tm, pl, dev, stream);
}

template <int NB, int G, int FMT, int NM>
cudaError_t launch_h(const CUtensorMap* tm, const Plan& pl, int dev, cudaStream_t stream) {
    if constexpr (NB == 2) {
        return launch_t<NB, G, 1, FMT, NM>(tm, pl, dev, stream);
    } else {
        switch (pl.H) {
            case 1: return launch_t<NB, G, 1, FMT, NM>(tm, pl, dev, stream);
            case 2:
                if constexpr (256 / G >= 2) return launch_t<NB, G, 2, FMT, NM>(tm, pl, dev, stream);
                break;
            case 4:
                if constexpr (256 / G >= 4) return launch_t<NB, G, 4, FMT, NM>(tm, pl, dev, stream);
                break;
        }
        return cudaErrorInvalidValue;
    }
}

template <int NB, int NM>
cudaError_t launch_nb(const CUtensorMap* tm, const Plan& pl, int dev, cudaStream_t stream) {
    switch (pl.p.G) {
        case 32: return launch_h<NB, 32, kFmt4, NM>(tm, pl, dev, stream);
        case 64: return launch_h<NB, 64, kFmt4, NM>(tm, pl, dev, stream);
        case 128: return launch_h<NB, 128, kFmt4, NM>(tm, pl, dev, stream);
        case 256: return launch_h<NB, 256, kFmt4, NM>(tm, pl, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

// The K split (one matrix; 4-bit codes or super-blocks; one segment per row, H group parities).
cudaError_t launch_ks(const CUtensorMap* tm, const Plan& pl, int dev, cudaStream_t stream, bool kq) {
    if (kq) {                                  // make_plan: M <= 8, one column block, G = 32
        switch (pl.H) {
            case 1: return launch_m<1, 32, 1, false, 0, kFmtQ4K, 1, false, true>(tm, pl, dev, stream);
            case 2: return launch_m<1, 32, 2, false, 0, kFmtQ4K, 1, false, true>(tm, pl, dev, stream);
            case 4: return launch_m<1, 32, 4, false, 0, kFmtQ4K, 1, false, true>(tm, pl, dev, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    if (pl.nb == 2) {
        switch (pl.p.G) {
            case 32: return launch_m<2, 32, 1, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
            case 64: return launch_m<2, 64, 1, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
            case 128: return launch_m<2, 128, 1, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
            case 256: return launch_m<2, 256, 1, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (pl.p.G * 8 + pl.H) {
        case 32 * 8 + 1: return launch_m<1, 32, 1, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        case 32 * 8 + 2: return launch_m<1, 32, 2, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        case 32 * 8 + 4: return launch_m<1, 32, 4, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        case 64 * 8 + 1: return launch_m<1, 64, 1, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        case 64 * 8 + 2: return launch_m<1, 64, 2, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        case 64 * 8 + 4: return launch_m<1, 64, 4, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        case 128 * 8 + 1: return launch_m<1, 128, 1, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        case 128 * 8 + 2: return launch_m<1, 128, 2, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        case 256 * 8 + 1: return launch_m<1, 256, 1, false, 0, kFmt4, 1, false, true>(tm, pl, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Two-CTA clusters of the K-split kernel that the device runs at once, one CTA per SM (the
// SMs pair up within their GPCs, so this can be below SMs / 2); asked once per device, 0
// when the device cannot say.
int ks_clusters(const DeviceInfo& di, int64_t M, int nmat, bool kq, bool w8, int G) {
    if (M < 2 || nmat != 1 || w8) return 0;                      // plans that never split
    static std::atomic<int> cached[kMaxDevices];
    const int v = cached[di.dev].load(std::memory_order_relaxed);
    if (v != 0) return v > 0 ? v : 0;
    // one CTA per SM, as in every K-split plan; the attribute is set to the device's opt-in
    // maximum, which is never below what a launch of this instance has set (launch_m only raises
    // it to a plan's size), so a launch on another thread cannot be left short
    auto kern = gemv_kernel<2, 128, 1, false, 0, kFmt4, 1, false, true>;
    const int smem = (int)di.smem_optin;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = 2;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2u);
        cfg.blockDim = dim3((unsigned)(cta_warps(2, 128) * 32));
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    if (n > di.sms / 2) n = di.sms / 2;
    cached[di.dev].store(n > 0 ? n : -1, std::memory_order_relaxed);
    return n > 0 ? n : 0;
}

// The 8-bit word layout (one column block; G' = 2G in {64, 128, 256}).
cudaError_t launch_w8(const CUtensorMap* tm, const Plan& pl, int dev, cudaStream_t stream) {
    switch (pl.p.G) {
        case 64: return launch_h<1, 64, kFmt8, 1>(tm, pl, dev, stream);
        case 128: return launch_h<1, 128, kFmt8, 1>(tm, pl, dev, stream);
        case 256: return launch_h<1, 256, kFmt8, 1>(tm, pl, dev, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t gemv_take_status(uint32_t* word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_gemv_status, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof(uint32_t));
}

bool gemv_fits(int64_t M, const int64_t* Ns, int nmat, int64_t K, int G, bool kq, bool w8) {
    Plan pl;
    DeviceInfo di;
    int kcl;
    if (current_device(di) != cudaSuccess) {   // no device: the B300's figures
        di.sms = 148;
        di.smem_optin = 227 * 1024;
        kcl = 74;
    } else {
        kcl = ks_clusters(di, M, nmat, kq, w8, G);
    }
    return w8 ? make_plan(M, Ns, nmat, 2 * K, 2 * G, di.sms, di.smem_optin, pl, false, true)
              : make_plan(M, Ns, nmat, K, G, di.sms, di.smem_optin, pl, kq, false, kcl);
}

bool gemv_runs_full(int64_t M, const int64_t* Ns, int nmat, int64_t K, int G) {
    Plan pl;
    DeviceInfo di;
    int kcl = 74;
    if (current_device(di) != cudaSuccess) {   // no device: the B300's figures
        di.sms = 148;
        di.smem_optin = 227 * 1024;
    } else {
        kcl = ks_clusters(di, M, nmat, false, false, G);
    }
    // groups of 32 split along K run behind the tensor cores at M = 16 (5120 -> 13824: 30.5
    // against 29.1 us), so only their plain plans count there
    return make_plan(M, Ns, nmat, K, G, di.sms, di.smem_optin, pl, false, false, kcl) &&
           pl.p.nw == cta_warps(pl.nb, G) && !(pl.p.ks && G == 32 && M > 8);
}

bool gemv_describe(int64_t M, int64_t N, int64_t K, int G, int mode, int32_t* plan) {
    Plan pl;
    DeviceInfo di;
    int kcl = 74;
    if (current_device(di) != cudaSuccess) {   // no device: the B300's figures
        di.sms = 148;
        di.smem_optin = 227 * 1024;
    } else {
        kcl = ks_clusters(di, M, 1, false, false, G);
    }
    const int64_t Ns[1] = {N};
    const bool ok = mode == 0 ? make_plan(M, Ns, 1, K, G, di.sms, di.smem_optin, pl, false, false, kcl)
                              : plan_one(M, Ns, 1, K, G, di.sms, di.smem_optin, pl, false, false, mode == 2 ? kcl : 0);
    if (!ok) return false;
    plan[0] = pl.p.P;
    plan[1] = pl.H;
    plan[2] = pl.p.nw;
    plan[3] = pl.p.ks;
    plan[4] = pl.grid;
    plan[5] = pl.p.nst;
    return true;
}

bool gemv_fits(int64_t M, int64_t N, int64_t K, int G, int nmat, bool kq) {
    int64_t Ns[kMaxMat];
    for (int i = 0; i < kMaxMat; ++i) Ns[i] = N;
    return gemv_fits(M, Ns, nmat, K, G, kq);
}

cudaError_t launch_gemv(const void* x, const GemvMat* mats, int nmat, int64_t M, int64_t N, int64_t K, int G,
                        cudaStream_t stream, const float* xsc, int64_t kx, bool kq, bool yf32, bool w8) {
    if (kx == 0) kx = K;
    if (kx != K && (kx * 2 != K || kx % 8 != 0)) return cudaErrorInvalidValue;
    if (kq && (G != 32 || xsc != nullptr || kx != K)) return cudaErrorInvalidValue;
    if (w8 && (kq || xsc != nullptr || kx != K)) return cudaErrorInvalidValue;
    if (nmat < 1 || nmat > kMaxMat) return cudaErrorInvalidValue;
    DeviceInfo di;
    const cudaError_t e = current_device(di);
    if (e != cudaSuccess) return e;
    int64_t Ns[kMaxMat];
    for (int i = 0; i < nmat; ++i) Ns[i] = mats[i].n > 0 ? mats[i].n : N;
    // the 8-bit word layout runs as a 4-bit layer of 2K channels and groups of 2G over the
    // same words; x keeps its K channels
    const int64_t Kv = w8 ? 2 * K : K;
    const int Gv = w8 ? 2 * G : G;
    Plan pl;
    if (!make_plan(M, Ns, nmat, Kv, Gv, di.sms, di.smem_optin, pl, kq, w8, ks_clusters(di, M, nmat, kq, w8, G)))
        return cudaErrorNotSupported;
    GemvParams& p = pl.p;
    p.x = static_cast<const __nv_bfloat16*>(x);
    p.xsc = xsc;
    p.kx = (int)kx;
    p.yf32 = yf32 ? 1 : 0;
    p.spin_limit = wait_limit();
    p.withhold = take_withhold(1) ? 1 : 0;
    CUtensorMap tm[2 * kMaxMat];
    for (int i = 0; i < kMaxMat; ++i) {
        const GemvMat& mt = mats[i < nmat ? i : 0];
        p.q[i] = mt.q;
        p.s[i] = static_cast<const unsigned short*>(mt.s);
        p.z[i] = mt.z;
        p.y[i] = mt.y;
        if (i < nmat) {
            if (!make_code_map(&tm[i], mt.q, Ns[i], Kv, p.P, di.dev)) return cudaErrorInvalidValue;
            if (p.mstream && !make_meta_map(&tm[kMaxMat + i], mt.s, Ns[i], p.lds, p.P, di.dev))
                return cudaErrorInvalidValue;
        } else {
            tm[i] = tm[0];
            tm[kMaxMat + i] = tm[kMaxMat];
        }
    }
    // instances by matrix count: one map for one matrix (no per-tile matrix lookup), two for a
    // pair, four for three or four (4-bit only); the super-block layout takes one or two, the
    // 8-bit word layout one
    if ((kq && nmat > 2) || (w8 && nmat > 1)) return cudaErrorInvalidValue;
    if (p.duo)                                                // make_plan: M = 1, G = 128, P = 4, H = 2
        return nmat == 1 ? launch_m<1, 128, 2, true, 4, kFmt4, 1, true>(tm, pl, di.dev, stream)
                         : launch_m<1, 128, 2, true, 4, kFmt4, 4, true>(tm, pl, di.dev, stream);
    if (p.ks) return launch_ks(tm, pl, di.dev, stream, kq);  // make_plan: one matrix, M >= 2
    if (kq)                                                   // make_plan: M <= 8, one column block
        return nmat == 1 ? launch_h<1, 32, kFmtQ4K, 1>(tm, pl, di.dev, stream)
                         : launch_h<1, 32, kFmtQ4K, 2>(tm, pl, di.dev, stream);
    if (w8) return launch_w8(tm, pl, di.dev, stream);
    if (nmat > 2)
        return pl.nb == 1 ? launch_nb<1, 4>(tm, pl, di.dev, stream) : launch_nb<2, 4>(tm, pl, di.dev, stream);
    if (nmat == 2)
        return pl.nb == 1 ? launch_nb<1, 2>(tm, pl, di.dev, stream) : launch_nb<2, 2>(tm, pl, di.dev, stream);
    return pl.nb == 1 ? launch_nb<1, 1>(tm, pl, di.dev, stream) : launch_nb<2, 1>(tm, pl, di.dev, stream);
}

}  // namespace w4a16
