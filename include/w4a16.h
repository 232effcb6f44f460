/*
 * w4a16.h -- C ABI of the B300 (sm_103a) W4A16 weight-only linear library.
 *
 * The library computes the fused dequantise-and-multiply linear layer of
 * W4A16 weight-only quantisation: weights are stored as 4-bit codes with one
 * FP16 scale and one 4-bit zero point per group of G input channels of each
 * output column; activations stay BF16, accumulation is FP32 and the output
 * is BF16.  The weights stay packed in device memory and are only expanded
 * inside the kernels (klaylearn.com glossary "Weight-Only Quantisation", main
 * body; zhuai.tech "Quantization Is Not a Zip File", section 8 "Engineering
 * pitfalls": packed data stays packed until the kernel).
 *
 * ---------------------------------------------------------------------------
 * Data layout (all row-major, all buffers owned by the caller):
 *
 *   W        FP16 [N, K]     weight in linear-layer orientation: row n is the
 *                            K input channels of output column n.
 *   x        BF16 [M, K]     activations, row pitch K.
 *   y        BF16 [M, N]     output, y = x * W_hat^T, row pitch N.
 *   qweight  uint32 [N, K/8] code of (n, k) in bits 4*(k%8) .. 4*(k%8)+3 of
 *                            word qweight[n][k/8] (low nibble first).
 *   scales   FP16 [N, ldS]   scales[n][g] = scale of group g = k / G;
 *                            ldS = w4a16_scales_ld(K, G) (K/G rounded up to
 *                            8 halves so each row starts on 16 bytes).
 *   zeros    uint32 [N, ldZ] zero point of group g in bits 4*(g%8).. of word
 *                            zeros[n][g/8]; ldZ = w4a16_zeros_ld(K, G).
 *
 *   W_hat[n][k] = (q[n][k] - z[n][k/G]) * s[n][k/G]        (exact in FP32)
 *
 * Reconstruction (q - zero_point) * scale is the asymmetric rule of instagit
 * "Comparison of Quantization Methods: INT8 vs GPTQ vs AWQ vs GGUF", section
 * "Practical Code Examples"; per-group scales of 32/64/128/256 weights follow
 * zhuai.tech section 3 "The core idea: local structure, not global rounding".
 *
 * ---------------------------------------------------------------------------
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless stated; the caller owns them.  All
 *     must be 16-byte aligned.  The library keeps no pointer after a call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued asynchronously; results are valid once the stream reaches the
 *     point of the call.  Calls on distinct streams may run concurrently.
 *   - The decode kernel, the tensor-core kernel and its x conversion are
 *     launched with programmatic stream serialisation: each may begin
 *     (initialise its barriers, allocate tensor memory) while the previous
 *     kernel on the stream finishes, but it reads and writes no global memory
 *     before that kernel has completed, so stream order keeps its usual
 *     meaning.  For long rows the decode kernel runs as clusters of two CTAs.
 *   - Scratch memory: the tensor-core path takes each call's scratch (the
 *     FP16 copy of x; FP32 partial sums when tiles are split along K: a
 *     narrow layer's tiles, or the last, partial wave of wider tiles)
 *     from the current device's current memory pool with cudaMallocAsync and
 *     frees it on the stream after the call's kernels; the library keeps no
 *     device memory of its own between calls (the no-allocation entry point
 *     below excepted).  What the pool keeps is the application's policy: a
 *     pool with release threshold 0 (the default pool's default) hands the
 *     memory back to the driver at every synchronisation, and the next call
 *     maps it again (measured on a B300: about 3 us per call on a 5120 ->
 *     13824 layer at M = 32).  A process that calls the layer in a loop
 *     should raise the threshold of that pool or make its own pool current.
 *   - Errors in arguments are reported before anything is launched, as a
 *     status code; no entry point aborts, throws, traps or asserts.  A CUDA
 *     launch error is reported as W4A16_ERR_CUDA.
 *   - Preconditions: G in {32, 64, 128, 256}; K > 0 and K % G == 0;
 *     N % 8 == 0; weights and activations finite; |x| < 65504.
 *     M == 0 or N == 0 is an empty problem: W4A16_OK, nothing is launched.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stdint.h>

#if defined(__GNUC__)
#define W4A16_API __attribute__((visibility("default")))
#else
#define W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* w4a16_stream_t;

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,   /* null pointer, bad size or shape mismatch */
    W4A16_ERR_UNSUPPORTED = 2,   /* group size or shape outside what is built */
    W4A16_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    W4A16_ERR_CUDA = 4,          /* the CUDA runtime reported an error */
    W4A16_ERR_TIMEOUT = 5,       /* a kernel's bounded wait expired (see
                                    w4a16_device_status) */
    W4A16_ERR_NO_DEVICE = 6      /* no usable sm_103 device is current */
} w4a16_status;

/* Human-readable name of a status code (static string, never NULL). */
W4A16_API const char* w4a16_status_string(w4a16_status status);

/* ---- layout helpers (elements per row; pure host functions) ------------- */

/* uint32 words per qweight row: K / 8. */
W4A16_API int64_t w4a16_qweight_ld(int64_t K);
/* FP16 halves per scales row: K/G rounded up to a multiple of 8. */
W4A16_API int64_t w4a16_scales_ld(int64_t K, int G);
/* uint32 words per zeros row: ceil(K/G / 8) rounded up to a multiple of 4. */
W4A16_API int64_t w4a16_zeros_ld(int64_t K, int G);

/* ---- packer ------------------------------------------------------------------
 * w4a16_pack: quantise FP16 W [N,K] to (qweight, scales, zeros), asymmetric
 * min-max per group of G consecutive input channels of one output column:
 *   lo = min(0, min w), hi = max(0, max w)            (range holds 0)
 *   s  = RNE_fp16( fp32(hi - lo) / 15 )               (IEEE binary32 ops)
 *   if s == 0: s = 1, z = 0                          (all-zero group)
 *   z  = clamp(rne(-lo / s), 0, 15)
 *   q  = clamp(rne(w / s) + z, 0, 15)
 * Codes are taken against the stored FP16 scale.  The groupwise min-max
 * scheme is the one the klaylearn glossary's main body describes (small
 * integers plus scale and zero-point per group); the zero point and its
 * reconstruction follow instagit's asymmetric example.
 * Every element of qweight, scales and zeros is written, row padding as 0.
 * Errors: W4A16_ERR_INVALID_ARG / _UNSUPPORTED / _MISALIGNED as above.
 */
W4A16_API w4a16_status w4a16_pack(const void* w_f16, int64_t N, int64_t K, int G,
                        uint32_t* qweight, void* scales_f16, uint32_t* zeros,
                        w4a16_stream_t stream);

/* ---- dequantise (checking aids) ----------------------------------------------
 * Each aid expands every packed word with one layer kernel's own inline
 * routine (the same functions the kernel calls, not a separate
 * implementation), so a bit-exact comparison of its output with the
 * definition W_hat = (q - z) * s checks the instructions the layer runs: the
 * nibble-to-FP16 expansion, the zero-point and scale extraction, and the
 * order in which codes land in registers.  The linear entry points never call
 * them and never expand weights in device memory.
 *
 * w4a16_dequant: w_out FP32 [N,K] = (q - z) * s through the decode kernel's
 *   expansion (codes as the exact FP16 values 1024 + q and 64 + q, zero point
 *   and scale as that kernel extracts them).  Exact in FP32.
 * w4a16_dequant_debug: the same call under its checking-aid name (identical
 *   arguments, behaviour and errors).
 * w4a16_dequant_f16: w_out FP16 [N,K] = RN_fp16((q - z) * s) through the
 *   tensor-core kernel's expansion: the FP16 operand it writes into tensor
 *   memory (one rounding of the exact product).
 * Errors: as w4a16_pack (shape, group size, null or misaligned pointers).
 */
W4A16_API w4a16_status w4a16_dequant(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros,
                           int64_t N, int64_t K, int G, float* w_out, w4a16_stream_t stream);
W4A16_API w4a16_status w4a16_dequant_debug(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros,
                                           int64_t N, int64_t K, int G, float* w_out, w4a16_stream_t stream);
W4A16_API w4a16_status w4a16_dequant_f16(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros,
                                         int64_t N, int64_t K, int G, void* w_out_f16, w4a16_stream_t stream);

/* ---- the layer ---------------------------------------------------------------
 * w4a16_linear: y[M,N] (BF16) = x[M,K] (BF16) * W_hat^T, FP32 accumulation,
 * one round-to-nearest-even to BF16 per output.  Dispatch: M <= 8 runs the
 * bandwidth-bound decode GEMV (when x of M rows, or half of it on each SM of
 * a two-CTA cluster splitting K, fits the kernel's shared memory), and so
 * does M = 9..16 where the GEMV runs with all its warps and also takes M = 8
 * (measured on a 5120 -> 13824 layer at M = 16: 24.9 us against 29.1 us for
 * the GEMM); anything else runs the tcgen05 tensor-core GEMM.  Decode is
 * weight-bandwidth bound and prefill compute bound (klaylearn glossary, FAQ
 * "Why is it especially useful for decode?"; multigrid.ai, section "Where it
 * stops being the right answer").
 * x and y must not overlap the weight buffers.
 */
W4A16_API w4a16_status w4a16_linear(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                          const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G,
                          void* y_bf16, w4a16_stream_t stream);

/*
 * w4a16_linear_dual: two projections of the same x (e.g. the gate and up
 * projections of a gated FFN) in one launch that stages x once:
 *   y_gate = x * W_hat_gate^T,  y_up = x * W_hat_up^T.
 * Both weights share K, N and G.  Paired gate/up traversal is the zhuai.tech
 * page's section 2 ("Moving fewer bytes can make decode faster") workload.
 * The dual GEMV runs where one matrix of twice the rows would (M <= 8, or
 * 9..16 with all its warps); otherwise the GEMM runs once per projection.
 */
W4A16_API w4a16_status w4a16_linear_dual(const void* x_bf16,
                               const uint32_t* qweight_gate, const void* scales_gate,
                               const uint32_t* zeros_gate,
                               const uint32_t* qweight_up, const void* scales_up,
                               const uint32_t* zeros_up,
                               int64_t M, int64_t N, int64_t K, int G,
                               void* y_gate_bf16, void* y_up_bf16, w4a16_stream_t stream);

/*
 * w4a16_linear_multi: up to four projections of the same x in one pass, each
 * with its own output size (e.g. the q, k and v projections of an attention
 * layer, grouped-query k/v included):  y_i = x * W_hat_i^T,  i < nmat.
 * At decode a layer's fixed per-launch cost (staging x, the first weights'
 * latency, the tail) is paid once for all the matrices instead of once each,
 * the multi-matrix generalisation of the paired gate/up traversal (zhuai.tech
 * "Quantization Is Not a Zip File", section 2 "Moving fewer bytes can make
 * decode faster").
 *   nmat        1..4
 *   qweight[i], scales_f16[i], zeros[i], y_bf16[i]
 *               HOST arrays of nmat DEVICE pointers: matrix i packed as
 *               above for [N[i], K] (same K and G for all), output y_i BF16
 *               [M, N[i]]
 *   N           HOST array of nmat output sizes (multiples of 8; 0 = skip)
 * M <= 8 runs one decode launch over all the matrices (when their rows fit
 * the kernel's shared memory), and so does M = 9..16 where that launch runs
 * with all its warps; otherwise the tensor-core kernel runs once per matrix on
 * one FP16 copy of x.  The arrays are read during the call only.
 * Errors: W4A16_ERR_INVALID_ARG for nmat outside 1..4 or a null array, else
 * as w4a16_linear for each matrix.
 */
W4A16_API w4a16_status w4a16_linear_multi(const void* x_bf16, int nmat, const uint32_t* const* qweight,
                                          const void* const* scales_f16, const uint32_t* const* zeros,
                                          const int64_t* N, int64_t M, int64_t K, int G, void* const* y_bf16,
                                          w4a16_stream_t stream);

/*
 * Explicit-path variants of w4a16_linear, same arguments and result, for
 * measuring both kernels on the same shape (e.g. the batch at which the
 * decode kernel stops being bandwidth bound).
 *   w4a16_linear_gemv: the decode kernel; W4A16_ERR_UNSUPPORTED if M > 16 or
 *                      x does not fit the kernel's shared memory.
 *   w4a16_linear_gemm: the tensor-core kernel, any M >= 1.
 */
W4A16_API w4a16_status w4a16_linear_gemv(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                               const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G,
                               void* y_bf16, w4a16_stream_t stream);
W4A16_API w4a16_status w4a16_linear_gemm(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                               const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G,
                               void* y_bf16, w4a16_stream_t stream);

/*
 * w4a16_linear_f32: the layer with an FP32 output y_f32 [M,N]: the kernels'
 * FP32 sums without the final BF16 rounding (for a caller that accumulates a
 * residual in FP32, and to check the kernels' arithmetic against a bound
 * tighter than the BF16 output allows).  path: 0 = the kernel w4a16_linear
 * would choose, 1 = the decode kernel (as w4a16_linear_gemv), 2 = the
 * tensor-core kernel.  Other arguments and errors as w4a16_linear; a path
 * outside 0..2 is W4A16_ERR_INVALID_ARG.
 */
W4A16_API w4a16_status w4a16_linear_f32(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                                        const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G, int path,
                                        float* y_f32, w4a16_stream_t stream);

/*
 * w4a16_linear_gemm_noalloc: the tensor-core path of w4a16_linear_gemm for
 * callers that may not allocate device memory while they run the layer: an
 * engine that reserves its whole memory budget at start-up and forbids any
 * later allocation, so that a running model never fails half-way on an
 * out-of-memory error or fragments a pool it manages itself.  The pages this
 * library follows have no counterpart to this entry point; it is a
 * deployment variant of the same computation.
 *
 * Same arguments and result as w4a16_linear_gemm.  The per-call FP16 copy of
 * x, which the allocating entry points take from a stream-ordered pool, here
 * lives in one file-scope device array of W4A16_NOALLOC_MAX_X_ELEMS FP16
 * values (16 MiB), which every GPU that loads the library holds until the
 * process exits.  The call itself allocates and frees nothing.
 *   - M * K > W4A16_NOALLOC_MAX_X_ELEMS: W4A16_ERR_UNSUPPORTED, nothing runs.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current).  Make that first call before
 *     any stream capture on the device.
 *   - All calls share the array: two calls whose kernels may overlap on the
 *     GPU (different streams with no ordering between them) race on it and
 *     give undefined results.  Calls ordered on one stream are safe; each
 *     call overwrites the part of the array it uses before reading it.
 */
#define W4A16_NOALLOC_MAX_X_ELEMS (8u * 1024u * 1024u)
W4A16_API w4a16_status w4a16_linear_gemm_noalloc(const void* x_bf16, const uint32_t* qweight,
                                       const void* scales_f16, const uint32_t* zeros, int64_t M, int64_t N,
                                       int64_t K, int G, void* y_bf16, w4a16_stream_t stream);

/*
 * w4a16_linear_act_scaled: the layer with a per-input-channel activation
 * scale fused into the staging of x:
 *   y[m,n] = bf16_rn( sum_k fp16_rn(fp32(x[m,k] * x_scale[k])) * W_hat[n,k] ).
 * This is the deployed form of activation-aware weight quantisation: the
 * weights of salient input channels (those that meet large activations) are
 * scaled up by alpha_k before packing and the activations scaled down by the
 * same factor, so the kernel stays an ordinary groupwise INT4 layer
 * (instagit.com "Comparison of Quantization Methods: INT8 vs GPTQ vs AWQ vs
 * GGUF", section "AWQ: Activation-Aware Weight Quantization"; klaylearn.com
 * glossary "Weight-Only Quantisation", FAQ "What is the difference between AWQ
 * and GPTQ?").  The caller packs W * diag(alpha) with w4a16_pack and passes
 * x_scale[k] = 1 / alpha_k.
 *   x_scale  FP32 [K], device, 16-byte aligned, owned by the caller; any
 *            finite values (|x * x_scale| must stay in the FP16 range).
 * Dispatch, layouts and the other arguments as for w4a16_linear.  The
 * product is formed in FP32 and rounded to FP16 once, on both kernels.
 * Errors: as w4a16_linear, plus W4A16_ERR_INVALID_ARG for a null x_scale and
 * W4A16_ERR_MISALIGNED for a misaligned one.
 */
W4A16_API w4a16_status w4a16_linear_act_scaled(const void* x_bf16, const float* x_scale, const uint32_t* qweight,
                                     const void* scales_f16, const uint32_t* zeros, int64_t M, int64_t N,
                                     int64_t K, int G, void* y_bf16, w4a16_stream_t stream);

/*
 * w4a16_linear_dual_act_scaled: w4a16_linear_dual with the same activation
 * scale applied to the shared x (both projections see x[m,k] * x_scale[k]).
 */
W4A16_API w4a16_status w4a16_linear_dual_act_scaled(const void* x_bf16, const float* x_scale,
                                          const uint32_t* qweight_gate, const void* scales_gate,
                                          const uint32_t* zeros_gate, const uint32_t* qweight_up,
                                          const void* scales_up, const uint32_t* zeros_up, int64_t M, int64_t N,
                                          int64_t K, int G, void* y_gate_bf16, void* y_up_bf16,
                                          w4a16_stream_t stream);

/* ---- the 8-bit variant (W8A16) ---------------------------------------------
 * The same group-wise asymmetric min-max quantiser with 255 steps:
 *   s8 = RNE_fp16( fp32(hi - lo) / 255 ); s8 == 0 -> s8 = 1, z8 = 0
 *   z8 = clamp(rne(-lo / s8), 0, 255),  q8 = clamp(rne(w / s8) + z8, 0, 255)
 * (weights stored as INT8 or INT4 with 16-bit activations: klaylearn.com
 * glossary "Weight-Only Quantisation", first FAQ answer).  Two storages:
 *
 * The word layout (w8a16_*): four codes per 32-bit word, one FP16 scale and
 * one 8-bit zero point per group:
 *   qweight  uint32 [N, K/4]   code of (n, k) in bits 8*(k%4) .. 8*(k%4)+7 of
 *                              word k/4 (low byte first)
 *   scales   FP16 [N, ldS]     as the 4-bit layout (ldS = w8a16_scales_ld)
 *   zeros    uint32 [N, ldZ8]  zero point of group g in bits 8*(g%4) .. of word
 *                              g/4; ldZ8 = ceil(K/G / 4) rounded up to a
 *                              multiple of 4 (w8a16_zeros_ld)
 *   W_hat = (q8 - z8) * s8, 8.125 bits per weight at G = 128.
 * w8a16_linear runs the decode kernel for M <= 8 and G <= 128 (where its rows
 * fit), which expands each code as its two nibbles against one FP16 exponent,
 * else the tensor-core kernel, which expands four codes per word with two byte
 * permutes.  w8a16_linear_gemv / _gemm force one kernel (the decode kernel
 * takes M <= 8 and G <= 128; W4A16_ERR_UNSUPPORTED otherwise).
 * w8a16_dequant (FP32) and w8a16_dequant_f16 (the tensor-core kernel's FP16
 * operand) are checking aids through the kernels' own 8-bit expansions, as
 * w4a16_dequant and w4a16_dequant_f16 are for the 4-bit layout.
 *
 * The two-plane storage (w8a16_planes_*): each 8-bit code as two 4-bit planes
 * of a 4-bit layer with 2K input channels, so the 4-bit kernels compute the
 * 8-bit layer exactly (16 s8 (q8>>4 - z8>>4) + s8 (q8&15 - z8&15) = s8 (q8 - z8)):
 *   qweight  uint32 [N, K/4]   row n: the K codes' high nibbles (channels
 *                              0..K-1) then their low nibbles (K..2K-1), in the
 *                              4-bit layout (8 bits per weight)
 *   scales   FP16 [N, ldS8]    the K/G hi-plane scales 16*s8, then the K/G
 *                              lo-plane scales s8 (ldS8 = w4a16_scales_ld(2K, G))
 *   zeros    uint32 [N, ldZ8]  z8 >> 4 per group, then z8 & 15 per group, packed
 *                              as 4-bit zeros of 2K/G groups (ldZ8 = w4a16_zeros_ld(2K, G))
 * (8.25 bits per weight at G = 128: each scale is stored twice.)  Its dispatch
 * is w4a16_linear_path(M, N, 2K, G).
 * Preconditions and errors as for the 4-bit calls.
 */
W4A16_API int64_t w8a16_qweight_ld(int64_t K);
W4A16_API int64_t w8a16_scales_ld(int64_t K, int G);
W4A16_API int64_t w8a16_zeros_ld(int64_t K, int G);
W4A16_API w4a16_status w8a16_pack(const void* w_f16, int64_t N, int64_t K, int G, uint32_t* qweight,
                                  void* scales_f16, uint32_t* zeros, w4a16_stream_t stream);
/* y[M,N] (BF16) = x[M,K] (BF16) * W_hat8^T, FP32 accumulation, one BF16 rounding per output. */
W4A16_API w4a16_status w8a16_linear(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                                    const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G,
                                    void* y_bf16, w4a16_stream_t stream);
W4A16_API w4a16_status w8a16_linear_gemv(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                                         const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G,
                                         void* y_bf16, w4a16_stream_t stream);
W4A16_API w4a16_status w8a16_linear_gemm(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                                         const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G,
                                         void* y_bf16, w4a16_stream_t stream);
W4A16_API w4a16_status w8a16_dequant(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros,
                                     int64_t N, int64_t K, int G, float* w_out, w4a16_stream_t stream);
W4A16_API w4a16_status w8a16_dequant_f16(const uint32_t* qweight, const void* scales_f16, const uint32_t* zeros,
                                         int64_t N, int64_t K, int G, void* w_out_f16, w4a16_stream_t stream);

W4A16_API int64_t w8a16_planes_qweight_ld(int64_t K);
W4A16_API int64_t w8a16_planes_scales_ld(int64_t K, int G);
W4A16_API int64_t w8a16_planes_zeros_ld(int64_t K, int G);
W4A16_API w4a16_status w8a16_planes_pack(const void* w_f16, int64_t N, int64_t K, int G, uint32_t* qweight,
                                         void* scales_f16, uint32_t* zeros, w4a16_stream_t stream);
W4A16_API w4a16_status w8a16_planes_linear(const void* x_bf16, const uint32_t* qweight, const void* scales_f16,
                                           const uint32_t* zeros, int64_t M, int64_t N, int64_t K, int G,
                                           void* y_bf16, w4a16_stream_t stream);

/* ---- the super-block variant (Q4_K-style) ------------------------------------
 * K-quants keep 4-bit codes in 256-weight super-blocks whose sub-blocks carry
 * their own scale and minimum, quantised in turn against per-super-block
 * factors (zhuai.tech "Quantization Is Not a Zip File", section 3, table "How
 * to read common GGUF quantization names", K-quants row; section 2 "Moving
 * fewer bytes can make decode faster" on packed Q4_K decode dot products and
 * the paired gate/up traversal).  A super-block is 256 consecutive input
 * channels of one row, cut into 8 sub-blocks of 32; sub-block j reconstructs
 * as  W_hat = d*sc_j*q - dmin*m_j  with q in [0,15], 6-bit sc_j, m_j and FP16
 * d, dmin.  Quantiser (min-max per sub-block, range widened to hold 0, all
 * decisions in IEEE binary32):
 *   a_j = (hi - lo) / 15, b_j = -lo;  d = RNE_fp16(max a_j / 63) (0 -> 1),
 *   dmin = RNE_fp16(max b_j / 63);  sc_j = clamp(rne(a_j / d), 0, 63),
 *   m_j = dmin == 0 ? 0 : clamp(rne(b_j / dmin), 0, 63),
 *   q = d*sc_j > 0 ? clamp(rne((w + dmin*m_j) / (d*sc_j)), 0, 15) : 0
 * Storage (4.5 bits per weight):
 *   qweight  uint32 [N, K/8]         the codes in the 4-bit layout
 *   meta     uint32 [N, K/256 * 4]   one 16-byte record per super-block:
 *            word 0 = d bits | dmin bits << 16;  word 1 = sc_j & 15 at bit 4j;
 *            word 2 = m_j & 15 at bit 4j;  word 3 = sc_j >> 4 at bit 2j and
 *            m_j >> 4 at bit 16 + 2j
 * Preconditions: K a positive multiple of 256, N a multiple of 8, every
 * pointer 16-byte aligned (W4A16_ERR_INVALID_ARG / W4A16_ERR_MISALIGNED).
 * The layer runs the decode kernel: up to 8 activation rows per launch, as
 * many as its shared memory holds for this K (x staged as M*K FP16); larger M
 * is split into row blocks, each of which reads the weights again.  Each CTA
 * also holds the records of all its weight rows; where even one activation
 * row does not fit that way (N*K above about 3e8 at M = 1, e.g. N = 28672
 * with K > 13824), the weight rows are cut into slices that fit and the call
 * runs one activation row per launch.  W4A16_ERR_UNSUPPORTED if K exceeds
 * 77312 (not even 8 weight rows and one activation row fit).
 */
W4A16_API int64_t q4k_meta_ld(int64_t K);   /* uint32 words per meta row: K/256*4 (0 if K % 256) */
/* Checking aid: w_out FP32 [N,K] = d*sc_j*q - dmin*m_j through the decode kernel's super-block
 * decoding (its code expansion and record fields), s = d*sc_j and mn = dmin*m_j exact, then s*q
 * (exact) minus mn rounded once.  Errors as q4k_pack. */
W4A16_API w4a16_status q4k_dequant(const uint32_t* qweight, const uint32_t* meta, int64_t N, int64_t K,
                                   float* w_out, w4a16_stream_t stream);
W4A16_API w4a16_status q4k_pack(const void* w_f16, int64_t N, int64_t K, uint32_t* qweight, uint32_t* meta,
                                w4a16_stream_t stream);
/* y[M,N] (BF16) = x[M,K] (BF16) * W_hat^T, FP32 accumulation, one BF16 rounding per output. */
W4A16_API w4a16_status q4k_linear(const void* x_bf16, const uint32_t* qweight, const uint32_t* meta, int64_t M,
                                  int64_t N, int64_t K, void* y_bf16, w4a16_stream_t stream);
/* Two matrices of the same shape sharing x (gate and up projections) in one launch per row block, or
 * one launch per matrix where the pair's super-block records do not fit a CTA's shared memory (at
 * N = 28672, K = 8192 for instance). */
W4A16_API w4a16_status q4k_linear_dual(const void* x_bf16, const uint32_t* qweight_gate, const uint32_t* meta_gate,
                                       const uint32_t* qweight_up, const uint32_t* meta_up, int64_t M, int64_t N,
                                       int64_t K, void* y_gate_bf16, void* y_up_bf16, w4a16_stream_t stream);

/*
 * Which kernel w4a16_linear would run for this shape: 1 = GEMV, 2 = GEMM,
 * 0 = the shape is rejected.  Host-only, no device access.
 */
W4A16_API int w4a16_linear_path(int64_t M, int64_t N, int64_t K, int G);

/*
 * Every wait inside the kernels on an asynchronous copy or a pipeline barrier
 * is bounded: after a spin budget (default 2^31 SM cycles, about 1 s) the
 * waiting warp records a code in a per-device status word, the kernel stops
 * issuing work, waits (again bounded) for the copies and MMAs it did issue,
 * frees its tensor memory and returns; nothing traps.  This call synchronises
 * the current device, returns W4A16_ERR_TIMEOUT if any kernel recorded a
 * give-up since the last call (and clears the word), else W4A16_OK.  *detail
 * (optional) receives the raw word: bit 0 tensor-core producer, 1 its MMA
 * issuer, 2 its dequantisers, 3 its epilogue, 4 a tensor-core drain that also
 * ran out, 8 the decode kernel, 9 a decode drain that also ran out.
 */
W4A16_API w4a16_status w4a16_device_status(uint32_t* detail);

/*
 * Testing hooks for the give-up path above (not needed in normal use).  The
 * pages this library follows have no counterpart; they exist so that a test
 * can make a wait run out without faulting, trapping or hanging the GPU.
 * w4a16_debug_set_wait_limit: the spin budget, in SM cycles, of every bounded
 *   wait in launches made after the call (any device, any thread); cycles <= 0
 *   restores the default.
 * w4a16_debug_withhold_copy: arms the NEXT launch of one kernel (1 = decode
 *   kernel, 2 = tensor-core kernel; 0 disarms) to withhold one copy by
 *   construction: the decode kernel's first warp of its first block never
 *   issues its first unit of weights, the tensor-core kernel's first block
 *   never issues its first slice of codes.  No copy or MMA is ever in flight
 *   against the withheld barrier, so the waiting warps give up after the spin
 *   budget, the kernel drains what it did issue and returns; that launch's
 *   outputs are undefined and w4a16_device_status reports the timeout.
 *   W4A16_ERR_INVALID_ARG for a kernel outside 0..2.
 */
W4A16_API void w4a16_debug_set_wait_limit(int64_t cycles);
W4A16_API w4a16_status w4a16_debug_withhold_copy(int kernel);

/*
 * w4a16_debug_gemv_plan: how the decode kernel would run one 4-bit matrix
 * [N, K] at M activation rows on the current device (host only, launches
 * nothing): plan[0] = segments per row P, plan[1] = group parities H,
 * plan[2] = warps per CTA, plan[3] = 1 when K is split across two-CTA
 * clusters, plan[4] = CTAs, plan[5] = ring units per warp.  mode 0: the plan
 * the layer takes; 1: the plain kernel's; 2: the K split's.  plan is a HOST
 * array of 6 int32.  Returns W4A16_OK, W4A16_ERR_UNSUPPORTED when that plan
 * cannot take the shape, W4A16_ERR_INVALID_ARG for a null plan, a mode
 * outside 0..2 or a bad shape.  For tests of the planner; the layer calls
 * plan by themselves.
 */
W4A16_API w4a16_status w4a16_debug_gemv_plan(int64_t M, int64_t N, int64_t K, int G, int mode, int32_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
