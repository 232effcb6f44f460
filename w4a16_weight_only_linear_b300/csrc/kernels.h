// kernels.h -- internal launchers behind the C ABI (not part of the public header).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace w4a16 {

constexpr int kMaxDevices = 64;

// The current device and its attributes, read once per device (host.cu).
struct DeviceInfo {
    int dev;
    int sms;
    size_t smem_optin;   // largest dynamic shared memory a block may opt into
};
cudaError_t current_device(DeviceInfo& info);

// Cycles a kernel's bounded wait spins before it gives up (host.cu; settable for tests).
long long wait_limit();
void set_wait_limit(long long cycles);   // <= 0 restores the default
// Test hook: arm (kernel 1 = decode, 2 = tensor-core, 0 = off) one launch that withholds
// one copy; take_withhold returns true once for the armed kernel and disarms it.
void arm_withhold(int kernel);
bool take_withhold(int kernel);

// 2-D row-major tensor [outer][inner] with 128-byte swizzled (or plain) boxes;
// encoded maps are cached by every argument (host.cu).  False if the driver's
// encoder is unavailable or rejects the arguments.
bool tmap_encoder_available();
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, int dev, bool swizzle128 = true);

cudaError_t launch_pack(const void* w, int64_t N, int64_t K, int G, uint32_t* qw, void* sc, uint32_t* zr,
                        cudaStream_t stream);
// The 8-bit packer: codes as two 4-bit planes of a 2K-channel 4-bit layer (see pack.cu).
cudaError_t launch_pack8(const void* w, int64_t N, int64_t K, int G, uint32_t* qw, void* sc, uint32_t* zr,
                         cudaStream_t stream);
// Checking aids through the layer kernels' expansion routines (see pack.cu):
// FP32 W_hat via the decode kernel's, FP16 RN(W_hat) via the tensor-core
// kernel's, FP32 W_hat of the super-block layout via the decode kernel's.
// The 8-bit packer in the word layout (four codes per word, 8-bit zeros; see pack.cu).
cudaError_t launch_pack8w(const void* w, int64_t N, int64_t K, int G, uint32_t* qw, void* sc, uint32_t* zr,
                          cudaStream_t stream);
cudaError_t launch_dequant(const uint32_t* qw, const void* sc, const uint32_t* zr, int64_t N, int64_t K, int G,
                           float* out, cudaStream_t stream);
cudaError_t launch_dequant_f16(const uint32_t* qw, const void* sc, const uint32_t* zr, int64_t N, int64_t K, int G,
                               void* out, cudaStream_t stream);
// The same aids for the 8-bit word layout (decode kernel: FP32; tensor-core kernel: FP16).
cudaError_t launch_dequant8w(const uint32_t* qw, const void* sc, const uint32_t* zr, int64_t N, int64_t K, int G,
                             float* out, cudaStream_t stream);
cudaError_t launch_dequant8w_f16(const uint32_t* qw, const void* sc, const uint32_t* zr, int64_t N, int64_t K, int G,
                                 void* out, cudaStream_t stream);
cudaError_t launch_dequant_q4k(const uint32_t* qw, const uint32_t* meta, int64_t N, int64_t K, float* out,
                               cudaStream_t stream);
// The super-block (Q4_K-style) packer: codes in the 4-bit layout, one 16-byte record per 256 channels
// (see pack.cu).  K a multiple of 256.
cudaError_t launch_pack_q4k(const void* w, int64_t N, int64_t K, uint32_t* qw, uint32_t* meta, cudaStream_t stream);

// Matrices one decode launch takes (sharing x).
constexpr int kMaxMat = 4;

// One packed weight matrix and the output it feeds; n = its rows (0: the call's N).
struct GemvMat {
    const uint32_t* q;
    const void* s;
    const uint32_t* z;
    void* y;
    int64_t n = 0;
};

// Whether the decode GEMV takes this shape (M <= 16 and its x staging plus
// stream rings fit the device's shared memory).  Host only.
// kq: the super-block layout (G = 32, M <= 8).
bool gemv_fits(int64_t M, int64_t N, int64_t K, int G, int nmat, bool kq = false);
// The same for nmat matrices of Ns[i] rows each.
// w8: the 8-bit word layout (K, G its real channels and group size; G <= 128, M <= 8).
bool gemv_fits(int64_t M, const int64_t* Ns, int nmat, int64_t K, int G, bool kq = false, bool w8 = false);
// Whether the 4-bit decode GEMV takes these matrices with all the warps of its instance (its
// launch bound; fewer when x leaves too little shared memory for the weight rings).  Host only.
bool gemv_runs_full(int64_t M, const int64_t* Ns, int nmat, int64_t K, int G);
// The plan of one 4-bit matrix: {P, H, warps, K split, CTAs, ring units per warp}; mode 0 the
// chosen plan, 1 the plain kernel's, 2 the K split's; false when that plan cannot take it.
bool gemv_describe(int64_t M, int64_t N, int64_t K, int G, int mode, int32_t* plan);

// y_i = x * W_hat_i^T for nmat (1..kMaxMat) matrices sharing x; matrix i has mats[i].n rows
// (0: N).
// xsc (optional, FP32 [K], 16-byte aligned): x_k is taken as x_k * xsc_k.
// kx (optional, 0 = K): row length of x; input channel k of the layer reads x[k mod kx]
// (the two-plane 8-bit layer is a 4-bit layer of K = 2 kx channels over x repeated).
// kq: the matrices are in the super-block layout (GemvMat.s = records, .z unused; G = 32,
// M <= 8, no xsc or kx).
// yf32: the outputs are FP32 [M, N] (the sums without the BF16 rounding).
cudaError_t launch_gemv(const void* x, const GemvMat* mats, int nmat, int64_t M, int64_t N, int64_t K, int G,
                        cudaStream_t stream, const float* xsc = nullptr, int64_t kx = 0, bool kq = false,
                        bool yf32 = false, bool w8 = false);

// Tensor-core path (any M): y_i = x * W_hat_i^T for nmat (1..kMaxMat) matrices
// sharing x, matrix i of mats[i].n rows (0: N); x is converted to FP16 once,
// into stream-ordered scratch.
// w8: 8-bit codes in the word layout (four per word, 8-bit zero points).
cudaError_t launch_gemm(const void* x, const GemvMat* mats, int nmat, int64_t M, int64_t N, int64_t K, int G,
                        cudaStream_t stream, const float* xsc = nullptr, int64_t kx = 0, bool yf32 = false,
                        bool w8 = false);
// The same tensor-core path for one matrix with the FP16 copy of x in a
// fixed-size file-scope device array (no allocation; M * K bounded by the
// header's W4A16_NOALLOC_MAX_X_ELEMS, else cudaErrorNotSupported).
cudaError_t launch_gemm_noalloc(const void* x, const GemvMat& mat, int64_t M, int64_t N, int64_t K, int G,
                                cudaStream_t stream);
// Activation rows per tensor-core tile for M rows.
int gemm_tile_n(int64_t M);

// Per-device status words written by kernels whose bounded waits gave up:
// synchronise, return the OR of both paths' words and clear them.
cudaError_t read_and_clear_status(uint32_t* word);
// The decode kernel's word (read and cleared; no synchronisation).
cudaError_t gemv_take_status(uint32_t* word);

}  // namespace w4a16
