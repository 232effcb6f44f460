// host.cu -- host-side state the launchers share: per-device attributes and a
// cache of TMA tensor maps.
//
// A decode launch moves tens of microseconds of weights; its host cost (device
// queries, two tensor-map encodes, the launch itself) is paid by every call,
// and in a decode loop that host time bounds the end-to-end rate once the
// kernels are fast.  So the attributes are read once per device and the
// encoded tensor maps are kept, keyed by everything that goes into them
// (base address, sizes, strides, box, swizzle).  A map depends on nothing
// else, so a hit is always the map a fresh encode would give, whatever
// happened to the memory in between; the library keeps no pointer it
// dereferences.  Both caches are guarded for calls from several host threads.
//
// It also holds the spin budget of the kernels' bounded waits and the one-shot
// test hook that makes one launch withhold a copy (see include/w4a16.h).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "kernels.h"

namespace w4a16 {

namespace {

std::atomic<int> g_sms[kMaxDevices];
std::atomic<long long> g_smem_optin[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

struct MapKey {
    const void* base;
    uint64_t inner, outer, row_bytes;
    uint32_t box_inner, box_outer;
    int dtype;
    int dev;
    int swizzle;
    bool operator==(const MapKey& o) const {
        return base == o.base && inner == o.inner && outer == o.outer && row_bytes == o.row_bytes &&
               box_inner == o.box_inner && box_outer == o.box_outer && dtype == o.dtype && dev == o.dev &&
               swizzle == o.swizzle;
    }
};

constexpr int kMapSlots = 512;   // direct-mapped; a miss re-encodes and replaces the slot
struct MapSlot {
    bool used = false;
    MapKey key{};
    CUtensorMap map{};
};
MapSlot g_maps[kMapSlots];
std::mutex g_maps_mu;

uint32_t key_hash(const MapKey& k) {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    h ^= (k.inner * 0xC2B2AE3D27D4EB4Full) ^ (k.outer * 0x165667B19E3779F9ull) ^ (k.row_bytes << 7);
    h ^= ((uint64_t)k.box_inner << 32) ^ ((uint64_t)k.box_outer << 16) ^
         (uint64_t)(k.dtype * 131 + k.dev * 7 + k.swizzle * 1031);
    h ^= h >> 29;
    return (uint32_t)(h % kMapSlots);
}

constexpr long long kDefaultWaitLimit = 1ll << 31;   // SM cycles, about 1 s at 2 GHz
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};
std::atomic<int> g_withhold{0};

}  // namespace

long long wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

void set_wait_limit(long long cycles) {
    g_wait_limit.store(cycles > 0 ? cycles : kDefaultWaitLimit, std::memory_order_relaxed);
}

void arm_withhold(int kernel) { g_withhold.store(kernel, std::memory_order_relaxed); }

bool take_withhold(int kernel) {
    int want = kernel;
    return g_withhold.load(std::memory_order_relaxed) == kernel &&
           g_withhold.compare_exchange_strong(want, 0, std::memory_order_relaxed);
}

cudaError_t current_device(DeviceInfo& info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    info.dev = dev;
    int sms = g_sms[dev].load(std::memory_order_relaxed);
    long long cap = g_smem_optin[dev].load(std::memory_order_relaxed);
    if (sms <= 0 || cap <= 0) {
        int v = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
        cap = v;
        g_sms[dev].store(sms, std::memory_order_relaxed);
        g_smem_optin[dev].store(cap, std::memory_order_relaxed);
    }
    info.sms = sms;
    info.smem_optin = (size_t)cap;
    return cudaSuccess;
}

bool tmap_encoder_available() { return encoder() != nullptr; }

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, int dev, bool swizzle128) {
    auto enc = encoder();
    if (!enc) return false;
    const MapKey key{base, inner, outer, row_bytes, box_inner, box_outer, (int)dt, dev, swizzle128 ? 1 : 0};
    const uint32_t h = key_hash(key);
    {
        std::lock_guard<std::mutex> lock(g_maps_mu);
        if (g_maps[h].used && g_maps[h].key == key) {
            std::memcpy(map, &g_maps[h].map, sizeof(CUtensorMap));
            return true;
        }
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    if (enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(g_maps_mu);
    g_maps[h].used = true;
    g_maps[h].key = key;
    std::memcpy(&g_maps[h].map, map, sizeof(CUtensorMap));
    return true;
}

}  // namespace w4a16
