// noalloc.cu - routing without a handle and without any device allocation.
//
// Some callers cannot allocate device memory themselves: a serving process
// whose device heap is owned by a pooling allocator with a fixed budget, or a
// latency-critical path that must not take cudaMalloc's implicit device-wide
// synchronisation. moe_route_noalloc gives them the routing step (router,
// expert offsets, stable permutation) using the same kernels as moe_route,
// with all intermediate data in one file-scope device array instead of a
// handle's workspace. The caller passes only inputs and outputs.
//
// The array is part of the library image: every GPU that loads the library
// holds it (about 1.3 MB) until the process exits. All calls share it, so
// calls that overlap on the GPU race; the caller orders them (one stream, or
// events). Its contents persist between calls; everything a call reads is
// written earlier in the same call, except the device error word, which each
// call clears first.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

using namespace moe;

namespace {

constexpr size_t align256(size_t v) { return (v + 255) / 256 * 256; }

constexpr int kMaxTokens = MOE_ROUTE_NOALLOC_MAX_TOKENS;
constexpr int kMaxBlocks = (kMaxTokens + kRouterTokens - 1) / kRouterTokens;
constexpr size_t kErrOff = 0;
constexpr size_t kHistOff = 256;
constexpr size_t kBaseOff = kHistOff + align256((size_t)kMaxBlocks * kMaxExperts * 4);
constexpr size_t kInvOff = kBaseOff + align256((size_t)kMaxBlocks * kMaxExperts * 4);
constexpr size_t kTilesTcOff = kInvOff + align256((size_t)kMaxTokens * kMaxTopK * 4);
constexpr size_t kTilesSimtOff = kTilesTcOff + align256((kMaxExperts + 1) * 4);
constexpr size_t kSharedOff = kTilesSimtOff + align256((kMaxExperts + 1) * 4);
constexpr size_t kScratchBytes = kSharedOff + 256;

__device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

// Device address of g_route_scratch per device, looked up once per device.
// The address belongs to the device's primary context; the cache assumes that
// context lives as long as the process (no cudaDeviceReset in between).
std::mutex g_mu;
constexpr int kMaxDevices = 64;
void* g_addr[kMaxDevices] = {};

cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_route_noalloc(const void* x, const void* router_w, const float* router_bias, int32_t T,
                                        int32_t hidden, int32_t num_experts, int32_t top_k, int32_t dtype,
                                        int32_t* topk_ids, float* topk_w, int32_t* perm, int32_t* offsets,
                                        void* stream) {
    if (T < 0 || T > kMaxTokens || hidden <= 0 || hidden % (dtype == MOE_BF16 ? 64 : 32) != 0 || num_experts <= 0 ||
        num_experts > kMaxExperts || top_k <= 0 || top_k > num_experts || top_k > kMaxTopK ||
        (dtype != MOE_F32 && dtype != MOE_BF16))
        return MOE_ERR_INVALID_ARG;
    if (offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (x == nullptr || router_w == nullptr || topk_ids == nullptr || topk_w == nullptr || perm == nullptr))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(router_w)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return MOE_ERR_CUDA;
    unsigned char* b = static_cast<unsigned char*>(base);
    int* err = reinterpret_cast<int*>(b + kErrOff);
    if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (T == 0) {
        return cudaMemsetAsync(offsets, 0, (size_t)(num_experts + 1) * 4, s) == cudaSuccess ? MOE_OK
                                                                                            : MOE_ERR_CUDA;
    }
    int32_t* hist = reinterpret_cast<int32_t*>(b + kHistOff);
    int32_t* blk_base = reinterpret_cast<int32_t*>(b + kBaseOff);
    int32_t* inv = reinterpret_cast<int32_t*>(b + kInvOff);
    int32_t* tiles_tc = reinterpret_cast<int32_t*>(b + kTilesTcOff);
    int32_t* tiles_simt = reinterpret_cast<int32_t*>(b + kTilesSimtOff);
    int32_t* shared = reinterpret_cast<int32_t*>(b + kSharedOff);
    RoutingJob j{x, router_w, router_bias, T, hidden, num_experts, top_k, dtype == MOE_BF16, topk_ids, topk_w,
                 nullptr, perm, inv, offsets, tiles_tc, tiles_simt, shared, hist, blk_base, err,
                 2000000000ull, nullptr, 0};
    if (enqueue_routing(j, s, nullptr) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

extern "C" moe_status moe_route_noalloc_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int word = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_route_scratch, sizeof word, kErrOff, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (word & kErrTimeout) return MOE_ERR_TIMEOUT;
    if (word & kErrCheck) return MOE_ERR_DEVICE_CHECK;
    return MOE_OK;
}
