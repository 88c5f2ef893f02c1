// routing.cu - the routing launch sequence and tensor-map encoding shared by
// every entry point that routes (moe_route, moe_forward, moe_route_noalloc).
#include "kernels.h"

namespace moe {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// SMs of the current device, looked up once per device.
int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev);
    return cached[dev];
}

template <typename F>
cudaError_t hooked(const LaunchHook* hook, int slot, cudaStream_t s, F&& launch) {
    if (hook && hook->before) hook->before(hook->ctx, slot, s);
    cudaError_t e = launch();
    if (hook && hook->after) hook->after(hook->ctx, slot, s, e);
    return e;
}

}  // namespace

bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                    uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)kTcBK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_u8_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_nd(CUtensorMap* m, bool bf16, const void* base, int rank, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box, bool swizzle128) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank,
               const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap* m, bool bf16, const void* base, const uint64_t dims[3], const uint64_t strides[2],
               const uint32_t box[3], bool swizzle128) {
    return encode_nd(m, bf16, base, 3, dims, strides, box, swizzle128);
}

cudaError_t enqueue_routing(const RoutingJob& j, cudaStream_t s, const LaunchHook* hook) {
    cudaError_t e;
    int NB, tpb;
    if (j.bf16) {
        const bool small = j.T <= kSmallTokens;
        CUtensorMap tmX, tmW;
        if (!encode_bf16_2d(&tmX, j.x, j.H, j.T, (uint64_t)j.H * 2, small ? kSmallTokens : kRouterTokensTc) ||
            !encode_bf16_2d(&tmW, j.wr, j.H, j.E, (uint64_t)j.H * 2, 64))
            return cudaErrorInvalidValue;
        RouterTcArgs ra{j.bias, j.T, j.H, j.E, j.k, j.ids, j.w, j.logits, j.blk_hist, j.offsets, j.tiles_tc,
                        j.tiles_simt, j.shared_meta, j.shared_meta + 2, j.shared_meta + 4, j.perm, j.inv,
                        j.zero_counters, j.zero_count, j.err, j.limit_ns};
        // one CTA (T <= 128) also scans and places; batches whose 4-CTA
        // clusters fit the GPU at once split K; larger ones keep one CTA per
        // 128 tokens, several waves of which already fill the GPU
        const bool single = j.T <= kRouterTokensTc;
        const bool split = !single && (int64_t)(j.T + kRouterTokensTc - 1) / kRouterTokensTc * 4 <= num_sms();
        e = hooked(hook, kSlotRouter, s, [&] {
            return small ? launch_router_tc_small(ra, tmX, tmW, s)
                   : split ? launch_router_tc_split(ra, tmX, tmW, s) : launch_router_tc(ra, tmX, tmW, s);
        });
        if (e != cudaSuccess) return e;
        if (single) return cudaSuccess;
        tpb = kRouterTokensTc;
        NB = (j.T + tpb - 1) / tpb;
    } else {
        tpb = kRouterTokens;
        NB = (j.T + tpb - 1) / tpb;
        RouterArgs ra{j.x, j.wr, j.bias, j.T, j.H, j.E, j.k, false, j.ids, j.w, j.logits, j.blk_hist, j.err};
        if ((e = hooked(hook, kSlotRouter, s, [&] { return launch_router(ra, s); })) != cudaSuccess) return e;
    }
    ScanArgs sa{j.blk_hist, NB, j.E, j.T, j.k, j.blk_base, j.offsets, j.tiles_tc, j.tiles_simt, j.shared_meta,
                j.shared_meta + 2, j.shared_meta + 4};
    PlaceArgs pa{j.ids, j.blk_base, j.T, j.k, j.E, NB, tpb, j.perm, j.inv, j.err};
    if ((int64_t)NB * j.E <= kScanPlaceMaxInts)
        return hooked(hook, kSlotPlace, s, [&] { return launch_scan_place(sa, pa, s); });
    if ((e = hooked(hook, kSlotScan, s, [&] { return launch_scan(sa, s); })) != cudaSuccess) return e;
    return hooked(hook, kSlotPlace, s, [&] { return launch_place(pa, s); });
}

}  // namespace moe
