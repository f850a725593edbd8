// xt_tmap.cu -- host-side TMA tensor-map encoding (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry-point query, so the library
// needs no link-time dependency on libcuda), and the cached SM count that
// sizes the persistent grids.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "xt_internal.h"

namespace xt {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    });
    return fn;
}

}  // namespace

namespace {

cudaError_t encode_tmap(CUtensorMap *map, CUtensorMapDataType type, const void *base, int rank,
                        const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                        int swizzle_bytes) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; es[i] = 1; }
    for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
    CUresult r = enc(map, type, (cuuint32_t)rank, const_cast<void *>(base), d, s, b, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int sm_count() {
    static int cache[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms < 1)
            return 148;
        cache[dev] = sms;
    }
    return cache[dev];
}

// A tensor of `rank` dims (innermost first), byte strides of dims 1..rank-1,
// box sizes per dim, 128- or 64-byte swizzle, zero fill out of bounds.
cudaError_t encode_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                             const uint64_t *strides_bytes, const uint32_t *box,
                             int swizzle_bytes) {
    return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes,
                       box, swizzle_bytes);
}

cudaError_t encode_tmap_f32(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                            const uint64_t *strides_bytes, const uint32_t *box,
                            int swizzle_bytes) {
    return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, rank, dims, strides_bytes,
                       box, swizzle_bytes);
}

}  // namespace xt
