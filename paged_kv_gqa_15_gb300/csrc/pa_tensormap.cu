// pa_tensormap.cu -- TMA tensor maps for the kernels, with a small cache.
//
// Encoding a map goes through the driver and costs the calling thread several
// microseconds; a decode step encodes three.  Serving calls repeat the same
// (pointer, shape, strides) again and again, so encoded maps are kept in a small
// table keyed by every input of the encoding and copied out on a hit.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

struct MapKey {
    const void *base;
    int rank;
    int dtype;
    cuuint64_t dims[5];
    cuuint64_t strides[4];
    cuuint32_t box[5];
};

struct MapEntry {
    bool used;
    MapKey key;
    CUtensorMap map;
};

constexpr int kCacheSize = 32;
std::mutex cache_mu;
MapEntry cache[kCacheSize];
int cache_next = 0;

}  // namespace

namespace {

bool encode_tensor_map(CUtensorMap *tm, CUtensorMapDataType dtype, const void *base, int rank,
                       const cuuint64_t *dims, const cuuint64_t *strides_bytes,
                       const cuuint32_t *box) {
    if (rank < 1 || rank > 5) return false;
    MapKey key;
    std::memset(&key, 0, sizeof key);
    key.base = base;
    key.rank = rank;
    key.dtype = static_cast<int>(dtype);
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank) key.strides[i] = strides_bytes[i];
    }
    {
        std::lock_guard<std::mutex> lock(cache_mu);
        for (int i = 0; i < kCacheSize; ++i) {
            if (cache[i].used && std::memcmp(&cache[i].key, &key, sizeof key) == 0) {
                *tm = cache[i].map;
                return true;
            }
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (fn(tm, dtype, rank, const_cast<void *>(base), dims,
           strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(cache_mu);
    MapEntry &e = cache[cache_next];
    cache_next = (cache_next + 1) % kCacheSize;
    e.used = true;
    e.key = key;
    e.map = *tm;
    return true;
}

}  // namespace

bool encode_tensor_map_bf16(CUtensorMap *tm, const void *base, int rank, const cuuint64_t *dims,
                            const cuuint64_t *strides_bytes, const cuuint32_t *box) {
    return encode_tensor_map(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims,
                             strides_bytes, box);
}

bool encode_tensor_map_u8(CUtensorMap *tm, const void *base, int rank, const cuuint64_t *dims,
                          const cuuint64_t *strides_bytes, const cuuint32_t *box) {
    return encode_tensor_map(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rank, dims, strides_bytes,
                             box);
}

}  // namespace pa
