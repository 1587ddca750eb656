// pa_blocks.cu -- whole-page copies between KV pools for sm_103a.
//
// What it computes ("paged_attn.py", PagedAttention.swap_blocks and
// PagedAttention.copy_blocks): for each (src, dst) pair of a block mapping, the
// bytes of page src of one pool become the bytes of page dst of another pool
// (swap_blocks: device <-> host for preemption) or of the same pool
// (copy_blocks: copy-on-write duplication of a shared page, for every layer's K
// and V pool at once).  A page is block_bytes contiguous bytes at byte offset
// page * block_bytes of its pool, as in a dense [num_blocks][...] pool of
// either page layout.
//
// The pages' own backend issues one copy-engine memcpy per pair.  Here every
// (pair, pool, 16 KB segment) is one unit of a single grid-stride kernel:
// small pages (a 16-token page is 1-64 KB) then cost no per-copy launch or
// engine set-up, and host pages move by plain loads and stores through the
// device's view of pinned host memory, over the CPU-GPU link.  Each thread keeps
// four 16-byte loads in flight before it stores, which hides the link's latency.
#include <cstring>

#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyVecs = 4;                                  // 16-byte vectors per thread
constexpr int64_t kSegBytes = kCopyThreads * kCopyVecs * 16;  // 16 KB per unit
constexpr int kMaxPoolsPerLaunch = 128;

struct BlockCopyParams {
    const uint8_t *src[kMaxPoolsPerLaunch];
    uint8_t *dst[kMaxPoolsPerLaunch];
    const int64_t *mapping;  // [num_pairs][2] (src page, dst page)
    int64_t num_pairs, src_blocks, dst_blocks, block_bytes, segs_per_page;
    int num_pools;
    int *status;
};

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}

__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__global__ void __launch_bounds__(kCopyThreads)
    block_copy_kernel(const __grid_constant__ BlockCopyParams p) {
    const int64_t per_pair = p.segs_per_page * p.num_pools;
    const int64_t units = p.num_pairs * per_pair;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t pair = u / per_pair;
        const int64_t rest = u - pair * per_pair;
        const int pool = static_cast<int>(rest / p.segs_per_page);
        const int64_t seg = rest - static_cast<int64_t>(pool) * p.segs_per_page;
        const int64_t s = p.mapping[2 * pair];
        const int64_t d = p.mapping[2 * pair + 1];
        if (s < 0 || d < 0) continue;  // padding pair
        if (s >= p.src_blocks || d >= p.dst_blocks) {
            if (threadIdx.x == 0 && rest == 0) atomicOr(p.status, kStatusBounds);
            continue;
        }
        const int64_t off = seg * kSegBytes;
        const int64_t nvec = min(kSegBytes, p.block_bytes - off) / 16;
        const uint4 *sp = reinterpret_cast<const uint4 *>(p.src[pool] + s * p.block_bytes + off);
        uint4 *dp = reinterpret_cast<uint4 *>(p.dst[pool] + d * p.block_bytes + off);
        uint4 r[kCopyVecs];
#pragma unroll
        for (int i = 0; i < kCopyVecs; ++i) {
            const int k = i * kCopyThreads + threadIdx.x;
            if (k < nvec) r[i] = ld_stream(sp + k);
        }
#pragma unroll
        for (int i = 0; i < kCopyVecs; ++i) {
            const int k = i * kCopyThreads + threadIdx.x;
            if (k < nvec) st_stream(dp + k, r[i]);
        }
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Enqueues the copies of pools [0, n) in launches of at most kMaxPoolsPerLaunch pools.
int launch_block_copies(const void *const *src, void *const *dst, int n, const int64_t *mapping,
                        int64_t num_pairs, int64_t src_blocks, int64_t dst_blocks,
                        int64_t block_bytes, cudaStream_t stream) {
    int *status = nullptr;
    int rc = api_status_ptr(&status);
    if (rc) return rc;
    BlockCopyParams p;
    std::memset(&p, 0, sizeof p);
    p.mapping = mapping;
    p.num_pairs = num_pairs;
    p.src_blocks = src_blocks;
    p.dst_blocks = dst_blocks;
    p.block_bytes = block_bytes;
    p.segs_per_page = (block_bytes + kSegBytes - 1) / kSegBytes;
    p.status = status;
    for (int first = 0; first < n; first += kMaxPoolsPerLaunch) {
        p.num_pools = n - first < kMaxPoolsPerLaunch ? n - first : kMaxPoolsPerLaunch;
        for (int i = 0; i < p.num_pools; ++i) {
            p.src[i] = static_cast<const uint8_t *>(src[first + i]);
            p.dst[i] = static_cast<uint8_t *>(dst[first + i]);
        }
        const int64_t units = num_pairs * p.num_pools * p.segs_per_page;
        const int64_t grid = units < 152 * 8 ? units : 152 * 8;  // 8 CTAs of 256 per SM
        block_copy_kernel<<<static_cast<unsigned>(grid), kCopyThreads, 0, stream>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return api_cuda_fail(e, "block_copy_kernel launch");
    }
    return PA_OK;
}

int check_copy_args(int num_pools, const int64_t *mapping, int64_t num_pairs,
                    int64_t block_bytes) {
    if (num_pools < 0) return api_fail(PA_ERR_INVALID, "num_pools %d", num_pools);
    if (num_pairs < 0) return api_fail(PA_ERR_INVALID, "num_pairs %lld", (long long)num_pairs);
    if (block_bytes <= 0 || block_bytes % 16)
        return api_fail(PA_ERR_INVALID, "block_bytes %lld must be a positive multiple of 16",
                        (long long)block_bytes);
    if (num_pairs > 0 && num_pools > 0 && !mapping)
        return api_fail(PA_ERR_INVALID, "block_mapping is NULL");
    return PA_OK;
}

// The device's address for `ptr`: device memory of the current device, pinned
// host memory mapped into the device's address space, or (where the device can
// read pageable host memory) any host address.
int device_view(const void *ptr, const char *what, int device, const void **out) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) return api_cuda_fail(e, "cudaPointerGetAttributes");
    switch (a.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            if (a.type == cudaMemoryTypeDevice && a.device != device)
                return api_fail(PA_ERR_INVALID, "%s is memory of device %d, not of device %d",
                                what, a.device, device);
            *out = a.devicePointer ? a.devicePointer : ptr;
            return PA_OK;
        case cudaMemoryTypeHost:
            if (!a.devicePointer)
                return api_fail(PA_ERR_INVALID,
                                "%s is pinned host memory that device %d cannot address", what,
                                device);
            *out = a.devicePointer;
            return PA_OK;
        default: {
            int pageable = 0;
            e = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, device);
            if (e != cudaSuccess) return api_cuda_fail(e, "cudaDeviceGetAttribute");
            if (!pageable)
                return api_fail(PA_ERR_INVALID,
                                "%s is pageable host memory; pin it (cudaHostAlloc or "
                                "cudaHostRegister)",
                                what);
            *out = ptr;
            return PA_OK;
        }
    }
}

}  // namespace
}  // namespace pa

extern "C" int pa_copy_blocks(void *const *pools, int num_pools, const int64_t *block_mapping,
                              int64_t num_pairs, int64_t num_blocks, int64_t block_bytes,
                              void *stream) {
    int rc = pa::check_copy_args(num_pools, block_mapping, num_pairs, block_bytes);
    if (rc) return rc;
    if (num_pairs == 0 || num_pools == 0) return PA_OK;
    if (num_blocks <= 0) return pa::api_fail(PA_ERR_INVALID, "num_blocks %lld", (long long)num_blocks);
    if (!pools) return pa::api_fail(PA_ERR_INVALID, "pools is NULL");
    for (int i = 0; i < num_pools; ++i) {
        if (!pools[i]) return pa::api_fail(PA_ERR_INVALID, "pools[%d] is NULL", i);
        if (!pa::aligned16(pools[i]))
            return pa::api_fail(PA_ERR_INVALID, "pools[%d] is not 16-byte aligned", i);
    }
    return pa::launch_block_copies(pools, pools, num_pools, block_mapping, num_pairs, num_blocks,
                                   num_blocks, block_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int pa_swap_blocks(const void *const *src_pools, void *const *dst_pools, int num_pools,
                              const int64_t *block_mapping, int64_t num_pairs,
                              int64_t src_num_blocks, int64_t dst_num_blocks,
                              int64_t block_bytes, void *stream) {
    int rc = pa::check_copy_args(num_pools, block_mapping, num_pairs, block_bytes);
    if (rc) return rc;
    if (num_pairs == 0 || num_pools == 0) return PA_OK;
    if (src_num_blocks <= 0 || dst_num_blocks <= 0)
        return pa::api_fail(PA_ERR_INVALID, "src_num_blocks %lld, dst_num_blocks %lld",
                            (long long)src_num_blocks, (long long)dst_num_blocks);
    if (!src_pools || !dst_pools) return pa::api_fail(PA_ERR_INVALID, "pool list is NULL");
    if (num_pools > 4096) return pa::api_fail(PA_ERR_UNSUPPORTED, "num_pools %d > 4096", num_pools);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return pa::api_cuda_fail(e, "cudaGetDevice");
    const void *map = nullptr;
    rc = pa::device_view(block_mapping, "block_mapping", device, &map);
    if (rc) return rc;
    if (reinterpret_cast<uintptr_t>(map) & 7u)
        return pa::api_fail(PA_ERR_INVALID, "block_mapping is not 8-byte aligned");
    static thread_local const void *src_v[4096];
    static thread_local void *dst_v[4096];
    for (int i = 0; i < num_pools; ++i) {
        if (!src_pools[i] || !dst_pools[i])
            return pa::api_fail(PA_ERR_INVALID, "pool %d is NULL", i);
        const void *sv = nullptr, *dv = nullptr;
        rc = pa::device_view(src_pools[i], "a source pool", device, &sv);
        if (rc) return rc;
        rc = pa::device_view(dst_pools[i], "a destination pool", device, &dv);
        if (rc) return rc;
        if (!pa::aligned16(sv) || !pa::aligned16(dv))
            return pa::api_fail(PA_ERR_INVALID, "pool %d is not 16-byte aligned", i);
        src_v[i] = sv;
        dst_v[i] = const_cast<void *>(dv);
    }
    return pa::launch_block_copies(src_v, dst_v, num_pools, static_cast<const int64_t *>(map),
                                   num_pairs, src_num_blocks, dst_num_blocks, block_bytes,
                                   static_cast<cudaStream_t>(stream));
}
