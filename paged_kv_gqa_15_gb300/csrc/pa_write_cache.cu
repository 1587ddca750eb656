// pa_write_cache.cu -- reshape_and_cache for sm_103a.
//
// What it computes ("paged_attn.py", PagedAttention.write_to_paged_cache,
// which hands key / value / slot_mapping.flatten() to reshape_and_cache): for
// each new token t with slot = slot_mapping[t] >= 0, the K and V rows of every
// kv head go to page slot / block_size, row slot % block_size -- a bit copy.
//
// One thread moves one 16-byte chunk of one (token, kv head) row of K and the
// same chunk of V: loads from the contiguous [T][nkv][hd] inputs are fully
// coalesced, and each page row is written as whole 16-byte vectors.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) write_cache_kernel(const __grid_constant__ WriteCacheParams p) {
    // a decode launched next in the stream may start up now; it waits for this grid
    // to complete before reading the cache
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int cpr = p.head_dim / 8;                  // 16-byte chunks per row
    const int64_t per_tok = static_cast<int64_t>(p.num_kv_heads) * cpr;
    const int64_t total = p.num_tokens * per_tok;
    const int64_t capacity = p.num_blocks * p.block_size;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = idx / per_tok;
        const int64_t rem = idx - t * per_tok;
        const int h = static_cast<int>(rem / cpr);
        const int c = static_cast<int>(rem - static_cast<int64_t>(h) * cpr);
        const int64_t slot = __ldg(p.slot_mapping + t);
        if (slot < 0) continue;  // padding token
        if (slot >= capacity) {
            if (rem == 0) atomicOr(p.status, kStatusBounds);
            continue;
        }
        const int64_t page = slot / p.block_size;
        const int64_t row = slot - page * p.block_size;
        const int64_t dst = page * p.s_block + h * p.s_head + row * p.s_token + c * 8;
        const int64_t src = idx * 8;  // == ((t * nkv + h) * hd + c * 8)
        const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.k) + src));
        const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.v) + src));
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.k_cache) + dst) = kv;
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.v_cache) + dst) = vv;
    }
}

}  // namespace

cudaError_t launch_write_cache(const WriteCacheParams &p, cudaStream_t stream) {
    const int64_t total = p.num_tokens * p.num_kv_heads * (p.head_dim / 8);
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;  // grid-stride beyond 16 CTAs per SM
    write_cache_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pa
