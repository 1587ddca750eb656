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
//
// With an FP8 E4M3 cache (kv_cache_dtype "fp8" with k_scale / v_scale, the same
// function of "paged_attn.py") the thread stores its 8 elements as the 8 codes of
// x / scale: the quotient in fp32 (IEEE division), rounded to the nearest E4M3
// value with ties to even and saturation at +-448 by the hardware conversion.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// E4M3 codes of x[0..7] / scale, packed little-endian into 8 bytes.
__device__ __forceinline__ uint2 quantize8_e4m3(const uint4 &bf, float scale) {
    const uint32_t w[4] = {bf.x, bf.y, bf.z, bf.w};
    uint32_t out[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint16_t h[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t pair = w[2 * i + j];
            const float lo = __fdiv_rn(__uint_as_float(pair << 16), scale);
            const float hi = __fdiv_rn(__uint_as_float(pair & 0xffff0000u), scale);
            // the first source operand goes to the upper byte
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h[j]) : "f"(hi), "f"(lo));
        }
        out[i] = static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16);
    }
    return make_uint2(out[0], out[1]);
}

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
        if (p.kv_fp8) {   // byte elements: dst is an 8-byte-aligned byte offset
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(p.k_cache) + dst) =
                quantize8_e4m3(kv, p.k_scale);
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(p.v_cache) + dst) =
                quantize8_e4m3(vv, p.v_scale);
        } else {
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.k_cache) + dst) = kv;
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.v_cache) + dst) = vv;
        }
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
