// pa_device.cuh -- device-side building blocks shared by the kernels:
// mbarrier operations with bounded waits, bulk (TMA) copies, bf16 unpacking,
// and the device status word bits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kBlockSize = 16;     // tokens per KV page
constexpr int kPartition = 512;    // tokens per split-KV partition
constexpr int kStatusUnsupported = 1 << 2;   // bit of PA_ERR_UNSUPPORTED (2)
constexpr int kStatusTimeout = 1 << 5;   // bit of PA_ERR_TIMEOUT (5)
constexpr int kStatusBounds = 1 << 6;    // bit of PA_ERR_DEVICE_BOUNDS (6)
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Sliding window of `window` keys ("paged_attn.py", forward_prefix's sliding_window):
// a query at position pos sees keys j > pos - window.  First visible key of the query
// at position L - 1 (decode); 0 when there is no window (window <= 0).
__device__ __forceinline__ int window_start(int L, int window) {
    return (window > 0 && L > window) ? L - window : 0;
}

// Partitions a split-KV call with this window can have per sequence (the partitions
// from the one holding key L - window to the last), capped at max_parts.
__host__ __device__ __forceinline__ int active_partitions_cap(int max_parts, int window) {
    if (window <= 0) return max_parts;
    const int cap = (window - 1) / kPartition + 2;
    return cap < max_parts ? cap : max_parts;
}

// Two FP8 E4M3 codes (low 16 bits: the first in the low byte) as floats.  Every
// E4M3 value is exactly an f16 value, and every f16 value a float.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two)));
    float lo, hi;
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
    return make_float2(lo, hi);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Brings lines [idx * 128, bytes) of `base`, every stride-th 128-byte line, into L2.  A
// dependent launch may issue it before griddepcontrol.wait even for data the kernel
// before it writes: L2 is where writes become visible, so a later load sees them.
__device__ __forceinline__ void prefetch_l2_lines(const void *base, size_t bytes, unsigned idx,
                                                  unsigned stride) {
    const char *p = static_cast<const char *>(base);
    for (size_t off = static_cast<size_t>(idx) * 128; off < bytes;
         off += static_cast<size_t>(stride) * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
}

// The decode kernels' first reads after the dependency wait -- sequence lengths, block
// tables and q -- into L2 beforehand, spread over the grid (up to 4 MB of tables).
__device__ __forceinline__ void prefetch_decode_inputs(const int32_t *seq_lens,
                                                       const int32_t *block_tables,
                                                       const void *q, int num_seqs,
                                                       int max_blocks, size_t q_bytes,
                                                       unsigned t, unsigned nt) {
    const unsigned idx = blockIdx.x * nt + t, stride = gridDim.x * nt;
    prefetch_l2_lines(seq_lens, static_cast<size_t>(num_seqs) * 4, idx, stride);
    const size_t tb = static_cast<size_t>(num_seqs) * max_blocks * 4;
    if (tb <= (4u << 20)) prefetch_l2_lines(block_tables, tb, idx, stride);
    if (q_bytes <= (4u << 20)) prefetch_l2_lines(q, q_bytes, idx, stride);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// after kWaitLimitNs (records PA_ERR_TIMEOUT and raises the CTA's abort flag)
// or as soon as another thread of the CTA has raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status,
                                          volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, kStatusTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}

// One bulk (non-tensor TMA) copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on `bar`.  Addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (KV pages are streamed once per call).
__device__ __forceinline__ void bulk_copy_g2s_hint(void *dst, const void *src, uint32_t bytes,
                                                   uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Named barrier over `nthreads` threads (a multiple of 32) with id `id` (1..15).
// Cluster-wide barrier: every thread of every CTA of the cluster arrives (release) and
// waits (acquire); called by all threads of each warp together.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// The shared::cluster address of this CTA's shared-memory address `addr` in CTA `rank`
// of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t res;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(res)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return res != 0;
}

// 8 bf16 packed in a uint4 -> 8 floats (exact widening).
__device__ __forceinline__ void unpack_bf16x8(const uint4 &raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

}  // namespace pa
