// pa_decode.cu -- bf16-cache instantiation of the paged GQA decode kernel
// (pa_decode_kernel.cuh), the log-sum-exp merge of the split partitions, and the
// decode / merge dispatch.
#include <initializer_list>

#include "pa_decode_kernel.cuh"

namespace pa {
namespace {

// Log-sum-exp merge of the split partitions of one (sequence, query head):
// M = max m_p, w_p = l_p exp(m_p - M), out = sum w_p o_p / sum w_p.
template <int HD>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int DG = HD / 4;     // float4 groups of a row
    constexpr int PL = 256 / DG;   // partition lanes
    __shared__ float red[PL][HD];
    __shared__ float stat[8];
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the partials are complete
    const int h = blockIdx.x, b = blockIdx.y;
    const int nq = p.num_q_heads;
    int L = p.seq_lens[b];
    if (L < 0) L = 0;
    if (L > p.max_seq_len) L = p.max_seq_len;
    // the partitions from the window's first one (all of them without a window)
    const int p0 = window_start(L, p.window) / kPartition;
    const int np = (L + kPartition - 1) / kPartition - p0;
    const int64_t row0 = (static_cast<int64_t>(b) * nq + h) * p.max_parts + p0;
    const float *pm = p.part_m + row0;
    const float *pl = p.part_l + row0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    float mx = -INFINITY;
    for (int i = tid; i < np; i += 256) mx = fmaxf(mx, pm[i]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    if (lane == 0) stat[warp] = mx;
    __syncthreads();
    float M = stat[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) M = fmaxf(M, stat[w]);
    __syncthreads();
    float wsum = 0.f;
    for (int i = tid; i < np; i += 256)
        wsum += (pm[i] == -INFINITY) ? 0.f : pl[i] * exp2f((pm[i] - M) * kLog2e);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) wsum += __shfl_xor_sync(kFull, wsum, off);
    if (lane == 0) stat[warp] = wsum;
    __syncthreads();
    float W = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) W += stat[w];

    const int dg = tid % DG, pi = tid / DG;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = pi; i < np; i += PL) {
        const float wi = (pm[i] == -INFINITY) ? 0.f : pl[i] * exp2f((pm[i] - M) * kLog2e);
        const float4 o = reinterpret_cast<const float4 *>(p.part_o + (row0 + i) * HD)[dg];
        a.x = fmaf(wi, o.x, a.x);
        a.y = fmaf(wi, o.y, a.y);
        a.z = fmaf(wi, o.z, a.z);
        a.w = fmaf(wi, o.w, a.w);
    }
    reinterpret_cast<float4 *>(&red[pi][0])[dg] = a;
    __syncthreads();
    if (tid < HD) {
        float o = 0.f;
#pragma unroll
        for (int i = 0; i < PL; ++i) o += red[i][tid];
        const float inv = W > 0.f ? 1.f / W : 0.f;
        static_cast<__nv_bfloat16 *>(p.out)[(static_cast<int64_t>(b) * nq + h) * HD + tid] =
            __float2bfloat16_rn(o * inv);
    }
}

// The same merge with one warp per (sequence, query head), for calls whose sequences
// have at most 32 partitions: lane i holds partition i's (m, l), the max and the
// weight sum are warp reductions, and each lane accumulates HD / 32 output dims over
// the partitions -- no block-wide syncs, so short-sequence batches are not bound by
// the latency of a 256-thread reduction per (sequence, head).
template <int HD>
__global__ void __launch_bounds__(256) merge_warp_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int DPL = HD / 32;   // output dims per lane
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the partials are complete
    const int lane = threadIdx.x & 31;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int nq = p.num_q_heads;
    if (gw >= static_cast<int64_t>(p.num_seqs) * nq) return;
    const int b = static_cast<int>(gw / nq), h = static_cast<int>(gw % nq);
    int L = p.seq_lens[b];
    if (L < 0) L = 0;
    if (L > p.max_seq_len) L = p.max_seq_len;
    const int p0 = window_start(L, p.window) / kPartition;
    const int np = (L + kPartition - 1) / kPartition - p0;   // <= 32 for this kernel
    const int64_t row0 = (static_cast<int64_t>(b) * nq + h) * p.max_parts + p0;
    // Every load is issued before any result is needed: m_p and l_p of partition `lane`,
    // and the partial outputs of the first kChunk partitions, so the merge costs one
    // memory round trip rather than one per dependent step.
    constexpr int kChunk = 8;
    const bool mine = lane < np;
    const float mi = mine ? p.part_m[row0 + lane] : -INFINITY;
    const float li = mine ? p.part_l[row0 + lane] : 0.f;
    float2 ov[kChunk][DPL / 2];
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
#pragma unroll
        for (int d = 0; d < DPL; d += 2)
            ov[i][d / 2] = i < np ? *reinterpret_cast<const float2 *>(
                                        p.part_o + (row0 + i) * HD + lane * DPL + d)
                                  : make_float2(0.f, 0.f);
    float M = mi;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    const float wi = (mine && mi != -INFINITY) ? li * exp2f((mi - M) * kLog2e) : 0.f;
    float W = wi;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) W += __shfl_xor_sync(kFull, W, off);
    float acc[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
        const float w = __shfl_sync(kFull, wi, i);
#pragma unroll
        for (int d = 0; d < DPL; d += 2) {
            acc[d] = fmaf(w, ov[i][d / 2].x, acc[d]);
            acc[d + 1] = fmaf(w, ov[i][d / 2].y, acc[d + 1]);
        }
    }
    for (int i = kChunk; i < np; ++i) {           // more than kChunk partitions
        const float w = __shfl_sync(kFull, wi, i);
        const float *o = p.part_o + (row0 + i) * HD + lane * DPL;
#pragma unroll
        for (int d = 0; d < DPL; d += 2) {
            const float2 v = *reinterpret_cast<const float2 *>(o + d);
            acc[d] = fmaf(w, v.x, acc[d]);
            acc[d + 1] = fmaf(w, v.y, acc[d + 1]);
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) + (static_cast<int64_t>(b) * nq + h) * HD +
                         lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; d += 2)
        *reinterpret_cast<__nv_bfloat162 *>(out + d) = __floats2bfloat162_rn(acc[d] * inv, acc[d + 1] * inv);
}

}  // namespace


namespace {

// The call's kv heads as kernel groups of g query heads: each pool kv head then serves
// G / g groups (kv_rep), which read its pages through L2.
DecodeParams regroup(const DecodeParams &p, int g) {
    DecodeParams r = p;
    const int G = p.num_q_heads / p.num_kv_heads;
    r.num_kv_heads = p.num_q_heads / g;
    r.kv_rep = G / g;
    r.pool_kv_heads = p.num_kv_heads;
    return r;
}

// The largest of cands (descending) that divides G, or 0.
int largest_divisor(int G, std::initializer_list<int> cands) {
    for (int c : cands)
        if (G % c == 0) return c;
    return 0;
}

}  // namespace

// Any GQA group size G = nq / nkv ("paged_attn.py", forward_decode's num_queries_per_kv).
// Kernels exist for some group sizes: the bf16 tensor-core decode for 3-16 query heads at
// head_dim 128 (its MMA's N) and 3-8 at head_dim 64, the fp8 one for 3-8 at head_dim 128
// (hi and lo rows fill N), the CUDA-core decode for 1, 2, 4 and 8.  A call runs on the first path with a kernel for G, else for
// the largest divisor of G it has: bf16 G = 32 as two groups of 16 per kv head, fp8
// G = 12 as two of 6, and a prime G above 16 (above 8 with fp8) on the CUDA cores as G
// groups of one.  Groups of 1 and 2 stay on the CUDA cores, which stream them at the
// copy peak.
cudaError_t launch_decode(const DecodeParams &p0, int head_dim, bool split, cudaStream_t stream) {
    if (p0.num_seqs == 0) return cudaSuccess;
    const int G = p0.num_q_heads / p0.num_kv_heads;
    const int g_max = p0.kv_fp8 ? 8 : decode_tc_max_group(head_dim);
    int g_tc = 0;
    for (int c = g_max; G > 2 && c >= 3 && !g_tc; --c)
        if (G % c == 0) g_tc = c;
    if (g_tc) {
        const DecodeParams p = regroup(p0, g_tc);
        if (decode_tc_supported(p, head_dim))
            return split ? launch_decode_tc(p, head_dim, stream)
                         : launch_decode_tc_single(p, head_dim, stream);
        if (decode_tc8_supported(p, head_dim))
            return split ? launch_decode_tc8(p, stream) : launch_decode_tc8_single(p, stream);
    }
    const DecodeParams p = regroup(p0, largest_divisor(G, {8, 4, 2, 1}));
    if (p.kv_fp8) return launch_decode_fp8(p, head_dim, split, stream);
    return launch_decode_cache<false>(p, head_dim, split, stream);
}

cudaError_t launch_merge(const DecodeParams &p, int head_dim, cudaStream_t stream) {
    if (p.num_seqs == 0) return cudaSuccess;
    if (active_partitions_cap(p.max_parts, p.window) <= 32) {   // one warp per (sequence, head)
        const int64_t warps = static_cast<int64_t>(p.num_seqs) * p.num_q_heads;
        const dim3 wgrid(static_cast<unsigned>((warps + 7) / 8));
        switch (head_dim) {
            case 64: return launch_dependent(merge_warp_kernel<64>, wgrid, dim3(256), 0, stream, p);
            case 128: return launch_dependent(merge_warp_kernel<128>, wgrid, dim3(256), 0, stream, p);
            case 256: return launch_dependent(merge_warp_kernel<256>, wgrid, dim3(256), 0, stream, p);
            default: return cudaErrorNotSupported;
        }
    }
    const dim3 grid(p.num_q_heads, p.num_seqs);
    switch (head_dim) {
        case 64: return launch_dependent(merge_kernel<64>, grid, dim3(256), 0, stream, p);
        case 128: return launch_dependent(merge_kernel<128>, grid, dim3(256), 0, stream, p);
        case 256: return launch_dependent(merge_kernel<256>, grid, dim3(256), 0, stream, p);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
