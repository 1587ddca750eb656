// pa_decode.cu -- paged GQA decode for sm_103a: single pass and split-KV
// partition pass, plus the log-sum-exp merge of the partitions.
//
// What it computes ("paged_attn.py", PagedAttention._forward_decode_pytorch
// and the V1 / V2 branches of forward_decode): for sequence b and kv head kh,
// the g = nq / nkv query heads kh*g .. kh*g+g-1 attend over the seq_lens[b]
// tokens of the sequence, token j living at page block_tables[b][j / 16],
// row j % 16.  The V2 branch splits the tokens into 512-token partitions and
// keeps per-partition max / sum / partial output, merged afterwards.
//
// GB300 design (not the pages' design):
//  * One CTA per (partition, kv head, sequence) serves the whole GQA group from
//    one read of each K / V page: every KV byte leaves HBM once per call.
//  * A producer warp streams the partition's pages into a shared-memory ring
//    with one bulk TMA copy per (page, kv head) -- a contiguous 4 KiB run for
//    head_dim 128 in the HND page layout -- so tens of KB per SM are in flight
//    without spending registers; mbarriers (full / empty) hand stages over.
//  * Consumer warps: thread (row r, chunk c) owns 8 dims of one token row of a
//    page.  Q for its 8 dims x g heads stays in registers for the whole CTA.
//    Partial dot products of U = 16 / g pages are reduced across the row's
//    lanes with a transposing butterfly (15 shuffles for 16 sums instead of 64).
//  * The 512 scaled scores of the partition go to shared memory; the max and
//    the exp-sum are block reductions; P then weights the V pages, still one
//    16-byte shared load per thread per page.  Between 512-token chunks of the
//    single-pass kernel the running (m, l, acc) are rescaled (online softmax).
//  * All waits are bounded; bad block ids are never dereferenced.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int HD, int G>
struct DecodeCfg {
    static constexpr int TPR = HD / 8;                 // threads per token row (16 B each)
    static constexpr int NC = kBlockSize * TPR;        // consumer threads: one page per pass
    static constexpr int NCW = NC / 32;                // consumer warps
    static constexpr int NT = NC + 32;                 // + one producer warp
    static constexpr int PAGE_BYTES = kBlockSize * HD * 2;
    static constexpr int RING_BYTES = (HD == 256 ? 96 : 64) * 1024;
    static constexpr int S = RING_BYTES / PAGE_BYTES;  // ring stages
    static constexpr int U = 16 / G;                   // pages per score-reduction group
    static constexpr int V = U * G;                    // partial sums per lane (= 16)
    static constexpr int NV = (V / TPR) > 0 ? (V / TPR) : 1;  // sums a lane keeps
    // shared memory layout (bytes)
    static constexpr int OFF_SC = RING_BYTES;                   // float [512][G]
    static constexpr int OFF_RED = OFF_SC + kPartition * G * 4;  // float [NCW][HD]
    static constexpr int OFF_RSTAT = OFF_RED + NCW * HD * 4;     // float [NCW][G]
    static constexpr int OFF_BAR = OFF_RSTAT + NCW * G * 4;      // uint64 full[S], empty[S]
    static constexpr int OFF_OK = OFF_BAR + 2 * S * 8;           // int [S]
    static constexpr int OFF_ABORT = OFF_OK + S * 4;             // int
    static constexpr int SMEM = OFF_ABORT + 16;
    static_assert(V == 16, "group sizes 1, 2, 4, 8");
    static_assert(OFF_BAR % 8 == 0, "barrier alignment");
};

// Reduces V partial sums across the TPR lanes of a token row.  Each of the
// first log2(min(V, TPR)) butterfly steps hands half of the remaining sums to
// the partner lane and keeps the other half, so lane l ends with the complete
// sums of indices [base, base + NV); further steps are plain butterflies.
template <int V, int TPR>
__device__ __forceinline__ int transpose_reduce(float (&v)[V], int lane) {
    int base = 0;
    int n = V;
#pragma unroll
    for (int mask = TPR / 2; mask >= 1; mask >>= 1) {
        if (n > 1) {
            const int half = n / 2;
            const bool upper = (lane & mask) != 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(kFull, send, mask);
                }
            }
            if (upper) base += half;
            n = half;
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], mask);
        }
    }
    return base;
}

template <int HD, int G, bool SPLIT>
__global__ void __launch_bounds__(DecodeCfg<HD, G>::NT, (HD == 256 || G == 8) ? 1 : 2)
    decode_kernel(const __grid_constant__ DecodeParams p) {
    using C = DecodeCfg<HD, G>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *ring = smem;
    float *sc = reinterpret_cast<float *>(smem + C::OFF_SC);
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);
    float *rstat = reinterpret_cast<float *>(smem + C::OFF_RSTAT);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::S;
    int *stage_ok = reinterpret_cast<int *>(smem + C::OFF_OK);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_ABORT);

    const int b = blockIdx.z;
    const int kh = blockIdx.y;
    int L = p.seq_lens[b];
    if (L < 0) L = 0;
    int cap = p.max_blocks * kBlockSize;
    if (SPLIT && p.max_seq_len < cap) cap = p.max_seq_len;
    if (L > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusBounds);
        L = cap;
    }
    const int n_chunks = (L + kPartition - 1) / kPartition;
    int ch_begin = 0, ch_end = n_chunks;
    if (SPLIT) {
        ch_begin = blockIdx.x;
        ch_end = blockIdx.x + 1;
        if (ch_begin >= n_chunks) return;  // partition past the sequence: nothing to do
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::NCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == C::NCW) {
        // ------------------------------ producer warp ------------------------------
        const uint64_t policy = l2_policy_evict_first();
        uint32_t it = 0;
        int stop = 0;  // warp-uniform
        const int32_t *bt_row = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
        for (int ch = ch_begin; ch < ch_end && !stop; ++ch) {
            const int t0 = ch * kPartition;
            const int n_tok = min(kPartition, L - t0);
            const int np = (n_tok + kBlockSize - 1) / kBlockSize;
            const int my_page = lane < np ? bt_row[t0 / kBlockSize + lane] : -1;
            for (int kv = 0; kv < 2 && !stop; ++kv) {
                const __nv_bfloat16 *base =
                    static_cast<const __nv_bfloat16 *>(kv ? p.v_cache : p.k_cache);
                for (int j = 0; j < np; ++j) {
                    const int page = __shfl_sync(kFull, my_page, j);
                    if (lane == 0) {
                        const int s = it % C::S;
                        const uint32_t ph = (it / C::S) & 1u;
                        if (!mbar_wait(&empty[s], ph ^ 1u, p.status, abort_flag)) {
                            stop = 1;
                        } else {
                            const bool ok = page >= 0 && page < p.num_blocks;
                            stage_ok[s] = ok ? 1 : 0;
                            if (ok) {
                                const __nv_bfloat16 *src =
                                    base + static_cast<int64_t>(page) * p.s_block +
                                    static_cast<int64_t>(kh) * p.s_head;
                                uint8_t *dst = ring + s * C::PAGE_BYTES;
                                mbar_arrive_expect_tx(&full[s], C::PAGE_BYTES);
                                if (p.rows_contiguous) {
                                    bulk_copy_g2s_hint(dst, src, C::PAGE_BYTES, &full[s], policy);
                                } else {
                                    for (int t = 0; t < kBlockSize; ++t)
                                        bulk_copy_g2s_hint(dst + t * HD * 2, src + t * p.s_token,
                                                           HD * 2, &full[s], policy);
                                }
                            } else {
                                atomicOr(p.status, kStatusBounds);
                                mbar_arrive(&full[s]);
                            }
                        }
                    }
                    stop = __shfl_sync(kFull, stop, 0);
                    if (stop) break;
                    ++it;  // stages issued so far
                }
            }
        }
        // Drain: never leave the CTA with bulk copies still landing in its smem.
        if (lane == 0 && (stop || *abort_flag)) {
            const uint32_t issued = it;
            for (uint32_t k = (issued > C::S ? issued - C::S : 0); k < issued; ++k) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&full[k % C::S], (k / C::S) & 1u)) {
                    if (global_timer_ns() - t0 > kWaitLimitNs) break;
                }
            }
        }
        return;
    }

    // -------------------------------- consumer warps --------------------------------
    const int tid = threadIdx.x;          // 0 .. NC-1
    const int r = tid / C::TPR;           // token row within a page
    const int c = tid % C::TPR;           // 16-byte chunk of the row
    const int nq = p.num_q_heads;

    float qf[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int h = kh * G + g;
        const uint4 raw = *reinterpret_cast<const uint4 *>(
            static_cast<const __nv_bfloat16 *>(p.q) + (static_cast<int64_t>(b) * nq + h) * HD +
            c * 8);
        unpack_bf16x8(raw, qf[g]);
#pragma unroll
        for (int i = 0; i < 8; ++i) qf[g][i] *= p.scale_log2;
    }

    float acc[G][8];
    float m_run[G], l_run[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[g][i] = 0.f;
    }

    uint32_t it = 0;
    bool aborted = false;
    for (int ch = ch_begin; ch < ch_end && !aborted; ++ch) {
        const int t0 = ch * kPartition;
        const int n_tok = min(kPartition, L - t0);
        const int np = (n_tok + kBlockSize - 1) / kBlockSize;

        // ---- K pages: scaled scores (log2 units) into sc ----
        for (int pg0 = 0; pg0 < np; pg0 += C::U) {
            float part[C::V];
            uint32_t okmask = 0;
#pragma unroll
            for (int u = 0; u < C::U; ++u) {
                if (pg0 + u < np) {
                    const int s = it % C::S;
                    const uint32_t ph = (it / C::S) & 1u;
                    ++it;
                    if (!mbar_wait(&full[s], ph, p.status, abort_flag)) {
                        aborted = true;
                    }
                    const int ok = aborted ? 0 : stage_ok[s];
                    const uint4 raw = *reinterpret_cast<const uint4 *>(
                        ring + s * C::PAGE_BYTES + r * HD * 2 + c * 16);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    float kf[8];
                    unpack_bf16x8(raw, kf);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float d = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) d = fmaf(qf[g][i], kf[i], d);
                        part[u * G + g] = d;
                    }
                    okmask |= static_cast<uint32_t>(ok) << u;
                } else {
#pragma unroll
                    for (int g = 0; g < G; ++g) part[u * G + g] = 0.f;
                }
            }
            const int base = transpose_reduce<C::V, C::TPR>(part, lane);
#pragma unroll
            for (int j = 0; j < C::NV; ++j) {
                const int idx = base + j;
                const int u = idx / G, g = idx % G;
                const int tok = (pg0 + u) * kBlockSize + r;
                if (pg0 + u < np) {
                    const bool valid = tok < n_tok && ((okmask >> u) & 1u);
                    sc[tok * G + g] = valid ? part[j] : -INFINITY;
                }
            }
        }
        if (named_barrier_or(1, C::NC, aborted)) {
            aborted = true;
            break;
        }

        // ---- softmax statistics of this chunk ----
        float cm[G];
#pragma unroll
        for (int g = 0; g < G; ++g) cm[g] = -INFINITY;
        for (int t = tid; t < n_tok; t += C::NC) {
#pragma unroll
            for (int g = 0; g < G; ++g) cm[g] = fmaxf(cm[g], sc[t * G + g]);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                cm[g] = fmaxf(cm[g], __shfl_xor_sync(kFull, cm[g], off));
        }
        if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) rstat[warp * G + g] = cm[g];
        }
        named_barrier(1, C::NC);
        float m_new[G], corr[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = m_run[g];
            for (int w = 0; w < C::NCW; ++w) mx = fmaxf(mx, rstat[w * G + g]);
            m_new[g] = mx;
            corr[g] = (m_run[g] == -INFINITY) ? 0.f : exp2f(m_run[g] - mx);
        }
        named_barrier(1, C::NC);  // rstat is reused below
        float ls[G];
#pragma unroll
        for (int g = 0; g < G; ++g) ls[g] = 0.f;
        for (int t = tid; t < n_tok; t += C::NC) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float sv = sc[t * G + g];
                const float pv = (sv == -INFINITY) ? 0.f : exp2f(sv - m_new[g]);
                sc[t * G + g] = pv;
                ls[g] += pv;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) ls[g] += __shfl_xor_sync(kFull, ls[g], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) rstat[warp * G + g] = ls[g];
        }
        named_barrier(1, C::NC);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float sum = 0.f;
            for (int w = 0; w < C::NCW; ++w) sum += rstat[w * G + g];
            l_run[g] = l_run[g] * corr[g] + sum;
            m_run[g] = m_new[g];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[g][i] *= corr[g];
        }

        // ---- V pages: acc += p * V ----
        for (int pg = 0; pg < np; ++pg) {
            const int s = it % C::S;
            const uint32_t ph = (it / C::S) & 1u;
            ++it;
            if (!mbar_wait(&full[s], ph, p.status, abort_flag)) {
                aborted = true;
            }
            const int ok = aborted ? 0 : stage_ok[s];
            const uint4 raw =
                *reinterpret_cast<const uint4 *>(ring + s * C::PAGE_BYTES + r * HD * 2 + c * 16);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            const int tok = pg * kBlockSize + r;
            if (ok && tok < n_tok) {
                float vf[8];
                unpack_bf16x8(raw, vf);
                float pw[G];
                if constexpr (G == 4) {
                    const float4 p4 = *reinterpret_cast<const float4 *>(sc + tok * 4);
                    pw[0] = p4.x; pw[1] = p4.y; pw[2] = p4.z; pw[3] = p4.w;
                } else {
#pragma unroll
                    for (int g = 0; g < G; ++g) pw[g] = sc[tok * G + g];
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[g][i] = fmaf(pw[g], vf[i], acc[g][i]);
                }
            }
        }
        if (named_barrier_or(1, C::NC, aborted)) {  // sc is rewritten by the next chunk
            aborted = true;
            break;
        }
    }
    if (aborted) return;

    // ---- reduce acc over the 16 rows: lanes of a warp, then warps via smem ----
#pragma unroll
    for (int mask = C::TPR; mask < 32; mask <<= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[g][i] += __shfl_xor_sync(kFull, acc[g][i], mask);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (lane < C::TPR) {
            float4 *dst = reinterpret_cast<float4 *>(red + warp * HD + c * 8);
            dst[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
            dst[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
        }
        named_barrier(1, C::NC);
        if (tid < HD) {
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < C::NCW; ++w) o += red[w * HD + tid];
            const int h = kh * G + g;
            const float inv = l_run[g] > 0.f ? 1.f / l_run[g] : 0.f;
            if constexpr (SPLIT) {
                const int64_t row = (static_cast<int64_t>(b) * nq + h) * p.max_parts + ch_begin;
                p.part_o[row * HD + tid] = o * inv;
                if (tid == 0) {
                    p.part_m[row] = m_run[g] * kLn2;
                    p.part_l[row] = l_run[g];
                }
            } else {
                static_cast<__nv_bfloat16 *>(p.out)[(static_cast<int64_t>(b) * nq + h) * HD + tid] =
                    __float2bfloat16_rn(o * inv);
            }
        }
        named_barrier(1, C::NC);
    }
}

// Log-sum-exp merge of the split partitions of one (sequence, query head):
// M = max m_p, w_p = l_p exp(m_p - M), out = sum w_p o_p / sum w_p.
template <int HD>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int DG = HD / 4;     // float4 groups of a row
    constexpr int PL = 256 / DG;   // partition lanes
    __shared__ float red[PL][HD];
    __shared__ float stat[8];
    const int h = blockIdx.x, b = blockIdx.y;
    const int nq = p.num_q_heads;
    int L = p.seq_lens[b];
    if (L < 0) L = 0;
    if (L > p.max_seq_len) L = p.max_seq_len;
    const int np = (L + kPartition - 1) / kPartition;
    const int64_t row0 = (static_cast<int64_t>(b) * nq + h) * p.max_parts;
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

template <int HD, int G, bool SPLIT>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t stream) {
    using C = DecodeCfg<HD, G>;
    auto kern = decode_kernel<HD, G, SPLIT>;
    static int configured_device = -1;  // cache of the smem opt-in (per process, last device)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const dim3 grid(SPLIT ? p.max_parts : 1, p.num_kv_heads, p.num_seqs);
    kern<<<grid, C::NT, C::SMEM, stream>>>(p);
    return cudaGetLastError();
}

template <int HD, bool SPLIT>
cudaError_t dispatch_group(const DecodeParams &p, cudaStream_t stream) {
    switch (p.num_q_heads / p.num_kv_heads) {
        case 1: return launch_decode_t<HD, 1, SPLIT>(p, stream);
        case 2: return launch_decode_t<HD, 2, SPLIT>(p, stream);
        case 4: return launch_decode_t<HD, 4, SPLIT>(p, stream);
        case 8: return launch_decode_t<HD, 8, SPLIT>(p, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, int head_dim, bool split, cudaStream_t stream) {
    if (p.num_seqs == 0) return cudaSuccess;
    switch (head_dim) {
        case 64: return split ? dispatch_group<64, true>(p, stream) : dispatch_group<64, false>(p, stream);
        case 128: return split ? dispatch_group<128, true>(p, stream) : dispatch_group<128, false>(p, stream);
        case 256: return split ? dispatch_group<256, true>(p, stream) : dispatch_group<256, false>(p, stream);
        default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_merge(const DecodeParams &p, int head_dim, cudaStream_t stream) {
    if (p.num_seqs == 0) return cudaSuccess;
    const dim3 grid(p.num_q_heads, p.num_seqs);
    switch (head_dim) {
        case 64: merge_kernel<64><<<grid, 256, 0, stream>>>(p); break;
        case 128: merge_kernel<128><<<grid, 256, 0, stream>>>(p); break;
        case 256: merge_kernel<256><<<grid, 256, 0, stream>>>(p); break;
        default: return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

}  // namespace pa
