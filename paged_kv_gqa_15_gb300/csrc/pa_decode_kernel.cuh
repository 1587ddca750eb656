#pragma once

#include <type_traits>

// pa_decode_kernel.cuh -- the paged GQA decode kernel (single pass and split-KV
// partition pass) and its launchers, templated on the KV cache element type; included
// by pa_decode.cu (bf16 caches) and pa_decode_fp8.cu (FP8 E4M3 caches), each of which
// instantiates one cache type.
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
//  * FP8 E4M3 caches (kv_cache_dtype "fp8"): pages move as bytes, half the bf16
//    ring bytes per stage, so the ring holds twice the stages; a thread's 8 dims
//    arrive as 8 bytes and become floats through exact e4m3 -> f16 conversions.
//    k_scale is folded into the pre-scaled Q and v_scale into the normalisation.
//  * Sliding window (keys j >= L - window): chunks wholly before the window are
//    skipped, and in the chunk holding L - window the pages wholly before it are
//    neither looked up nor loaded; the earlier rows of its first page are masked.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {


constexpr unsigned kFull = 0xffffffffu;

// Decode launch modes: one work item per CTA (single pass over all chunks, or
// one split partition), a persistent split grid that walks a compact list of
// (sequence, partition, kv head) items round-robin, or the single pass spread over
// a thread-block cluster: the cluster's CTAs each take a contiguous share of the
// sequence's pages and merge their (max, sum, output) through distributed shared
// memory, so one (sequence, kv head) no longer streams through one CTA alone and
// the call still needs no workspace.
enum DecodeMode { kSingle = 0, kSplitDirect = 1, kSplitPersistent = 2, kSingleCluster = 3 };
constexpr int kDecodeCluster = 4;   // CTAs per (sequence, kv head) in kSingleCluster

template <int HD, int G, bool FP8 = false>
struct DecodeCfg {
    static constexpr int ELEM = FP8 ? 1 : 2;           // bytes per cache element
    static constexpr int TPR = HD / 8;                 // threads per token row (8 dims each)
    static constexpr int LOG_TPR = HD == 64 ? 3 : (HD == 128 ? 4 : 5);
    static constexpr int NC = kBlockSize * TPR;        // consumer threads: one page per pass
    static constexpr int NCW = NC / 32;                // consumer warps
    static constexpr int NT = NC + 32;                 // + one producer warp
    static constexpr int PAGE_BYTES = kBlockSize * HD * ELEM;
    static constexpr int SP = 4;                       // pages per ring stage
    static constexpr int STAGE_BYTES = SP * PAGE_BYTES;
    static constexpr int S = (HD == 64 ? 8 : (HD == 128 ? 5 : 4)) * (FP8 ? 2 : 1);  // stages
    static constexpr int RING_BYTES = S * STAGE_BYTES;
    static constexpr int LOG_G = G == 1 ? 0 : (G == 2 ? 1 : (G == 4 ? 2 : 3));
    static constexpr int LOG_V = 2 + LOG_G;            // a stage's SP pages x G heads
    static constexpr int V = 1 << LOG_V;               // partial sums per lane
    static constexpr int NV = (V / TPR) > 0 ? (V / TPR) : 1;  // sums a lane keeps
    static constexpr int MAXB = 2048;                  // sequences for the persistent grid
    // shared memory layout (bytes)
    static constexpr int OFF_SC = RING_BYTES;                   // float [512][G]
    static constexpr int OFF_RED = OFF_SC + kPartition * G * 4;  // float [NCW][HD]
    static constexpr int OFF_RSTAT = OFF_RED + NCW * HD * 4;     // float [NCW][G]
    static constexpr int OFF_PREF = OFF_RSTAT + NCW * G * 4;     // int [MAXB + 1]
    static constexpr int OFF_BAR = OFF_PREF + (MAXB + 8) * 4;    // uint64 full[S], empty[S]
    static constexpr int OFF_OK = OFF_BAR + 2 * S * 8;           // int [S]: valid-page bits
    static constexpr int OFF_ABORT = OFF_OK + S * 4;             // int
    // kSingleCluster: this CTA's unnormalised output [G][HD], then max [G] and sum [G]
    static constexpr int OFF_CL = OFF_ABORT + 16;
    static constexpr int CL_FLOATS = G * HD + 2 * G;
    static constexpr int SMEM = OFF_CL + CL_FLOATS * 4;
    static_assert(OFF_BAR % 8 == 0, "barrier alignment");
    static_assert(G * HD * 2 <= STAGE_BYTES, "a query group fits in one ring stage");
    static_assert(kPartition % (SP * kBlockSize) == 0, "stages tile a partition");
};

// Sums V partial dot products across the TPR lanes of a token row with shuffles
// and adds only.  Each lane holds its partials in a lane-dependent order -- slot
// s holds physical index s ^ perm(lane), where the bit of perm that a butterfly
// step splits on equals the lane bit that step exchanges -- so every step just
// adds the partner's upper half to its own lower half.  Afterwards lane l holds
// the complete sums of physical indices perm(l) ^ j for j < NV.
template <int V, int TPR>
__device__ __forceinline__ void row_reduce(float (&v)[V]) {
    int n = V;
#pragma unroll
    for (int mask = TPR / 2; mask >= 1; mask >>= 1) {
        if (n > 1) {
            const int half = n / 2;
#pragma unroll
            for (int i = 0; i < V / 2; ++i)
                if (i < half) v[i] += __shfl_xor_sync(kFull, v[i + half], mask);
            n = half;
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], mask);
        }
    }
}

// Physical-index permutation of lane chunk c for row_reduce (see above).
template <int LOG_V, int LOG_TPR>
__device__ __forceinline__ int reduce_perm(int c) {
    if constexpr (LOG_TPR <= LOG_V) return c << (LOG_V - LOG_TPR);
    else return c >> (LOG_TPR - LOG_V);
}

// Work item of the k-th iteration of this CTA; false when there is none.  ch_begin /
// ch_end select the item's partition (split) or stand for "all of it" (single pass).
template <int MODE>
__device__ __forceinline__ bool decode_item(const DecodeParams &p, const int *pref, long long total,
                                            int k, int &b, int &kh, int &ch_begin, int &ch_end) {
    if constexpr (MODE == kSplitPersistent) {
        const long long i = static_cast<long long>(blockIdx.x) + static_cast<long long>(k) * gridDim.x;
        if (i >= total) return false;
        kh = static_cast<int>(i % p.num_kv_heads);
        const int j = static_cast<int>(i / p.num_kv_heads);
        int lo = 0, hi = p.num_seqs;          // largest b with pref[b] <= j
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pref[mid] <= j) lo = mid; else hi = mid;
        }
        b = lo;
        ch_begin = j - pref[b];
        ch_end = ch_begin + 1;
        return true;
    } else {
        if (k > 0) return false;
        b = blockIdx.z;
        kh = blockIdx.y;
        ch_begin = MODE == kSplitDirect ? static_cast<int>(blockIdx.x) : 0;
        ch_end = MODE == kSplitDirect ? ch_begin + 1 : 1 << 30;  // clipped by the length
        return true;
    }
}

// The token range [t_begin, t_end) an item covers in a sequence of L tokens whose window
// starts at token ws; it is processed in chunks of up to kPartition tokens from t_begin
// (a page boundary).  A split item is one partition (a persistent split item's index
// counts from the window's first partition); a single-pass item runs from the window's
// first partition to the end; a cluster item is the CTA's share of the pages from the
// window's first page, split evenly over the cluster's ranks.
template <int MODE>
__device__ __forceinline__ void item_range(int L, int ws, int ch_begin, int &t_begin,
                                           int &t_end) {
    if constexpr (MODE == kSplitPersistent || MODE == kSplitDirect) {
        const int ch = MODE == kSplitPersistent ? ch_begin + ws / kPartition : ch_begin;
        t_begin = ch * kPartition;
        t_end = min(L, t_begin + kPartition);
    } else if constexpr (MODE == kSingle) {
        t_begin = ws / kPartition * kPartition;
        t_end = L;
    } else {
        const int p0 = ws / kBlockSize;
        const int np = (L + kBlockSize - 1) / kBlockSize - p0;
        const int rank = static_cast<int>(blockIdx.x), cs = static_cast<int>(gridDim.x);
        t_begin = (p0 + np * rank / cs) * kBlockSize;
        t_end = min(L, (p0 + np * (rank + 1) / cs) * kBlockSize);
    }
    if (t_end < t_begin) t_end = t_begin;
}

// Effective length of sequence b (negative -> 0, clamped to the table / max_seq_len).
template <int MODE>
__device__ __forceinline__ int seq_len_clamped(const DecodeParams &p, int b, bool flag) {
    int L = p.seq_lens[b];
    if (L < 0) L = 0;
    int cap = p.max_blocks * kBlockSize;
    if ((MODE == kSplitDirect || MODE == kSplitPersistent) && p.max_seq_len < cap)
        cap = p.max_seq_len;
    if (L > cap) {
        if (flag) atomicOr(p.status, kStatusBounds);
        L = cap;
    }
    return L;
}

// The 8 cache elements a thread owns in a token row, raw (16 bytes of bf16 or 8
// bytes of E4M3), and their float values in (low, high) pairs.
template <bool FP8>
using Raw8 = typename std::conditional<FP8, uint2, uint4>::type;

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w);

__device__ __forceinline__ void unpack8(const uint4 &raw, float2 (&f)[4]) {
    f[0] = bf16x2_to_float2(raw.x);
    f[1] = bf16x2_to_float2(raw.y);
    f[2] = bf16x2_to_float2(raw.z);
    f[3] = bf16x2_to_float2(raw.w);
}

__device__ __forceinline__ void unpack8(const uint2 &raw, float2 (&f)[4]) {
    f[0] = e4m3x2_to_float2(raw.x & 0xffffu);
    f[1] = e4m3x2_to_float2(raw.x >> 16);
    f[2] = e4m3x2_to_float2(raw.y & 0xffffu);
    f[3] = e4m3x2_to_float2(raw.y >> 16);
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int HD, int G, int MODE, bool FP8>
__global__ void __launch_bounds__(DecodeCfg<HD, G, FP8>::NT, (HD == 256 || G == 8) ? 1 : 2)
    decode_kernel(const __grid_constant__ DecodeParams p) {
    using C = DecodeCfg<HD, G, FP8>;
    constexpr bool SPLIT = MODE == kSplitDirect || MODE == kSplitPersistent;
    constexpr bool CLUSTER = MODE == kSingleCluster;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *ring = smem;
    float *sc = reinterpret_cast<float *>(smem + C::OFF_SC);
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);
    float *rstat = reinterpret_cast<float *>(smem + C::OFF_RSTAT);
    int *pref = reinterpret_cast<int *>(smem + C::OFF_PREF);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::S;
    int *stage_ok = reinterpret_cast<int *>(smem + C::OFF_OK);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_ABORT);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Launched as a programmatic dependent of the previous kernel in the stream (the
    // cache write): the launch and CTA start-up overlap it, nothing it may have
    // written is read before it has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    long long total = 0;
    if constexpr (MODE == kSplitPersistent) {
        // prefix over sequences of their partition counts (compact item list)
        for (int b = threadIdx.x; b < p.num_seqs; b += C::NT) {
            const int L = seq_len_clamped<MODE>(p, b, blockIdx.x == 0);
            pref[b + 1] = (L + kPartition - 1) / kPartition - window_start(L, p.window) / kPartition;
        }
        if (threadIdx.x == 0) pref[0] = 0;
        __syncthreads();
        if (warp == 0) {
            int carry = 0;
            for (int base = 1; base <= p.num_seqs; base += 32) {
                const int idx = base + lane;
                int v = idx <= p.num_seqs ? pref[idx] : 0;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int u = __shfl_up_sync(kFull, v, off);
                    if (lane >= off) v += u;
                }
                if (idx <= p.num_seqs) pref[idx] = v + carry;
                carry += __shfl_sync(kFull, v, 31);
            }
        }
        __syncthreads();
        total = static_cast<long long>(pref[p.num_seqs]) * p.num_kv_heads;
        if (static_cast<long long>(blockIdx.x) >= total) return;
    } else if constexpr (MODE == kSplitDirect) {
        const int L = seq_len_clamped<MODE>(p, blockIdx.z, blockIdx.x == 0 && threadIdx.x == 0);
        if (static_cast<int>(blockIdx.x) * kPartition >= L) return;  // partition past the end
        if (static_cast<int>(blockIdx.x) < window_start(L, p.window) / kPartition) return;
    } else {
        // flags an over-long seq_len (once per sequence)
        seq_len_clamped<MODE>(p, blockIdx.z, threadIdx.x == 0 && blockIdx.x == 0);
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

    if (warp == C::NCW) {
        // ------------------------------ producer warp ------------------------------
        const uint64_t policy = l2_policy_evict_first();
        uint32_t it = 0;
        int stop = 0;  // warp-uniform
        // Claims the next ring stage (waits until the consumers released it).
        auto claim = [&]() -> int {
            int s = -1;
            if (lane == 0) {
                s = it % C::S;
                if (!mbar_wait(&empty[s], ((it / C::S) & 1u) ^ 1u, p.status, abort_flag)) s = -1;
            }
            s = __shfl_sync(kFull, s, 0);
            if (s < 0) stop = 1;
            return s;
        };
        int b, kh, ch_begin, ch_end;
        for (int k = 0; !stop && decode_item<MODE>(p, pref, total, k, b, kh, ch_begin, ch_end);
             ++k) {
            const int L = seq_len_clamped<MODE>(p, b, false);
            const int ws = window_start(L, p.window);
            int t_begin, t_end;
            item_range<MODE>(L, ws, ch_begin, t_begin, t_end);
            // stage 1 of an item: its query group (G heads x HD, contiguous)
            {
                const int s = claim();
                if (s < 0) break;
                if (lane == 0) {
                    stage_ok[s] = 1;
                    mbar_arrive_expect_tx(&full[s], G * HD * 2);
                    bulk_copy_g2s_hint(ring + s * C::STAGE_BYTES,
                                       static_cast<const __nv_bfloat16 *>(p.q) +
                                           (static_cast<int64_t>(b) * p.num_q_heads + kh * G) * HD,
                                       G * HD * 2, &full[s], policy);
                }
                ++it;
            }
            const int32_t *bt_row = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;
            for (int t0 = t_begin; t0 < t_end && !stop; t0 += kPartition) {
                const int np = (min(kPartition, t_end - t0) + kBlockSize - 1) / kBlockSize;
                const int pg_lo = max(0, ws - t0) / kBlockSize;   // first page in the window
                const bool mine = lane >= pg_lo && lane < np;
                const int my_page = mine ? bt_row[t0 / kBlockSize + lane] : -1;
                const bool my_ok = mine && my_page >= 0 && my_page < p.num_blocks;
                if (__any_sync(kFull, mine && !my_ok) && lane == 0)
                    atomicOr(p.status, kStatusBounds);
                for (int kv = 0; kv < 2 && !stop; ++kv) {
                    const uint8_t *base = static_cast<const uint8_t *>(kv ? p.v_cache : p.k_cache);
                    for (int pg0 = pg_lo; pg0 < np; pg0 += C::SP) {
                        const int s = claim();
                        if (s < 0) break;
                        const int npg = min(C::SP, np - pg0);
                        // lane u < npg copies page pg0 + u of the stage (row by row if needed)
                        const int page = __shfl_sync(kFull, my_page, (pg0 + (lane & (C::SP - 1))) & 31);
                        const bool ok = (lane & (C::SP - 1)) < npg && page >= 0 && page < p.num_blocks;
                        const uint32_t okbits = __ballot_sync(kFull, ok && lane < C::SP) & ((1u << C::SP) - 1);
                        if (lane == 0) {
                            stage_ok[s] = static_cast<int>(okbits);
                            mbar_arrive_expect_tx(&full[s], __popc(okbits) * C::PAGE_BYTES);
                        }
                        __syncwarp();
                        if (lane < C::SP && ok) {
                            const uint8_t *src = base + (static_cast<int64_t>(page) * p.s_block +
                                                         static_cast<int64_t>(kh / p.kv_rep) * p.s_head) * C::ELEM;
                            uint8_t *dst = ring + s * C::STAGE_BYTES + lane * C::PAGE_BYTES;
                            if (p.rows_contiguous) {
                                bulk_copy_g2s_hint(dst, src, C::PAGE_BYTES, &full[s], policy);
                            } else {
                                for (int t = 0; t < kBlockSize; ++t)
                                    bulk_copy_g2s_hint(dst + t * HD * C::ELEM,
                                                       src + t * p.s_token * C::ELEM, HD * C::ELEM,
                                                       &full[s], policy);
                            }
                        }
                        ++it;
                    }
                }
            }
        }
        // Drain: never leave the CTA with bulk copies still landing in its smem.
        if (lane == 0 && (stop || *abort_flag)) {
            const uint32_t issued = it;  // stages claimed and filled
            for (uint32_t k = (issued > C::S ? issued - C::S : 0); k < issued; ++k) {  // last S stages
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&full[k % C::S], (k / C::S) & 1u)) {
                    if (global_timer_ns() - t0 > kWaitLimitNs) break;
                }
            }
        }
        __syncwarp();
        if constexpr (CLUSTER) {   // every thread of the cluster takes part in both syncs
            cluster_sync_all();
            cluster_sync_all();
        }
        return;
    }

    // -------------------------------- consumer warps --------------------------------
    const int tid = threadIdx.x;          // 0 .. NC-1
    const int r = tid / C::TPR;           // token row within a page
    const int c = tid % C::TPR;           // 16-byte chunk of the row
    const int perm = reduce_perm<C::LOG_V, C::LOG_TPR>(c);
    const int pu = perm >> C::LOG_G;      // page order of this lane within a group
    const int pg = perm & (G - 1);        // head order of this lane
    const int nq = p.num_q_heads;
    // scores in log2 units; an FP8 cache's k_scale scales every score, its v_scale
    // every output
    const float q_mul = p.scale_log2 * (FP8 ? p.k_scale : 1.f);
    const float v_mul = FP8 ? p.v_scale : 1.f;
    uint32_t it = 0;
    bool aborted = false;

    int b, kh, ch_begin, ch_end;
    for (int k = 0; !aborted && decode_item<MODE>(p, pref, total, k, b, kh, ch_begin, ch_end); ++k) {
        const int L = seq_len_clamped<MODE>(p, b, false);
        const int ws = window_start(L, p.window);
        int t_begin, t_end;
        item_range<MODE>(L, ws, ch_begin, t_begin, t_end);

        // ---- the item's query group: Q x scale (heads in this lane's order) in registers ----
        float2 q2[G][4];
        {
            const int s = it % C::S;
            if (!mbar_wait(&full[s], (it / C::S) & 1u, p.status, abort_flag)) aborted = true;
            const __nv_bfloat16 *qs =
                reinterpret_cast<const __nv_bfloat16 *>(ring + s * C::STAGE_BYTES);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(qs + (g ^ pg) * HD + c * 8);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = bf16x2_to_float2(w[i]);
                    q2[g][i] = make_float2(f.x * q_mul, f.y * q_mul);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++it;
        }

        float2 acc[G][4];
        float m_run[G], l_run[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m_run[g] = -INFINITY;
            l_run[g] = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[g][i] = make_float2(0.f, 0.f);
        }

        // One chunk of up to 512 tokens from t0 (a page boundary): scores, softmax
        // statistics, then P.V; false on abort.
        auto chunk = [&](int t0) -> bool {
            const int n_tok = min(kPartition, t_end - t0);
            const int np = (n_tok + kBlockSize - 1) / kBlockSize;
            const int t_lo = max(0, ws - t0);              // first token in the window
            const int pg_lo = t_lo / kBlockSize;           // pages before it are not loaded
            const int t_first = pg_lo * kBlockSize;

            // ---- K pages, one 4-page stage at a time: scaled scores (log2 units) into sc ----
            for (int pg0 = pg_lo; pg0 < np; pg0 += C::SP) {
                const int npg = min(C::SP, np - pg0);
                const int s = it % C::S;
                if (!mbar_wait(&full[s], (it / C::S) & 1u, p.status, abort_flag)) aborted = true;
                const uint32_t okbits = aborted ? 0u : static_cast<uint32_t>(stage_ok[s]);
                const uint8_t *st = ring + s * C::STAGE_BYTES + (r * HD + c * 8) * C::ELEM;
                float part[C::V];
#pragma unroll
                for (int u = 0; u < C::SP; ++u) {
                    const int up = u ^ pu;           // page this lane handles in slot u
                    if (up < npg) {
                        float2 kf[4];
                        unpack8(*reinterpret_cast<const Raw8<FP8> *>(st + up * C::PAGE_BYTES), kf);
                        const float2 k0 = kf[0], k1 = kf[1], k2 = kf[2], k3 = kf[3];
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            float2 d = __fmul2_rn(q2[g][0], k0);
                            d = __ffma2_rn(q2[g][1], k1, d);
                            d = __ffma2_rn(q2[g][2], k2, d);
                            d = __ffma2_rn(q2[g][3], k3, d);
                            part[u * G + g] = d.x + d.y;
                        }
                    } else {
#pragma unroll
                        for (int g = 0; g < G; ++g) part[u * G + g] = 0.f;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                ++it;
                row_reduce<C::V, C::TPR>(part);
#pragma unroll
                for (int j = 0; j < C::NV; ++j) {
                    const int idx = perm ^ j;
                    const int u = idx >> C::LOG_G, g = idx & (G - 1);
                    if (u < npg) {
                        const int tok = (pg0 + u) * kBlockSize + r;
                        const bool valid = tok < n_tok && tok >= t_lo && ((okbits >> u) & 1u);
                        sc[tok * G + g] = valid ? part[j] : -INFINITY;
                    }
                }
            }
            if (named_barrier_or(1, C::NC, aborted)) return false;

            // ---- softmax statistics of this chunk ----
            float cm[G];
#pragma unroll
            for (int g = 0; g < G; ++g) cm[g] = -INFINITY;
            for (int t = t_first + tid; t < n_tok; t += C::NC) {
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
            for (int t = t_first + tid; t < n_tok; t += C::NC) {
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
                if constexpr (SPLIT) {
                    // a split item is one chunk: the accumulator starts here, so it
                    // (and Q before it) need not stay live across the other phase
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[g][i] = make_float2(0.f, 0.f);
                } else {
                    const float2 cc = make_float2(corr[g], corr[g]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[g][i] = __fmul2_rn(acc[g][i], cc);
                }
            }

            // ---- V pages, one 4-page stage at a time: acc += p * V ----
            for (int pg0 = pg_lo; pg0 < np; pg0 += C::SP) {
                const int s = it % C::S;
                if (!mbar_wait(&full[s], (it / C::S) & 1u, p.status, abort_flag)) aborted = true;
                const uint32_t okbits = aborted ? 0u : static_cast<uint32_t>(stage_ok[s]);
                const uint8_t *st = ring + s * C::STAGE_BYTES + (r * HD + c * 8) * C::ELEM;
                Raw8<FP8> raw[C::SP];
                float pw[C::SP][G];
#pragma unroll
                for (int u = 0; u < C::SP; ++u) {
                    const int tok = (pg0 + u) * kBlockSize + r;
                    const bool use = ((okbits >> u) & 1u) && tok < n_tok && tok >= t_lo;
                    raw[u] = use ? *reinterpret_cast<const Raw8<FP8> *>(st + u * C::PAGE_BYTES)
                                 : Raw8<FP8>{};
                    if constexpr (G == 4) {
                        const float4 p4 = use ? *reinterpret_cast<const float4 *>(sc + tok * 4)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                        pw[u][0] = p4.x; pw[u][1] = p4.y; pw[u][2] = p4.z; pw[u][3] = p4.w;
                    } else if constexpr (G == 2) {
                        const float2 p2 = use ? *reinterpret_cast<const float2 *>(sc + tok * 2)
                                              : make_float2(0.f, 0.f);
                        pw[u][0] = p2.x; pw[u][1] = p2.y;
                    } else {
#pragma unroll
                        for (int g = 0; g < G; ++g) pw[u][g] = use ? sc[tok * G + g] : 0.f;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                ++it;
#pragma unroll
                for (int u = 0; u < C::SP; ++u) {
                    float2 vf[4];
                    unpack8(raw[u], vf);
                    const float2 v0 = vf[0], v1 = vf[1], v2 = vf[2], v3 = vf[3];
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float2 pp = make_float2(pw[u][g], pw[u][g]);
                        acc[g][0] = __ffma2_rn(v0, pp, acc[g][0]);
                        acc[g][1] = __ffma2_rn(v1, pp, acc[g][1]);
                        acc[g][2] = __ffma2_rn(v2, pp, acc[g][2]);
                        acc[g][3] = __ffma2_rn(v3, pp, acc[g][3]);
                    }
                }
            }
            return !named_barrier_or(1, C::NC, aborted);  // sc is rewritten next chunk
        };
        for (int t0 = t_begin; t0 < t_end; t0 += kPartition) {
            if (!chunk(t0)) {
                aborted = true;
                break;
            }
        }
        if (aborted) break;

        // ---- reduce acc over the 16 rows: lanes of a warp, then warps via smem ----
#pragma unroll
        for (int mask = C::TPR; mask < 32; mask <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[g][i].x += __shfl_xor_sync(kFull, acc[g][i].x, mask);
                    acc[g][i].y += __shfl_xor_sync(kFull, acc[g][i].y, mask);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (lane < C::TPR) {
                float4 *dst = reinterpret_cast<float4 *>(red + warp * HD + c * 8);
                dst[0] = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
                dst[1] = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
            }
            named_barrier(1, C::NC);
            if (tid < HD) {
                float o = 0.f;
#pragma unroll
                for (int w = 0; w < C::NCW; ++w) o += red[w * HD + tid];
                const int h = kh * G + g;
                const float inv = l_run[g] > 0.f ? 1.f / l_run[g] : 0.f;
                if constexpr (CLUSTER) {
                    float *cl = reinterpret_cast<float *>(smem + C::OFF_CL);
                    cl[g * HD + tid] = o;                  // unnormalised
                    if (tid == 0) {
                        cl[G * HD + g] = m_run[g];         // log2 units
                        cl[G * HD + G + g] = l_run[g];
                    }
                } else if constexpr (SPLIT) {
                    const int64_t row = (static_cast<int64_t>(b) * nq + h) * p.max_parts +
                                        t_begin / kPartition;
                    p.part_o[row * HD + tid] = o * inv * v_mul;
                    if (tid == 0) {
                        p.part_m[row] = m_run[g] * kLn2;
                        p.part_l[row] = l_run[g];
                    }
                } else {
                    static_cast<__nv_bfloat16 *>(p.out)[(static_cast<int64_t>(b) * nq + h) * HD + tid] =
                        __float2bfloat16_rn(o * inv * v_mul);
                }
            }
            named_barrier(1, C::NC);
        }
    }

    if constexpr (CLUSTER) {
        // Merge the cluster's partial results: with M the largest of the ranks' maxima,
        // out = sum_r 2^(m_r - M) o_r / sum_r 2^(m_r - M) l_r.  Every thread of every CTA
        // of the cluster reaches both syncs (an aborted CTA too; its status is flagged).
        __syncwarp();
        cluster_sync_all();   // each rank's partials are in its shared memory
        const uint32_t cl = smem_addr(smem + C::OFF_CL);
        const int rank = static_cast<int>(blockIdx.x);
        const int b = blockIdx.z, kh = blockIdx.y;
        for (int e = rank * C::NC + tid; e < G * HD; e += kDecodeCluster * C::NC) {
            const int g = e / HD;
            float mr[kDecodeCluster];
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < kDecodeCluster; ++q) {
                mr[q] = ld_shared_cluster_f32(mapa_shared(cl + (G * HD + g) * 4, q));
                M = fmaxf(M, mr[q]);
            }
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int q = 0; q < kDecodeCluster; ++q) {
                    const float wq = exp2f(mr[q] - M);
                    den += wq * ld_shared_cluster_f32(mapa_shared(cl + (G * HD + G + g) * 4, q));
                    num += wq * ld_shared_cluster_f32(mapa_shared(cl + e * 4, q));
                }
            }
            static_cast<__nv_bfloat16 *>(p.out)[(static_cast<int64_t>(b) * nq + kh * G + g) * HD +
                                                e % HD] =
                __float2bfloat16_rn(den > 0.f ? num / den * v_mul : 0.f);
        }
        cluster_sync_all();   // no rank leaves while another still reads its shared memory
    }
}

// Launches a kernel as a programmatic dependent of the previous work in the stream:
// its CTAs may start while that work finishes, and wait for it (griddepcontrol.wait)
// before reading anything.
template <typename... Args>
cudaError_t launch_dependent(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, const DecodeParams &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<DecodeParams *>(&p)};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// launch_dependent for a grid of thread-block clusters of `cluster` CTAs along x.
template <typename... Args>
cudaError_t launch_dependent_cluster(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, const DecodeParams &p, int cluster) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *args[] = {const_cast<DecodeParams *>(&p)};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

int sm_count() {
    static int count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (!count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        count[dev] = n;
    }
    return count[dev];
}

template <int HD, int G, int MODE, bool FP8>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t stream) {
    using C = DecodeCfg<HD, G, FP8>;
    auto kern = decode_kernel<HD, G, MODE, FP8>;
    static int configured_device = -1;  // cache of the smem opt-in (per process, last device)
    static int blocks_per_sm = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        // ask for the largest shared-memory carveout so two CTAs fit per SM
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, kern, C::NT, C::SMEM);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    dim3 grid;
    if (MODE == kSingleCluster) {
        grid = dim3(kDecodeCluster, p.num_kv_heads, p.num_seqs);
        return launch_dependent_cluster(kern, grid, dim3(C::NT), C::SMEM, stream, p,
                                        kDecodeCluster);
    }
    if (MODE == kSplitPersistent) {
        const long long slots = static_cast<long long>(p.num_seqs) * p.num_kv_heads *
                                active_partitions_cap(p.max_parts, p.window);
        long long n = static_cast<long long>(sm_count()) * (blocks_per_sm > 0 ? blocks_per_sm : 1);
        if (slots < n) n = slots;
        grid = dim3(static_cast<unsigned>(n > 0 ? n : 1), 1, 1);
    } else {
        grid = dim3(MODE == kSplitDirect ? p.max_parts : 1, p.num_kv_heads, p.num_seqs);
    }
    return launch_dependent(kern, grid, dim3(C::NT), C::SMEM, stream, p);
}

template <int HD, int G, bool FP8>
cudaError_t launch_mode(const DecodeParams &p, bool split, cudaStream_t stream) {
    using C = DecodeCfg<HD, G, FP8>;
    // The single pass spreads each (sequence, kv head) over a cluster when there are too
    // few of them to give every SM two CTAs and sequences may span more than two 512-token
    // chunks: 8 sequences of 32k-131k tokens, 8 kv heads: 2.54 -> 0.89 ms.  With enough
    // items one CTA each is as fast or faster (64 sequences x 8 kv heads of 0.5k-4k tokens:
    // 0.188 vs 0.183 ms; 32 x 32 ungrouped: 0.195 vs 0.220 ms).
    if (!split) {
        const long long items = static_cast<long long>(p.num_seqs) * p.num_kv_heads;
        const bool spread = items < 2LL * sm_count() && p.max_blocks * kBlockSize > 2 * kPartition;
        return spread ? launch_decode_t<HD, G, kSingleCluster, FP8>(p, stream)
                      : launch_decode_t<HD, G, kSingle, FP8>(p, stream);
    }
    if (p.num_seqs <= C::MAXB) return launch_decode_t<HD, G, kSplitPersistent, FP8>(p, stream);
    return launch_decode_t<HD, G, kSplitDirect, FP8>(p, stream);
}

template <int HD, bool FP8>
cudaError_t dispatch_group(const DecodeParams &p, bool split, cudaStream_t stream) {
    switch (p.num_q_heads / p.num_kv_heads) {
        case 1: return launch_mode<HD, 1, FP8>(p, split, stream);
        case 2: return launch_mode<HD, 2, FP8>(p, split, stream);
        case 4: return launch_mode<HD, 4, FP8>(p, split, stream);
        case 8: return launch_mode<HD, 8, FP8>(p, split, stream);
        default: return cudaErrorNotSupported;
    }
}

// The CUDA-core decode over caches of one element type (bf16, or FP8 E4M3).
template <bool FP8>
cudaError_t launch_decode_cache(const DecodeParams &p, int head_dim, bool split,
                                cudaStream_t stream) {
    switch (head_dim) {
        case 64: return dispatch_group<64, FP8>(p, split, stream);
        case 128: return dispatch_group<128, FP8>(p, split, stream);
        case 256: return dispatch_group<256, FP8>(p, split, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace
}  // namespace pa
