// pa_prefill.cu -- ragged (varlen) causal prefill on the Blackwell tensor cores.
//
// What it computes ("spark_runtime/flashinfer.rs", ragged_prefill_bf16_hd256
// and its CPU reference; "paged_attn.py", _forward_prefix_pytorch): request r
// owns query rows [qo_indptr[r], qo_indptr[r+1]) and kv_len keys; query row i,
// head h attends to keys j < kv_len of kv head h / g, and under the causal mask
// only to j <= i + (kv_len - qo_len).  Keys come from contiguous rows
// kv_indptr[r] + j (ragged mode) or from token j of block_tables[r] (paged
// mode, 16-token pages).
//
// GB300 design (FlashAttention-style, not the pages' SM80 design):
//  * Persistent CTAs (two per SM at head_dim <= 128) claim work items -- one
//    (request, 128-row query tile, query head) each -- from a heaviest-first
//    list through a global counter; the producer decodes each claimed item once
//    and hands it to the other warps through a 4-deep shared-memory queue.
//    6 warps per CTA (7 for paged K/V at head_dim 256, see warp 6):
//      warp 0   TMA producer: Q once per item, then K_j / V_j tiles (128-byte
//               swizzle) into 2-stage rings, K one tile ahead of V (the order the
//               MMA warp consumes them); paged mode issues one box per 16-token
//               page and looks each page id up once per tile, a tile early
//      warp 1   TMEM allocator + single-thread tcgen05.mma issuer:
//               S_j = Q K_j^T (M=128, N=BN, K=head_dim) into TMEM buffer j%2,
//               then O += P_{j-1} V_{j-1} with P read straight from TMEM; two
//               tcgen05.commits per key tile (S done, P.V done), everything else
//               (K / Q reuse, O rescale, O final) is read off those two barriers
//      warps 2-5  softmax: one query row per thread, read S from TMEM, mask,
//               exp2, write P (bf16) over S in TMEM; epilogue O / l -> bf16
//      warp 6   paged head_dim 256 only: a second TMA producer that issues the V
//               tiles (a tile there is 32 two-kilobyte boxes), taking the items
//               from the queue; warp 0 then issues Q and K only
//  * Online softmax with lazy rescaling: O is rescaled (in TMEM) only when a
//    row max grows by more than 2^8, so the correction is rare; the final
//    normalisation uses the same running max, which keeps the result exact.
//  * Causal tile skipping: a query tile stops at the last key tile any of its
//    rows can see; per-element masking only on tiles that cross the diagonal
//    or the end of the keys.
//  * The (request, q-tile) work items are ordered by their number of key tiles,
//    heaviest first: on the host for up to 1024 query tiles (the list then travels
//    in the kernel's parameters), otherwise by a one-CTA kernel into the caller's
//    workspace.  The producer claims item k + 1 once item k's first K tile is on its
//    way, and the last CTA to finish clears the work counters for the next launch.
//  * Every mbarrier wait is bounded (PA_ERR_TIMEOUT instead of a hang).
#include <algorithm>

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kBM = 128;              // query rows per tile (MMA M)
constexpr int kSchedBuckets = 2048;

constexpr uint32_t pow2_at_least(uint32_t x) {
    uint32_t v = 32;
    while (v < x) v <<= 1;
    return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 32-byte store (one full L2 sector per thread); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_32B(void *ptr, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t a4, uint32_t a5, uint32_t a6,
                                              uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(ptr), "r"(a0), "r"(a1),
                 "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// max(a, b, c) in one instruction (three-input max.f32 of the sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Online-softmax state of one query row; m is a running max of s * scale (log2 units).
struct RowSoftmax {
    float m, l;
};

// Masks the columns outside [lo, lim) of a key tile (when need_mask: the visible keys
// of a row are a run of the tile's columns -- lo > 0 only under a sliding window),
// takes the row max and makes the lazy-rescale decision: m moves only when the max
// grows by more than 2^8.  Returns whether it moves; m_use is the max the tile's P is
// then taken against and corr the factor O and l are scaled by.
template <int BN>
__device__ __forceinline__ bool tile_max(uint32_t (&sr)[BN], bool need_mask, int lo, int lim,
                                         float scale, const RowSoftmax &rs, float &m_use,
                                         float &corr) {
    if (need_mask) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
            if (c >= lim || c < lo) sr[c] = __float_as_uint(-INFINITY);
    }
    // row max of the raw scores (sm_scale > 0, so it scales to the max of s * scale);
    // eight partial maxima, each taking two new columns per three-input max, keep the
    // dependency chains short
    static_assert(BN % 16 == 0, "row max works in groups of 16 columns");
    float pmax[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) pmax[e] = fmaxf(__uint_as_float(sr[e]), __uint_as_float(sr[8 + e]));
#pragma unroll
    for (int c = 16; c < BN; c += 16)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            pmax[e] = fmax3(pmax[e], __uint_as_float(sr[c + e]), __uint_as_float(sr[c + 8 + e]));
    const float tmax = fmax3(fmax3(pmax[0], pmax[1], pmax[2]), fmax3(pmax[3], pmax[4], pmax[5]),
                             fmaxf(pmax[6], pmax[7]));
    const float m_new = fmaxf(rs.m, tmax * scale);   // -inf stays -inf
    const bool grow = m_new > rs.m + 8.0f;
    m_use = grow ? m_new : rs.m;
    corr = (rs.m == -INFINITY) ? 0.f : fast_exp2(rs.m - m_use);
    return grow;
}

// P = 2^(s * scale - m) for a key tile, packed to bf16 pairs, and its row sum added
// to l.  All exponentials go to the MUFU unit: the softmax is bound by its issue
// slots and latency, not by MUFU throughput, so moving some of them to an FMA-pipe
// polynomial (more instructions per exponential) measured slower.
template <int BN>
__device__ __forceinline__ void tile_exp(const uint32_t (&sr)[BN], float scale, RowSoftmax &rs,
                                         uint32_t (&pk)[BN / 2]) {
    float2 lsum[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
    if (rs.m != -INFINITY) {
        const float2 sc2 = make_float2(scale, scale), nm2 = make_float2(-rs.m, -rs.m);
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, nm2);
            const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            lsum[c & 3] = __fadd2_rn(lsum[c & 3], e);
            pk[c] = pack_bf16x2(e.x, e.y);
        }
    } else {
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) pk[c] = 0u;
    }
    const float2 ls01 = __fadd2_rn(lsum[0], lsum[1]), ls23 = __fadd2_rn(lsum[2], lsum[3]);
    const float2 lsum_t = __fadd2_rn(ls01, ls23);
    rs.l += lsum_t.x + lsum_t.y;
}

// Paged K/V at head_dim 256: a key tile is 32 two-kilobyte TMA boxes (K and V: 4
// pages x 4 column chunks), and one warp issuing them all set the pace, so a second
// producer warp (warp 6) issues the V tiles.  Contiguous K/V move as 8 KB boxes and
// do not need it (a split measured 7 % slower there); at head_dim <= 128 two CTAs
// share an SM and their registers leave no room for a seventh warp.
// At head_dim 256 (one CTA per SM) two threads issue the MMAs: warp 1 the scores
// S_j = Q K_j^T, warp 6 the P_j V_j (tcgen05.commit tracks each thread's own MMAs), so
// the scores of tile j + 1 never queue behind the issue of P_j V_j in one thread's
// program order, nor P_j V_j behind a K tile the score issuer waits for: chunked paged
// prefill 0.246 -> 0.221 ms.  At head_dim <= 128 two CTAs share an SM, and the seventh
// warp's registers (128 per thread, with spills) made it 5 % slower there.
template <int HD, bool PAGED>
struct ProducerSplit {
    static constexpr bool value = HD == 256 && PAGED;
    static constexpr bool two_issuers = HD == 256;
    static constexpr int PV_WARP = two_issuers ? 6 : -1;
    static constexpr int V_WARP = two_issuers ? 7 : 6;   // the V producer (split only)
    static constexpr int threads = 32 * (6 + (two_issuers ? 1 : 0) + (value ? 1 : 0));
};

template <int HD, int BN>
struct PrefillCfg {
    static constexpr int QCH = HD / 64;                       // 128-byte column chunks
    static constexpr uint32_t Q_BYTES = QCH * kBM * 128;
    static constexpr uint32_t KV_CHUNK = BN * 128;            // one chunk of a K / V tile
    static constexpr uint32_t KV_BYTES = QCH * KV_CHUNK;
    // K ring stages.  With two, stage j % 2 is S buffer j % 2 and K_j is free once S_j
    // is done (s_full); head_dim 256 runs one CTA per SM, where a third stage (freed
    // by a softmax-side arrival on k_empty) hides more of the TMA latency.  (A third
    // stage at head_dim 128, with two CTAs per SM, measured no faster.)
    static constexpr int KS = HD == 256 ? 3 : 2;
    static constexpr int VS = 2;                              // V ring stages

    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + KS * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + VS * KV_BYTES;
    static constexpr uint32_t SMEM_USED = OFF_BAR + 512;   // barriers + item queue
    // TMEM: S / P double buffer at columns [0, BN) and [BN, 2 BN), O after them
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_O = 2 * BN;
    static constexpr uint32_t TMEM_COLS = pow2_at_least(2 * BN + HD);
    // Two CTAs share an SM when both fit in its 512 TMEM columns (and in shared
    // memory): their MMA and softmax phases then interleave on the tensor core.
    // A CTA that needs all 512 columns asks for enough shared memory to be alone.
    // 1024 bytes of slack realign the base for the 128-byte-swizzled tiles (the kernel
    // checks that the realigned tiles fit before touching shared memory).
    static constexpr int CTAS_PER_SM = TMEM_COLS <= 256 ? 2 : 1;
    static constexpr uint32_t SLACK = 1024;
    static constexpr uint32_t SMEM_MIN = CTAS_PER_SM == 2 ? 0 : 118 * 1024;
    static constexpr uint32_t SMEM = (SMEM_USED + SLACK > SMEM_MIN) ? SMEM_USED + SLACK : SMEM_MIN;
    static_assert(HD % 64 == 0 && BN % 16 == 0 && BN <= 128, "tile shape");
    static_assert(KS >= 2 && KS <= 4 && VS >= 2 && VS <= 4, "ring stages");
    static_assert(TMEM_COLS <= 512, "TMEM budget");
    // two CTAs, each with the 1 KB the runtime reserves per CTA, in the SM's 228 KB
    static_assert(CTAS_PER_SM == 1 || 2 * (SMEM + 1024) <= 228 * 1024, "two CTAs per SM");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// First key any row of the query tile at q0 sees under a sliding window of `window`
// keys (row i at position i + kv_len - qo_len sees keys j > position - window); 0
// without a window.
__host__ __device__ __forceinline__ int window_first_key(int q0, int qo_len, int kv_len, int window) {
    if (window <= 0) return 0;
    const int k = q0 + (kv_len - qo_len) - window + 1;
    return k > 0 ? k : 0;
}

// Number of key tiles a query tile needs (its work): bottom-right causal, from the
// tile holding the window's first key.
__host__ __device__ __forceinline__ int key_tiles(int q0, int qo_len, int kv_len, int causal,
                                                  int window, int bn) {
    int kv_end = kv_len;
    if (causal) {
        const int last = q0 + kBM + (kv_len - qo_len);   // one past the last row's last key
        kv_end = last < 0 ? 0 : (last < kv_len ? last : kv_len);
    }
    const int n = (kv_end + bn - 1) / bn - window_first_key(q0, qo_len, kv_len, window) / bn;
    return n > 0 ? n : 0;
}

// Heaviest-first order of the (request, query tile) work items.
__global__ void __launch_bounds__(1024) prefill_schedule_kernel(
    const int32_t *qo_indptr, const int32_t *kv_indptr, int batch, int causal, int window,
    int bn, int n_tiles, int2 *tiles, int *item_counter, int *status) {
    __shared__ int hist[kSchedBuckets];
    __shared__ int total_sh;
    const int tid = threadIdx.x;
    // the prefill kernel may launch now (it sets up, then waits for this grid)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {   // the prefill kernel claims items from [0]; [1] counts its CTAs done
        item_counter[0] = 0;
        item_counter[1] = 0;
    }
    for (int i = tid; i < kSchedBuckets; i += blockDim.x) hist[i] = 0;
    if (tid == 0) total_sh = 0;
    __syncthreads();
    for (int r = tid; r < batch; r += blockDim.x) {
        const int qo_len = qo_indptr[r + 1] - qo_indptr[r];
        const int kv_len = kv_indptr[r + 1] - kv_indptr[r];
        const int nt = (max(qo_len, 0) + kBM - 1) / kBM;
        for (int t = 0; t < nt; ++t) {
            const int key =
                min(key_tiles(t * kBM, qo_len, kv_len, causal, window, bn), kSchedBuckets - 1);
            atomicAdd(&hist[kSchedBuckets - 1 - key], 1);
        }
        atomicAdd(&total_sh, nt);
    }
    __syncthreads();
    if (tid < 32) {  // exclusive scan of the histogram by one warp
        constexpr int PER = kSchedBuckets / 32;
        int local = 0;
        for (int i = 0; i < PER; ++i) local += hist[tid * PER + i];
        int incl = local;
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(kFullMask, incl, off);
            if (tid >= off) incl += v;
        }
        int run = incl - local;
        for (int i = 0; i < PER; ++i) {
            const int c = hist[tid * PER + i];
            hist[tid * PER + i] = run;
            run += c;
        }
    }
    __syncthreads();
    const int total = total_sh;
    if (tid == 0 && total != n_tiles) atomicOr(status, kStatusBounds);
    for (int r = tid; r < batch; r += blockDim.x) {
        const int qo_len = qo_indptr[r + 1] - qo_indptr[r];
        const int kv_len = kv_indptr[r + 1] - kv_indptr[r];
        const int nt = (max(qo_len, 0) + kBM - 1) / kBM;
        for (int t = 0; t < nt; ++t) {
            const int key =
                min(key_tiles(t * kBM, qo_len, kv_len, causal, window, bn), kSchedBuckets - 1);
            const int pos = atomicAdd(&hist[kSchedBuckets - 1 - key], 1);
            if (pos < n_tiles) tiles[pos] = make_int2(r, t);
        }
    }
    for (int i = total + tid; i < n_tiles; i += blockDim.x) tiles[i] = make_int2(-1, -1);
}

// One work item: a 128-row query tile of one request for one query head.
struct PrefillItem {
    int r, h, qo_start, qo_len, kv_start, kv_len, q0;
    int n_kv;   // key tiles; -1 marks the end of the work list
    int work;   // the tile holds query rows (it is written, possibly with zeros)
    int kv_lo;  // first key any row of the tile sees (> 0 only under a sliding window)
    int j0;     // first key tile, kv_lo / BN: the item's key tiles are j0 .. j0 + n_kv - 1
};

template <bool PAGED, int BN, bool WINDOW>
__device__ __forceinline__ PrefillItem prefill_item(const PrefillParams &p, long long i) {
    PrefillItem w;
    int2 tile;
    if (p.n_inline > 0) {
        const uint32_t v = p.inline_tiles[i / p.nq];
        tile = make_int2(static_cast<int>(v & 0xffffu), static_cast<int>(v >> 16));
    } else {
        tile = p.tiles[i / p.nq];
    }
    w.h = static_cast<int>(i % p.nq);
    w.r = tile.x;
    w.qo_start = w.qo_len = w.kv_start = w.kv_len = 0;
    const bool ok = w.r >= 0 && w.r < p.batch;
    if (ok) {
        w.qo_start = p.qo_indptr[w.r];
        w.qo_len = p.qo_indptr[w.r + 1] - w.qo_start;
        w.kv_start = p.kv_indptr[w.r];
        w.kv_len = p.kv_indptr[w.r + 1] - w.kv_start;
        if (PAGED && w.kv_len > p.max_blocks * kBlockSize) w.kv_len = p.max_blocks * kBlockSize;
    }
    w.q0 = ok ? tile.y * kBM : 0;
    w.work = ok && w.q0 < w.qo_len;
    const int window = WINDOW ? p.window : 0;
    w.n_kv = w.work ? key_tiles(w.q0, w.qo_len, w.kv_len, p.causal, window, BN) : 0;
    w.kv_lo = w.work ? window_first_key(w.q0, w.qo_len, w.kv_len, window) : 0;
    w.j0 = w.kv_lo / BN;
    return w;
}

// The item queue (4 entries) follows the 40 barrier words in the 512 bytes at OFF_BAR.
static_assert(40 * 8 + 4 * sizeof(PrefillItem) <= 512, "item queue fits its shared memory");

__device__ __forceinline__ PrefillItem end_item() {
    PrefillItem w{};
    w.n_kv = -1;
    return w;
}

// Persistent: each CTA claims items of the heaviest-first list (item i = query
// tile i / nq, head i % nq) one at a time from a global counter, so the load
// balances itself; TMEM and barriers are set up once and the next item's
// Q / K / V loads overlap the current item's tail.  WINDOW instantiates the
// sliding-window form (items start at their window's key tile, rows get a lower
// column bound); without it the window terms are compiled out.
template <int HD, int BN, bool PAGED, bool WINDOW>
__global__ void __launch_bounds__(ProducerSplit<HD, PAGED>::threads, PrefillCfg<HD, BN>::CTAS_PER_SM)
    prefill_kernel(const __grid_constant__ PrefillParams p) {
    using C = PrefillCfg<HD, BN>;
    constexpr bool SPLIT = ProducerSplit<HD, PAGED>::value;
    const int window = WINDOW ? p.window : 0;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    {   // the realigned tiles must fit the dynamic shared memory this launch has
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        if (static_cast<uint32_t>(smem - smem_raw) + C::SMEM_USED > dyn) {
            if (threadIdx.x == 0) atomicOr(p.status, kStatusUnsupported);
            return;   // uniform over the CTA, before any barrier or TMEM is set up
        }
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    // A tcgen05.commit costs the single MMA thread far more than an MMA, so each key
    // tile g (counted over all items of the CTA) has exactly two: s_full[g % 2] when
    // S_g = Q K_g^T is done and v_empty[g % VS] when O += P_g V_g is done.  Everything
    // else is read off those two: K_g's stage and (after an item's last tile) Q are
    // free once S_g is done; O is final, or may be rescaled, once the last issued
    // P.V is done.  Each of these parity waits is unambiguous because the barrier
    // can be neither two phases behind the awaited one (the waiter's own previous
    // wait on it, or the in-order completion of S_g after P_{g-2} V, saw the phase
    // before) nor one ahead (the next phase needs work the waiter has not released).
    uint64_t *q_full = bars + 0;
    uint64_t *q_empty = bars + 1;   // head_dim 256: an item's last S is done (score issuer)
    uint64_t *k_full = bars + 2;    // [KS]
    uint64_t *k_empty = bars + 6;   // [KS] (KS != 2): one softmax thread arrives once S_g is done
    uint64_t *v_full = bars + 10;   // [VS]
    uint64_t *v_empty = bars + 14;  // [VS]
    uint64_t *s_full = bars + 18;   // [2]
    // p_full and o_free take one arrival per softmax warp (lane 0, after the warp's
    // tcgen05 fences and a __syncwarp): 128 per-thread arrivals on one mbarrier are
    // serialised and sat on the softmax -> MMA critical path.
    uint64_t *p_full = bars + 20;   // [2]: P_j is in TMEM
    uint64_t *o_free = bars + 24;   // the epilogue has read O
    uint64_t *drain = bars + 25;     // [S issuer], and bars + 23 for the P.V issuer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 26);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 27);
    // Work items are claimed dynamically (atomicAdd on a global counter) by the
    // producer, decoded once (the tile list and indptr reads are two dependent
    // global round trips) and handed to the MMA and softmax warps, decoded, through
    // a 4-deep queue in shared memory.
    uint64_t *item_full = bars + 28;   // [4]
    uint64_t *item_empty = bars + 32;  // [4]: released by the MMA thread + 4 softmax warps
    PrefillItem *item_q = reinterpret_cast<PrefillItem *>(bars + 40);  // [4]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long n_items = static_cast<long long>(p.n_tiles) * p.nq;
    const int group = p.nq / p.nkv;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 4);
        }
        mbar_init(o_free, 4);
        mbar_init(drain, 1);
        mbar_init(bars + 23, 1);
        for (int k = 0; k < 4; ++k) {
            mbar_init(&item_full[k], 1);
            mbar_init(&item_empty[k], 5 + (ProducerSplit<HD, PAGED>::two_issuers ? 1 : 0) +
                                          (SPLIT ? 1 : 0));
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || (SPLIT && warp == ProducerSplit<HD, PAGED>::V_WARP)) {
        // ------------------------------- TMA producers -------------------------------
        // Warp 0 claims the items and loads Q, K (and, unless split, V); with a split
        // producer warp 6 loads V, taking the items from the queue like the consumers.
        const bool v_only = SPLIT && warp == ProducerSplit<HD, PAGED>::V_WARP;
        const bool loads_v = !SPLIT || v_only;
        if (lane == 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
        }
        // This grid is launched as a programmatic dependent of the kernel before it
        // (the schedule kernel, when the work list is built on the device): the
        // set-up above overlaps it, and nothing it may write (the work list, the
        // counters, q, k, v, the pools) is read before it has completed.  The other
        // warps see items only through this warp.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        uint32_t kv_it = 0;
        uint32_t n_q = 0, n_k = 0, n_v = 0;   // copies issued (for the drain on an abort)
        int stop = 0;
        // Claims the k-th item of this CTA, decodes it and publishes it to the MMA
        // and softmax warps; an item with n_kv == -1 ends the list.
        auto claim = [&](uint32_t k) -> PrefillItem {
            const int slot = k & 3;
            if (lane == 0) {
                if (!mbar_wait(&item_empty[slot], ((k >> 2) & 1) ^ 1u, p.status, abort_flag)) {
                    stop = 1;
                } else {
                    const long long claimed = atomicAdd(p.item_counter, 1);
                    item_q[slot] = claimed >= 0 && claimed < n_items
                                       ? prefill_item<PAGED, BN, WINDOW>(p, claimed)
                                       : end_item();
                    mbar_arrive(&item_full[slot]);
                }
            }
            __syncwarp();
            stop = __shfl_sync(kFullMask, stop, 0);
            return stop ? end_item() : item_q[slot];
        };
        // The V-only producer's k-th item, read from the queue the claimer fills.
        auto take = [&](uint32_t k) -> PrefillItem {
            const int slot = k & 3;
            if (lane == 0 && !mbar_wait(&item_full[slot], (k >> 2) & 1, p.status, abort_flag))
                stop = 1;
            // The shuffle carries the flag but orders no memory: the warp barrier makes
            // lane 0's acquire on item_full cover the other lanes' reads of the slot.
            __syncwarp();
            stop = __shfl_sync(kFullMask, stop, 0);
            if (stop) return end_item();
            const PrefillItem it = item_q[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            return it;
        };
        // Block-table entry of page `lane` of key tile j (lanes < BN / 16); -2 for
        // lanes and pages past the sequence or wholly before the window (those entries
        // are never looked up).  Issued a tile early, checked at use.
        auto page_raw = [&](int r, int j, int pages_seq, int page_lo) -> int {
            const int pidx = j * (BN / kBlockSize) + lane;
            if (lane >= BN / kBlockSize || pidx >= pages_seq || pidx < page_lo) return -2;
            return p.block_tables[static_cast<int64_t>(r) * p.max_blocks + pidx];
        };
        // Bad ids are flagged; they and pages past the sequence become num_blocks, an
        // out-of-range box that reads zeros.
        auto page_fix = [&](int raw) -> int {
            const bool bad = raw != -2 && (raw < 0 || raw >= p.num_blocks);
            if (__any_sync(kFullMask, bad) && lane == 0) atomicOr(p.status, kStatusBounds);
            return (raw == -2 || bad) ? static_cast<int>(p.num_blocks) : raw;
        };
        // Item k + 1 is claimed and published once item k's first K tile is on its way,
        // so the claim's atomic and the item's indptr reads overlap item k's loads
        // instead of stalling the producer between items.
        PrefillItem w = v_only ? take(0) : claim(0);
        for (uint32_t k = 0; !stop; ++k) {
            if (stop || w.n_kv < 0) break;
            if (w.n_kv == 0) {
                w = v_only ? take(k + 1) : claim(k + 1);
                continue;
            }
            const int kh = w.h / group;

            if (!v_only && lane == 0) {
                // Q is reused once the previous item's last S (tile kv_it - 1) is done.
                // With one MMA issuer and no split, this warp's own V loads keep it close
                // behind the MMA: it issued V_{kv_it-1} after P_{kv_it-3} V was done, which
                // in that thread's issue order means S_{kv_it-2} was done too, so
                // s_full[(kv_it - 1) & 1] is at most one phase from the awaited one and its
                // parity wait is exact.  At head_dim 256 neither holds (a split producer is
                // throttled only by its 3-stage K ring; two issuers have no common order),
                // so the wait is on q_empty, which the score issuer commits once per item
                // after the item's last S.
                constexpr bool Q_EMPTY = ProducerSplit<HD, PAGED>::two_issuers;
                bool ok_q = true;
                if constexpr (Q_EMPTY) {
                    if (n_q > 0) ok_q = mbar_wait(q_empty, (n_q - 1) & 1u, p.status, abort_flag);
                } else {
                    if (kv_it > 0)
                        ok_q = mbar_wait(&s_full[(kv_it - 1) & 1], ((kv_it - 1) >> 1) & 1,
                                         p.status, abort_flag);
                }
                if (!ok_q)
                    stop = 1;
                else
                    mbar_arrive_expect_tx(q_full, C::Q_BYTES);
            }
            stop = __shfl_sync(kFullMask, stop, 0);
            if (stop) break;
            if (!v_only) {
                if (lane < C::QCH)   // one 64-column chunk of Q per lane
                    tma_load_3d(smem + C::OFF_Q + lane * kBM * 128, &p.tm_q, lane * 64, w.h,
                                w.qo_start + w.q0, q_full);
                ++n_q;
            }
            const int pages_seq = (w.kv_len + kBlockSize - 1) / kBlockSize;
            const int j0 = WINDOW ? w.j0 : 0;
            const int page_lo = WINDOW ? w.kv_lo / kBlockSize : 0;
            // Loads key tile j (kv = 0) or value tile j (kv = 1) of this item into its
            // ring stage; g is the tile's index over all items of this CTA.
            auto load_tile = [&](int kv, int j, uint32_t g, int page) {
                const int ns = kv ? C::VS : C::KS;
                const int s = g % ns;
                const uint32_t ph = ((g / ns) & 1) ^ 1u;
                uint64_t *full = kv ? &v_full[s] : &k_full[s];
                uint64_t *empty = kv ? &v_empty[s] : (C::KS == 2 ? &s_full[s] : &k_empty[s]);
                const CUtensorMap *tm = kv ? &p.tm_v : &p.tm_k;
                uint8_t *dst = smem + (kv ? C::OFF_V : C::OFF_K) + s * C::KV_BYTES;
                if (lane == 0) {
                    if (!mbar_wait(empty, ph, p.status, abort_flag))
                        stop = 1;
                    else
                        mbar_arrive_expect_tx(full, C::KV_BYTES);   // before any copy lands
                }
                stop = __shfl_sync(kFullMask, stop, 0);   // also orders lane 0 before the copies
                if (stop) return;
                ++(kv ? n_v : n_k);
                // One box per lane, so a tile's boxes leave in one warp instruction: lane
                // l copies 64-column chunk l % QCH of page l / QCH (paged) or chunk l.
                if constexpr (PAGED) {
                    const int pg = __shfl_sync(kFullMask, page, (lane / C::QCH) & 31);
                    if (lane < (BN / kBlockSize) * C::QCH) {
                        const int e = lane / C::QCH, c = lane % C::QCH;
                        tma_load_4d(dst + c * C::KV_CHUNK + e * kBlockSize * 128, tm, c * 64, 0, kh,
                                    pg, full);
                    }
                } else {
                    if (lane < C::QCH)
                        tma_load_3d(dst + lane * C::KV_CHUNK, tm, lane * 64, kh,
                                    w.kv_start + (j0 + j) * BN, full);
                }
            };
            // The MMA warp consumes K_{j+1} (for S_{j+1}) before V_j (for P_j V_j), so K
            // runs one tile ahead: a K load then never waits behind a V stage, whose
            // release depends on the softmax of an earlier tile.
            // Pages are looked up once per tile (K_j and V_j share them), one tile
            // ahead of their use.
            int pg_cur = 0, raw_next = -2;
            if constexpr (PAGED) {
                pg_cur = page_fix(page_raw(w.r, j0, pages_seq, page_lo));
                if (w.n_kv > 1) raw_next = page_raw(w.r, j0 + 1, pages_seq, page_lo);
            }
            if (!v_only) load_tile(0, 0, kv_it, pg_cur);
            const PrefillItem next = (stop || v_only) ? end_item() : claim(k + 1);
            for (int j = 0; j < w.n_kv && !stop; ++j) {
                int pg_next = 0;
                if (j + 1 < w.n_kv) {
                    if constexpr (PAGED) {
                        pg_next = page_fix(raw_next);
                        if (j + 2 < w.n_kv)
                            raw_next = page_raw(w.r, j0 + j + 2, pages_seq, page_lo);
                    }
                    if (!v_only) load_tile(0, j + 1, kv_it + j + 1, pg_next);
                }
                if (!stop && loads_v) load_tile(1, j, kv_it + j, pg_cur);
                pg_cur = pg_next;
            }
            kv_it += w.n_kv;
            // the V-only producer takes its next item only after this one's tiles
            w = v_only ? (stop ? end_item() : take(k + 1)) : next;
        }
        // never leave the CTA with copies still landing in its shared memory
        if (lane == 0 && (stop || *abort_flag)) {
            auto settle = [&](uint64_t *full, int ns, uint32_t n) {
                for (uint32_t g = n > static_cast<uint32_t>(ns) ? n - ns : 0; g < n; ++g) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(&full[g % ns], (g / ns) & 1u))
                        if (global_timer_ns() - t0 > kWaitLimitNs) break;
                }
            };
            if (!v_only) {
                settle(q_full, 1, n_q);
                settle(k_full, C::KS, n_k);
            }
            if (loads_v) settle(v_full, C::VS, n_v);
        }
        // This CTA claims nothing more; the last CTA to get here clears the claim and
        // done counters, so every launch leaves them zero for the next one.
        if (!v_only && lane == 0) {
            __threadfence();
            if (atomicAdd(p.item_counter + 1, 1) == static_cast<int>(gridDim.x) - 1) {
                p.item_counter[0] = 0;
                p.item_counter[1] = 0;
            }
        }
    } else if (warp == 1 || warp == ProducerSplit<HD, PAGED>::PV_WARP) {
        // ------------------ MMA issuers: warp 1 the scores, warp 6 the P.V ------------------
        constexpr bool TWO = ProducerSplit<HD, PAGED>::two_issuers;
        const bool s_role = warp == 1;
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, BN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, HD, false, true);
            // Operand descriptors are built once: within a 128-byte-swizzled operand a
            // byte offset moves only the start-address field (address / 16, 14 bits,
            // never carried out of for shared-memory addresses), so each MMA adds a
            // constant to a base descriptor instead of rebuilding it -- the single
            // issuing thread otherwise spends more time on descriptor arithmetic than
            // the tensor core spends on a 128 x 64 x 16 MMA.
            const uint64_t q_desc = smem_desc_sw128(smem_addr(smem + C::OFF_Q), 16, 1024);
            const uint64_t k_desc = smem_desc_sw128(smem_addr(smem + C::OFF_K), 16, 1024);
            const uint64_t v_desc =
                smem_desc_sw128(smem_addr(smem + C::OFF_V), C::KV_CHUNK, 1024);
            uint32_t kv_it = 0, q_it = 0, o_items = 0;
            bool ok = true;
            // O += P_g V_g for global key tile g: the item's tile jj, whose first row is
            // key j0 * BN + jj * BN; kv_rel = kv_len - j0 * BN is the key count from the
            // item's first tile and head the first row of that tile in the window
            auto issue_pv = [&](uint32_t g, int jj, int kv_rel, int head) {
                if (!ok) return;
                const int b = g & 1;          // S / P buffer
                const int s = g % C::VS;      // V stage
                if (jj == 0 && o_items > 0)  // the previous item's epilogue has read O
                    ok = mbar_wait(o_free, (o_items - 1) & 1, p.status, abort_flag);
                ok = ok && mbar_wait(&p_full[b], (g >> 1) & 1, p.status, abort_flag) &&
                     mbar_wait(&v_full[s], (g / C::VS) & 1, p.status, abort_flag);
                if (!ok) return;
                tc_fence_after_sync();
                if constexpr (PAGED) {
                    // Rows past kv_len in the sequence's last page, and rows before the
                    // window in its first page, hold whatever the pool held; P is 0
                    // there, but 0 x NaN would still poison O, so zero them.  (Whole
                    // pages outside were read as zero boxes.)
                    const int first_stale = kv_rel - jj * BN;
                    const int head_end = jj == 0 ? head : 0;
                    if (first_stale < BN || head_end > 0) {
                        uint8_t *vt = smem + C::OFF_V + s * C::KV_BYTES;
                        const int head_begin = head_end / kBlockSize * kBlockSize;
                        for (int c = 0; c < C::QCH; ++c) {
                            for (int row = max(first_stale, 0); row < BN; ++row) {
                                uint4 *dst =
                                    reinterpret_cast<uint4 *>(vt + c * C::KV_CHUNK + row * 128);
#pragma unroll
                                for (int e = 0; e < 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
                            }
                            for (int row = head_begin; row < head_end; ++row) {
                                uint4 *dst =
                                    reinterpret_cast<uint4 *>(vt + c * C::KV_CHUNK + row * 128);
#pragma unroll
                                for (int e = 0; e < 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                        fence_proxy_async_smem();
                    }
                }
                const uint64_t vd = v_desc + ((s * C::KV_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_bf16_ts(tmem + C::TM_O, tmem + C::TM_S + b * BN + kk * 8,
                                vd + ((kk * 16 * 128) >> 4), idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&v_empty[s]);
            };
            for (uint32_t k = 0; ok; ++k) {
                const int slot = k & 3;
                ok = mbar_wait(&item_full[slot], (k >> 2) & 1, p.status, abort_flag);
                if (!ok) break;
                const PrefillItem w = item_q[slot];
                mbar_arrive(&item_empty[slot]);
                if (w.n_kv < 0) break;
                if (w.n_kv == 0) continue;
                const uint32_t base = kv_it;
                // keys from the item's first tile on, and its first row in the window
                const int kv_rel = WINDOW ? w.kv_len - w.j0 * BN : w.kv_len;
                const int head = WINDOW ? w.kv_lo - w.j0 * BN : 0;
                if (TWO && !s_role) {
                    for (int j = 0; j < w.n_kv && ok; ++j) issue_pv(base + j, j, kv_rel, head);
                    kv_it += w.n_kv;
                    ++o_items;
                    continue;
                }
                ok = mbar_wait(q_full, q_it & 1, p.status, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                for (int j = 0; j < w.n_kv && ok; ++j) {
                    const uint32_t g = base + j;
                    const int s = g % C::KS;      // K stage
                    const int b = g & 1;          // S / P buffer
                    ok = mbar_wait(&k_full[s], (g / C::KS) & 1, p.status, abort_flag);
                    // S buffer b held P_{g-2}: with two issuers its P.V (the other thread's)
                    // must be done; one issuer's MMAs run in issue order
                    if (TWO && ok && g >= 2)
                        ok = mbar_wait(&v_empty[(g - 2) % C::VS], ((g - 2) / C::VS) & 1, p.status,
                                       abort_flag);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint64_t kd = k_desc + ((s * C::KV_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t c = kk / 4, inner = (kk % 4) * 32;
                        mma_bf16_ss(tmem + C::TM_S + b * BN, q_desc + ((c * kBM * 128 + inner) >> 4),
                                    kd + ((c * C::KV_CHUNK + inner) >> 4), idesc_s, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&s_full[b]);
                    if (TWO && j == w.n_kv - 1) tc_commit(q_empty);   // the item's Q is free
                    if (!TWO && j >= 1) issue_pv(g - 1, j - 1, kv_rel, head);
                }
                if (!TWO) issue_pv(base + w.n_kv - 1, w.n_kv - 1, kv_rel, head);
                kv_it += w.n_kv;
                ++q_it;
                if (!TWO) ++o_items;
            }
            // never release TMEM / smem with tensor-core work still in flight
            uint64_t *my_drain = s_role ? drain : bars + 23;
            tc_commit(my_drain);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(my_drain, 0)) {
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp >= 2 && warp <= 5) {
        // ----------------------------- softmax + epilogue -----------------------------
        const int quad = warp & 3;                  // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;           // query row within the tile
        const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
        const float scale = p.scale_log2;
        uint32_t kv_it = 0;
        bool ok = true;
        for (uint32_t k = 0; ok; ++k) {
            const int slot = k & 3;
            ok = mbar_wait(&item_full[slot], (k >> 2) & 1, p.status, abort_flag);
            if (__any_sync(kFullMask, !ok)) break;
            const PrefillItem w = item_q[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (w.n_kv < 0) break;
            if (!w.work) continue;
            const int off = w.kv_len - w.qo_len;
            const int q_pos = w.q0 + row + off;     // last key this row may see (causal)
            RowSoftmax rs{-INFINITY, 0.f};
            for (int j = 0; j < w.n_kv && ok; ++j) {
                const uint32_t g = kv_it + j;
                const int s = g & 1;
                ok = mbar_wait(&s_full[s], (g >> 1) & 1, p.status, abort_flag);
                if (__any_sync(kFullMask, !ok)) {
                    ok = false;
                    break;
                }
                if (C::KS != 2 && warp == 2 && lane == 0) mbar_arrive(&k_empty[g % C::KS]);   // K_g read
                tc_fence_after_sync();
                uint32_t sr[BN];
                if constexpr (BN == 64) {
                    tmem_load_64(tmem + t_lane + C::TM_S + s * BN, sr);
                } else {
#pragma unroll
                    for (int c = 0; c < BN / 64; ++c) {
                        uint32_t (&chunk)[64] = *reinterpret_cast<uint32_t (*)[64]>(&sr[c * 64]);
                        tmem_load_64(tmem + t_lane + C::TM_S + s * BN + c * 64, chunk);
                    }
                }
                const int jj = WINDOW ? w.j0 + j : j;  // key tile of the request
                // under a window, row q_pos sees keys j > q_pos - window only; the tile
                // needs the lower mask when it starts before the last row's window
                const bool need_lo = WINDOW && jj * BN < w.q0 + kBM + off - window;
                const bool need_mask = (jj + 1) * BN > w.kv_len ||
                                       (p.causal && (jj + 1) * BN - 1 > w.q0 + off) || need_lo;
                const int lim = min(w.kv_len, p.causal ? q_pos + 1 : w.kv_len) - jj * BN;
                const int lo = WINDOW ? q_pos - window + 1 - jj * BN : 0;
                float m_use, corr;
                const bool grow = tile_max<BN>(sr, need_mask, lo, lim, scale, rs, m_use, corr);
                if (j > 0 && __any_sync(kFullMask, grow)) {
                    // O holds P_0..P_{j-1} V: wait for the last P.V, then rescale in TMEM
                    ok = mbar_wait(&v_empty[(g - 1) % C::VS], ((g - 1) / C::VS) & 1, p.status,
                                   abort_flag);
                    if (__any_sync(kFullMask, !ok)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const float f = grow ? corr : 1.f;
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t o[32];
                        tmem_load_32(tmem + t_lane + C::TM_O + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_store_32(tmem + t_lane + C::TM_O + c * 32, o);
                    }
                    tmem_store_wait();
                }
                if (grow) {
                    rs.l *= corr;
                    rs.m = m_use;
                }
                uint32_t pk[BN / 2];
                tile_exp<BN>(sr, scale, rs, pk);
                if constexpr (BN == 128) {
                    tmem_store_64(tmem + t_lane + C::TM_S + s * BN, pk);
                } else {
                    tmem_store_32(tmem + t_lane + C::TM_S + s * BN,
                                  *reinterpret_cast<uint32_t (*)[32]>(pk));
                }
                tmem_store_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[s]);
            }
            if (!ok) break;
            kv_it += w.n_kv;
            if (w.n_kv > 0) {   // O is final once the item's last P.V (tile kv_it - 1) is done
                ok = mbar_wait(&v_empty[(kv_it - 1) % C::VS], ((kv_it - 1) / C::VS) & 1, p.status,
                               abort_flag);
                if (__any_sync(kFullMask, !ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
            }
            const float inv = rs.l > 0.f ? 1.f / rs.l : 0.f;
            // O / l -> bf16, 32 columns at a time (o_free is released as soon as the
            // last columns have left TMEM)
            auto o_chunk = [&](int c, uint32_t (&wv)[16]) {
                uint32_t o[32];
                if (w.n_kv > 0) {
                    tmem_load_32(tmem + t_lane + C::TM_O + c * 32, o);
                    if (c == HD / 32 - 1) {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(o_free);   // O may be overwritten next
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    wv[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv,
                                        __uint_as_float(o[2 * e + 1]) * inv);
            };
            // Each thread owns one output row, so a warp's store touches 32 rows; 32-byte
            // stores (when o is 32-byte aligned: rows are multiples of 32 bytes) fill
            // whole sectors.  Staging through shared memory for wider coalescing, or a
            // TMA store of full tiles, measured slower here (the epilogue sits on the
            // softmax warps' critical path and both add latency).
            const bool row_ok = w.q0 + row < w.qo_len;
            const bool o_32B = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.o) +
                                  (static_cast<int64_t>(w.qo_start + w.q0 + row) * p.nq + w.h) * HD;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t wv[16];
                o_chunk(c, wv);
                if (row_ok && o_32B) {
                    st_global_32B(orow + c * 32, wv[0], wv[1], wv[2], wv[3], wv[4], wv[5], wv[6],
                                  wv[7]);
                    st_global_32B(orow + c * 32 + 16, wv[8], wv[9], wv[10], wv[11], wv[12], wv[13],
                                  wv[14], wv[15]);
                } else if (row_ok) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
                    dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
                    dst[2] = make_uint4(wv[8], wv[9], wv[10], wv[11]);
                    dst[3] = make_uint4(wv[12], wv[13], wv[14], wv[15]);
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ---- host side ----------------------------------------------------------------------

template <int HD, int BN, bool PAGED, bool WINDOW>
cudaError_t launch_prefill_t(PrefillParams &p, const PrefillLaunch &L, cudaStream_t stream) {
    using C = PrefillCfg<HD, BN>;
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(p.nq),
                                    static_cast<cuuint64_t>(L.total_qo)};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(HD) * 2,
                                   static_cast<cuuint64_t>(p.nq) * HD * 2};
        const cuuint32_t box[3] = {64, 1, kBM};
        if (!encode_tensor_map_bf16(&p.tm_q, L.q, 3, dims, str, box)) return cudaErrorInvalidValue;
    }
    if constexpr (!PAGED) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(p.nkv),
                                    static_cast<cuuint64_t>(L.total_kv > 0 ? L.total_kv : 1)};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(HD) * 2,
                                   static_cast<cuuint64_t>(p.nkv) * HD * 2};
        const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(BN)};
        if (!encode_tensor_map_bf16(&p.tm_k, L.k, 3, dims, str, box)) return cudaErrorInvalidValue;
        if (!encode_tensor_map_bf16(&p.tm_v, L.v, 3, dims, str, box)) return cudaErrorInvalidValue;
    } else {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(HD), 16,
                                    static_cast<cuuint64_t>(p.nkv),
                                    static_cast<cuuint64_t>(p.num_blocks)};
        const cuuint64_t str[3] = {static_cast<cuuint64_t>(L.s_token) * 2,
                                   static_cast<cuuint64_t>(L.s_head) * 2,
                                   static_cast<cuuint64_t>(L.s_block) * 2};
        const cuuint32_t box[4] = {64, 16, 1, 1};
        if (!encode_tensor_map_bf16(&p.tm_k, L.k, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!encode_tensor_map_bf16(&p.tm_v, L.v, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    // The heaviest-first work list: for up to kPrefillInlineTiles query tiles it is built
    // here, from the host indptrs, and travels in the kernel's parameters (a stable sort
    // by key-tile count, heaviest first); longer lists are built on the device by a
    // one-CTA kernel, which also clears the counters.
    cudaError_t e = cudaSuccess;
    if (p.n_tiles <= kPrefillInlineTiles && p.batch <= 65536) {
        struct Tile {
            int key;
            uint32_t code;
        };
        Tile list[kPrefillInlineTiles];
        int n = 0;
        for (int r = 0; r < p.batch; ++r) {
            const int qo_len = L.qo_indptr_h[r + 1] - L.qo_indptr_h[r];
            const int kv_len = L.kv_indptr_h[r + 1] - L.kv_indptr_h[r];
            const int nt = (qo_len + kBM - 1) / kBM;
            for (int t = 0; t < nt && n < kPrefillInlineTiles; ++t)
                list[n++] = {key_tiles(t * kBM, qo_len, kv_len, p.causal, p.window, BN),
                             static_cast<uint32_t>(r) | (static_cast<uint32_t>(t) << 16)};
        }
        std::stable_sort(list, list + n, [](const Tile &a, const Tile &b) { return a.key > b.key; });
        for (int i = 0; i < n; ++i) p.inline_tiles[i] = list[i].code;
        p.n_inline = n;
    } else {
        p.n_inline = 0;
        prefill_schedule_kernel<<<1, 1024, 0, stream>>>(p.qo_indptr, p.kv_indptr, p.batch,
                                                        p.causal, p.window, BN, p.n_tiles,
                                                        const_cast<int2 *>(p.tiles),
                                                        p.item_counter, p.status);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const void *kern = reinterpret_cast<const void *>(prefill_kernel<HD, BN, PAGED, WINDOW>);
    const uint32_t smem = C::SMEM;
    const int per_sm = C::CTAS_PER_SM, threads = ProducerSplit<HD, PAGED>::threads;
    static int configured_device = -1;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    static int sms = 0;
    if (!sms && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 152;
    const long long items = static_cast<long long>(p.n_tiles) * p.nq;
    long long ctas = static_cast<long long>(sms) * per_sm;
    if (items < ctas) ctas = items;
    void *args[] = {&p};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, kern, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int HD, bool WINDOW>
cudaError_t launch_prefill_hd(PrefillParams &p, const PrefillLaunch &L, cudaStream_t stream) {
    return p.block_tables != nullptr ? launch_prefill_t<HD, 64, true, WINDOW>(p, L, stream)
                                     : launch_prefill_t<HD, 64, false, WINDOW>(p, L, stream);
}

template <bool WINDOW>
cudaError_t launch_prefill_w(PrefillParams &p, const PrefillLaunch &L, cudaStream_t stream) {
    switch (L.head_dim) {
        case 64: return launch_prefill_hd<64, WINDOW>(p, L, stream);
        case 128: return launch_prefill_hd<128, WINDOW>(p, L, stream);
        case 256: return launch_prefill_hd<256, WINDOW>(p, L, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_prefill(PrefillParams &p, const PrefillLaunch &L, cudaStream_t stream) {
    if (p.n_tiles == 0) return cudaSuccess;
    return p.window > 0 ? launch_prefill_w<true>(p, L, stream)
                        : launch_prefill_w<false>(p, L, stream);
}

}  // namespace pa
