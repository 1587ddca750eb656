// pa_decode_tc.cu -- split-KV paged GQA decode on the Blackwell tensor cores, for
// head_dim 128 with GQA groups of 3 to 16 query heads per kv head, and head_dim 64 with
// groups of 3 to 8.
//
// What it computes is the partition pass of the split decode ("paged_attn.py",
// the V2 branch of forward_decode): for sequence b, kv head kh and 512-token
// partition p, the g query heads kh*g .. kh*g+g-1 attend over the partition's
// tokens (token j at page block_tables[b][j / 16], row j % 16); the pass keeps the
// partition's max and exp-sum per head and its normalised partial output, which
// the log-sum-exp merge combines.
//
// GB300 design: the CUDA-core decode kernel spends a quarter of its time on the
// q.k and p.v multiply-adds (measured: the same page stream with the arithmetic
// removed runs 30 % faster), so here both contractions run on the tensor cores
// and the CUDA cores only do the softmax of 512 x g scores per partition:
//  * a partition is 4 tiles of 128 tokens; a tile is 8 pages, loaded by TMA with
//    one box per (page, 64-column chunk) -- 128-byte swizzle, ready for the MMA;
//  * S^T = K Q^T per tile: tcgen05.mma M = 128 tokens, N = 16 (the group's query
//    heads, zero-padded), K = head_dim, accumulated in TMEM (lane = token);
//  * four warps take the partition's softmax from TMEM (one token per thread and
//    tile), reduce max and sum over the 512 tokens, and write P (bf16) to shared
//    memory in the MMA's K-major layout;
//  * O^T = V^T P: tcgen05.mma M = 128 dims, N = 16, K = 128 tokens per tile, with V
//    read as an MN-major operand straight from the TMA tile; the epilogue reads
//    O^T from TMEM (lane = dim) and writes the partials, coalesced.  At head_dim 64
//    the V tiles' second 64-dim chunk stays zero, so M stays 128 and rows 64-127 of
//    O^T are zero and unread.
//  * Persistent CTAs walk the compact (sequence, partition, kv head) item list;
//    S, P and O are double-buffered across items.  K and V tiles stream through
//    separate rings, each filled by its own producer warp: an item's V tiles wait
//    in their ring for its softmax while the next item's K tiles (and score MMAs)
//    go ahead, so HBM keeps streaming through the softmax.  Two threads issue the
//    MMAs -- warp 1 the scores, warp 7 the P.V (tcgen05.commit tracks each thread's
//    own MMAs) -- so the score MMAs of later items never queue behind the P.V of an
//    item whose softmax is still running.  Every wait is bounded.
//  * Sliding window (keys j >= L - window): the item list holds only partitions
//    that reach into the window; in the one holding L - window, tiles wholly before
//    it are skipped, pages before it inside its first tile are read as zero boxes
//    (their table entries are never looked up), and its earlier rows are masked.
//  * The same kernel runs the single pass (pa_decode, "paged_attn.py" V1 branch),
//    which has no workspace for partials: there a CTA owns whole (sequence, kv head)
//    pairs and walks their partitions in order, and the epilogue merges each
//    partition's (max, sum, output) into running registers (the log-sum-exp rule of
//    the split's merge) and writes the bf16 output after the pair's last partition.
//    Pairs go to CTAs in a snake over the sequences sorted by partition count
//    (heaviest first: CTA c takes ranks c, 2C - 1 - c, 2C + c, ...), so the loads
//    even out without a work counter; every CTA sorts the same way (a stable counting
//    sort in shared memory), so they agree on the assignment.
#include <cuda.h>

#include "pa_decode_pairs.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr unsigned kFullMaskTc = 0xffffffffu;
constexpr int kHD = 128;
constexpr int kTok = 128;                      // tokens per tile (MMA M of S^T)
constexpr int kTiles = kPartition / kTok;      // tiles per partition
constexpr int kPagesPerTile = kTok / kBlockSize;
constexpr int kN = 16;                         // MMA N: query heads, zero-padded
constexpr int kThreadsTc = 256;                // K producer, MMA, 4 softmax, V producer, P.V MMA
// Tile rings: 3 K and 3 V stages (a partition is 4 tiles).  Against 2 K / 4 V stages
// this measured ~0.5 % faster on the Llama-8B batch, ~1 % on the 4096-key window and
// ~1.2 % on the long-context batch: a partition's first three K tiles are in flight at
// once, so its softmax starts a round trip earlier.
constexpr int kKStages = 3;                    // K tile ring
constexpr int kVStages = 3;                    // V tile ring
constexpr uint32_t kTileChunk = kTok * 128;    // one 64-column chunk of a tile
constexpr uint32_t kTileBytes = 2 * kTileChunk;
constexpr uint32_t kSmallChunk = kN * 128;     // one 64-column chunk of Q^T or P
constexpr uint32_t kQBytes = 2 * kSmallChunk;  // Q^T of one item: [2 chunks][16 rows]
constexpr uint32_t kPTile = 2 * kSmallChunk;   // P of one tile: [2 chunks][16 rows]
constexpr uint32_t kPBytes = kTiles * kPTile;
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffQ = kOffV + kVStages * kTileBytes;     // two Q^T buffers
// One P buffer: the softmax warps write item e + 1's P only after their epilogue of
// item e has seen O^T of item e complete, i.e. after every P.V read of P.
constexpr uint32_t kOffP = kOffQ + 2 * kQBytes;
constexpr uint32_t kOffRed = kOffP + kPBytes;                // float [2][4 warps][16]
constexpr uint32_t kOffPref = kOffRed + 2 * 4 * kN * 4;      // int [MAXB + 1]
constexpr int kMaxSeqsTc = 2048;
static_assert(kPairSortKeys * 4 <= kPBytes, "the single pass's sort histogram fits in P");
constexpr uint32_t kOffBar = kOffPref + (kMaxSeqsTc + 8) * 4;
constexpr uint32_t kSmemTc = kOffBar + 256 + 1024;           // + realignment slack
constexpr uint32_t kTmemCols = 256;            // S: 2 x 4 tiles x 16; O: 2 x 16
constexpr uint32_t kTmS = 0, kTmO = 128;
static_assert(kSmemTc <= 227 * 1024, "shared memory");
static_assert(kKStages <= 3 && kVStages <= 3, "the barrier layout holds 3 stages per ring");

struct DecodeTcParams {
    CUtensorMap tm_q;   // q as (hd, nq, B), box {64, g, 1}
    CUtensorMap tm_k;   // pool as (hd, 16 rows, nkv, blocks), box {64, 16, 1, 1}
    CUtensorMap tm_v;
    DecodeParams d;
};

__device__ __forceinline__ int tc_seq_len(const DecodeParams &p, int b, bool flag);

// The k-th item of this CTA: (b, kh, partition); false when there is none.
__device__ __forceinline__ bool tc_item(const DecodeParams &p, const int *pref, long long total,
                                        int k, int &b, int &kh, int &part) {
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
    part = j - pref[b];
    if (p.window > 0)   // items count from the partition holding the window's first key
        part += window_start(tc_seq_len(p, b, false), p.window) / kPartition;
    return true;
}

// The k-th item of this CTA in either mode.
template <bool SINGLE>
struct TcItems {
    const int *pref;  // split: prefix of partition counts; single: sequences by weight
    long long total;
    PairWalk walk;
    __device__ __forceinline__ bool at(const DecodeParams &p, int e, int &b, int &kh, int &part) {
        if constexpr (SINGLE) return walk.at(p, pref, e, b, kh, part);
        else return tc_item(p, pref, total, e, b, kh, part);
    }
};

// The part of item (b, part) inside the sequence and its window: tokens
// [t0 + t_lo, t0 + n_tok) of the partition starting at t0, in tiles i_lo .. n_tiles-1.
struct TcSpan {
    int t0, n_tok, t_lo, i_lo, n_tiles;
};

__device__ __forceinline__ TcSpan tc_span(const DecodeParams &p, int b, int part) {
    const int L = tc_seq_len(p, b, false);
    TcSpan s;
    s.t0 = part * kPartition;
    s.n_tok = min(kPartition, L - s.t0);
    s.t_lo = max(0, window_start(L, p.window) - s.t0);
    s.i_lo = s.t_lo / kTok;
    s.n_tiles = (s.n_tok + kTok - 1) / kTok;
    return s;
}

__device__ __forceinline__ int tc_seq_len(const DecodeParams &p, int b, bool flag) {
    return pair_seq_len(p, b, flag);
}

template <int HD, int G, bool SINGLE>
__global__ void __launch_bounds__(kThreadsTc, 1)
    decode_tc_kernel(const __grid_constant__ DecodeTcParams prm) {
    // head_dim 64 runs the head_dim-128 pipeline on the first 64-column chunk of every
    // row: the score MMAs cover only that chunk, and O^T = V^T P keeps M = 128 over V
    // tiles whose second chunk stays zero (its output rows 64-127 are zero and unread)
    static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
    constexpr int kCh = HD / 64;   // 64-column chunks of a row that carry data
    const DecodeParams &p = prm.d;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    int *pref = reinterpret_cast<int *>(smem + kOffPref);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    // Items are numbered e per CTA; item e uses Q^T, S, P and O buffers e % 2.
    //   k_full/k_empty[2], v_full/v_empty[3]  tile stages (TMA fill / MMA done reading)
    //   q_full/q_empty[2]        Q^T filled / its score MMAs done
    //   s_full[2]   S^T of all the item's tiles done (commit)
    //   s_free[2]   softmax has read S^T (one arrival per softmax warp)
    //   p_full[2]   P written to shared memory (one arrival per softmax warp)
    //   o_full[2]   O^T done (commit);  o_free[2]: epilogue has read O^T
    uint64_t *k_full = bars + 0;     // [kKStages <= 3]
    uint64_t *k_empty = bars + 3;    // [kKStages]
    uint64_t *v_full = bars + 6;     // [kVStages <= 3]
    uint64_t *v_empty = bars + 9;    // [kVStages]
    uint64_t *q_full = bars + 12;
    uint64_t *q_empty = bars + 14;
    uint64_t *s_full = bars + 16;
    uint64_t *s_free = bars + 18;
    uint64_t *p_full = bars + 20;
    uint64_t *o_full = bars + 22;
    uint64_t *o_free = bars + 24;
    uint64_t *drain = bars + 26;   // [2] S issuer, P.V issuer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 28);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 29);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The set-up that reads no global memory (barriers, the zeroed padding, TMEM, the
    // tensor maps, which are launch parameters) runs before the wait; as a programmatic
    // dependent of the cache write it then overlaps that kernel.  Everything that reads
    // global memory (sequence lengths, block tables, q, the pools) comes after it.
    // rows g .. 15 of the Q^T and P buffers stay zero (padding of the MMA's N)
    for (uint32_t i = threadIdx.x; i < (2 * kQBytes + kPBytes) / 16; i += kThreadsTc)
        reinterpret_cast<uint4 *>(smem + kOffQ)[i] = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (kCh == 1)   // the V tiles' unused second chunk reads zero
        for (uint32_t i = threadIdx.x; i < kVStages * (kTileChunk / 16); i += kThreadsTc)
            reinterpret_cast<uint4 *>(smem + kOffV + (i / (kTileChunk / 16)) * kTileBytes +
                                      kTileChunk)[i % (kTileChunk / 16)] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&q_full[b], 1);
            mbar_init(&q_empty[b], 1);
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], 4);
            mbar_init(&p_full[b], 4);
            mbar_init(&o_full[b], 1);
            mbar_init(&o_free[b], 4);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();   // the zeroed padding is read by the tensor core
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        prefetch_tensormap(&prm.tm_k);
        prefetch_tensormap(&prm.tm_v);
        prefetch_tensormap(&prm.tm_q);
    }
    if (warp >= 2 && warp < 6)   // the softmax warps are idle until the first scores
        prefetch_decode_inputs(p.seq_lens, p.block_tables, p.q, p.num_seqs, p.max_blocks,
                               static_cast<size_t>(p.num_seqs) * p.num_q_heads * HD * 2,
                               threadIdx.x - 64, 128);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if constexpr (!SINGLE) {
    // prefix over sequences of their partition counts (the compact item list)
    for (int b = threadIdx.x; b < p.num_seqs; b += kThreadsTc) {
        const int L = tc_seq_len(p, b, blockIdx.x == 0);
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
                const int u = __shfl_up_sync(kFullMaskTc, v, off);
                if (lane >= off) v += u;
            }
            if (idx <= p.num_seqs) pref[idx] = v + carry;
            carry += __shfl_sync(kFullMaskTc, v, 31);
        }
    }
    } else {
        // the sequences by partition count, heaviest first, into pref[] (the sort's
        // histogram lives in the P buffer, whose zero padding it restores)
        pair_sort<kThreadsTc>(p, pref, reinterpret_cast<int *>(smem + kOffP), HD);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const long long total = SINGLE ? 0 : static_cast<long long>(pref[p.num_seqs]) * p.num_kv_heads;

    if (warp == 0 || warp == 6) {
        // --------------------- TMA producers: warp 0 Q and K, warp 6 V ---------------------
        const bool is_v = warp == 6;
        const int NS = is_v ? kVStages : kKStages;
        uint64_t *full = is_v ? v_full : k_full;
        uint64_t *empty = is_v ? v_empty : k_empty;
        uint8_t *ring = smem + (is_v ? kOffV : kOffK);
        const CUtensorMap *tm = is_v ? &prm.tm_v : &prm.tm_k;
        const uint64_t policy = l2_policy_evict_first();
        uint32_t it = 0;   // ring uses
        int stop = 0;
        int b, kh, part;
        TcItems<SINGLE> items{pref, total};
        for (int e = 0; !stop && items.at(p, e, b, kh, part); ++e) {
            const TcSpan sp = tc_span(p, b, part);
            const int t0 = sp.t0;
            const int n_tiles = sp.n_tiles;
            const int kvh = p.kv_rep == 1 ? kh : kh / p.kv_rep;   // the pool's kv head
            // page ids of the partition, one per lane (past the sequence, before the
            // window or bad: an out-of-range box that reads zeros); read before the Q load
            // is issued, so the read and that load overlap
            const int np = (sp.n_tok + kBlockSize - 1) / kBlockSize;
            const int pg_lo = sp.t_lo / kBlockSize;
            int page = (lane >= pg_lo && lane < np)
                           ? p.block_tables[static_cast<int64_t>(b) * p.max_blocks +
                                            t0 / kBlockSize + lane]
                           : -2;
            if (!is_v) {
                const int qb = e & 1;
                if (lane == 0) {
                    if (!mbar_wait(&q_empty[qb], ((e >> 1) & 1) ^ 1u, p.status, abort_flag))
                        stop = 1;
                    else
                        mbar_arrive_expect_tx(&q_full[qb], kCh * G * 128);
                }
                stop = __shfl_sync(kFullMaskTc, stop, 0);
                if (stop) break;
                if (lane < kCh)   // Q rows of the group: one 64-column chunk per lane
                    tma_load_3d(smem + kOffQ + qb * kQBytes + lane * kSmallChunk, &prm.tm_q,
                                lane * 64, kh * G, b, &q_full[qb]);
            }
            // bad ids are flagged by the K producer only
            const bool bad = page != -2 && (page < 0 || page >= p.num_blocks);
            if (!is_v && __any_sync(kFullMaskTc, bad) && lane == 0) atomicOr(p.status, kStatusBounds);
            if (page == -2 || bad) page = static_cast<int>(p.num_blocks);
            for (int i = sp.i_lo; i < n_tiles; ++i, ++it) {
                const int s = it % NS;
                if (lane == 0) {
                    if (!mbar_wait(&empty[s], ((it / NS) & 1) ^ 1u, p.status, abort_flag))
                        stop = 1;
                    else
                        mbar_arrive_expect_tx(&full[s], kCh * kTileChunk);
                }
                stop = __shfl_sync(kFullMaskTc, stop, 0);
                if (stop) break;
                // lane l: page l / kCh of the tile, 64-column chunk l % kCh
                const int pg = __shfl_sync(kFullMaskTc, page, (i * kPagesPerTile + lane / kCh) & 31);
                if (lane < kCh * kPagesPerTile)   // K / V are read once: evict them first
                    tma_load_4d_hint(ring + s * kTileBytes + (lane % kCh) * kTileChunk +
                                         (lane / kCh) * kBlockSize * 128,
                                     tm, (lane % kCh) * 64, 0, kvh, pg, &full[s], policy);
            }
        }
        // never leave the CTA with copies still landing in its shared memory
        if (lane == 0 && (stop || *abort_flag)) {
            for (uint32_t k = (it > static_cast<uint32_t>(NS) ? it - NS : 0); k < it; ++k) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&full[k % NS], (k / NS) & 1u))
                    if (global_timer_ns() - t0 > kWaitLimitNs) break;
            }
        }
    } else if (warp == 1 || warp == 7) {
        // ------------- MMA issuers: warp 1 the scores, warp 7 the P.V -------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kTok, kN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kHD, kN, true, false);
            const uint64_t ring_k = smem_desc_sw128(smem_addr(smem + kOffK), 16, 1024);
            const uint64_t ring_v = smem_desc_sw128(smem_addr(smem + kOffV), kTileChunk, 1024);
            const uint64_t q_desc = smem_desc_sw128(smem_addr(smem + kOffQ), 16, 1024);
            const uint64_t p_desc = smem_desc_sw128(smem_addr(smem + kOffP), 16, 1024);
            uint32_t kit = 0, vit = 0;   // K / V ring uses
            bool ok = true;
            // The token span of item e; n_tiles = -1 when there is none.
            TcItems<SINGLE> items{pref, total};
            auto item_span = [&](int e) -> TcSpan {
                int b, kh, part;
                if (!items.at(p, e, b, kh, part)) {
                    TcSpan none = {};
                    none.n_tiles = -1;
                    return none;
                }
                return tc_span(p, b, part);
            };
            // S^T = K Q^T for every tile of item e, into S buffer e % 2
            auto issue_s = [&](int e, const TcSpan &sp) {
                const int n_tiles = sp.n_tiles;
                const int x = e & 1;
                const uint32_t use = e >> 1;
                ok = ok && mbar_wait(&q_full[x], use & 1, p.status, abort_flag);
                // S^T of item e - 2 has been read from TMEM before it is overwritten
                if (ok && e >= 2) ok = mbar_wait(&s_free[x], (use - 1) & 1, p.status, abort_flag);
                if (!ok) return;
                tc_fence_after_sync();
                const uint64_t qd = q_desc + ((x * kQBytes) >> 4);
                for (int i = sp.i_lo; i < n_tiles && ok; ++i, ++kit) {
                    const int s = kit % kKStages;
                    ok = mbar_wait(&k_full[s], (kit / kKStages) & 1, p.status, abort_flag);
                    if (!ok) return;
                    tc_fence_after_sync();
                    const uint64_t kd = ring_k + ((s * kTileBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off = (kk % 4) * 32;
                        mma_bf16_ss(tmem + kTmS + x * 64 + i * kN,
                                    kd + (((kk / 4) * kTileChunk + off) >> 4),
                                    qd + (((kk / 4) * kSmallChunk + off) >> 4), idesc_s,
                                    kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&k_empty[s]);
                }
                if (!ok) return;
                tc_commit(&s_full[x]);
                tc_commit(&q_empty[x]);
            };
            // O^T = V^T P over the tiles of item e, once P is in shared memory and the
            // epilogue of item e - 2 has read O buffer e % 2
            auto issue_pv = [&](int e, const TcSpan &sp) {
                const int n_tiles = sp.n_tiles, n_tok = sp.n_tok;
                const int x = e & 1;
                const uint32_t use = e >> 1;
                ok = ok && mbar_wait(&p_full[x], use & 1, p.status, abort_flag);
                if (ok && e >= 2) ok = mbar_wait(&o_free[x], (use - 1) & 1, p.status, abort_flag);
                if (!ok) return;
                tc_fence_after_sync();
                for (int i = sp.i_lo; i < n_tiles && ok; ++i, ++vit) {
                    const int s = vit % kVStages;
                    ok = mbar_wait(&v_full[s], (vit / kVStages) & 1, p.status, abort_flag);
                    if (!ok) return;
                    tc_fence_after_sync();
                    // rows outside [t_lo, n_tok) in a page that was loaded hold whatever
                    // the pool held (whole pages outside read as zeros); P is 0 there,
                    // but 0 x NaN would poison O, so zero those V rows: past the sequence
                    // in its last page, and before the window in its first page
                    const int stale = n_tok - i * kTok;   // first row past the tokens
                    const int head = sp.t_lo - i * kTok;  // first row in the window
                    if (stale < kTok || (head > 0 && head < kTok)) {
                        uint8_t *vt = smem + kOffV + s * kTileBytes;
                        const int tail_end = min(kTok, (stale + kBlockSize - 1) / kBlockSize * kBlockSize);
                        const int head_begin = max(0, head / kBlockSize * kBlockSize);
                        for (int c = 0; c < kCh; ++c) {
                            for (int row = stale; row < tail_end; ++row) {
                                uint4 *dst = reinterpret_cast<uint4 *>(vt + c * kTileChunk + row * 128);
#pragma unroll
                                for (int q = 0; q < 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
                            }
                            for (int row = head_begin; row < head && row < kTok; ++row) {
                                uint4 *dst = reinterpret_cast<uint4 *>(vt + c * kTileChunk + row * 128);
#pragma unroll
                                for (int q = 0; q < 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                        fence_proxy_async_smem();
                    }
                    const uint64_t vd = ring_v + ((s * kTileBytes) >> 4);
                    const uint64_t pd = p_desc + ((i * kPTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTok / 16; ++kk)
                        mma_bf16_ss(tmem + kTmO + x * kN, vd + ((kk * 16 * 128) >> 4),
                                    pd + (((kk / 4) * kSmallChunk + (kk % 4) * 32) >> 4), idesc_o,
                                    (i > sp.i_lo || kk > 0) ? 1u : 0u);
                    tc_commit(&v_empty[s]);
                }
                if (!ok) return;
                tc_commit(&o_full[x]);
            };
            // Software pipeline: the scores of item e + 1 are issued before the P.V of
            // item e, so they run while item e's softmax does and the K ring keeps
            // draining (the S buffers alternate; s_free guards their reuse).
            for (int e = 0; ok; ++e) {
                const TcSpan cur = item_span(e);
                if (cur.n_tiles <= 0) break;
                if (warp == 1) issue_s(e, cur); else issue_pv(e, cur);
            }
            uint64_t *my_drain = &drain[warp == 1 ? 0 : 1];
            tc_commit(my_drain);   // never release TMEM / smem with MMAs in flight
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(my_drain, 0)) {
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
            }
        }
        __syncwarp();
    } else {
        // --------------------------- softmax + epilogue ---------------------------
        // Thread row (0..127) is TMEM lane `row`: token `row` of every tile for S^T,
        // dim `row` for O^T.  The 4 warps reduce over the partition through shared
        // memory and named barrier 1; all 4 always run the same barrier sequence.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
        const float scale = p.scale_log2;
        const int nq = p.num_q_heads;
        bool ok = true;
        int b, kh, part;
        TcItems<SINGLE> items{pref, total};
        // single pass: the pair's running max (log2 units), sum and unnormalised output
        // (this thread's dim) over the partitions merged so far
        float run_m[G], run_l[G], run_o[G];
        for (int e = 0; items.at(p, e, b, kh, part); ++e) {
            const TcSpan sp = tc_span(p, b, part);
            const int n_tok = sp.n_tok;
            const int x = e & 1;
            const uint32_t use = e >> 1;
            // scores of this thread's token in each tile, in log2 units
            float sc[kTiles][G];
            bool got = mbar_wait(&s_full[x], use & 1, p.status, abort_flag);
            got = !__any_sync(kFullMaskTc, !got);
            if (got) tc_fence_after_sync();
#pragma unroll
            for (int i = 0; i < kTiles; ++i) {
                const bool tile = got && i >= sp.i_lo && i * kTok < n_tok;
                constexpr int NL = G > 8 ? 16 : 8;   // S^T columns loaded: one per head
                uint32_t v[NL];
                if (tile) {
                    if constexpr (NL == 16) {
                        tmem_load_16(tmem + t_lane + kTmS + x * 64 + i * kN, v);
                    } else {
                        tmem_load_8(tmem + t_lane + kTmS + x * 64 + i * kN, v);
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < NL; ++g) v[g] = 0u;
                }
                const bool valid = tile && i * kTok + row < n_tok && i * kTok + row >= sp.t_lo;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    sc[i][g] = valid ? __uint_as_float(v[g]) * scale : -INFINITY;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[x]);   // S^T buffer x may be rewritten
            // partition max and sum per head: warp shuffles, then the 4 warps
            float* rm = red + quad * kN;               // [4][16] maxima, then [4][16] sums
            float* rl = red + 4 * kN + quad * kN;
            float mx[G], sm[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float m = fmaxf(fmaxf(sc[0][g], sc[1][g]), fmaxf(sc[2][g], sc[3][g]));
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(kFullMaskTc, m, off));
                mx[g] = m;
            }
            if (lane == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) rm[g] = mx[g];
            }
            named_barrier(1, 128);
#pragma unroll
            for (int g = 0; g < G; ++g)
                mx[g] = fmaxf(fmaxf(red[g], red[kN + g]), fmaxf(red[2 * kN + g], red[3 * kN + g]));
            float pv[kTiles][G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < kTiles; ++i) {
                    pv[i][g] = sc[i][g] == -INFINITY ? 0.f : exp2f(sc[i][g] - mx[g]);
                    s += pv[i][g];
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(kFullMaskTc, s, off);
                sm[g] = s;
            }
            if (lane == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) rl[g] = sm[g];
            }
            // P (bf16), K-major by head: tile i, chunk row / 64, head row g, 16-byte
            // chunk (row % 64) / 8 swizzled by g % 8 (rows 8-15 are the second 8-row swizzle
            // atom), element row % 8.  The previous item's P.V has completed: this warp's
            // epilogue of it waited for O^T.
            uint8_t *pb = smem + kOffP + (row / 64) * kSmallChunk + (row % 8) * 2;
#pragma unroll
            for (int i = 0; i < kTiles; ++i)
#pragma unroll
                for (int g = 0; g < G; ++g)
                    *reinterpret_cast<__nv_bfloat16 *>(pb + i * kPTile + g * 128 +
                                                       ((((row % 64) / 8) ^ (g & 7)) << 4)) =
                        __float2bfloat16_rn(pv[i][g]);
            fence_proxy_async_smem();
            named_barrier(1, 128);   // also publishes the sums
#pragma unroll
            for (int g = 0; g < G; ++g)
                sm[g] = red[4 * kN + g] + red[5 * kN + g] + red[6 * kN + g] + red[7 * kN + g];
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
            // epilogue: O^T (lane = dim) -> partial output, normalised by the sum
            bool done = got && mbar_wait(&o_full[x], use & 1, p.status, abort_flag);
            done = !__any_sync(kFullMaskTc, !done);
            uint32_t o[G > 8 ? 16 : 8];   // O^T columns: one per head
            if (done) {
                tc_fence_after_sync();
                if constexpr (G > 8) {
                    tmem_load_16(tmem + t_lane + kTmO + x * kN, o);
                } else {
                    tmem_load_8(tmem + t_lane + kTmO + x * kN, o);
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[x]);
            if constexpr (SINGLE) {
                if (items.walk.first(e)) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        run_m[g] = -INFINITY;
                        run_l[g] = 0.f;
                        run_o[g] = 0.f;
                    }
                }
                if (done) {
                    // log-sum-exp merge of this partition into the running state
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float M = fmaxf(run_m[g], mx[g]);
                        if (M != -INFINITY) {
                            const float fa = run_m[g] == -INFINITY ? 0.f : exp2f(run_m[g] - M);
                            const float fb = mx[g] == -INFINITY ? 0.f : exp2f(mx[g] - M);
                            run_o[g] = run_o[g] * fa + __uint_as_float(o[g]) * fb;
                            run_l[g] = run_l[g] * fa + sm[g] * fb;
                            run_m[g] = M;
                        }
                    }
                    if (items.walk.last(e) && row < HD) {   // the pair's last partition
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            static_cast<__nv_bfloat16 *>(p.out)[(static_cast<int64_t>(b) * nq +
                                                                 kh * G + g) * HD + row] =
                                __float2bfloat16_rn(run_l[g] > 0.f ? run_o[g] / run_l[g] : 0.f);
                    }
                }
            } else if (done) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int64_t r =
                        (static_cast<int64_t>(b) * nq + kh * G + g) * p.max_parts + part;
                    if (row < HD) p.part_o[r * HD + row] = __uint_as_float(o[g]) / sm[g];
                    if (row == 0) {
                        p.part_m[r] = mx[g] * kLn2;
                        p.part_l[r] = sm[g];
                    }
                }
            }
            // every softmax warp leaves the item loop at the same item
            ok = !named_barrier_or(1, 128, !(got && done));
            if (!ok) break;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int HD, int G, bool SINGLE>
cudaError_t launch_tc(const DecodeParams &p, cudaStream_t stream) {
    DecodeTcParams prm;
    prm.d = p;
    {
        const cuuint64_t dims[3] = {HD, static_cast<cuuint64_t>(p.num_q_heads),
                                    static_cast<cuuint64_t>(p.num_seqs)};
        const cuuint64_t str[2] = {HD * 2, static_cast<cuuint64_t>(p.num_q_heads) * HD * 2};
        const cuuint32_t box[3] = {64, G, 1};
        if (!encode_tensor_map_bf16(&prm.tm_q, p.q, 3, dims, str, box))
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {HD, kBlockSize, static_cast<cuuint64_t>(p.pool_kv_heads),
                                    static_cast<cuuint64_t>(p.num_blocks)};
        const cuuint64_t str[3] = {static_cast<cuuint64_t>(p.s_token) * 2,
                                   static_cast<cuuint64_t>(p.s_head) * 2,
                                   static_cast<cuuint64_t>(p.s_block) * 2};
        const cuuint32_t box[4] = {64, kBlockSize, 1, 1};
        if (!encode_tensor_map_bf16(&prm.tm_k, p.k_cache, 4, dims, str, box) ||
            !encode_tensor_map_bf16(&prm.tm_v, p.v_cache, 4, dims, str, box))
            return cudaErrorInvalidValue;
    }
    auto kern = decode_tc_kernel<HD, G, SINGLE>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    static int sms = 0;
    if (!sms && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 152;
    // split: one CTA per item at most; single pass: one per (sequence, kv head) pair
    const long long slots = static_cast<long long>(p.num_seqs) * p.num_kv_heads *
                            (SINGLE ? 1 : active_partitions_cap(p.max_parts, p.window));
    long long n = sms;
    if (slots < n) n = slots;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n > 0 ? n : 1));
    cfg.blockDim = dim3(kThreadsTc);
    cfg.dynamicSmemBytes = kSmemTc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&prm};
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kern), args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// The largest group size with a kernel at this head_dim.
int decode_tc_max_group(int head_dim) { return head_dim == kHD ? kN : (head_dim == 64 ? 8 : 0); }

bool decode_tc_supported(const DecodeParams &p, int head_dim) {
    const int g = p.num_kv_heads > 0 ? p.num_q_heads / p.num_kv_heads : 0;
    return !p.kv_fp8 && g >= 3 && g <= decode_tc_max_group(head_dim) &&
           p.num_seqs <= kMaxSeqsTc &&
           (p.s_token * 2) % 16 == 0 && (p.s_head * 2) % 16 == 0 && (p.s_block * 2) % 16 == 0 &&
           (reinterpret_cast<uintptr_t>(p.k_cache) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(p.v_cache) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(p.q) & 15) == 0;
}

namespace {

template <bool SINGLE>
cudaError_t launch_tc_any(const DecodeParams &p, int head_dim, cudaStream_t stream) {
    if (p.num_seqs == 0) return cudaSuccess;
    const int g = p.num_q_heads / p.num_kv_heads;
    if (head_dim == 64) {
        switch (g) {
            case 3: return launch_tc<64, 3, SINGLE>(p, stream);
            case 4: return launch_tc<64, 4, SINGLE>(p, stream);
            case 5: return launch_tc<64, 5, SINGLE>(p, stream);
            case 6: return launch_tc<64, 6, SINGLE>(p, stream);
            case 7: return launch_tc<64, 7, SINGLE>(p, stream);
            case 8: return launch_tc<64, 8, SINGLE>(p, stream);
            default: return cudaErrorNotSupported;
        }
    }
    switch (g) {
        case 3: return launch_tc<kHD, 3, SINGLE>(p, stream);
        case 4: return launch_tc<kHD, 4, SINGLE>(p, stream);
        case 5: return launch_tc<kHD, 5, SINGLE>(p, stream);
        case 6: return launch_tc<kHD, 6, SINGLE>(p, stream);
        case 7: return launch_tc<kHD, 7, SINGLE>(p, stream);
        case 8: return launch_tc<kHD, 8, SINGLE>(p, stream);
        case 9: return launch_tc<kHD, 9, SINGLE>(p, stream);
        case 10: return launch_tc<kHD, 10, SINGLE>(p, stream);
        case 11: return launch_tc<kHD, 11, SINGLE>(p, stream);
        case 12: return launch_tc<kHD, 12, SINGLE>(p, stream);
        case 13: return launch_tc<kHD, 13, SINGLE>(p, stream);
        case 14: return launch_tc<kHD, 14, SINGLE>(p, stream);
        case 15: return launch_tc<kHD, 15, SINGLE>(p, stream);
        case 16: return launch_tc<kHD, 16, SINGLE>(p, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeParams &p, int head_dim, cudaStream_t stream) {
    return launch_tc_any<false>(p, head_dim, stream);
}

cudaError_t launch_decode_tc_single(const DecodeParams &p, int head_dim, cudaStream_t stream) {
    return launch_tc_any<true>(p, head_dim, stream);
}

}  // namespace pa
