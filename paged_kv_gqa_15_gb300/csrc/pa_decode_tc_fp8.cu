// pa_decode_tc_fp8.cu -- split-KV paged GQA decode on the Blackwell tensor cores over
// an FP8 E4M3 KV cache, for head_dim 128 and GQA groups of 3 to 8 query heads.
//
// What it computes is the partition pass of the split decode ("paged_attn.py", the V2
// branch of forward_decode, with kv_cache_dtype "fp8", k_scale and v_scale): as the
// bf16 tensor-core decode (pa_decode_tc.cu), with every K element worth its E4M3 code
// value times k_scale and every V element its code value times v_scale.
//
// GB300 design, on top of the bf16 tensor-core decode:
//  * Pages stream as bytes: a 128-token tile is 16 KB, half the bf16 traffic.
//  * S^T = K Q^T runs on the 8-bit tensor cores (tcgen05.mma kind::f8f6f4) straight
//    from the TMA tile.  Q is split per head into two E4M3 rows, hi = e4m3(q s) and
//    lo = e4m3(q s - hi), with s a power of two that puts max|q s| in [128, 256): the
//    pair holds q to about 2^-8 relative, close to its bf16 input, so K needs no
//    conversion.  The MMA's N = 16 columns hold the G hi rows and the G lo rows; the
//    softmax adds each pair and divides by s.
//  * O^T = V^T P also runs on the 8-bit tensor cores, straight from the TMA tile: V^T
//    is read as an MN-major E4M3 operand (a tile's 128-byte rows are tokens, its bytes
//    dims), and P is carried like Q, as two E4M3 rows per head, hi = e4m3(256 p) and
//    lo = e4m3(256 p - hi), which hold p to 2^-8 relative (R17); the epilogue adds each
//    head's hi and lo columns and divides by 256.  Rows outside the partition's tokens
//    in a loaded page are zeroed in the tile before the MMA (0 x NaN would poison O).
//    An earlier design converted every V tile to f16 with four converter warps into a
//    2-stage f16 ring, and that convert -> P.V chain set the pace; dropping it frees
//    the ring's 64 KB for deeper fp8 rings.  k_scale scales the scores, v_scale
//    the outputs.
//  * Warps: 0 K producer, 1 score-MMA issuer, 2-5 softmax, Q rows and epilogue, 6 V
//    producer, 7 P.V-MMA issuer.  With two issuing threads the score MMAs of later
//    items never queue behind the P.V of an item whose softmax is still running
//    (tcgen05.commit tracks each thread's own MMAs).  P is double buffered and each
//    item's epilogue waits until the next item's P is written, so one item's P.V
//    overlaps the next item's softmax.  The softmax warps also split q into the Q rows,
//    two items ahead, so the K producer does nothing but stream tiles: with the split
//    on the producer, that warp's serial work per item set the whole kernel's pace.
//    Every wait is bounded.
//  * The same kernel runs the single pass (pa_decode) as the bf16 one does: a CTA owns
//    whole (sequence, kv head) pairs (pa_decode_pairs.cuh) and its epilogue merges the
//    pair's partitions in registers, writing the bf16 output after the last one.
#include <cuda.h>
#include <cuda_fp16.h>

#include "pa_decode_pairs.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr unsigned kMask = 0xffffffffu;
constexpr int kHD = 128;
constexpr int kTok = 128;                      // tokens per tile (MMA M of S^T)
constexpr int kTiles = kPartition / kTok;      // tiles per partition
constexpr int kPagesPerTile = kTok / kBlockSize;
constexpr int kN = 16;                         // MMA N: G hi and G lo rows (Q or P), padded
constexpr int kThreads = 256;                  // 8 warps
// Tile rings: 6 K and 6 V stages of 16 KB, as many tiles as shared memory holds.  Against
// 4 K / 6 V this measured ~2.4 % faster on the Llama-8B batch and ~2.3 % on the long-context
// one (4 K / 8 V: -2.6 % and -0.7 %; 5 K / 7 V: 0 and -1.5 %): the scores of the next
// partition start while the last one's tiles are still in use.
constexpr int kKStages = 6;                    // fp8 K tile ring
constexpr int kV8Stages = 6;                   // fp8 V tile ring
constexpr uint32_t kTile8Bytes = kTok * 128;   // 128 tokens x 128 one-byte dims
constexpr uint32_t kQBytes = kN * 128;         // Q rows: 16 x 128 bytes
constexpr uint32_t kPTile = kN * 128;          // P rows of one tile: 16 x 128 tokens, bytes
constexpr uint32_t kPBytes = kTiles * kPTile;
constexpr float kPScale = 256.f;               // P is carried as E4M3 codes of 256 p
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV8 = kOffK + kKStages * kTile8Bytes;
constexpr uint32_t kOffQ = kOffV8 + kV8Stages * kTile8Bytes;     // two Q buffers
constexpr uint32_t kOffP = kOffQ + 2 * kQBytes;                  // two P buffers
constexpr uint32_t kOffRed = kOffP + 2 * kPBytes;                // float [2][4 warps][16]
constexpr uint32_t kOffQinv = kOffRed + 2 * 4 * kN * 4;          // float [2][16]
constexpr uint32_t kOffPref = kOffQinv + 2 * kN * 4;             // int [MAXB + 1]
constexpr int kMaxSeqs = 2048;
constexpr uint32_t kOffBar = kOffPref + (kMaxSeqs + 8) * 4;
constexpr uint32_t kSmem = kOffBar + 512 + 1024;                 // + realignment slack
constexpr uint32_t kTmemCols = 256;            // S: 2 x 4 tiles x 16; O: 2 x 16
constexpr uint32_t kTmS = 0, kTmO = 128;
static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
static_assert((2 * (kKStages + kV8Stages) + 16) * 8 <= 512, "barriers fit");
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms on 1 KB boundaries");
static_assert(kPairSortKeys * 4 <= kPBytes, "the single pass's sort histogram fits in P");

struct DecodeTc8Params {
    CUtensorMap tm_k;   // pool bytes as (hd, 16 rows, nkv, blocks), box {128, 16, 1, 1}
    CUtensorMap tm_v;
    DecodeParams d;
};

__device__ __forceinline__ int seq_len8(const DecodeParams &p, int b, bool flag) {
    return pair_seq_len(p, b, flag);
}

// The k-th item of this CTA: (b, kh, partition); false when there is none.
__device__ __forceinline__ bool item8(const DecodeParams &p, const int *pref, long long total,
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
        part += window_start(seq_len8(p, b, false), p.window) / kPartition;
    return true;
}

// The k-th item of this CTA in either mode (split: the compact partition list; single
// pass: the walk over this CTA's pairs).
template <bool SINGLE>
struct Items8 {
    const int *pref;  // split: prefix of partition counts; single: sequences by weight
    long long total;
    PairWalk walk;
    __device__ __forceinline__ bool at(const DecodeParams &p, int e, int &b, int &kh, int &part) {
        if constexpr (SINGLE) return walk.at(p, pref, e, b, kh, part);
        else return item8(p, pref, total, e, b, kh, part);
    }
};

// Tokens [t0 + t_lo, t0 + n_tok) of the partition at t0, in tiles i_lo .. n_tiles - 1.
struct Span8 {
    int t0, n_tok, t_lo, i_lo, n_tiles;
};

__device__ __forceinline__ Span8 span8(const DecodeParams &p, int b, int part) {
    const int L = seq_len8(p, b, false);
    Span8 s;
    s.t0 = part * kPartition;
    s.n_tok = min(kPartition, L - s.t0);
    s.t_lo = max(0, window_start(L, p.window) - s.t0);
    s.i_lo = s.t_lo / kTok;
    s.n_tiles = (s.n_tok + kTok - 1) / kTok;
    return s;
}

// The power of two s with max|q| * s in [128, 256) (1 for a zero or NaN maximum):
// q * s then spans E4M3's top binades, and the hi / lo split keeps ~8 bits of q.
__device__ __forceinline__ float q_split_scale(float m) {
    if (!(m > 0.f)) return 1.f;
    int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xffu);
    if (e == 0) e = 1;                    // subnormal maximum: treat as 2^-126
    int k = 7 - (e - 127);
    k = max(-126, min(127, k));
    return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

// Max |x| over one 16-byte chunk (8 bf16) of q, then over the 16 lanes of a half warp
// (the 16 chunks of one head's 128 dims).  Every lane of the warp must call it.
__device__ __forceinline__ float head_max(const uint4 &raw) {
    float f[8];
    unpack_bf16x8(raw, f);
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    if (f[0] != f[0] || f[1] != f[1] || f[2] != f[2] || f[3] != f[3] || f[4] != f[4] ||
        f[5] != f[5] || f[6] != f[6] || f[7] != f[7])
        m = __int_as_float(0x7fc00000);   // NaN: the scale stays 1, NaN flows on
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
        const float o = __shfl_xor_sync(kMask, m, off);
        m = (m != m || o != o) ? __int_as_float(0x7fc00000) : fmaxf(m, o);
    }
    return m;
}

// E4M3 codes of (x1, x0) packed as (high byte, low byte), round to nearest, saturating.
__device__ __forceinline__ uint16_t e4m3x2(float x1, float x0) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(x1), "f"(x0));
    return h;
}

// Chunk c (head c / 16, dims (c % 16) * 8 .. + 7) of one item's q, already scaled by s,
// as E4M3 hi / lo codes into the Q rows at qb: row g = hi of head g, row G + g its lo;
// the bytes of each 128-byte row are swizzled in 16-byte units by row % 8.
template <int G>
__device__ __forceinline__ void store_q_split(uint8_t *qb, int c, const uint4 &raw, float s) {
    float f[8];
    unpack_bf16x8(raw, f);
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint16_t hp[2], lp[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float a0 = f[4 * h + 2 * j] * s, a1 = f[4 * h + 2 * j + 1] * s;
            hp[j] = e4m3x2(a1, a0);
            const float2 back = e4m3x2_to_float2(hp[j]);
            lp[j] = e4m3x2(a1 - back.y, a0 - back.x);
        }
        hw[h] = hp[0] | (static_cast<uint32_t>(hp[1]) << 16);
        lw[h] = lp[0] | (static_cast<uint32_t>(lp[1]) << 16);
    }
    const int g = c >> 4, d0 = (c & 15) * 8;
    const int rh = g, rl = G + g;
    *reinterpret_cast<uint2 *>(qb + rh * 128 + (((d0 >> 4) ^ (rh & 7)) << 4) + (d0 & 15)) =
        make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2 *>(qb + rl * 128 + (((d0 >> 4) ^ (rl & 7)) << 4) + (d0 & 15)) =
        make_uint2(lw[0], lw[1]);
}

template <int G, bool SINGLE>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc8_kernel(const __grid_constant__ DecodeTc8Params prm) {
    const DecodeParams &p = prm.d;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    float *qinv = reinterpret_cast<float *>(smem + kOffQinv);
    int *pref = reinterpret_cast<int *>(smem + kOffPref);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    // Items are numbered e per CTA; item e uses the Q, S and O buffers e % 2.
    uint64_t *k_full = bars;                       // fp8 K tile landed (TMA)
    uint64_t *k_empty = k_full + kKStages;         // its score MMAs are done (commit)
    uint64_t *v8_full = k_empty + kKStages;        // fp8 V tile landed (TMA)
    uint64_t *v8_empty = v8_full + kV8Stages;      // its P.V MMAs are done (commit)
    uint64_t *q_full = v8_empty + kV8Stages;       // [2] Q rows written (4 arrivals)
    uint64_t *s_full = q_full + 2;                 // [2] S^T of all the item's tiles (commit)
    uint64_t *s_free = s_full + 2;                 // [2] softmax has read S^T (4 arrivals)
    uint64_t *p_full = s_free + 2;                 // [2] P written (4 arrivals)
    uint64_t *o_full = p_full + 2;                 // [2] O^T done (commit)
    uint64_t *o_free = o_full + 2;                 // [2] epilogue has read O^T (4 arrivals)
    uint64_t *drain = o_free + 2;                  // [2] S issuer, P.V issuer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(drain + 3);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The set-up that reads no global memory (barriers, the zeroed padding, TMEM, the
    // tensor maps, which are launch parameters) runs before the wait; as a programmatic
    // dependent of the cache write it then overlaps that kernel.  Everything that reads
    // global memory (sequence lengths, block tables, q, the pools) comes after it.
    // Q and P rows 2G .. 15 stay zero (padding of the MMA's N)
    for (uint32_t i = threadIdx.x; i < (2 * kQBytes + 2 * kPBytes) / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + kOffQ)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kV8Stages; ++s) {
            mbar_init(&v8_full[s], 1);
            mbar_init(&v8_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&q_full[x], 4);
            mbar_init(&s_full[x], 1);
            mbar_init(&s_free[x], 4);
            mbar_init(&p_full[x], 4);
            mbar_init(&o_full[x], 1);
            mbar_init(&o_free[x], 4);
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
    }
    if (warp >= 2 && warp < 6)   // the softmax warps are idle until the first scores
        prefetch_decode_inputs(p.seq_lens, p.block_tables, p.q, p.num_seqs, p.max_blocks,
                               static_cast<size_t>(p.num_seqs) * p.num_q_heads * kHD * 2,
                               threadIdx.x - 64, 128);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if constexpr (!SINGLE) {
    for (int b = threadIdx.x; b < p.num_seqs; b += kThreads) {
        const int L = seq_len8(p, b, blockIdx.x == 0);
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
                const int u = __shfl_up_sync(kMask, v, off);
                if (lane >= off) v += u;
            }
            if (idx <= p.num_seqs) pref[idx] = v + carry;
            carry += __shfl_sync(kMask, v, 31);
        }
    }
    } else {
        // the sequences by partition count, heaviest first, into pref[] (the sort's
        // histogram lives in the P buffer, whose zero padding it restores)
        pair_sort<kThreads>(p, pref, reinterpret_cast<int *>(smem + kOffP), kHD);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const long long total = SINGLE ? 0 : static_cast<long long>(pref[p.num_seqs]) * p.num_kv_heads;
    const int nq = p.num_q_heads;

    if (warp == 0 || warp == 6) {
        // ------------------- producers: warp 0 K tiles, warp 6 V tiles -------------------
        const bool is_v = warp == 6;
        const int NS = is_v ? kV8Stages : kKStages;
        uint64_t *full = is_v ? v8_full : k_full;
        uint64_t *empty = is_v ? v8_empty : k_empty;
        uint8_t *ring = smem + (is_v ? kOffV8 : kOffK);
        const CUtensorMap *tm = is_v ? &prm.tm_v : &prm.tm_k;
        const uint64_t policy = l2_policy_evict_first();
        uint32_t it = 0;
        int stop = 0;
        int b, kh, part;
        Items8<SINGLE> items{pref, total};
        for (int e = 0; !stop && items.at(p, e, b, kh, part); ++e) {
            const Span8 sp = span8(p, b, part);
            const int kvh = p.kv_rep == 1 ? kh : kh / p.kv_rep;   // the pool's kv head
            // page ids of the partition, one per lane (past the sequence, before the window
            // or bad: an out-of-range box that reads zeros); the V producer flags nothing
            const int np = (sp.n_tok + kBlockSize - 1) / kBlockSize;
            const int pg_lo = sp.t_lo / kBlockSize;
            int page = (lane >= pg_lo && lane < np)
                           ? p.block_tables[static_cast<int64_t>(b) * p.max_blocks +
                                            sp.t0 / kBlockSize + lane]
                           : -2;
            const bool bad = page != -2 && (page < 0 || page >= p.num_blocks);
            if (!is_v && __any_sync(kMask, bad) && lane == 0) atomicOr(p.status, kStatusBounds);
            if (page == -2 || bad) page = static_cast<int>(p.num_blocks);
            for (int i = sp.i_lo; i < sp.n_tiles; ++i, ++it) {
                const int s = it % NS;
                if (lane == 0) {
                    if (!mbar_wait(&empty[s], ((it / NS) & 1) ^ 1u, p.status, abort_flag))
                        stop = 1;
                    else
                        mbar_arrive_expect_tx(&full[s], kTile8Bytes);
                }
                stop = __shfl_sync(kMask, stop, 0);
                if (stop) break;
                // lane l < 8 loads page l of the tile: 16 rows of 128 bytes
                const int pg = __shfl_sync(kMask, page, (i * kPagesPerTile + (lane & 7)) & 31);
                if (lane < kPagesPerTile)   // K / V are read once: evict them first
                    tma_load_4d_hint(ring + s * kTile8Bytes + lane * kBlockSize * 128, tm, 0, 0,
                                     kvh, pg, &full[s], policy);
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
            constexpr uint32_t idesc_s = idesc_f32(kTok, kN, 0, 0, false, false);   // E4M3 x E4M3
            // E4M3 V^T, MN-major: a tile's 128 dims of one token are one 128-byte row
            constexpr uint32_t idesc_o = idesc_f32(kHD, kN, 0, 0, true, false);
            const uint64_t ring_k = smem_desc_sw128(smem_addr(smem + kOffK), 16, 1024);
            const uint64_t ring_v = smem_desc_sw128(smem_addr(smem + kOffV8), kTile8Bytes, 1024);
            const uint64_t q_desc = smem_desc_sw128(smem_addr(smem + kOffQ), 16, 1024);
            const uint64_t p_desc = smem_desc_sw128(smem_addr(smem + kOffP), 16, 1024);
            uint32_t kit = 0, vit = 0;
            bool ok = true;
            Items8<SINGLE> items{pref, total};
            auto item_span = [&](int e) -> Span8 {
                int b, kh, part;
                if (!items.at(p, e, b, kh, part)) {
                    Span8 none = {};
                    none.n_tiles = -1;
                    return none;
                }
                return span8(p, b, part);
            };
            // S^T = K Q^T for every tile of item e, into S buffer e % 2
            auto issue_s = [&](int e, const Span8 &sp) {
                const int x = e & 1;
                const uint32_t use = e >> 1;
                ok = ok && mbar_wait(&q_full[x], use & 1, p.status, abort_flag);
                if (ok && e >= 2) ok = mbar_wait(&s_free[x], (use - 1) & 1, p.status, abort_flag);
                if (!ok) return;
                tc_fence_after_sync();
                const uint64_t qd = q_desc + ((x * kQBytes) >> 4);
                for (int i = sp.i_lo; i < sp.n_tiles && ok; ++i, ++kit) {
                    const int s = kit % kKStages;
                    ok = mbar_wait(&k_full[s], (kit / kKStages) & 1, p.status, abort_flag);
                    if (!ok) return;
                    tc_fence_after_sync();
                    const uint64_t kd = ring_k + ((s * kTile8Bytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kHD / 32; ++kk)   // 32 one-byte dims per MMA
                        mma_f8_ss(tmem + kTmS + x * 64 + i * kN, kd + ((kk * 32) >> 4),
                                  qd + ((kk * 32) >> 4), idesc_s, kk > 0 ? 1u : 0u);
                    tc_commit(&k_empty[s]);
                }
                if (!ok) return;
                tc_commit(&s_full[x]);
            };
            // O^T = V^T P over the fp8 V tiles of item e, with P's E4M3 hi / lo rows
            auto issue_pv = [&](int e, const Span8 &sp) {
                const int x = e & 1;
                const uint32_t use = e >> 1;
                ok = ok && mbar_wait(&p_full[x], use & 1, p.status, abort_flag);
                if (ok && e >= 2) ok = mbar_wait(&o_free[x], (use - 1) & 1, p.status, abort_flag);
                if (!ok) return;
                tc_fence_after_sync();
                for (int i = sp.i_lo; i < sp.n_tiles && ok; ++i, ++vit) {
                    const int s = vit % kV8Stages;
                    ok = mbar_wait(&v8_full[s], (vit / kV8Stages) & 1, p.status, abort_flag);
                    if (!ok) return;
                    tc_fence_after_sync();
                    // rows outside [t_lo, n_tok) in a page that was loaded hold whatever
                    // the pool held (whole pages outside read as zeros); P is 0 there,
                    // but 0 x NaN would poison O, so zero those V rows: past the sequence
                    // in its last page, and before the window in its first page
                    const int stale = sp.n_tok - i * kTok;   // first row past the tokens
                    const int head = sp.t_lo - i * kTok;     // first row in the window
                    if (stale < kTok || (head > 0 && head < kTok)) {
                        uint8_t *vt = smem + kOffV8 + s * kTile8Bytes;
                        const int tail_end = min(kTok, (stale + kBlockSize - 1) / kBlockSize * kBlockSize);
                        const int head_begin = max(0, head / kBlockSize * kBlockSize);
                        for (int r = stale; r < tail_end; ++r) {
                            uint4 *dst = reinterpret_cast<uint4 *>(vt + r * 128);
#pragma unroll
                            for (int q = 0; q < 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
                        }
                        for (int r = head_begin; r < head && r < kTok; ++r) {
                            uint4 *dst = reinterpret_cast<uint4 *>(vt + r * 128);
#pragma unroll
                            for (int q = 0; q < 8; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                    const uint64_t vd = ring_v + ((s * kTile8Bytes) >> 4);
                    const uint64_t pd = p_desc + ((x * kPBytes + i * kPTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTok / 32; ++kk)   // 32 one-byte tokens per MMA
                        mma_f8_ss(tmem + kTmO + x * kN, vd + ((kk * 32 * 128) >> 4),
                                  pd + ((kk * 32) >> 4), idesc_o, (i > sp.i_lo || kk > 0) ? 1u : 0u);
                    tc_commit(&v8_empty[s]);
                }
                if (!ok) return;
                tc_commit(&o_full[x]);
            };
            // two issuing threads: the scores of later items never queue behind the P.V
            // of an item whose softmax is still running
            for (int e = 0; ok; ++e) {
                const Span8 cur = item_span(e);
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
        // dim `row` for O^T.  The 4 warps always run the same barrier sequence.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int sid = (warp - 2) * 32 + lane;          // 0..127 across the softmax warps
        const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
        const float q_mul = p.scale_log2 * p.k_scale;    // log2 units, k_scale folded in
        bool ok = true;
        int b, kh, part;
        // These warps also write each item's Q rows (E4M3 hi / lo, R16) into Q buffer
        // e % 2 and its per-head scales into qinv[e % 2]: items 0 and 1 here, item e + 2
        // once item e's P is written (item e's score MMAs, the last reader of that
        // buffer, are complete: this warp has waited for them), so the producer warp
        // does nothing but stream K tiles.  Thread sid < 16 G holds one 16-byte chunk of
        // q, loaded an item before it is split so that the load's latency stays off
        // this chain.
        // each of q_chunk, q_write and the item loop walks the items in its own order
        Items8<SINGLE> items_qc{pref, total}, items_qw{pref, total}, items{pref, total};
        auto q_chunk = [&](int e) -> uint4 {
            int bb, kk, pp;
            if (sid >= 16 * G || !items_qc.at(p, e, bb, kk, pp)) return make_uint4(0u, 0u, 0u, 0u);
            const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q) +
                                      (static_cast<int64_t>(bb) * nq + kk * G) * kHD;
            return __ldg(reinterpret_cast<const uint4 *>(qg) + sid);
        };
        auto q_write = [&](int e, const uint4 &raw) {
            int bb, kk, pp;
            if (!items_qw.at(p, e, bb, kk, pp)) return;   // uniform over the CTA
            // head_max shuffles over the whole warp, so every lane of a warp holding a head's
            // chunk takes part (with an odd G the last such warp's upper half holds zeros)
            if (sid < 32 * ((G + 1) / 2)) {
                const float s = q_split_scale(head_max(raw));
                if (sid < 16 * G) {
                    if ((lane & 15) == 0) qinv[(e & 1) * kN + (sid >> 4)] = 1.f / s;  // exact
                    store_q_split<G>(smem + kOffQ + (e & 1) * kQBytes, sid, raw, s);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_full[e & 1]);
        };
        q_write(0, q_chunk(0));
        q_write(1, q_chunk(1));
        uint4 q_ahead = q_chunk(2);
        named_barrier(1, 128);
        // The epilogue of an item (O^T from TMEM, normalised, to the partials) is deferred
        // until the next item's P is written, so that the P.V of one item overlaps the
        // softmax of the next; its inputs wait in these registers.
        bool have_prev = false, prev_got = false, prev_first = false, prev_last = false;
        int prev_b = 0, prev_kh = 0, prev_part = 0, prev_x = 0;
        uint32_t prev_use = 0;
        float prev_sm[G], prev_mx[G];
        // single pass: the pair's running max (log2 units), sum and unnormalised output
        // (this thread's dim, v_scale not yet applied) over the partitions merged so far
        float run_m[G], run_l[G], run_o[G];
        auto epilogue = [&]() -> bool {
            bool done = prev_got && mbar_wait(&o_full[prev_x], prev_use & 1, p.status, abort_flag);
            done = !__any_sync(kMask, !done);
            uint32_t o[16];   // column g: head g's hi part, column G + g its lo part
            if (done) {
                tc_fence_after_sync();
                if constexpr (2 * G > 8) {   // G hi and G lo columns
                    tmem_load_16(tmem + t_lane + kTmO + prev_x * kN, o);
                } else {
                    tmem_load_8(tmem + t_lane + kTmO + prev_x * kN,
                                *reinterpret_cast<uint32_t (*)[8]>(o));
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[prev_x]);
            if constexpr (SINGLE) {
                if (prev_first) {
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
                        const float og = (__uint_as_float(o[g]) + __uint_as_float(o[G + g])) *
                                         (1.f / kPScale);
                        const float M = fmaxf(run_m[g], prev_mx[g]);
                        if (M != -INFINITY) {
                            const float fa = run_m[g] == -INFINITY ? 0.f : exp2f(run_m[g] - M);
                            const float fb = prev_mx[g] == -INFINITY ? 0.f : exp2f(prev_mx[g] - M);
                            run_o[g] = run_o[g] * fa + og * fb;
                            run_l[g] = run_l[g] * fa + prev_sm[g] * fb;
                            run_m[g] = M;
                        }
                    }
                    if (prev_last) {   // the pair's last partition: its output
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            static_cast<__nv_bfloat16 *>(p.out)[(static_cast<int64_t>(prev_b) * nq +
                                                                 prev_kh * G + g) * kHD + row] =
                                __float2bfloat16_rn(
                                    run_l[g] > 0.f ? run_o[g] / run_l[g] * p.v_scale : 0.f);
                    }
                }
            } else if (done) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int64_t r =
                        (static_cast<int64_t>(prev_b) * nq + prev_kh * G + g) * p.max_parts + prev_part;
                    const float og = (__uint_as_float(o[g]) + __uint_as_float(o[G + g])) *
                                     (1.f / kPScale);
                    p.part_o[r * kHD + row] = og / prev_sm[g] * p.v_scale;
                    if (row == 0) {
                        p.part_m[r] = prev_mx[g] * kLn2;
                        p.part_l[r] = prev_sm[g];
                    }
                }
            }
            return done;
        };
        for (int e = 0; items.at(p, e, b, kh, part); ++e) {
            const Span8 sp = span8(p, b, part);
            const int x = e & 1;
            const uint32_t use = e >> 1;
            const float *qi = qinv + x * kN;
            float sc[kTiles][G];
            bool got = mbar_wait(&s_full[x], use & 1, p.status, abort_flag);
            got = !__any_sync(kMask, !got);
            if (got) tc_fence_after_sync();
#pragma unroll
            for (int i = 0; i < kTiles; ++i) {
                const bool tile = got && i >= sp.i_lo && i * kTok < sp.n_tok;
                uint32_t v[16];
                if (tile) {
                    if constexpr (2 * G > 8) {   // G hi and G lo columns
                        tmem_load_16(tmem + t_lane + kTmS + x * 64 + i * kN, v);
                    } else {
                        uint32_t (&v8)[8] = *reinterpret_cast<uint32_t (*)[8]>(v);
                        tmem_load_8(tmem + t_lane + kTmS + x * 64 + i * kN, v8);
                    }
                } else {
#pragma unroll
                    for (int g = 0; g < 16; ++g) v[g] = 0u;
                }
                const int tok = i * kTok + row;
                const bool valid = tile && tok < sp.n_tok && tok >= sp.t_lo;
#pragma unroll
                for (int g = 0; g < G; ++g)
                    sc[i][g] = valid ? (__uint_as_float(v[g]) + __uint_as_float(v[G + g])) *
                                           (qi[g] * q_mul)
                                     : -INFINITY;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[x]);
            float *rm = red + quad * kN;
            float *rl = red + 4 * kN + quad * kN;
            float mx[G], sm[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float m = fmaxf(fmaxf(sc[0][g], sc[1][g]), fmaxf(sc[2][g], sc[3][g]));
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kMask, m, off));
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
                for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(kMask, s, off);
                sm[g] = s;
            }
            if (lane == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) rl[g] = sm[g];
            }
            // P into buffer e % 2 as E4M3 rows, K-major (a row's bytes are the tile's
            // tokens, swizzled in 16-byte units by row % 8): row g holds hi = e4m3(256 p)
            // of head g, row G + g its lo = e4m3(256 p - hi) (R17).  The P.V of item e - 2
            // that read this buffer finished before that item's epilogue, which ran in the
            // previous iteration.
            uint8_t *pb = smem + kOffP + x * kPBytes + (row & 15);
#pragma unroll
            for (int i = 0; i < kTiles; ++i) {
#pragma unroll
                for (int g = 0; g < G; g += 2) {   // heads in pairs; an odd G's last alone
                    const bool pair = g + 1 < G;
                    const float a0 = pv[i][g] * kPScale;
                    const float a1 = pair ? pv[i][pair ? g + 1 : g] * kPScale : 0.f;
                    const uint16_t hi = e4m3x2(a1, a0);
                    const float2 back = e4m3x2_to_float2(hi);
                    const uint16_t lo = e4m3x2(a1 - back.y, a0 - back.x);
                    uint8_t *t = pb + i * kPTile;
                    const int u = row >> 4;   // 16-byte unit of this token within a row
                    t[g * 128 + ((u ^ (g & 7)) << 4)] = static_cast<uint8_t>(hi & 0xffu);
                    t[(G + g) * 128 + ((u ^ ((G + g) & 7)) << 4)] = static_cast<uint8_t>(lo & 0xffu);
                    if (pair) {
                        t[(g + 1) * 128 + ((u ^ ((g + 1) & 7)) << 4)] = static_cast<uint8_t>(hi >> 8);
                        t[(G + g + 1) * 128 + ((u ^ ((G + g + 1) & 7)) << 4)] =
                            static_cast<uint8_t>(lo >> 8);
                    }
                }
            }
            fence_proxy_async_smem();
            named_barrier(1, 128);   // also publishes the sums
#pragma unroll
            for (int g = 0; g < G; ++g)
                sm[g] = red[4 * kN + g] + red[5 * kN + g] + red[6 * kN + g] + red[7 * kN + g];
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
            q_write(e + 2, q_ahead);
            q_ahead = q_chunk(e + 3);
            // item e - 1's epilogue runs now, while the P.V of item e can start
            const bool done = !have_prev || epilogue();
            have_prev = true;
            prev_b = b;
            prev_kh = kh;
            prev_part = part;
            prev_x = x;
            prev_use = use;
            prev_got = got;
            prev_first = items.walk.first(e);
            prev_last = items.walk.last(e);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                prev_sm[g] = sm[g];
                prev_mx[g] = mx[g];
            }
            ok = !named_barrier_or(1, 128, !(got && done));
            if (!ok) break;
        }
        if (ok && have_prev) epilogue();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int G, bool SINGLE>
cudaError_t launch_tc8(const DecodeParams &p, cudaStream_t stream) {
    DecodeTc8Params prm;
    prm.d = p;
    {
        const cuuint64_t dims[4] = {kHD, kBlockSize, static_cast<cuuint64_t>(p.pool_kv_heads),
                                    static_cast<cuuint64_t>(p.num_blocks)};
        const cuuint64_t str[3] = {static_cast<cuuint64_t>(p.s_token),
                                   static_cast<cuuint64_t>(p.s_head),
                                   static_cast<cuuint64_t>(p.s_block)};
        const cuuint32_t box[4] = {128, kBlockSize, 1, 1};
        if (!encode_tensor_map_u8(&prm.tm_k, p.k_cache, 4, dims, str, box) ||
            !encode_tensor_map_u8(&prm.tm_v, p.v_cache, 4, dims, str, box))
            return cudaErrorInvalidValue;
    }
    auto kern = decode_tc8_kernel<G, SINGLE>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
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
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
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

bool decode_tc8_supported(const DecodeParams &p, int head_dim) {
    const int g = p.num_kv_heads > 0 ? p.num_q_heads / p.num_kv_heads : 0;
    // 2 g hi / lo rows fill the MMA's N of 16
    return p.kv_fp8 && head_dim == kHD && g >= 3 && g <= kN / 2 && p.num_seqs <= kMaxSeqs &&
           p.s_token % 16 == 0 && p.s_head % 16 == 0 && p.s_block % 16 == 0 &&
           (reinterpret_cast<uintptr_t>(p.k_cache) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(p.v_cache) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(p.q) & 15) == 0;
}

cudaError_t launch_decode_tc8(const DecodeParams &p, cudaStream_t stream) {
    if (p.num_seqs == 0) return cudaSuccess;
    switch (p.num_q_heads / p.num_kv_heads) {
        case 3: return launch_tc8<3, false>(p, stream);
        case 4: return launch_tc8<4, false>(p, stream);
        case 5: return launch_tc8<5, false>(p, stream);
        case 6: return launch_tc8<6, false>(p, stream);
        case 7: return launch_tc8<7, false>(p, stream);
        case 8: return launch_tc8<8, false>(p, stream);
        default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_decode_tc8_single(const DecodeParams &p, cudaStream_t stream) {
    if (p.num_seqs == 0) return cudaSuccess;
    switch (p.num_q_heads / p.num_kv_heads) {
        case 3: return launch_tc8<3, true>(p, stream);
        case 4: return launch_tc8<4, true>(p, stream);
        case 5: return launch_tc8<5, true>(p, stream);
        case 6: return launch_tc8<6, true>(p, stream);
        case 7: return launch_tc8<7, true>(p, stream);
        case 8: return launch_tc8<8, true>(p, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
