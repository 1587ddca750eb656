#pragma once
// pa_decode_pairs.cuh -- the single pass's work assignment, shared by the tensor-core
// decode kernels (bf16 and FP8 caches).
//
// pa_decode has no workspace for partials, so in its tensor-core form a CTA owns whole
// (sequence, kv head) pairs and runs their 512-token partitions one after another,
// merging them in registers.  Every CTA sorts the sequences by partition count, heaviest
// first, with the same stable counting sort in shared memory, so all CTAs agree on the
// order without a work counter; pair ranks then go to CTAs in a snake (CTA c takes ranks
// c, 2C - 1 - c, 2C + c, ...), which evens out the CTAs' loads.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kPairSortKeys = 1024;   // partition-count buckets of the sort

// Sequence b's length: negative -> 0, clamped to the table and to max_seq_len (flagged
// when `flag`).
__device__ __forceinline__ int pair_seq_len(const DecodeParams &p, int b, bool flag) {
    int L = p.seq_lens[b];
    if (L < 0) L = 0;
    int cap = p.max_blocks * kBlockSize;
    if (p.max_seq_len < cap) cap = p.max_seq_len;
    if (L > cap) {
        if (flag) atomicOr(p.status, kStatusBounds);
        L = cap;
    }
    return L;
}

// Active partitions of a sequence of L tokens (those reaching into the window).
__device__ __forceinline__ int pair_parts(int L, int window) {
    return (L + kPartition - 1) / kPartition - window_start(L, window) / kPartition;
}

// The walk over this CTA's pairs, one partition per step: order[] lists the sequences by
// partition count, heaviest first; pair position q is sequence order[q / nkv], kv head
// q % nkv.  Each role keeps its own walk and asks for its steps e = 0, 1, 2, ... in order.
struct PairWalk {
    int r = -1;       // rank of the current pair within this CTA (-1: none yet)
    int base = 0;     // step of the current pair's first partition
    int np = 0;       // its active partitions
    int b = 0, kh = 0, first_part = 0;

    __device__ __forceinline__ bool at(const DecodeParams &p, const int *order, int e, int &ob,
                                       int &okh, int &opart) {
        const int C = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
        const long long n_pairs = static_cast<long long>(p.num_seqs) * p.num_kv_heads;
        while (r < 0 || e >= base + np) {
            if (r >= 0) base += np;
            ++r;
            const long long q = static_cast<long long>(r) * C + ((r & 1) ? C - 1 - c : c);
            if (q >= n_pairs) return false;
            b = order[q / p.num_kv_heads];
            kh = static_cast<int>(q % p.num_kv_heads);
            const int L = pair_seq_len(p, b, false);
            np = pair_parts(L, p.window);
            first_part = window_start(L, p.window) / kPartition;
            if (np == 0) return false;   // sorted heaviest first: the rest are empty too
        }
        ob = b;
        okh = kh;
        opart = first_part + (e - base);
        return true;
    }
    // whether step e (the last one asked for) is its pair's first / last partition
    __device__ __forceinline__ bool first(int e) const { return e == base; }
    __device__ __forceinline__ bool last(int e) const { return e == base + np - 1; }
};

// The sequences in order[] by partition count, heaviest first (a stable counting sort by
// key kPairSortKeys - 1 - min(partitions, kPairSortKeys - 1)), with its histogram in hist
// (kPairSortKeys ints of shared memory, zero again on return), and zero output rows
// (num_q_heads x head_dim bf16) for the sequences of no visible token, which no pair's
// epilogue writes, each from one CTA.  All NT threads of the CTA call it together.
template <int NT>
__device__ __forceinline__ void pair_sort(const DecodeParams &p, int *order, int *hist,
                                          int head_dim) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr unsigned kAll = 0xffffffffu;
    for (int k = threadIdx.x; k < kPairSortKeys; k += NT) hist[k] = 0;
    __syncthreads();
    auto key_of = [&](int b) {
        return kPairSortKeys - 1 -
               min(pair_parts(pair_seq_len(p, b, false), p.window), kPairSortKeys - 1);
    };
    for (int b = threadIdx.x; b < p.num_seqs; b += NT) {
        const int L = pair_seq_len(p, b, blockIdx.x == 0);
        atomicAdd(&hist[key_of(b)], 1);
        if (pair_parts(L, p.window) == 0 &&
            b % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x)) {
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out) +
                               static_cast<int64_t>(b) * p.num_q_heads * head_dim;
            for (int i = 0; i < p.num_q_heads * head_dim; ++i) o[i] = __float2bfloat16_rn(0.f);
        }
    }
    __syncthreads();
    if (warp == 0) {   // exclusive prefix of the histogram, then the stable scatter
        constexpr int PER = kPairSortKeys / 32;
        int loc = 0;
        for (int i = 0; i < PER; ++i) loc += hist[lane * PER + i];
        int incl = loc;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(kAll, incl, off);
            if (lane >= off) incl += u;
        }
        int run = incl - loc;
        for (int i = 0; i < PER; ++i) {
            const int cnt = hist[lane * PER + i];
            hist[lane * PER + i] = run;
            run += cnt;
        }
        __syncwarp();
        for (int base = 0; base < p.num_seqs; base += 32) {
            const int b = base + lane;
            const bool v = b < p.num_seqs;
            const int key = v ? key_of(b) : -1 - lane;   // invalid lanes match no one
            const unsigned same = __match_any_sync(kAll, key);
            const int leader = __ffs(same) - 1;
            int start = 0;
            if (v && lane == leader) {
                start = hist[key];
                hist[key] = start + __popc(same);
            }
            start = __shfl_sync(kAll, start, leader);
            if (v) order[start + __popc(same & ((1u << lane) - 1u))] = b;
            __syncwarp();
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < kPairSortKeys; k += NT) hist[k] = 0;
}

}  // namespace
}  // namespace pa
