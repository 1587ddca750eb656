// pa_internal.h -- launch parameter blocks and launcher declarations shared
// between the C ABI layer (pa_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

struct WriteCacheParams {
    const void *k, *v;
    void *k_cache, *v_cache;
    const int64_t *slot_mapping;
    int64_t num_tokens, num_blocks;
    int64_t s_block, s_head, s_token;
    int num_kv_heads, head_dim, block_size;
    int kv_fp8;                   // store FP8 E4M3 codes of x / scale (else bf16 bits)
    float k_scale, v_scale;
    int *status;
};

struct DecodeParams {
    void *out;                    // bf16 [B][nq][hd]        (single pass)
    const void *q;                // bf16 [B][nq][hd]
    const void *k_cache, *v_cache;
    const int32_t *block_tables;  // [B][max_blocks]
    const int32_t *seq_lens;      // [B]
    float *part_o, *part_m, *part_l;  // split partials (split pass only)
    int64_t num_blocks;
    int64_t s_block, s_head, s_token;
    int num_seqs, num_q_heads, num_kv_heads, max_blocks;
    // The kernels serve num_kv_heads groups of num_q_heads / num_kv_heads query heads;
    // group kh reads pool kv head kh / kv_rep, of pool_kv_heads.  A call whose GQA group
    // has no kernel of its own runs as kv_rep groups per pool kv head (launch_decode).
    int kv_rep, pool_kv_heads;
    int max_parts;                // split: partitions per (b, h) in the workspace
    int max_seq_len;              // split: clamp for seq_lens
    float scale_log2;             // sm_scale * log2(e)
    int rows_contiguous;          // s_token == head_dim: one bulk copy per page
    int window;                   // sliding window in keys (> 0), or 0 for none
    int kv_fp8;                   // the pools hold FP8 E4M3 codes (else bf16)
    float k_scale, v_scale;       // FP8: element value = code value * scale
    int *status;
};

// Work lists of up to this many query tiles are ordered on the host and passed inline
// in the kernel's parameters (4 KB); longer ones are ordered by a one-CTA kernel.
constexpr int kPrefillInlineTiles = 1024;

struct PrefillParams {
    CUtensorMap tm_q;   // q [total_qo][nq][hd] as (hd, nq, rows), 128-row boxes
    CUtensorMap tm_k;   // ragged: (hd, nkv, rows); paged: (hd, 16, nkv, blocks)
    CUtensorMap tm_v;
    void *o;
    const int32_t *qo_indptr, *kv_indptr;  // device [batch + 1]
    const int32_t *block_tables;           // paged mode, else nullptr
    const int2 *tiles;                     // (request, q tile), heaviest first (device list)
    // [0] the next unclaimed work item, [1] CTAs done; zero when a launch starts (the
    // last CTA to finish clears both)
    int *item_counter;
    int64_t num_blocks;
    int batch, nq, nkv, max_blocks, n_tiles, causal;
    int window;                            // sliding window in keys (> 0), or 0 for none
    float scale_log2;
    int *status;
    // > 0: the work list is inline_tiles[0 .. n_inline - 1], each request | tile << 16,
    // heaviest first, and `tiles` is unused
    int n_inline;
    uint32_t inline_tiles[kPrefillInlineTiles];
};

struct PrefillLaunch {
    const void *q, *k, *v;
    const int32_t *qo_indptr_h, *kv_indptr_h;   // host copies of the indptrs
    int64_t total_qo, total_kv;
    int64_t s_block, s_head, s_token;
    int head_dim;
};

// Set the thread's last-error message and return `code` (or PA_ERR_CUDA).
int api_fail(int code, const char *fmt, ...);
int api_cuda_fail(cudaError_t e, const char *what);

// Tiled tensor map of a bf16 tensor with 128-byte swizzle, out-of-range reads as
// zeros; false when the driver entry point or the encoding fails.
bool encode_tensor_map_bf16(CUtensorMap *tm, const void *base, int rank, const cuuint64_t *dims,
                            const cuuint64_t *strides_bytes, const cuuint32_t *box);
// The same for a tensor of bytes (FP8 E4M3 codes).
bool encode_tensor_map_u8(CUtensorMap *tm, const void *base, int rank, const cuuint64_t *dims,
                          const cuuint64_t *strides_bytes, const cuuint32_t *box);

cudaError_t launch_write_cache(const WriteCacheParams &p, cudaStream_t stream);
// Tensor-core partition pass of the split decode (head_dim 128, GQA group 4 or 8).
bool decode_tc_supported(const DecodeParams &p, int head_dim);
int decode_tc_max_group(int head_dim);
cudaError_t launch_decode_tc(const DecodeParams &p, int head_dim, cudaStream_t stream);
cudaError_t launch_decode_tc_single(const DecodeParams &p, int head_dim, cudaStream_t stream);
// The same over an FP8 E4M3 cache (pa_decode_tc_fp8.cu).
bool decode_tc8_supported(const DecodeParams &p, int head_dim);
cudaError_t launch_decode_tc8(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_decode_tc8_single(const DecodeParams &p, cudaStream_t stream);
// Returns cudaErrorNotSupported for an unsupported (head_dim, group) pair.
cudaError_t launch_decode(const DecodeParams &p, int head_dim, bool split, cudaStream_t stream);
// The CUDA-core decode over FP8 E4M3 caches (pa_decode_fp8.cu).
cudaError_t launch_decode_fp8(const DecodeParams &p, int head_dim, bool split,
                              cudaStream_t stream);
cudaError_t launch_merge(const DecodeParams &p, int head_dim, cudaStream_t stream);
cudaError_t launch_prefill(PrefillParams &p, const PrefillLaunch &L, cudaStream_t stream);

// Records `msg` as this thread's pa_last_error() text and returns `code`.
int set_error(int code, const char *msg);
// Device address of the current device's status word (PA_OK or an error status).
int api_status_ptr(int **out);
// Unique id of the CUDA context current on this thread, or 0 if there is none or the
// driver cannot say.  A device address cached under one id is stale under another
// (cudaDeviceReset tears the context down; the next one may load the module elsewhere).
unsigned long long current_context_id();

}  // namespace pa
