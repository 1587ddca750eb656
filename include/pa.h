/*
 * pa.h -- C ABI of the paged-KV GQA attention library for GB300 (sm_103a).
 *
 * Operations (each cites the page section that defines it):
 *   pa_write_cache      reshape_and_cache scatter of new K/V rows into pages
 *                       ("paged_attn.py", PagedAttention.write_to_paged_cache)
 *   pa_decode           single-pass paged GQA decode
 *                       ("paged_attn.py", PagedAttention._forward_decode_pytorch
 *                        and the paged_attention_v1 call in forward_decode)
 *   pa_decode_split     split-KV decode: 512-token partitions with fp32
 *                       per-partition max / sum / partial output, then a
 *                       log-sum-exp merge ("paged_attn.py", forward_decode, V2
 *                       branch; "libmir-cuda attention/mod.rs",
 *                       SplitPagedAttention and its workspace); its two halves
 *                       are also exposed as pa_decode_partitions and
 *                       pa_decode_merge, and pa_decode_split_static runs it on a
 *                       library-owned scratch buffer (no caller workspace)
 *   pa_ragged_prefill   ragged (varlen) causal prefill of many requests in one
 *                       launch through qo_indptr / kv_indptr, over contiguous
 *                       or paged K/V ("spark_runtime/flashinfer.rs",
 *                       ragged_prefill_bf16_hd256; "paged_attn.py",
 *                       _forward_prefix_pytorch)
 *   pa_block_table_sync upload of the changed rows of a block table, for
 *                       CUDA-graph replays of the decode ("libmir-cuda
 *                       attention/mod.rs", captured decode nodes)
 *   pa_copy_blocks      copy-on-write page copies inside every layer's K and
 *                       V pools ("paged_attn.py", PagedAttention.copy_blocks)
 *   pa_swap_blocks      page copies between pools on the device and in pinned
 *                       host memory ("paged_attn.py", PagedAttention.swap_blocks)
 *   pa_selftest_wait_timeout  one bounded pipeline wait run out on purpose, to
 *                       check the PA_ERR_TIMEOUT path (no page defines it)
 *
 * The decode entry points take kv_dtype (PA_KV_BF16 or PA_KV_FP8_E4M3) with
 * k_scale / v_scale; pa_write_cache quantises into an FP8 pool with the same
 * arguments ("paged_attn.py", kv_cache_dtype, k_scale and v_scale).
 *
 * Conventions shared by every entry point:
 *  - All data pointers are DEVICE pointers of the current CUDA device unless
 *    the name ends in _h (host).  The caller owns all memory; no entry point
 *    allocates, frees or synchronises (except pa_get_device_status, which
 *    synchronises `stream`).  Work is enqueued on `stream` (a cudaStream_t,
 *    NULL = legacy default stream) and returns immediately.
 *  - bf16 tensors are passed as void pointers to IEEE bfloat16 data.
 *  - KV pools are addressed by element strides (stride_block, stride_head,
 *    stride_token) in elements of the pool's type (bytes for an FP8 pool), each
 *    a multiple of 16 bytes; the head_dim axis is contiguous.  The default layout is
 *    HND per page, [num_blocks][num_kv_heads][block_size][head_dim], i.e.
 *    strides (nkv*bs*hd, bs*hd, hd).  The NHD page layout
 *    [num_blocks][block_size][num_kv_heads][head_dim] is (bs*nkv*hd, hd, nkv*hd).
 *    K and V pools share one set of strides.
 *  - Supported shapes: head_dim in {64, 128, 256}; block_size == 16;
 *    num_q_heads % num_kv_heads == 0, with any group size g = num_q_heads /
 *    num_kv_heads ("paged_attn.py", num_queries_per_kv).  Query head h reads kv
 *    head h / g.  The decode kernels serve some group sizes directly (on the
 *    tensor cores bf16 3-16 at head_dim 128 and 3-8 at head_dim 64, fp8 3-8 at
 *    head_dim 128; the CUDA-core kernel 1, 2, 4 and 8); any other g runs as
 *    several groups of a divisor of g per kv head, each reading that kv head's
 *    pages (through L2).
 *    Pointers must be 16-byte aligned.
 *  - sliding_window (decode and prefill): a query at position pos attends only
 *    to keys j > pos - sliding_window, the sliding_window most recent keys
 *    including its own position ("paged_attn.py", forward_prefix's
 *    sliding_window; "libmir-cuda attention/mod.rs", active_partitions(token
 *    count, window)).  sliding_window <= 0 means no window.  A decode query sits
 *    at position seq_len - 1.  Block-table entries of pages that lie wholly
 *    before a query's window are never read, so a caller may recycle them.
 *  - Return value: PA_OK or an error status; on error nothing was enqueued and
 *    pa_last_error() (thread-local) describes the problem.
 *  - Device-side guards: a block-table entry outside [0, num_blocks), a
 *    seq_len larger than max_blocks_per_seq * block_size, or a slot outside
 *    the pool is never dereferenced: the affected tokens contribute nothing and
 *    a device status word records PA_ERR_DEVICE_BOUNDS.  Every pipeline wait
 *    is bounded; a wait that runs out records PA_ERR_TIMEOUT and the kernel
 *    returns.  A kernel that finds its launch unusable on the device (its
 *    realigned shared-memory tiles not fitting the launch's shared memory) does
 *    no work and records PA_ERR_UNSUPPORTED.  Read (and clear) that word with
 *    pa_get_device_status().
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID = 1,       /* bad argument (null pointer, negative size, ...) */
    PA_ERR_UNSUPPORTED = 2,   /* valid but unsupported shape or layout */
    PA_ERR_CUDA = 3,          /* a CUDA runtime call failed */
    PA_ERR_WORKSPACE = 4,     /* workspace too small or misaligned */
    PA_ERR_TIMEOUT = 5,       /* device-side bounded wait ran out */
    PA_ERR_DEVICE_BOUNDS = 6  /* device-side index guard fired */
} pa_status;

/*
 * KV cache element types ("paged_attn.py": kv_cache_dtype, k_scale, v_scale on
 * write_to_paged_cache and forward_decode).  PA_KV_FP8_E4M3 pools hold one byte
 * per element, an OCP FP8 E4M3 code (sign, 4 exponent bits with bias 7, 3
 * mantissa bits, largest finite 448, no infinities): the cache write stores the
 * code nearest to the fp32 quotient x / k_scale (v_scale for V), ties to even,
 * saturating at +-448; the decode reads code value * k_scale (v_scale).  The
 * scales must be positive and finite.  With PA_KV_BF16 they are ignored.
 * Paged prefill reads bf16 pools only.
 */
typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1 } pa_kv_dtype;

/* Tokens per split-KV partition ("paged_attn.py", _PARTITION_SIZE). */
#define PA_PARTITION_TOKENS 512

/*
 * pa_write_cache -- reshape_and_cache.
 * For each token t in [0, num_tokens) with slot = slot_mapping[t] >= 0, copies
 * k[t][h][:] into k_cache at page slot / block_size, head h, row
 * slot % block_size (and v likewise): bit for bit into a PA_KV_BF16 pool, or as
 * the E4M3 codes of the elements divided by k_scale (v_scale) into a
 * PA_KV_FP8_E4M3 pool (see pa_kv_dtype).  slot < 0 skips the token
 * (padding).  Slots >= num_blocks * block_size are not written and set
 * PA_ERR_DEVICE_BOUNDS in the device status word.  Two tokens with the same
 * slot in one call give an unspecified winner.
 *   k, v          [num_tokens][num_kv_heads][head_dim] bf16, contiguous
 *   k_cache, v_cache  pools of kv_dtype addressed by the strides (see conventions)
 *   slot_mapping  [num_tokens] int64
 */
int pa_write_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                   const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                   int head_dim, int block_size, int64_t num_blocks,
                   int64_t stride_block, int64_t stride_head, int64_t stride_token,
                   int kv_dtype, float k_scale, float v_scale, void *stream);

/*
 * pa_decode -- single-pass paged GQA decode (one query token per sequence).
 * For sequence b and query head h (kv head kh = h / (num_q_heads/num_kv_heads)):
 *   out[b][h] = softmax(sm_scale * q[b][h] . K_j) weighted sum of V_j over
 *   j < seq_lens[b], with token j at page block_tables[b][j / block_size],
 *   row j % block_size.  seq_lens[b] == 0 gives a zero row.
 *   out, q        [num_seqs][num_q_heads][head_dim] bf16
 *   block_tables  [num_seqs][max_blocks_per_seq] int32 (entries past
 *                 ceil(seq_len / block_size) are never read)
 *   seq_lens      [num_seqs] int32
 *   k_cache, v_cache, kv_dtype, k_scale, v_scale  the pools and their element
 *                 type (see pa_kv_dtype)
 * One CTA walks the whole sequence of its (b, kv head); suited to short
 * contexts or large batches.  Allocates nothing.
 */
int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
              int max_blocks_per_seq, int64_t num_blocks, int64_t stride_block,
              int64_t stride_head, int64_t stride_token, float sm_scale, int sliding_window,
              int kv_dtype, float k_scale, float v_scale, void *stream);

/*
 * Bytes of workspace pa_decode_split needs (256-byte aligned sub-buffers):
 *   P = ceil(max_seq_len / 512) partitions
 *   partial_out [num_seqs][num_q_heads][P][head_dim] fp32   at offset 0
 *   partial_max [num_seqs][num_q_heads][P] fp32  (natural-log units)  next
 *   partial_sum [num_seqs][num_q_heads][P] fp32                         next
 * Offsets are given by pa_decode_split_workspace_offsets().
 */
size_t pa_decode_split_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                      int max_seq_len);
void pa_decode_split_workspace_offsets(int num_seqs, int num_q_heads, int head_dim,
                                       int max_seq_len, size_t *off_out, size_t *off_max,
                                       size_t *off_sum);

/*
 * pa_decode_split -- split-KV paged GQA decode.  Same result as pa_decode.
 * Pass 1: one CTA per (partition p, kv head, sequence) computes for its group
 * of query heads m_p = max of the scaled scores over tokens
 * [512 p, min(512 (p+1), L)), l_p = sum exp(s - m_p) and
 * o_p = sum exp(s - m_p) V / l_p, into the workspace (fp32).  Partitions at or
 * past ceil(L / 512) are neither written nor read; under a sliding window, neither
 * are those before the partition holding key L - sliding_window, whose tokens
 * before the window are left out of its m_p, l_p and o_p.
 * Pass 2 (merge): M = max_p m_p, w_p = l_p exp(m_p - M),
 * out = sum_p w_p o_p / sum_p w_p, rounded to bf16; L == 0 gives zeros.
 * max_seq_len must be >= every seq_lens[b]; a larger seq_len is clamped to it
 * and flagged PA_ERR_DEVICE_BOUNDS.  workspace is caller-owned device memory
 * of at least pa_decode_split_workspace_size() bytes, 256-byte aligned.
 */
int pa_decode_split(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                    int max_blocks_per_seq, int64_t num_blocks, int64_t stride_block,
                    int64_t stride_head, int64_t stride_token, float sm_scale,
                    int sliding_window, int kv_dtype, float k_scale, float v_scale,
                    int max_seq_len, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The two passes of pa_decode_split as separate calls (same arguments and
 * workspace): pa_decode_partitions writes the per-partition (m_p, l_p, o_p)
 * into the workspace; pa_decode_merge reads them and writes out.  Both passes
 * must be given the same sliding_window.
 * pa_decode_split == pa_decode_partitions followed by pa_decode_merge.
 */
int pa_decode_partitions(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int max_blocks_per_seq, int64_t num_blocks, int64_t stride_block,
                         int64_t stride_head, int64_t stride_token, float sm_scale,
                         int sliding_window, int kv_dtype, float k_scale, float v_scale,
                         int max_seq_len, void *workspace, size_t workspace_bytes,
                         void *stream);
int pa_decode_merge(void *out, const int32_t *seq_lens, int num_seqs, int num_q_heads,
                    int head_dim, int max_seq_len, int sliding_window, const void *workspace,
                    size_t workspace_bytes, void *stream);

/*
 * pa_decode_split_static -- pa_decode_split for callers that cannot allocate.
 * (Not an operation from the reference pages: it has no counterpart there.)
 * Some callers may not call cudaMalloc and have no workspace to pass: e.g. a
 * plugin inside an engine that owns all device memory, or a latency-critical
 * decode loop where an allocation could synchronise the device or fail with
 * out-of-memory mid-step.  This entry point allocates nothing: the split
 * partials live in a device array of PA_STATIC_SCRATCH_BYTES compiled into the
 * library (every GPU that loads the library holds it until the process exits).
 * Arguments and result are those of pa_decode_split without the workspace.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address with cudaGetSymbolAddress; make that first call
 *    before any stream capture.  The address is cached per device together
 *    with the id of the CUDA context it was looked up in; after a
 *    cudaDeviceReset the next call looks it up again (so, after a reset, that
 *    call too must come before any capture).
 *  - A batch whose pa_decode_split_workspace_size() exceeds
 *    PA_STATIC_SCRATCH_BYTES is rejected with PA_ERR_WORKSPACE.  The 16 MiB
 *    fit a 64-sequence, 32-head, head_dim-128 batch with seq_lens up to 4096
 *    (about 8.1 MiB of partials); 8 such sequences of up to 131072 tokens need
 *    about 32.5 MiB and must use pa_decode_split with a workspace.
 *  - All calls on a device share the array, which keeps the last call's
 *    partials; nothing in it needs clearing (each call writes every partition
 *    it later merges).  Calls that overlap on the GPU (e.g. on two streams of
 *    one device) race on the array: order them on one stream or with events.
 */
#define PA_STATIC_SCRATCH_BYTES (16 * 1024 * 1024)
int pa_decode_split_static(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_blocks_per_seq, int64_t num_blocks, int64_t stride_block,
                           int64_t stride_head, int64_t stride_token, float sm_scale,
                           int sliding_window, int kv_dtype, float k_scale, float v_scale,
                           int max_seq_len, void *stream);

/*
 * Bytes of workspace pa_ragged_prefill needs: 256 bytes of work counters, then room
 * for a device-built tile schedule.
 */
size_t pa_ragged_prefill_workspace_size(int batch, int total_qo_rows, int num_q_heads,
                                        int head_dim);

/*
 * pa_ragged_prefill -- ragged causal (or full) prefill, N requests, one launch.
 * Request r owns query rows [qo_indptr[r], qo_indptr[r+1]) and
 * kv_len_r = kv_indptr[r+1] - kv_indptr[r] keys.  Query row i of request r,
 * head h, attends to keys j < kv_len_r of kv head h / (num_q_heads/num_kv_heads)
 * and, if causal != 0, only to j <= i + (kv_len_r - qo_len_r) (bottom-right
 * alignment: the query rows are the LAST qo_len_r positions).  Under a sliding
 * window, row i sees only keys j > i + (kv_len_r - qo_len_r) - sliding_window.
 * A row with no visible key is written as zeros.
 *   o, q  [total_qo_rows][num_q_heads][head_dim] bf16
 *   Contiguous mode (block_tables == NULL): k, v are
 *         [total_kv_rows][num_kv_heads][head_dim] bf16 and key j of request r
 *         is row kv_indptr[r] + j; the stride arguments are ignored.
 *   Paged mode (block_tables != NULL): k, v are the paged pools, key j of
 *         request r is token j of block_tables[r] (as in pa_decode); the
 *         kv_indptr values only give the lengths.
 *   qo_indptr_h, kv_indptr_h  [batch+1] int32 HOST copies (used to size and
 *         order the launch: up to 1024 query tiles, the heaviest-first work list
 *         is built from them on the host and passed with the launch); qo_indptr_d,
 *         kv_indptr_d the same on the device, which must hold the same values.
 *   workspace  >= pa_ragged_prefill_workspace_size() bytes, 256-byte aligned, owned
 *         by the caller and used by one call at a time.  Its first 8 bytes are the
 *         launch's work counters: they must be zero before the first call (allocate
 *         it zeroed), and every call leaves them zero.  After a call that reported
 *         PA_ERR_TIMEOUT through pa_get_device_status, zero them again.
 *   sm_scale must be positive and finite (PA_ERR_INVALID otherwise).
 */
int pa_ragged_prefill(void *o, const void *q, const void *k, const void *v,
                      const int32_t *qo_indptr_h, const int32_t *kv_indptr_h,
                      const int32_t *qo_indptr_d, const int32_t *kv_indptr_d,
                      const int32_t *block_tables, int max_blocks_per_seq, int block_size,
                      int64_t num_blocks, int64_t stride_block, int64_t stride_head,
                      int64_t stride_token, int batch, int total_qo_rows,
                      int total_kv_rows, int num_q_heads, int num_kv_heads, int head_dim,
                      float sm_scale, int causal, int sliding_window, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * Block-table upload for CUDA-graph replays ("libmir-cuda attention/mod.rs",
 * the captured decode nodes and their block-table snapshot; "paged_attn.py",
 * block tables padded for graph capture): a captured decode reads a fixed
 * device table, so between replays only the rows that changed need copying.
 *   host_table   [num_rows][row_len] int32, the table the caller wants on the
 *                device (any host memory);
 *   snapshot     [num_rows][row_len] int32 PINNED host memory owned by the
 *                caller, holding what was last uploaded.  Before the first
 *                call, fill it with -1 (a value no row holds), so that the
 *                first call finds every row changed and uploads the whole
 *                table;
 *   device_table [num_rows][row_len] int32 device memory.
 * Rows of host_table that differ from the snapshot are copied into it, and
 * each run of consecutive changed rows is enqueued on `stream` as one async
 * copy from the snapshot to device_table.  *rows_uploaded (if not NULL)
 * receives the number of rows copied.  The snapshot's rows must not change
 * again until the stream has executed those copies (for instance, sync once
 * per step, after the previous step's work on the stream is done).
 * Returns PA_OK, PA_ERR_INVALID or PA_ERR_CUDA.
 */
int pa_block_table_sync(const int32_t *host_table, int32_t *snapshot, int32_t *device_table,
                        int num_rows, int row_len, int *rows_uploaded, void *stream);

/*
 * Whole-page copies ("paged_attn.py", PagedAttention.copy_blocks and
 * PagedAttention.swap_blocks).  A page of a pool is the block_bytes contiguous
 * bytes at byte offset page * block_bytes (block_bytes = stride_block * element
 * size for a dense pool of either page layout); block_bytes must be a positive
 * multiple of 16 and every pool 16-byte aligned.
 * block_mapping is [num_pairs][2] int64 (source page, destination page).  For
 * each pair and each pool, the source page's bytes become the destination
 * page's bytes, bit for bit.  A pair with a negative entry is skipped (padding);
 * a pair with a source >= the source pool's block count or a destination >=
 * the destination pool's block count is skipped and sets PA_ERR_DEVICE_BOUNDS
 * in the device status word.  A destination that appears twice, or that is
 * also a source in the same call, gives an unspecified result.  One kernel
 * launch moves every (pair, pool) of a call (one launch per 128 pools); the
 * calls allocate nothing and return once the work is enqueued on `stream`.
 */

/*
 * pa_copy_blocks -- copy_blocks: the pairs are applied inside each of the
 * num_pools pools (pass every layer's key pool and value pool, e.g.
 * [k_0, v_0, k_1, v_1, ...]); all pools have num_blocks pages.
 *   pools          HOST array of num_pools device pointers
 *   block_mapping  device memory (or pinned host memory whose device address
 *                  equals its host address, as cudaHostAlloc gives), read by
 *                  the kernel; the call makes no CUDA runtime query, so it can
 *                  be captured into a CUDA graph.
 * Returns PA_OK, PA_ERR_INVALID or PA_ERR_CUDA.
 */
int pa_copy_blocks(void *const *pools, int num_pools, const int64_t *block_mapping,
                   int64_t num_pairs, int64_t num_blocks, int64_t block_bytes, void *stream);

/*
 * pa_swap_blocks -- swap_blocks: pool i of src_pools (src_num_blocks pages)
 * into pool i of dst_pools (dst_num_blocks pages), for i < num_pools <= 4096.
 * Each pool and block_mapping may be device memory of the current device or
 * pinned host memory (cudaHostAlloc / cudaHostRegister), or any host memory on
 * a device that can read pageable memory; host pages are read and written by
 * the kernel directly over the CPU-GPU link.  The host addresses are resolved
 * with cudaPointerGetAttributes on every call (capture this call only where that
 * query is allowed).  Memory that the device cannot address is rejected with
 * PA_ERR_INVALID.  Host memory must stay valid and unchanged until the stream
 * has run the copy.
 *   src_pools, dst_pools  HOST arrays of num_pools pointers
 * Returns PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED or PA_ERR_CUDA.
 */
int pa_swap_blocks(const void *const *src_pools, void *const *dst_pools, int num_pools,
                   const int64_t *block_mapping, int64_t num_pairs, int64_t src_num_blocks,
                   int64_t dst_num_blocks, int64_t block_bytes, void *stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word: *status_h receives PA_OK or the OR-ed PA_ERR_* bits recorded by the
 * device-side guards (bit (1 << code)).  Returns PA_OK or PA_ERR_CUDA.
 */
int pa_get_device_status(int *status_h, void *stream);

/*
 * pa_selftest_wait_timeout -- exercises the bounded wait that every kernel's
 * pipeline uses.  One thread waits on an mbarrier that nothing completes; after
 * about 1 s (the per-wait limit) it records PA_ERR_TIMEOUT in the device status
 * word and the kernel returns.  No memory is touched but that word; the context
 * stays usable.  Enqueued on `stream`; returns PA_OK, or PA_ERR_CUDA when the
 * launch fails.
 */
int pa_selftest_wait_timeout(void *stream);

/* Thread-local description of the last error returned on this thread. */
const char *pa_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
