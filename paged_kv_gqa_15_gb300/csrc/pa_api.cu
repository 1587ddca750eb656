// pa_api.cu -- the C ABI (include/pa.h): argument validation, workspace
// layout, the device status word, and kernel dispatch.  No entry point here
// allocates memory or synchronises (pa_get_device_status excepted).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

thread_local char g_last_error[512] = "no error";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

// Error reporting for entry points defined in other translation units.
int pa::api_fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

int pa::api_cuda_fail(cudaError_t e, const char *what) { return cuda_fail(e, what); }

namespace {

// Device status word (OR of 1 << PA_ERR_* bits), one per device.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
struct CachedStatus {
    unsigned long long ctx;   // context the address belongs to (0: do not reuse)
    int *ptr;
};
CachedStatus g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mutex;

int status_ptr(int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device %d", dev);
    std::lock_guard<std::mutex> lock(g_status_mutex);
    const unsigned long long ctx = pa::current_context_id();
    if (ctx == 0 || g_status_ptr[dev].ctx != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        g_status_ptr[dev] = {pa::current_context_id(), static_cast<int *>(p)};
    }
    *out = g_status_ptr[dev].ptr;
    return PA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_heads(int head_dim, int num_q_heads, int num_kv_heads) {
    if (num_q_heads <= 0 || num_kv_heads <= 0)
        return fail(PA_ERR_INVALID, "head counts must be positive (nq=%d, nkv=%d)", num_q_heads,
                    num_kv_heads);
    if (num_q_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    num_q_heads, num_kv_heads);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", head_dim);
    return PA_OK;
}

// Element size in bytes of a KV cache dtype (0 for an unknown one).
int kv_elem_bytes(int kv_dtype) {
    return kv_dtype == PA_KV_BF16 ? 2 : (kv_dtype == PA_KV_FP8_E4M3 ? 1 : 0);
}

int check_kv_dtype(int kv_dtype, float k_scale, float v_scale) {
    if (!kv_elem_bytes(kv_dtype)) return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d", kv_dtype);
    if (kv_dtype == PA_KV_FP8_E4M3 &&
        (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY))
        return fail(PA_ERR_INVALID, "fp8 cache scales must be positive and finite (%g, %g)",
                    (double)k_scale, (double)v_scale);
    return PA_OK;
}

int check_pool(int head_dim, int block_size, int64_t num_blocks, int num_kv_heads,
               int64_t sb, int64_t sh, int64_t st, int elem_bytes = 2) {
    if (block_size != 16)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d: only 16-token blocks", block_size);
    if (num_blocks <= 0) return fail(PA_ERR_INVALID, "num_blocks %lld", (long long)num_blocks);
    const int64_t q = 16 / elem_bytes;   // elements per 16 bytes
    if (sb <= 0 || sh <= 0 || st <= 0 || sb % q || sh % q || st % q)
        return fail(PA_ERR_INVALID,
                    "pool strides (%lld, %lld, %lld) must be positive multiples of 16 bytes",
                    (long long)sb, (long long)sh, (long long)st);
    if (st < head_dim)
        return fail(PA_ERR_INVALID, "token stride %lld < head_dim %d", (long long)st, head_dim);
    (void)num_kv_heads;
    return PA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int decode_common(pa::DecodeParams &p, void *out, const void *q, const void *k_cache,
                  const void *v_cache, const int32_t *block_tables, const int32_t *seq_lens,
                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int max_blocks_per_seq, int64_t num_blocks, int64_t sb, int64_t sh, int64_t st,
                  float sm_scale, int sliding_window, int kv_dtype, float k_scale, float v_scale) {
    if (num_seqs < 0) return fail(PA_ERR_INVALID, "num_seqs %d", num_seqs);
    int rc = check_heads(head_dim, num_q_heads, num_kv_heads);
    if (rc) return rc;
    rc = check_kv_dtype(kv_dtype, k_scale, v_scale);
    if (rc) return rc;
    rc = check_pool(head_dim, block_size, num_blocks, num_kv_heads, sb, sh, st,
                    kv_elem_bytes(kv_dtype));
    if (rc) return rc;
    if (max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID, "max_blocks_per_seq %d", max_blocks_per_seq);
    if (num_seqs > 0 && (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens))
        return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID, "out, q and the KV pools must be 16-byte aligned");
    if (!(sm_scale == sm_scale)) return fail(PA_ERR_INVALID, "sm_scale is NaN");
    std::memset(&p, 0, sizeof p);
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.num_blocks = num_blocks;
    p.s_block = sb;
    p.s_head = sh;
    p.s_token = st;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.kv_rep = 1;
    p.pool_kv_heads = num_kv_heads;
    p.max_blocks = max_blocks_per_seq;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.rows_contiguous = (st == head_dim) ? 1 : 0;
    p.max_seq_len = max_blocks_per_seq * 16;
    p.window = sliding_window > 0 ? sliding_window : 0;
    p.kv_fp8 = kv_dtype == PA_KV_FP8_E4M3 ? 1 : 0;
    p.k_scale = p.kv_fp8 ? k_scale : 1.f;
    p.v_scale = p.kv_fp8 ? v_scale : 1.f;
    return PA_OK;
}

}  // namespace

int pa::set_error(int code, const char *msg) { return fail(code, "%s", msg); }

int pa::api_status_ptr(int **out) { return status_ptr(out); }

unsigned long long pa::current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault,
                                             &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
                cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<GetCurrentFn>(a);
            get_id = reinterpret_cast<GetIdFn>(b);
        }
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

extern "C" {

const char *pa_last_error(void) { return g_last_error; }

int pa_get_device_status(int *status_h, void *stream) {
    if (!status_h) return fail(PA_ERR_INVALID, "status_h is NULL");
    int *ptr = nullptr;
    int rc = status_ptr(&ptr);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpy(status_h, ptr, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read status");
    e = cudaMemset(ptr, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
    return PA_OK;
}

namespace {
// One thread waits, bounded, on an mbarrier that nothing arrives on: the wait every
// kernel's pipeline uses, run out on purpose.
__global__ void wait_timeout_selftest_kernel(int *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        pa::mbar_init(&bar, 1);
        abort_flag = 0;
        pa::fence_mbar_init();
        (void)pa::mbar_wait(&bar, 0, status, &abort_flag);
    }
}
}  // namespace

int pa_selftest_wait_timeout(void *stream) {
    int *status = nullptr;
    int rc = status_ptr(&status);
    if (rc) return rc;
    wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return PA_OK;
}

int pa_write_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                   const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                   int head_dim, int block_size, int64_t num_blocks, int64_t stride_block,
                   int64_t stride_head, int64_t stride_token, int kv_dtype, float k_scale,
                   float v_scale, void *stream) {
    if (num_tokens < 0) return fail(PA_ERR_INVALID, "num_tokens %lld", (long long)num_tokens);
    if (num_kv_heads <= 0) return fail(PA_ERR_INVALID, "num_kv_heads %d", num_kv_heads);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", head_dim);
    int rc = check_kv_dtype(kv_dtype, k_scale, v_scale);
    if (rc) return rc;
    rc = check_pool(head_dim, block_size, num_blocks, num_kv_heads, stride_block, stride_head,
                    stride_token, kv_elem_bytes(kv_dtype));
    if (rc) return rc;
    if (num_tokens > 0 && (!k || !v || !k_cache || !v_cache || !slot_mapping))
        return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID, "k, v and the caches must be 16-byte aligned");
    pa::WriteCacheParams p;
    p.k = k;
    p.v = v;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.slot_mapping = slot_mapping;
    p.num_tokens = num_tokens;
    p.num_blocks = num_blocks;
    p.s_block = stride_block;
    p.s_head = stride_head;
    p.s_token = stride_token;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.block_size = block_size;
    p.kv_fp8 = kv_dtype == PA_KV_FP8_E4M3 ? 1 : 0;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    rc = status_ptr(&p.status);
    if (rc) return rc;
    cudaError_t e = pa::launch_write_cache(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "write_cache launch");
    return PA_OK;
}

int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
              int max_blocks_per_seq, int64_t num_blocks, int64_t stride_block,
              int64_t stride_head, int64_t stride_token, float sm_scale, int sliding_window,
              int kv_dtype, float k_scale, float v_scale, void *stream) {
    pa::DecodeParams p;
    int rc = decode_common(p, out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                           num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                           num_blocks, stride_block, stride_head, stride_token, sm_scale,
                           sliding_window, kv_dtype, k_scale, v_scale);
    if (rc) return rc;
    rc = status_ptr(&p.status);
    if (rc) return rc;
    cudaError_t e = pa::launch_decode(p, head_dim, false, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return PA_OK;
}

void pa_decode_split_workspace_offsets(int num_seqs, int num_q_heads, int head_dim,
                                       int max_seq_len, size_t *off_out, size_t *off_max,
                                       size_t *off_sum) {
    const size_t parts = max_seq_len > 0 ? (static_cast<size_t>(max_seq_len) + 511) / 512 : 0;
    const size_t rows = static_cast<size_t>(num_seqs > 0 ? num_seqs : 0) *
                        static_cast<size_t>(num_q_heads > 0 ? num_q_heads : 0) * parts;
    const size_t o_bytes = round256(rows * static_cast<size_t>(head_dim > 0 ? head_dim : 0) * 4);
    const size_t s_bytes = round256(rows * 4);
    if (off_out) *off_out = 0;
    if (off_max) *off_max = o_bytes;
    if (off_sum) *off_sum = o_bytes + s_bytes;
}

size_t pa_decode_split_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                      int max_seq_len) {
    size_t o, m, l;
    pa_decode_split_workspace_offsets(num_seqs, num_q_heads, head_dim, max_seq_len, &o, &m, &l);
    return l + (l - m);  // partial_out, then partial_max and partial_sum of equal size
}

namespace {

int split_setup(pa::DecodeParams &p, int num_seqs, int num_q_heads, int head_dim,
                int max_blocks_per_seq, int max_seq_len, const void *workspace,
                size_t workspace_bytes) {
    if (max_seq_len < 0) return fail(PA_ERR_INVALID, "max_seq_len %d", max_seq_len);
    if (max_blocks_per_seq > 0 && max_seq_len > max_blocks_per_seq * 16)
        return fail(PA_ERR_INVALID, "max_seq_len %d exceeds max_blocks_per_seq * 16 = %d",
                    max_seq_len, max_blocks_per_seq * 16);
    const size_t need =
        pa_decode_split_workspace_size(num_seqs, num_q_heads, head_dim, max_seq_len);
    if (workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
    if (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(PA_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
    size_t oo, om, ol;
    pa_decode_split_workspace_offsets(num_seqs, num_q_heads, head_dim, max_seq_len, &oo, &om,
                                      &ol);
    char *ws = static_cast<char *>(const_cast<void *>(workspace));
    p.part_o = reinterpret_cast<float *>(ws + oo);
    p.part_m = reinterpret_cast<float *>(ws + om);
    p.part_l = reinterpret_cast<float *>(ws + ol);
    p.max_parts = (max_seq_len + 511) / 512;
    p.max_seq_len = max_seq_len;
    return PA_OK;
}

}  // namespace

int pa_decode_partitions(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int max_blocks_per_seq, int64_t num_blocks, int64_t stride_block,
                         int64_t stride_head, int64_t stride_token, float sm_scale,
                         int sliding_window, int kv_dtype, float k_scale, float v_scale,
                         int max_seq_len, void *workspace, size_t workspace_bytes,
                         void *stream) {
    pa::DecodeParams p;
    // `out` is not written by this pass; q stands in for the alignment check.
    int rc = decode_common(p, const_cast<void *>(q), q, k_cache, v_cache, block_tables,
                           seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_blocks_per_seq, num_blocks, stride_block, stride_head,
                           stride_token, sm_scale, sliding_window, kv_dtype, k_scale, v_scale);
    if (rc) return rc;
    p.out = nullptr;
    rc = split_setup(p, num_seqs, num_q_heads, head_dim, max_blocks_per_seq, max_seq_len,
                     workspace, workspace_bytes);
    if (rc) return rc;
    if (num_seqs == 0 || p.max_parts == 0) return PA_OK;
    rc = status_ptr(&p.status);
    if (rc) return rc;
    cudaError_t e = pa::launch_decode(p, head_dim, true, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode partition launch");
    return PA_OK;
}

int pa_decode_merge(void *out, const int32_t *seq_lens, int num_seqs, int num_q_heads,
                    int head_dim, int max_seq_len, int sliding_window, const void *workspace,
                    size_t workspace_bytes, void *stream) {
    if (num_seqs < 0 || num_q_heads <= 0)
        return fail(PA_ERR_INVALID, "num_seqs %d, num_q_heads %d", num_seqs, num_q_heads);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", head_dim);
    if (num_seqs > 0 && (!out || !seq_lens)) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(out)) return fail(PA_ERR_INVALID, "out must be 16-byte aligned");
    pa::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.out = out;
    p.seq_lens = seq_lens;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.window = sliding_window > 0 ? sliding_window : 0;
    int rc = split_setup(p, num_seqs, num_q_heads, head_dim, 0, max_seq_len, workspace,
                         workspace_bytes);
    if (rc) return rc;
    if (num_seqs == 0) return PA_OK;
    rc = status_ptr(&p.status);
    if (rc) return rc;
    cudaError_t e = pa::launch_merge(p, head_dim, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return PA_OK;
}

int pa_decode_split(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                    int max_blocks_per_seq, int64_t num_blocks, int64_t stride_block,
                    int64_t stride_head, int64_t stride_token, float sm_scale,
                    int sliding_window, int kv_dtype, float k_scale, float v_scale,
                    int max_seq_len, void *workspace, size_t workspace_bytes, void *stream) {
    pa::DecodeParams p;
    int rc = decode_common(p, out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                           num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                           num_blocks, stride_block, stride_head, stride_token, sm_scale,
                           sliding_window, kv_dtype, k_scale, v_scale);
    if (rc) return rc;
    rc = split_setup(p, num_seqs, num_q_heads, head_dim, max_blocks_per_seq, max_seq_len,
                     workspace, workspace_bytes);
    if (rc) return rc;
    if (num_seqs == 0) return PA_OK;
    rc = status_ptr(&p.status);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.max_parts > 0) {
        cudaError_t e = pa::launch_decode(p, head_dim, true, s);
        if (e != cudaSuccess) return cuda_fail(e, "decode partition launch");
    }
    cudaError_t e = pa::launch_merge(p, head_dim, s);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return PA_OK;
}

size_t pa_ragged_prefill_workspace_size(int batch, int total_qo_rows, int num_q_heads,
                                        int head_dim) {
    (void)num_q_heads;
    (void)head_dim;
    const size_t tiles = static_cast<size_t>(total_qo_rows > 0 ? total_qo_rows : 0) / 128 +
                         static_cast<size_t>(batch > 0 ? batch : 0) + 1;
    return 256 + round256(tiles * 8);  // work counters, then room for a device-built list
}

int pa_ragged_prefill(void *o, const void *q, const void *k, const void *v,
                      const int32_t *qo_indptr_h, const int32_t *kv_indptr_h,
                      const int32_t *qo_indptr_d, const int32_t *kv_indptr_d,
                      const int32_t *block_tables, int max_blocks_per_seq, int block_size,
                      int64_t num_blocks, int64_t stride_block, int64_t stride_head,
                      int64_t stride_token, int batch, int total_qo_rows, int total_kv_rows,
                      int num_q_heads, int num_kv_heads, int head_dim, float sm_scale,
                      int causal, int sliding_window, void *workspace, size_t workspace_bytes,
                      void *stream) {
    if (batch < 0 || total_qo_rows < 0 || total_kv_rows < 0)
        return fail(PA_ERR_INVALID, "negative size (batch %d, qo %d, kv %d)", batch,
                    total_qo_rows, total_kv_rows);
    int rc = check_heads(head_dim, num_q_heads, num_kv_heads);
    if (rc) return rc;
    if (batch == 0) return PA_OK;
    if (!qo_indptr_h || !kv_indptr_h || !qo_indptr_d || !kv_indptr_d)
        return fail(PA_ERR_INVALID, "null indptr");
    if (!(sm_scale > 0.f) || sm_scale == INFINITY)
        return fail(PA_ERR_INVALID, "sm_scale must be positive and finite for prefill");
    const bool paged = block_tables != nullptr;
    if (paged) {
        rc = check_pool(head_dim, block_size, num_blocks, num_kv_heads, stride_block,
                        stride_head, stride_token);
        if (rc) return rc;
        if (max_blocks_per_seq <= 0)
            return fail(PA_ERR_INVALID, "max_blocks_per_seq %d", max_blocks_per_seq);
        if (num_blocks >= (int64_t(1) << 31) - 1)
            return fail(PA_ERR_UNSUPPORTED, "num_blocks %lld too large", (long long)num_blocks);
    }
    if (qo_indptr_h[0] != 0 || kv_indptr_h[0] != 0)
        return fail(PA_ERR_INVALID, "indptr must start at 0");
    int64_t n_tiles = 0;
    for (int r = 0; r < batch; ++r) {
        const int qo = qo_indptr_h[r + 1] - qo_indptr_h[r];
        const int kv = kv_indptr_h[r + 1] - kv_indptr_h[r];
        if (qo < 0 || kv < 0) return fail(PA_ERR_INVALID, "indptr not monotone at request %d", r);
        if (paged && kv > max_blocks_per_seq * 16)
            return fail(PA_ERR_INVALID, "request %d: %d keys exceed its block table (%d pages)", r,
                        kv, max_blocks_per_seq);
        n_tiles += (qo + 127) / 128;
    }
    if (qo_indptr_h[batch] != total_qo_rows)
        return fail(PA_ERR_INVALID, "qo_indptr[batch] %d != total_qo_rows %d", qo_indptr_h[batch],
                    total_qo_rows);
    if (!paged && kv_indptr_h[batch] != total_kv_rows)
        return fail(PA_ERR_INVALID, "kv_indptr[batch] %d != total_kv_rows %d", kv_indptr_h[batch],
                    total_kv_rows);
    if (n_tiles > 65535)
        return fail(PA_ERR_UNSUPPORTED, "%lld query tiles exceed one launch", (long long)n_tiles);
    if (total_qo_rows == 0) return PA_OK;
    if (!o || !q || !k || !v) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(o) || !aligned16(q) || !aligned16(k) || !aligned16(v))
        return fail(PA_ERR_INVALID, "o, q, k and v must be 16-byte aligned");
    const size_t need =
        pa_ragged_prefill_workspace_size(batch, total_qo_rows, num_q_heads, head_dim);
    if (workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(PA_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");

    pa::PrefillParams p;
    std::memset(&p, 0, sizeof p);
    p.o = o;
    p.qo_indptr = qo_indptr_d;
    p.kv_indptr = kv_indptr_d;
    p.block_tables = block_tables;
    p.item_counter = static_cast<int *>(workspace);
    p.tiles = reinterpret_cast<const int2 *>(static_cast<char *>(workspace) + 256);
    p.num_blocks = paged ? num_blocks : 0;
    p.batch = batch;
    p.nq = num_q_heads;
    p.nkv = num_kv_heads;
    p.max_blocks = paged ? max_blocks_per_seq : 0;
    p.n_tiles = static_cast<int>(n_tiles);
    p.causal = causal ? 1 : 0;
    p.window = sliding_window > 0 ? sliding_window : 0;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    rc = status_ptr(&p.status);
    if (rc) return rc;
    pa::PrefillLaunch L;
    L.q = q;
    L.k = k;
    L.v = v;
    L.qo_indptr_h = qo_indptr_h;
    L.kv_indptr_h = kv_indptr_h;
    L.total_qo = total_qo_rows;
    L.total_kv = total_kv_rows;
    L.s_block = stride_block;
    L.s_head = stride_head;
    L.s_token = stride_token;
    L.head_dim = head_dim;
    cudaError_t e = pa::launch_prefill(p, L, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue)
        return fail(PA_ERR_CUDA, "tensor map encoding failed (cuTensorMapEncodeTiled)");
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return PA_OK;
}

}  // extern "C"
