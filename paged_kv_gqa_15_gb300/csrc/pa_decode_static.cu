// pa_decode_static.cu -- pa_decode_split_static: the split-KV decode with its
// partial results kept in a fixed-size device array that is part of this
// library, for callers that cannot allocate device memory.
//
// Who needs it: code that is not allowed to call cudaMalloc (or any allocating
// routine) and has no workspace to hand over -- for example a plugin running
// inside an inference engine that owns the whole device memory budget, or a
// latency-critical decode loop where an allocation (which may synchronise the
// device or fail with out-of-memory halfway through a step) is unacceptable.
//
// How it works: the partials live in g_split_scratch, a file-scope __device__
// array of PA_STATIC_SCRATCH_BYTES.  Host code cannot pass the array's name to
// a kernel (on the host it only names a stand-in), so the first call on each
// device, with that device current, asks the runtime for the array's device
// address with cudaGetSymbolAddress and caches it with the id of the CUDA
// context it belongs to (a later context, after cudaDeviceReset, looks it up
// again); every call then runs the regular pa_decode_split with that address
// as its workspace.
//
// Size: the 16 MiB hold the split partials of the 64-sequence Llama-3-8B decode
// batch (seq_lens up to 4096: about 8.1 MiB) and of the 4-sequence tiny batch;
// the 8-sequence long-context batch (seq_lens up to 131072, about 32.5 MiB of
// partials) does not fit and must use pa_decode_split with a workspace.
#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

// Every GPU that loads this library keeps this array until the process exits.
static __device__ __align__(256) unsigned char g_split_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct CachedScratch {
    unsigned long long ctx;   // context the address belongs to (0: do not reuse)
    void *ptr;
};
CachedScratch g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_split_scratch on the current device, looked up once per device
// and context: after cudaDeviceReset the next context may place the array elsewhere,
// so an address cached under an earlier context is looked up again.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pa::set_error(PA_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices)
        return pa::set_error(PA_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    const unsigned long long ctx = pa::current_context_id();
    if (ctx == 0 || g_scratch_addr[dev].ctx != ctx) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_split_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return pa::set_error(PA_ERR_CUDA,
                                 "cudaGetSymbolAddress of the static split scratch failed");
        g_scratch_addr[dev] = {pa::current_context_id(), ptr};
    }
    *out = g_scratch_addr[dev].ptr;
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_split_static(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      const int32_t *seq_lens, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq, int64_t num_blocks,
                                      int64_t stride_block, int64_t stride_head,
                                      int64_t stride_token, float sm_scale, int sliding_window,
                                      int kv_dtype, float k_scale, float v_scale,
                                      int max_seq_len, void *stream) {
    const size_t need =
        pa_decode_split_workspace_size(num_seqs, num_q_heads, head_dim, max_seq_len);
    if (need > static_cast<size_t>(PA_STATIC_SCRATCH_BYTES))
        return pa::set_error(PA_ERR_WORKSPACE,
                             "pa_decode_split_static: this batch needs more split scratch than "
                             "the library's fixed PA_STATIC_SCRATCH_BYTES; use pa_decode_split "
                             "with a caller-provided workspace");
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != PA_OK) return rc;
    return pa_decode_split(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                           num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                           num_blocks, stride_block, stride_head, stride_token, sm_scale,
                           sliding_window, kv_dtype, k_scale, v_scale, max_seq_len, scratch,
                           static_cast<size_t>(PA_STATIC_SCRATCH_BYTES), stream);
}
