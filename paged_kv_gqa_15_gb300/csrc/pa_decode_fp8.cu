// pa_decode_fp8.cu -- FP8 E4M3-cache instantiation of the paged GQA decode kernel
// (pa_decode_kernel.cuh): kv_cache_dtype "fp8" with k_scale / v_scale ("paged_attn.py",
// forward_decode), compiled apart from the bf16 instantiation so the two build in
// parallel.
#include "pa_decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_fp8(const DecodeParams &p, int head_dim, bool split,
                              cudaStream_t stream) {
    if (p.num_seqs == 0) return cudaSuccess;
    return launch_decode_cache<true>(p, head_dim, split, stream);
}

}  // namespace pa
