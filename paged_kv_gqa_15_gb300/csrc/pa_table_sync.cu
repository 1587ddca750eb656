// pa_table_sync.cu -- block-table upload between CUDA-graph replays of the decode
// ("libmir-cuda attention/mod.rs": the captured decode reads a fixed device table and
// the host re-uploads it only when it changed).  The snapshot is the caller's pinned
// copy of what was last uploaded; each run of consecutive changed rows becomes one
// async copy from it.
#include <cuda_runtime.h>

#include <cstring>

#include "../../include/pa.h"
#include "pa_internal.h"

extern "C" int pa_block_table_sync(const int32_t *host_table, int32_t *snapshot,
                                   int32_t *device_table, int num_rows, int row_len,
                                   int *rows_uploaded, void *stream) {
    if (rows_uploaded) *rows_uploaded = 0;
    if (num_rows < 0 || row_len < 0)
        return pa::api_fail(PA_ERR_INVALID, "num_rows %d, row_len %d", num_rows, row_len);
    if (num_rows == 0 || row_len == 0) return PA_OK;
    if (!host_table || !snapshot || !device_table)
        return pa::api_fail(PA_ERR_INVALID, "null pointer argument");
    const size_t row_bytes = static_cast<size_t>(row_len) * sizeof(int32_t);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int copied = 0;
    int run_start = -1;   // first row of the current run of changed rows
    for (int r = 0; r <= num_rows; ++r) {
        bool changed = false;
        if (r < num_rows) {
            const int32_t *h = host_table + static_cast<size_t>(r) * row_len;
            int32_t *snap = snapshot + static_cast<size_t>(r) * row_len;
            if (std::memcmp(h, snap, row_bytes) != 0) {
                std::memcpy(snap, h, row_bytes);
                changed = true;
            }
        }
        if (changed && run_start < 0) run_start = r;
        if (!changed && run_start >= 0) {   // the run [run_start, r) ends here
            const size_t off = static_cast<size_t>(run_start) * row_len;
            const cudaError_t e =
                cudaMemcpyAsync(device_table + off, snapshot + off,
                                static_cast<size_t>(r - run_start) * row_bytes,
                                cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return pa::api_cuda_fail(e, "block table upload");
            copied += r - run_start;
            run_start = -1;
        }
    }
    if (rows_uploaded) *rows_uploaded = copied;
    return PA_OK;
}
