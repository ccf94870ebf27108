// reduce_finish.cu - second pass of the epilogue reductions.
//
// The GEMM kernel leaves one partial per (row, N tile) and per (32-row slab,
// column) of the epilogue value t, and an atomic abs-max word per batch.
// This pass adds the partials in index order (so the sums do not depend on
// which CTA finished first), writes the caller's fp32 outputs and resets the
// abs-max words to zero for the next launch.  What is reduced is the reading
// of "Technical Documentation: NVIDIA/cutlass", "What's New in CUTLASS 4.8"
// (per-row or per-column reductions in the epilogue): t before rounding.
#include "gemm_internal.h"

namespace gemm_sm103 {

__global__ void __launch_bounds__(256) reduce_finish_kernel(const FinishParams f) {
    const int64_t rows = f.row_ws ? (int64_t)f.L * f.M : 0;
    const int64_t cols = f.col_ws ? (int64_t)f.L * f.N : 0;
    const int64_t amax = f.amax_ws ? f.L : 0;
    const int64_t total = rows + cols + amax;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        if (i < rows) {
            const int64_t l = i / f.M, m = i - l * f.M;
            const float* src = f.row_ws + l * f.tiles_n * (int64_t)f.M + m;
            float s = 0.f;
            for (int t = 0; t < f.tiles_n; ++t) s += src[(int64_t)t * f.M];
            f.out_rows[i] = s;
        } else if (i < rows + cols) {
            const int64_t k = i - rows;
            const int64_t l = k / f.N, n = k - l * f.N;
            const float* src = f.col_ws + l * f.slabs * (int64_t)f.N + n;
            float s = 0.f;
            for (int t = 0; t < f.slabs; ++t) s += src[(int64_t)t * f.N];
            f.out_cols[k] = s;
        } else {
            const int64_t l = i - rows - cols;
            f.out_amax[l] = __uint_as_float(f.amax_ws[l]);
            f.amax_ws[l] = 0u;
        }
    }
}

cudaError_t launch_finish(const FinishParams& f, cudaStream_t stream) {
    const int64_t total = (f.row_ws ? (int64_t)f.L * f.M : 0) + (f.col_ws ? (int64_t)f.L * f.N : 0) +
                          (f.amax_ws ? f.L : 0);
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    reduce_finish_kernel<<<(unsigned)blocks, 256, 0, stream>>>(f);
    return cudaGetLastError();
}

}  // namespace gemm_sm103
