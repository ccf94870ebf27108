// gemm_internal.h - what the host planner (api.cpp) hands the sm_103a kernel
// (gemm_kernel.cuh).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "layout.hpp"

namespace gemm_sm103 {

// Fixed tile geometry.  A stage holds 128 bytes of K per operand row
// (64 16-bit or 128 8-bit elements), i.e. one 128-byte swizzle row, and the
// MMA consumes it in four 32-byte K steps (16 elements for kind::f16, 32 for
// kind::f8f6f4).
constexpr int kTileM = 128;
constexpr int kStageKBytes = 128;
constexpr int kKStepBytes = 32;
constexpr int kThreads = 192;          // warp 0 loads, warp 1 issues MMAs, warps 2-5 run the epilogue
                                       // (block-scaled kernels add warp 6: scale-factor copies)
constexpr int kEpiWarps = 4;
constexpr int kEpiRows = 32;           // rows per epilogue warp (one TMEM lane quadrant)
constexpr int kEpiBufBytes = kEpiRows * 128;
constexpr uint64_t kDefaultTimeoutNs = 2000ull * 1000ull * 1000ull;

// Status-word bits written by the kernel.
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusRoleLoad = 1u << 8;
constexpr uint32_t kStatusRoleMma = 1u << 9;
constexpr uint32_t kStatusRoleEpi = 1u << 10;
constexpr uint32_t kStatusRoleDrain = 1u << 11;
constexpr uint32_t kStatusRoleFixup = 1u << 12;   // a stream-K owner waiting for a partial sum
constexpr uint32_t kStatusRoleCopy = 1u << 13;    // the scale-factor copier waiting for a stage
// Diagnostic build with index checks (GEMM_DEBUG): a plain store whose index
// falls outside its buffer is skipped and this bit is recorded.
constexpr uint32_t kStatusBounds = 2u;

struct KernelParams {
    int32_t M, N, K, L;           // kernel orientation: D is M x N row-major
    int32_t tiles_m, tiles_n;
    int32_t tiles_per_batch, num_tiles;
    int32_t num_kb;               // K blocks of kStageKBytes
    // Persistent tile order: tile t of a batch -> linear index m_blk + tiles_m * n_blk.
    gl::FlatLayout raster_full;   // the groups of `raster_group` M tiles
    gl::FlatLayout raster_tail;   // the last, shorter group
    int32_t raster_full_count;    // tiles covered by raster_full
    int32_t raster_tail_offset;   // first M tile of the tail group
    int32_t a_kmajor, b_kmajor;
    int32_t elem_bytes;           // operand element size, 1 or 2
    int32_t kind_f8;              // 1: kind::f8f6f4, 0: kind::f16
    // MMA loop variant, one per instruction descriptor:
    // 8*kind_f8 + 4*(operands bf16) + 2*(A MN-major) + (B MN-major)
    int32_t mma_variant;
    int32_t a_batched, b_batched, c_batched;   // 0: operand shared by all batches
    float alpha, beta;
    int32_t has_c;
    int32_t bias_mode;            // 0 none, 1 per kernel column, 2 per kernel row
    const float* bias;
    int64_t bias_stride;
    int32_t act;                  // 0 none, 1 ReLU, 2 GELU (x * Phi(x))
    int32_t out_f16;              // 2-byte outputs: 1 fp16, 0 bf16
    // A TMA store clips the inner dimension only at 16-byte granules, so when
    // a D row does not end on a 16-byte boundary the subtile holding its last
    // columns is written with plain stores instead.
    int32_t d_ragged;
    void* d_ptr;
    int64_t ldd;                  // kernel orientation: row stride of D, elements
    int64_t d_bstride;            // batch stride of D, elements
    uint32_t* status;
    uint64_t timeout_ns;
    // Work split (stream-K hybrid).  Tiles [0, dp_tiles) of the raster are
    // computed whole, worker w taking tiles w, w + workers, ...; the K-block
    // iterations of the remaining tiles, sk_iters in all, are cut into one
    // contiguous range per worker.  A tile cut between workers is finished
    // by the worker that ran its first K block (its owner), which adds the
    // other workers' fp32 partial sums before the epilogue.  Without a split,
    // dp_tiles = num_tiles and sk_iters = 0.
    int32_t clc;                  // 1: dynamic schedule (cluster launch control), grid = every tile
    // Block scaling.  block_scaled = 1 (MXFP8): one ue8m0 factor per 32 K
    // elements; the factors of 128 rows x one K stage (4 factors each) form
    // one 512-byte block; a batch's tensor holds blocks (row/128) * num_kb + kb.
    // block_scaled = 2 (NVFP4): operands are planned as bytes (two e2m1 per
    // byte, K and num_kb in bytes), one ue4m3 factor per 16 elements, four
    // blocks per 128 rows and K stage, loaded through a map of their own.
    // MX output (out_f8 = 1): D in e4m3, factors written to sfd in the
    // basic-block layout (rows = M, one factor per 32 columns; sfd_kb4 =
    // ceil(ceil(N/32)/4) blocks along N; sfd_bstride bytes per batch).
    // NVFP4 output (out_f8 = 2): D in e2m1 (two per byte; ldd and d_bstride
    // then count bytes), one ue4m3 factor per 16 columns, global scale scale_d.
    int32_t out_f8;
    float scale_d;
    uint8_t* sfd;
    int64_t sfd_bstride;
    int32_t sfd_kb4;
    int32_t block_scaled;
    int32_t sf_mblocks, sf_nblocks;    // 128-row blocks of the kernel's A and B
    const uint8_t* sfa;                // (kept for reference; the kernel loads through tmSA / tmSB)
    const uint8_t* sfb;
    int32_t dp_tiles;
    int64_t sk_iters;
    int32_t sk_ranges;            // ranges the iterations are cut into (<= workers); range r
                                  // is [sk_iters*r/sk_ranges, sk_iters*(r+1)/sk_ranges)
    float* sk_part;               // per worker: one tile of fp32 partial sums
    uint32_t* sk_flags;           // per worker, CTA and epilogue warp: 1 = partial written
    // Reductions of the epilogue value t (fp32, before rounding to D's type),
    // kernel orientation.  Partials, each written once per launch:
    //   red_row_ws[(l * tiles_n + n_tile) * M + m]   sum of t over one tile's columns
    //   red_col_ws[(l * slabs + m / 32) * N + n]     sum of t over one 32-row slab
    //   red_amax_ws[l]                               max |t| as fp32 bits (atomicMax)
    int32_t red_rows, red_cols, red_amax;
    float* red_row_ws;
    float* red_col_ws;
    uint32_t* red_amax_ws;
    int32_t inject;               // 1: skip the first load (bounded-wait test)
    // Grouped GEMM (groups > 0): group g owns rows [group_rows[g],
    // group_rows[g+1]) of A, C and D (one matrix each; offsets clamped to
    // [0, M], each group starting where the previous one ends at the latest) and
    // batch g of B and of the bias.  Its tiles follow those of group g - 1,
    // M-block fastest; each CTA counts the tiles itself (data parallel only).
    int32_t groups;
    const int64_t* group_rows;    // device, groups + 1 entries
    // Diagnostic build with timestamps (GEMM_STAMPS): 8 %globaltimer values
    // per CTA (see gemm_kernel.cuh); null otherwise.
    unsigned long long* stamps;
};

struct LaunchArgs {
    CUtensorMap tmA, tmB, tmC, tmD;
    CUtensorMap tmSA, tmSB;       // scale-factor blocks (block-scaled kernel; else copies of tmA)
    KernelParams p;
    int cta_group;                // 1 or 2 (CTA pair, cluster of 2)
    int tile_n;                   // 128 or 256
    int out_bytes;                // 1 (e4m3 with MX factors), 2 or 4
    int block_scaled;             // 1: MXFP8, 2: NVFP4 block-scaled kernel
    int grid;                     // CTAs (a multiple of cta_group)
    cudaStream_t stream;
};

// Second pass of the reductions: sums the partials in a fixed order into the
// caller's outputs (kernel orientation) and resets the abs-max words.
struct FinishParams {
    int32_t L, M, N, tiles_n, slabs;
    const float* row_ws;          // null: no row sums
    const float* col_ws;          // null: no column sums
    uint32_t* amax_ws;            // null: no abs-max
    float* out_rows;              // [L][M]
    float* out_cols;              // [L][N]
    float* out_amax;              // [L]
};
cudaError_t launch_finish(const FinishParams& f, cudaStream_t stream);

int stages_for(int cta_group, int tile_n, int block_scaled);
size_t smem_bytes_for(int cta_group, int tile_n, int out_bytes, int block_scaled);
cudaError_t prepare_kernel(int cta_group, int tile_n, int out_bytes, int block_scaled);
int max_active_clusters(int cta_group, int tile_n, int out_bytes, int block_scaled);   // 0 if unknown
cudaError_t launch(const LaunchArgs& a);

// Launch set-up of the kernel variants (dynamic shared-memory attribute set,
// clusters that fit at once), kept per device by callers without a handle.
// One slot per variant without block scaling: CTA group x tile width x
// output bytes.
struct VariantCache {
    static constexpr int kSlots = 12;
    std::atomic<int> prepared[kSlots] = {};        // 1 once the attribute is set
    std::atomic<int> clusters_plus1[kSlots] = {};  // 0: not asked yet
    static int slot(int cta_group, int tile_n, int out_bytes) {
        return ((cta_group - 1) * 2 + (tile_n == 256)) * 3 + (out_bytes == 1 ? 0 : out_bytes == 2 ? 1 : 2);
    }
};

}  // namespace gemm_sm103
