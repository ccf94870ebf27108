// api.cpp - the C ABI of gemm.h: descriptor validation, planning (operand
// orientation, tile shape, raster order), TMA descriptor encoding and launch.
//
// Planning follows the pages' host-side steps: the BLAS argument set and
// "first kernel whose types, layouts and alignment fit" selection of
// "Technical Documentation: NVIDIA/cutlass" ("Launching a GEMM kernel in
// CUDA", "CUTLASS Library"); the alignment table of "Layouts, Tensor
// Alignment Requirements to Target tcgen05.mma Instructions"; and tile
// addressing and TMA metadata derived from shape:stride layouts ("CUTLASS"
// knowledge-base page, "CuTe and layouts").
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>

#include "../../include/gemm.h"
#include "gemm_internal.h"

using namespace gemm_sm103;

namespace {

int dtype_bytes(int dt) {
    switch (dt) {
        case GEMM_F32: return 4;
        case GEMM_F16: return 2;
        case GEMM_BF16: return 2;
        case GEMM_E4M3: return 1;
        default: return 0;
    }
}

// Layout of a stored matrix as seen through op(): logical (r, c) of the
// rows x cols operand.  op N: stored rows x cols; op T: stored cols x rows.
// Row-major storage puts (i, j) at i*ld + j, column-major at i + j*ld.
gl::Layout logical_layout(int op, int order, int64_t rows, int64_t cols, int64_t ld, int64_t batch,
                          int64_t bstride) {
    int64_t sr, sc;                              // strides of logical row / column index
    const bool row_major = order == GEMM_ROW_MAJOR;
    if (op == GEMM_OP_N) {
        sr = row_major ? ld : 1;
        sc = row_major ? 1 : ld;
    } else {
        sr = row_major ? 1 : ld;
        sc = row_major ? ld : 1;
    }
    gl::Layout parts[3] = {gl::leaf(rows > 0 ? rows : 1, sr), gl::leaf(cols > 0 ? cols : 1, sc),
                           gl::leaf(batch, bstride)};
    gl::Layout out;
    gl::concat(parts, 3, &out);
    return out;
}

// Stride of mode i of a rank-3 layout built by logical_layout.
int64_t mode_stride(const gl::Layout& l, int i) { return gl::mode(l, i).stride[0]; }
int64_t mode_extent(const gl::Layout& l, int i) { return gl::mode(l, i).shape[0]; }

// Swap the first two modes (a transpose view): composition with (c,r):(r,1)
// would do the same; swapping the leaves is the direct form.
gl::Layout transpose2(const gl::Layout& l) {
    gl::Layout parts[3] = {gl::mode(l, 1), gl::mode(l, 0), gl::mode(l, 2)};
    gl::Layout out;
    gl::concat(parts, 3, &out);
    return out;
}

struct Plan {
    gemm_desc_t d;
    gemm_plan_info_t info;
    // kernel orientation
    gl::Layout a, b, cd;     // a: (M', K, L), b: (N', K, L), cd: (M', N', L)
    int64_t Mk, Nk;
    int a_bytes, out_bytes;
    int cta_group;
    int tile_n;
    bool has_c;
    int bias_mode;           // 0 none, 1 per kernel column, 2 per kernel row
    KernelParams kp;
};

bool aligned16(int64_t elems, int bytes) { return ((elems * bytes) % 16) == 0; }

// groups > 0: a grouped GEMM (gemm_grouped_create); desc.batch must be 1,
// B and the bias get `groups` batches (strides stride_b, stride_bias).
gemm_status_t validate_and_plan(const gemm_desc_t* desc, Plan* out, int32_t groups = 0) {
    if (!desc || !out) return GEMM_ERR_INVALID_ARG;
    if (groups < 0 || groups > 65535) return GEMM_ERR_INVALID_ARG;
    if (groups > 0) {
        // one A, C and D split by rows; no swap (row-major D), no splits of K
        // across workers, none of the extensions that keep per-batch state
        if (desc->batch != 1 || desc->stride_a || desc->stride_c || desc->stride_d) return GEMM_ERR_INVALID_ARG;
        if (desc->order_d != GEMM_ROW_MAJOR || (desc->beta != 0.0f && desc->order_c != GEMM_ROW_MAJOR))
            return GEMM_ERR_UNSUPPORTED;
        if (desc->out_scale != GEMM_OUT_SCALE_NONE || desc->reduce || desc->bias == GEMM_BIAS_ROW)
            return GEMM_ERR_UNSUPPORTED;
        // A K-contiguous: a group's first row is any offset, and a tensor copy
        // may start at any row but only at 16-byte-aligned inner coordinates
        if ((desc->op_a == GEMM_OP_N) != (desc->order_a == GEMM_ROW_MAJOR)) return GEMM_ERR_UNSUPPORTED;
    }
    // NVFP4 operands are planned as bytes: two e2m1 elements per byte along
    // K (both operands K-contiguous), so K, the leading dimensions and the
    // batch strides of A and B are halved and the byte view is planned like
    // an 8-bit operand.  A stage's 128 bytes of K then hold 256 elements.
    gemm_desc_t view = *desc;
    const bool nv = desc->block_scale == GEMM_BLOCK_SCALE_NV;
    if (nv) {
        if (desc->dtype_a != GEMM_E2M1 || desc->dtype_b != GEMM_E2M1) return GEMM_ERR_UNSUPPORTED;
        if (desc->K < 0 || desc->lda < 0 || desc->ldb < 0) return GEMM_ERR_INVALID_ARG;
        if (desc->K % 2) return GEMM_ERR_UNSUPPORTED;
        // K-contiguous storage of both operands (the pages' TN layout)
        const bool a_k = (desc->op_a == GEMM_OP_N) == (desc->order_a == GEMM_ROW_MAJOR);
        const bool b_k = (desc->op_b == GEMM_OP_N) == (desc->order_b == GEMM_COL_MAJOR);
        if (!a_k || !b_k) return GEMM_ERR_UNSUPPORTED;
        if (desc->lda % 32 || desc->ldb % 32 || (desc->batch > 1 && (desc->stride_a % 32 || desc->stride_b % 32)) ||
            (groups > 1 && desc->stride_b % 32))
            return GEMM_ERR_MISALIGNED;
        view.K /= 2;
        view.lda /= 2;
        view.ldb /= 2;
        view.stride_a /= 2;
        view.stride_b /= 2;
        view.dtype_a = view.dtype_b = GEMM_E4M3;
    }
    const gemm_desc_t& d = view;
    if (d.M < 0 || d.N < 0 || d.K < 0 || d.batch < 1) return GEMM_ERR_INVALID_ARG;
    if (d.M > INT32_MAX || d.N > INT32_MAX || d.K > INT32_MAX || d.batch > 65535) return GEMM_ERR_UNSUPPORTED;
    if ((d.op_a != GEMM_OP_N && d.op_a != GEMM_OP_T) || (d.op_b != GEMM_OP_N && d.op_b != GEMM_OP_T))
        return GEMM_ERR_INVALID_ARG;
    for (int o : {d.order_a, d.order_b, d.order_c, d.order_d})
        if (o != GEMM_ROW_MAJOR && o != GEMM_COL_MAJOR) return GEMM_ERR_INVALID_ARG;
    if (d.act != GEMM_ACT_NONE && d.act != GEMM_ACT_RELU && d.act != GEMM_ACT_GELU) return GEMM_ERR_INVALID_ARG;
    if (d.reduce & ~(GEMM_REDUCE_ROW_SUM | GEMM_REDUCE_COL_SUM | GEMM_REDUCE_ABS_MAX)) return GEMM_ERR_INVALID_ARG;
    if (d.block_scale != GEMM_BLOCK_SCALE_NONE && d.block_scale != GEMM_BLOCK_SCALE_MX &&
        d.block_scale != GEMM_BLOCK_SCALE_NV)
        return GEMM_ERR_INVALID_ARG;
    if (d.block_scale == GEMM_BLOCK_SCALE_MX && (d.dtype_a != GEMM_E4M3 || d.dtype_b != GEMM_E4M3))
        return GEMM_ERR_UNSUPPORTED;
    if (d.bias != GEMM_BIAS_NONE && d.bias != GEMM_BIAS_COL && d.bias != GEMM_BIAS_ROW) return GEMM_ERR_INVALID_ARG;
    // e2m1 D exists only with its block factors (GEMM_OUT_SCALE_NV)
    if (d.out_scale != GEMM_OUT_SCALE_NONE && d.out_scale != GEMM_OUT_SCALE_MX && d.out_scale != GEMM_OUT_SCALE_NV)
        return GEMM_ERR_INVALID_ARG;
    const bool out_nv = d.out_scale == GEMM_OUT_SCALE_NV;
    if ((d.dtype_d == GEMM_E2M1) != out_nv) return GEMM_ERR_UNSUPPORTED;
    for (int t : {d.dtype_a, d.dtype_b})
        if (!dtype_bytes(t)) return GEMM_ERR_INVALID_ARG;
    if (!out_nv && !dtype_bytes(d.dtype_d)) return GEMM_ERR_INVALID_ARG;
    const bool has_c = d.beta != 0.0f;
    if (has_c && !dtype_bytes(d.dtype_c)) return GEMM_ERR_INVALID_ARG;

    // One operand type per MMA: both f16, both bf16 or both e4m3.
    if (d.dtype_a != d.dtype_b) return GEMM_ERR_UNSUPPORTED;
    if (d.dtype_a == GEMM_F32) return GEMM_ERR_UNSUPPORTED;
    if ((d.dtype_d == GEMM_E4M3) != (d.out_scale == GEMM_OUT_SCALE_MX)) return GEMM_ERR_UNSUPPORTED;
    if (d.out_scale != GEMM_OUT_SCALE_NONE && (d.order_d != GEMM_ROW_MAJOR || d.beta != 0.0f || d.reduce))
        return GEMM_ERR_UNSUPPORTED;
    if (out_nv) {
        // a normal fp32 (the kernel's exact rounding tests need g >= 2^-126)
        if (!(d.scale_d >= 1.17549435e-38f) || !(d.scale_d < 3.0e38f)) return GEMM_ERR_INVALID_ARG;
        if (d.N % 2) return GEMM_ERR_UNSUPPORTED;                  // whole bytes per row
        if (d.ldd % 32 || (d.batch > 1 && d.stride_d % 32)) return GEMM_ERR_MISALIGNED;
    }
    if (has_c && (d.dtype_c != d.dtype_d || d.order_c != d.order_d)) return GEMM_ERR_UNSUPPORTED;

    const int ab = dtype_bytes(d.dtype_a), ob = out_nv ? 1 : dtype_bytes(d.dtype_d);   // e2m1 D: the 1-byte kernel

    // Leading dimensions must cover the stored rows (BLAS rule).
    auto ld_ok = [](int order, int64_t srows, int64_t scols, int64_t ld) {
        const int64_t need = order == GEMM_ROW_MAJOR ? scols : srows;
        return ld >= (need > 1 ? need : 1);
    };
    const int64_t a_sr = d.op_a == GEMM_OP_N ? d.M : d.K, a_sc = d.op_a == GEMM_OP_N ? d.K : d.M;
    const int64_t b_sr = d.op_b == GEMM_OP_N ? d.K : d.N, b_sc = d.op_b == GEMM_OP_N ? d.N : d.K;
    if (!ld_ok(d.order_a, a_sr, a_sc, d.lda) || !ld_ok(d.order_b, b_sr, b_sc, d.ldb) ||
        !ld_ok(d.order_d, d.M, d.N, d.ldd) || (has_c && !ld_ok(d.order_c, d.M, d.N, d.ldc)))
        return GEMM_ERR_INVALID_ARG;
    if (d.stride_a < 0 || d.stride_b < 0 || d.stride_c < 0 || d.stride_d < 0 || d.stride_bias < 0)
        return GEMM_ERR_INVALID_ARG;
    // Batches of D must not overlap.
    if (d.batch > 1) {
        const int64_t outer = d.order_d == GEMM_ROW_MAJOR ? d.M : d.N;
        if (d.stride_d < outer * d.ldd) return GEMM_ERR_INVALID_ARG;
    }
    // TMA needs 16-byte strides: 8 elements for 16-bit, 16 for 8-bit types.
    if (!aligned16(d.lda, ab) || !aligned16(d.ldb, ab) || !aligned16(d.ldd, ob) || (has_c && !aligned16(d.ldc, ob)))
        return GEMM_ERR_MISALIGNED;
    if (d.batch > 1 && (!aligned16(d.stride_a, ab) || !aligned16(d.stride_b, ab) || !aligned16(d.stride_d, ob) ||
                        (has_c && !aligned16(d.stride_c, ob))))
        return GEMM_ERR_MISALIGNED;

    Plan& P = *out;
    memset(&P.info, 0, sizeof(P.info));
    P.d = d;
    P.has_c = has_c;
    P.a_bytes = ab;
    P.out_bytes = ob;

    const int64_t L = d.batch;
    const int64_t Lb = groups > 0 ? groups : L;             // batches of B (and of the bias)
    if (groups > 1 && (d.stride_b < 0 || !aligned16(d.stride_b, ab))) return GEMM_ERR_MISALIGNED;
    gl::Layout la = logical_layout(d.op_a, d.order_a, d.M, d.K, d.lda, L, L > 1 ? d.stride_a : 0);  // (M,K,L)
    gl::Layout lbt = transpose2(logical_layout(d.op_b, d.order_b, d.K, d.N, d.ldb, Lb, Lb > 1 ? d.stride_b : 0));  // (N,K,Lb)
    gl::Layout ld_ = logical_layout(GEMM_OP_N, d.order_d, d.M, d.N, d.ldd, L, d.stride_d);   // (M,N,L)

    // The kernel writes D with N contiguous.  A column-major D is the
    // row-major D^T = op(B)^T op(A)^T: swap the operands.
    const bool swap = mode_stride(ld_, 1) != 1;
    P.info.swapped = swap;
    if (!swap) {
        P.a = la;
        P.b = lbt;
        P.cd = ld_;
        P.Mk = d.M;
        P.Nk = d.N;
    } else {
        P.a = lbt;
        P.b = la;
        P.cd = transpose2(ld_);
        P.Mk = d.N;
        P.Nk = d.M;
    }
    // An operand is K-major when its K mode has unit stride.  Leading
    // dimensions are at least 16 bytes, so exactly one mode has unit stride.
    const bool a_kmaj = mode_stride(P.a, 1) == 1;
    const bool b_kmaj = mode_stride(P.b, 1) == 1;
    P.info.a_k_major = a_kmaj;
    P.info.b_k_major = b_kmaj;
    P.bias_mode = d.bias == GEMM_BIAS_NONE ? 0 : ((d.bias == GEMM_BIAS_COL) != swap ? 1 : 2);

    // Tile shape.  Default: a CTA pair (cta_group::2) computes 256 x 256, each
    // SM loading 128 rows of A and 128 of B per K block: 64 B/clk/SM of
    // L2->SM traffic at full MMA rate.  A single CTA's 128 x 256 tile needs
    // 96 B/clk/SM and 128 x 128 the whole 128 B/clk of shared-memory reads,
    // so one CTA is used only where pairs would leave most SMs idle (small
    // problems) or N fits in 128.
    const int64_t tiles2 = ((P.Mk + 255) / 256) * ((P.Nk + 255) / 256) * L;
    int cg = (P.Mk > 128 && P.Nk > 128 && tiles2 >= 64) ? 2 : 1;
    int tile_n = 256;
    if (cg == 1 && (P.Nk <= 128 || ((P.Mk + kTileM - 1) / kTileM) * ((P.Nk + 255) / 256) * L < 76)) tile_n = 128;
    // 0 dense, 1 MXFP8, 2 NVFP4
    const int bs = d.block_scale == GEMM_BLOCK_SCALE_NONE ? 0 : (nv ? 2 : 1);
    if (nv && (!a_kmaj || !b_kmaj)) return GEMM_ERR_UNSUPPORTED;     // the pages' TN layout only
    if (bs) {
        // The block-scaled kernel: CTA pairs with 256 x 256 tiles (one TMEM
        // accumulator beside the scale factors) where at least 64 of them fill
        // the GPU, else pairs with 256 x 128 tiles, else one CTA (128 x 128).
        // NVFP4 output takes the 256 x 128 pairs whenever 64 of them fill the
        // GPU: their two accumulators let the quantising epilogue run under
        // the next tile's MMAs (8192^3 NVFP4 -> NVFP4 2557 -> 2845 TFLOP/s;
        // with a bf16 or MX output the 256 x 256 tile is faster).
        // A pair CTA of a 256 x 128 tile holds 64 rows of B, narrower than one
        // 128-element MN-major e4m3 box, so an MN-major B stays on one CTA.
        const int64_t tiles_256 = ((P.Mk + 255) / 256) * ((P.Nk + 255) / 256) * L;
        const int64_t tiles_128 = ((P.Mk + 255) / 256) * ((P.Nk + 127) / 128) * L;
        if (P.Mk > 128 && P.Nk > 128 && tiles_256 >= 64 && !(out_nv && tiles_128 >= 64 && b_kmaj)) {
            cg = 2;
            tile_n = 256;
        } else {
            cg = (P.Mk > 128 && tiles_128 >= 64 && b_kmaj) ? 2 : 1;
            tile_n = 128;
        }
    }
    const int tile_m = kTileM * cg;
    P.cta_group = cg;
    P.tile_n = tile_n;
    const int64_t tiles_m = (P.Mk + tile_m - 1) / tile_m;
    const int64_t tiles_n = (P.Nk + tile_n - 1) / tile_n;

    P.info.tile_m = tile_m;
    P.info.tile_n = tile_n;
    P.info.tile_k = kStageKBytes / ab * (nv ? 2 : 1);
    P.info.cta_group = cg;
    P.info.stages = stages_for(cg, tile_n, bs);
    P.info.epi_cols = 128 / ob;
    P.info.tiles_m = tiles_m;
    P.info.tiles_n = tiles_n;
    P.info.tiles = tiles_m * tiles_n * L;
    P.info.kernel_m = P.Mk;
    P.info.kernel_n = P.Nk;
    if (P.info.tiles > INT32_MAX) return GEMM_ERR_UNSUPPORTED;

    // Grouped raster: walk `G` M tiles, then the next N tile, so CTAs that
    // run together share A and B panels in L2.  As layouts from the tile
    // counter t to the linear tile index m_blk + tiles_m * n_blk.
    const int64_t gmax = cg == 2 ? 8 : 16;
    const int64_t G = tiles_m < 1 ? 1 : (tiles_m < gmax ? tiles_m : gmax);
    const int64_t full_groups = tiles_m / G;
    const int64_t tail = tiles_m - full_groups * G;
    P.info.raster_group = (int32_t)G;

    KernelParams& k = P.kp;
    memset(&k, 0, sizeof(k));
    k.M = (int32_t)P.Mk;
    k.N = (int32_t)P.Nk;
    k.K = (int32_t)d.K;
    k.L = (int32_t)L;
    k.tiles_m = (int32_t)tiles_m;
    k.tiles_n = (int32_t)tiles_n;
    k.tiles_per_batch = (int32_t)(tiles_m * tiles_n);
    k.num_tiles = (int32_t)(tiles_m * tiles_n * L);
    const int kel = kStageKBytes / ab;
    k.num_kb = (int32_t)((d.K + kel - 1) / kel);
    k.dp_tiles = k.num_tiles;                 // data parallel until a schedule says otherwise
    {
        gl::Layout parts[3] = {gl::leaf(G, 1), gl::leaf(tiles_n, tiles_m), gl::leaf(full_groups > 0 ? full_groups : 1, G)};
        gl::Layout full;
        gl::concat(parts, 3, &full);
        gl::flatten(full, &k.raster_full);
        k.raster_full_count = (int32_t)(G * tiles_n * full_groups);
        gl::Layout tparts[2] = {gl::leaf(tail > 0 ? tail : 1, 1), gl::leaf(tiles_n, tiles_m)};
        gl::Layout tl;
        gl::concat(tparts, 2, &tl);
        gl::flatten(tl, &k.raster_tail);
        k.raster_tail_offset = (int32_t)(full_groups * G);
    }
    k.a_kmajor = a_kmaj;
    k.b_kmajor = b_kmaj;
    k.block_scaled = bs;
    // 1: e4m3 D with ue8m0 factors per 32; 2: e2m1 D with ue4m3 factors per 16
    k.out_f8 = d.out_scale == GEMM_OUT_SCALE_MX ? 1 : (out_nv ? 2 : 0);
    k.scale_d = d.scale_d;
    if (k.out_f8) {
        const int64_t sv = out_nv ? 16 : 32;
        const int64_t sfk = (P.Nk + sv - 1) / sv;
        k.sfd_kb4 = (int32_t)((sfk + 3) / 4);
        k.sfd_bstride = ((P.Mk + 127) / 128) * (int64_t)k.sfd_kb4 * 512;
    }
    k.sf_mblocks = (int32_t)((P.Mk + 127) / 128);
    k.sf_nblocks = (int32_t)((P.Nk + 127) / 128);
    k.elem_bytes = ab;
    k.kind_f8 = d.dtype_a == GEMM_E4M3;
    k.mma_variant = (d.dtype_a == GEMM_E4M3 ? 8 : 0) + (d.dtype_a == GEMM_BF16 ? 4 : 0) + (a_kmaj ? 0 : 2) +
                    (b_kmaj ? 0 : 1);
    k.a_batched = L > 1 && mode_stride(P.a, 2) != 0;
    k.b_batched = Lb > 1 && mode_stride(P.b, 2) != 0;
    k.groups = groups;
    k.c_batched = L > 1 && d.stride_c != 0;
    k.alpha = d.alpha * d.scale_a * d.scale_b;            // per-tensor dequantisation folded into alpha
    k.beta = d.beta;
    k.has_c = has_c;
    k.bias_mode = P.bias_mode;
    k.bias_stride = d.stride_bias;
    k.act = d.act;
    // reductions in kernel orientation: with D computed transposed, the
    // caller's rows are the kernel's columns
    const bool user_rows = (d.reduce & GEMM_REDUCE_ROW_SUM) != 0, user_cols = (d.reduce & GEMM_REDUCE_COL_SUM) != 0;
    k.red_rows = P.info.swapped ? user_cols : user_rows;
    k.red_cols = P.info.swapped ? user_rows : user_cols;
    k.red_amax = (d.reduce & GEMM_REDUCE_ABS_MAX) != 0;
    k.out_f16 = d.dtype_d == GEMM_F16;
    k.d_ragged = ((P.Nk * ob) % 16) != 0;
    k.ldd = mode_stride(P.cd, 0);
    k.d_bstride = mode_stride(P.cd, 2);
    if (out_nv) {                              // the kernel addresses e2m1 D in bytes
        k.ldd /= 2;
        k.d_bstride /= 2;
    }
    k.timeout_ns = kDefaultTimeoutNs;
    return GEMM_OK;
}

// ------------------------------------------------------------ TMA maps ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

CUtensorMapDataType tma_type(int dt) {
    switch (dt) {
        case GEMM_F32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
    }
}

// 3-D map over a kernel-orientation operand layout (rows, cols, batch): the
// unit-stride mode becomes TMA dimension 0 (as the layout's strides dictate),
// the other matrix mode dimension 1, the batch dimension 2.
bool encode_map(CUtensorMap* map, const gl::Layout& lay, int dt, const void* base, uint32_t box0, uint32_t box1,
                bool batched) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int es = dtype_bytes(dt);
    const int inner = mode_stride(lay, 0) == 1 ? 0 : 1;
    const int outer = 1 - inner;
    const int64_t e_in = mode_extent(lay, inner), e_out = mode_extent(lay, outer);
    const int64_t s_out = mode_stride(lay, outer);
    cuuint64_t dims[3] = {(cuuint64_t)e_in, (cuuint64_t)e_out, (cuuint64_t)(batched ? mode_extent(lay, 2) : 1)};
    const cuuint64_t row_bytes = (cuuint64_t)s_out * es;
    const cuuint64_t bs = batched ? (cuuint64_t)mode_stride(lay, 2) * es : row_bytes * dims[1];
    cuuint64_t strides[2] = {row_bytes, bs < row_bytes ? row_bytes : bs};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, tma_type(dt), 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Scale-factor tensor as TMA sees it: rows of 256 bytes, 2 rows (one
// 512-byte block) per box, `blocks` blocks in all.  A copy moves a box row
// at a time, so wide rows keep a block to two requests.
// Rank 3 (a unit third dimension) like the operand maps, since the kernel
// issues 3-D tensor copies for both.
bool encode_sf_map(CUtensorMap* map, const void* base, int64_t blocks) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {256, (cuuint64_t)(blocks * 2), 1};
    cuuint64_t strides[2] = {256, (cuuint64_t)(blocks * 512)};
    cuuint32_t box[3] = {256, 2, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MXFP8 factors of B for a tile of `per_tile` 128-column blocks: a 4-D view
// (256-byte row, the block's 2 rows, K block, 128-column block) whose box
// takes one K block of `per_tile` adjacent column blocks.
bool encode_sf_map_b4(CUtensorMap* map, const void* base, int64_t kblocks, int64_t nblocks, uint32_t per_tile) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {256, 2, (cuuint64_t)kblocks, (cuuint64_t)nblocks};
    cuuint64_t strides[3] = {256, 512, (cuuint64_t)(kblocks * 512)};
    cuuint32_t box[4] = {256, 2, 1, per_tile};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NVFP4 factors: one ue4m3 per 16 K elements, so a 256-element K stage
// takes four 512-byte blocks per 128 rows, adjacent in the tensor.  Seen as
// rows of 256 bytes: dimension 1 walks a 128-row block's K blocks (2 rows
// each, `kblocks` of them), dimension 2 the 128-row blocks; a box of 8 rows
// is one stage's four blocks (of `per_box` adjacent 128-row blocks: B's box
// covers a 256-wide tile's two), and blocks past the last K block read as
// zero.
bool encode_sf_map_nv(CUtensorMap* map, const void* base, int64_t kblocks, int64_t row_blocks, uint32_t per_box = 1) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {256, (cuuint64_t)(kblocks * 2), (cuuint64_t)row_blocks};
    cuuint64_t strides[2] = {256, (cuuint64_t)(kblocks * 512)};
    cuuint32_t box[3] = {256, 8, per_box};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Persistent grid: one CTA (or CTA pair) per SM (pair of SMs), never more
// than there are tiles.  A grouped launch counts its tiles on the device, so
// it takes every slot.
// Workers (CTAs, or CTA pairs) the GPU holds at once.
int64_t worker_slots(const Plan& P, int sm_count, int max_clusters) {
    int64_t slots = sm_count / P.cta_group;
    if (max_clusters > 0 && max_clusters < slots) slots = max_clusters;
    return slots < 1 ? 1 : slots;
}

// CTAs of a launch: one worker per slot, no more workers than tiles, except
// that a split single wave has one worker per K range.
int grid_for(const Plan& P, int sm_count, int max_clusters) {
    const int64_t tiles = P.info.tiles;
    const int cg = P.cta_group;
    if (P.kp.clc) return (int)(tiles * cg);          // dynamic: one cluster per tile
    const int64_t slots = worker_slots(P, sm_count, max_clusters);
    if (P.kp.groups > 0) return (int)(slots * cg);
    int64_t n = tiles < slots ? tiles : slots;
    if (P.kp.sk_ranges > n) n = P.kp.sk_ranges;
    return (int)(n * cg);
}

}  // namespace

struct gemm_handle_s {
    Plan plan;
    int device = -1;
    int sm_count = 0;
    int max_clusters = 0;     // co-resident clusters of the planned kernel (0: unknown)
    uint32_t* status = nullptr;
    int workers = 0;          // persistent CTAs (or CTA pairs) of a launch
    void* ws = nullptr;       // stream-K partial sums, then the flag words
    bool ws_dirty = false;    // a launch failed: flags / abs-max words may be left set
    void* red_ws = nullptr;   // reduction partials: rows, columns, abs-max words
    size_t red_amax_off = 0;  // byte offset of the abs-max words in red_ws
    cudaStream_t last_stream = nullptr;
    bool launched = false;
    uint64_t launches = 0;
    // map cache, keyed by the pointers of the last run
    const void* cached[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    bool cache_valid = false;
    CUtensorMap maps[6];
};

namespace {

// Work split for `mode` (gemm_sched_t) on the handle's device; allocates the
// stream-K workspace when the split cuts tiles.
gemm_status_t apply_schedule(gemm_handle_s* h, int mode) {
    Plan& P = h->plan;
    KernelParams& k = P.kp;
    if (h->ws) {
        cudaFree(h->ws);
        h->ws = nullptr;
    }
    k.dp_tiles = k.num_tiles;
    k.sk_iters = 0;
    k.sk_ranges = 0;
    k.sk_part = nullptr;
    k.sk_flags = nullptr;
    k.clc = 0;
    h->ws_dirty = false;
    int64_t workers = grid_for(P, h->sm_count, h->max_clusters) / P.cta_group;
    h->workers = (int)workers;
    if (mode == GEMM_SCHED_DYNAMIC) {      // whole tiles, one cluster launched per tile
        k.clc = 1;
        return GEMM_OK;
    }
    const int64_t T = k.num_tiles, kb = k.num_kb;
    if (mode == GEMM_SCHED_DATA_PARALLEL || k.groups > 0 || workers < 1 || kb < 1) return GEMM_OK;
    const int64_t slots = worker_slots(P, h->sm_count, h->max_clusters);
    int64_t dp, sk, ranges;
    if (mode == GEMM_SCHED_STREAM_K) {
        // the last full wave and the ragged one, one equal range per worker
        // (S workers: a single wave of fewer tiles is spread over all of them)
        const int64_t full = T / slots;
        dp = full >= 1 ? (full - 1) * slots : 0;
        sk = (T - dp) * kb;
        ranges = slots;
        workers = slots;
    } else {
        // the ragged last wave only: each of its tiles cut into `pieces`
        // equal K ranges, so that pieces * rest <= slots (a problem of less
        // than one wave then runs on pieces * rest workers)
        const int64_t full = T / slots, ragged = T % slots;
        if (ragged == 0) return GEMM_OK;
        int64_t pieces = slots / ragged;
        if (pieces > kb) pieces = kb;
        // (AUTO leaves a single wave whole: cutting 1000^3's 64 tiles in two
        // measured 11.2 -> 13.9 us, the partial sums' exchange costing more
        // than the halved K loop saves)
        if (mode == GEMM_SCHED_AUTO && (full < 1 || pieces < 2 || kb / pieces < 4)) return GEMM_OK;
        if (pieces < 1) pieces = 1;
        dp = full * slots;
        sk = ragged * kb;
        ranges = ragged * pieces;
        if (ranges > workers) workers = ranges;
    }
    const size_t part_bytes = (size_t)workers * P.cta_group * kTileM * P.tile_n * sizeof(float);
    const size_t flag_bytes = (size_t)workers * P.cta_group * kEpiWarps * sizeof(uint32_t);
    if (cudaMalloc(&h->ws, part_bytes + flag_bytes) != cudaSuccess ||
        cudaMemset(static_cast<char*>(h->ws) + part_bytes, 0, flag_bytes) != cudaSuccess) {
        cudaGetLastError();
        if (h->ws) cudaFree(h->ws);
        h->ws = nullptr;
        return GEMM_ERR_CUDA;
    }
    k.dp_tiles = (int32_t)dp;
    k.sk_iters = sk;
    k.sk_ranges = (int32_t)ranges;
    h->workers = (int)workers;
    k.sk_part = static_cast<float*>(h->ws);
    k.sk_flags = reinterpret_cast<uint32_t*>(static_cast<char*>(h->ws) + part_bytes);
    return GEMM_OK;
}

// Reduction partials (kernel orientation): rows [L][tiles_n][M], columns
// [L][ceil(M/32)][N], abs-max words [L] (zeroed here; the finishing pass
// zeroes them after each launch).
gemm_status_t alloc_reductions(gemm_handle_s* h) {
    KernelParams& k = h->plan.kp;
    if (!k.red_rows && !k.red_cols && !k.red_amax) return GEMM_OK;
    const int64_t L = k.L, M = k.M, N = k.N;
    const size_t row_b = k.red_rows ? (size_t)(L * k.tiles_n * M) * sizeof(float) : 0;
    const size_t col_b = k.red_cols ? (size_t)(L * ((M + 31) / 32) * N) * sizeof(float) : 0;
    const size_t amax_off = (row_b + col_b + 255) & ~(size_t)255;
    const size_t bytes = amax_off + (size_t)L * sizeof(uint32_t);
    if (cudaMalloc(&h->red_ws, bytes) != cudaSuccess ||
        cudaMemset(static_cast<char*>(h->red_ws) + amax_off, 0, (size_t)L * sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        if (h->red_ws) cudaFree(h->red_ws);
        h->red_ws = nullptr;
        return GEMM_ERR_CUDA;
    }
    char* base = static_cast<char*>(h->red_ws);
    k.red_row_ws = k.red_rows ? reinterpret_cast<float*>(base) : nullptr;
    k.red_col_ws = k.red_cols ? reinterpret_cast<float*>(base + row_b) : nullptr;
    k.red_amax_ws = k.red_amax ? reinterpret_cast<uint32_t*>(base + amax_off) : nullptr;
    h->red_amax_off = amax_off;
    return GEMM_OK;
}

size_t flag_bytes_of(const gemm_handle_s* h) {
    return (size_t)h->workers * h->plan.cta_group * kEpiWarps * sizeof(uint32_t);
}

}  // namespace

extern "C" {

gemm_status_t gemm_plan(const gemm_desc_t* desc, gemm_plan_info_t* info) {
    if (!info) return GEMM_ERR_INVALID_ARG;
    Plan* p = new (std::nothrow) Plan;
    if (!p) return GEMM_ERR_INVALID_ARG;
    const gemm_status_t s = validate_and_plan(desc, p);
    if (s == GEMM_OK) *info = p->info;
    delete p;
    return s;
}

static gemm_status_t create_impl(gemm_handle_t* out, const gemm_desc_t* desc, int32_t groups) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    gemm_handle_s* h = new (std::nothrow) gemm_handle_s;
    if (!h) return GEMM_ERR_INVALID_ARG;
    gemm_status_t s = validate_and_plan(desc, &h->plan, groups);
    if (s != GEMM_OK) {
        delete h;
        return s;
    }
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        cudaGetLastError();
        delete h;
        return GEMM_ERR_NO_DEVICE;
    }
    int major = 0, minor = 0;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return GEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {      // built for sm_103a only
        delete h;
        return GEMM_ERR_NO_DEVICE;
    }
    if (prepare_kernel(h->plan.cta_group, h->plan.tile_n, h->plan.out_bytes, h->plan.kp.block_scaled) != cudaSuccess ||
        cudaMalloc(&h->status, sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(h->status, 0, sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        if (h->status) cudaFree(h->status);
        delete h;
        return GEMM_ERR_CUDA;
    }
    h->plan.kp.status = h->status;
    h->max_clusters =
        max_active_clusters(h->plan.cta_group, h->plan.tile_n, h->plan.out_bytes, h->plan.kp.block_scaled);
    s = apply_schedule(h, GEMM_SCHED_AUTO);
    if (s == GEMM_OK) s = alloc_reductions(h);
    if (s != GEMM_OK) {
        if (h->ws) cudaFree(h->ws);
        cudaFree(h->status);
        delete h;
        return s;
    }
    *out = h;
    return GEMM_OK;
}

gemm_status_t gemm_create(gemm_handle_t* out, const gemm_desc_t* desc) { return create_impl(out, desc, 0); }

gemm_status_t gemm_grouped_create(gemm_handle_t* out, const gemm_desc_t* desc, int32_t groups) {
    if (groups < 1) {
        if (out) *out = nullptr;
        return GEMM_ERR_INVALID_ARG;
    }
    return create_impl(out, desc, groups);
}

static gemm_status_t run_impl(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
                              const float* bias, float* row_sum, float* col_sum, float* abs_max, const void* sfa,
                              const void* sfb, void* sfd, void* stream, const int64_t* group_rows = nullptr) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    Plan& P = h->plan;
    const gemm_desc_t& d = P.d;
    if ((P.kp.groups > 0) != (group_rows != nullptr)) return GEMM_ERR_INVALID_ARG;
    if (group_rows && (reinterpret_cast<uintptr_t>(group_rows) & 7u)) return GEMM_ERR_MISALIGNED;
    if (P.kp.out_f8 && !sfd) return GEMM_ERR_INVALID_ARG;
    if (P.kp.block_scaled && d.K > 0) {
        if (!sfa || !sfb) return GEMM_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(sfa) | reinterpret_cast<uintptr_t>(sfb)) & 15u) return GEMM_ERR_MISALIGNED;
    }
    if (((d.reduce & GEMM_REDUCE_ROW_SUM) && !row_sum) || ((d.reduce & GEMM_REDUCE_COL_SUM) && !col_sum) ||
        ((d.reduce & GEMM_REDUCE_ABS_MAX) && !abs_max))
        return GEMM_ERR_INVALID_ARG;
    if (d.M == 0 || d.N == 0) return GEMM_OK;
    if (!D || (d.K > 0 && (!A || !B)) || (P.has_c && !C) || (d.bias != GEMM_BIAS_NONE && !bias))
        return GEMM_ERR_INVALID_ARG;
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al16(D) || (A && !al16(A)) || (B && !al16(B)) || (P.has_c && !al16(C))) return GEMM_ERR_MISALIGNED;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return GEMM_ERR_MISALIGNED;

    // With K == 0 nothing is loaded; give the maps a valid placeholder base.
    const void* a_ptr = A ? A : D;
    const void* b_ptr = B ? B : D;
    const void* c_ptr = P.has_c ? C : D;
    const bool swap = P.info.swapped;
    const void* ka = swap ? b_ptr : a_ptr;
    const void* kb = swap ? a_ptr : b_ptr;
    const int ab = P.a_bytes;
    const uint32_t kel = kStageKBytes / ab;
    // kernel orientation: with D computed transposed, A's factors go with the kernel's B
    const void* ksfa = swap ? sfb : sfa;
    const void* ksfb = swap ? sfa : sfb;
    if (!h->cache_valid || h->cached[0] != ka || h->cached[1] != kb || h->cached[2] != c_ptr || h->cached[3] != D ||
        h->cached[4] != ksfa || h->cached[5] != ksfb) {
        const int tn = P.tile_n;
        const uint32_t epi_cols = 128u / P.out_bytes;
        const int adt = d.dtype_a;
        bool ok = true;
        // A: box {K: kel, M: 128} (K-major) or {M: kel, K: kel} (MN-major)
        ok = ok && encode_map(&h->maps[0], P.a, adt, ka, kel, P.kp.a_kmajor ? kTileM : kel, P.kp.a_batched);
        ok = ok && encode_map(&h->maps[1], P.b, adt, kb, kel, P.kp.b_kmajor ? (uint32_t)(tn / P.cta_group) : kel,
                              P.kp.b_batched);
        if (P.kp.out_f8 == 2) {
            // e2m1 D (stored by the kernel directly): a map over its bytes
            const gl::Layout lb = logical_layout(GEMM_OP_N, GEMM_ROW_MAJOR, d.M, d.N / 2, d.ldd / 2, d.batch,
                                                 d.stride_d / 2);
            ok = ok && encode_map(&h->maps[3], lb, GEMM_E4M3, D, epi_cols, kEpiRows, d.batch > 1);
        } else {
            ok = ok && encode_map(&h->maps[3], P.cd, d.dtype_d, D, epi_cols, kEpiRows, d.batch > 1);
        }
        if (P.has_c) {
            gl::Layout lc = logical_layout(GEMM_OP_N, d.order_c, d.M, d.N, d.ldc, d.batch, d.stride_c);
            if (swap) lc = transpose2(lc);
            ok = ok && encode_map(&h->maps[2], lc, d.dtype_c, C, epi_cols, kEpiRows, P.kp.c_batched);
        } else {
            h->maps[2] = h->maps[3];
        }
        if (P.kp.block_scaled && d.K > 0) {
            // grouped: A's factors in whole 128-row blocks per group (at most
            // one partial block per group on top of A's own), B's per group
            const int64_t groups = P.kp.groups;
            const int64_t la_n = P.kp.a_batched ? P.kp.L : 1;
            const int64_t lb_n = P.kp.b_batched ? (groups > 0 ? groups : P.kp.L) : 1;
            const int64_t a_rowblocks = la_n * P.kp.sf_mblocks + groups;
            if (P.kp.block_scaled == 2) {
                // K here counts bytes (two elements each): ceil(K/16) factors, four per block
                const int64_t kblocks = (2 * d.K + 63) / 64;
                ok = ok && encode_sf_map_nv(&h->maps[4], ksfa, kblocks, a_rowblocks);
                ok = ok && encode_sf_map_nv(&h->maps[5], ksfb, kblocks, lb_n * P.kp.sf_nblocks, (uint32_t)(tn / 128));
            } else {
                ok = ok && encode_sf_map(&h->maps[4], ksfa, a_rowblocks * (int64_t)P.kp.num_kb);
                ok = ok && encode_sf_map_b4(&h->maps[5], ksfb, P.kp.num_kb, lb_n * P.kp.sf_nblocks, (uint32_t)(tn / 128));
            }
        } else {
            h->maps[4] = h->maps[0];
            h->maps[5] = h->maps[0];
        }
        if (!ok) {
            h->cache_valid = false;
            return GEMM_ERR_CUDA;
        }
        h->cached[0] = ka;
        h->cached[1] = kb;
        h->cached[2] = c_ptr;
        h->cached[3] = D;
        h->cached[4] = ksfa;
        h->cached[5] = ksfb;
        h->cache_valid = true;
    }
    LaunchArgs la;
    la.tmA = h->maps[0];
    la.tmB = h->maps[1];
    la.tmC = h->maps[2];
    la.tmD = h->maps[3];
    la.tmSA = h->maps[4];
    la.tmSB = h->maps[5];
    la.p = P.kp;
    la.p.bias = bias;
    la.p.d_ptr = D;
    la.p.sfa = static_cast<const uint8_t*>(ksfa);
    la.p.sfb = static_cast<const uint8_t*>(ksfb);
    la.p.sfd = static_cast<uint8_t*>(sfd);
    la.p.group_rows = group_rows;
    la.cta_group = P.cta_group;
    la.tile_n = P.tile_n;
    la.out_bytes = P.out_bytes;
    la.block_scaled = P.kp.block_scaled;
    la.grid = grid_for(P, h->sm_count, h->max_clusters);
    la.stream = static_cast<cudaStream_t>(stream);
    if (la.grid < 1) return GEMM_OK;
    if (h->ws_dirty) {      // a failed launch may have left flags or abs-max words set
        if ((h->ws && cudaMemsetAsync(P.kp.sk_flags, 0, flag_bytes_of(h), la.stream) != cudaSuccess) ||
            (P.kp.red_amax_ws &&
             cudaMemsetAsync(P.kp.red_amax_ws, 0, (size_t)P.kp.L * sizeof(uint32_t), la.stream) != cudaSuccess)) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        h->ws_dirty = false;
    }
    cudaError_t e = launch(la);
    if (e == cudaSuccess && h->red_ws) {
        FinishParams f;
        f.L = P.kp.L;
        f.M = P.kp.M;
        f.N = P.kp.N;
        f.tiles_n = P.kp.tiles_n;
        f.slabs = (P.kp.M + 31) / 32;
        f.row_ws = P.kp.red_row_ws;
        f.col_ws = P.kp.red_col_ws;
        f.amax_ws = P.kp.red_amax_ws;
        // kernel rows are the caller's columns when D is computed transposed
        f.out_rows = P.info.swapped ? col_sum : row_sum;
        f.out_cols = P.info.swapped ? row_sum : col_sum;
        f.out_amax = abs_max;
        e = launch_finish(f, la.stream);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    h->last_stream = la.stream;
    h->launched = true;
    ++h->launches;
    return GEMM_OK;
}

gemm_status_t gemm_run(gemm_handle_t h, const void* A, const void* B, const void* C, void* D, const float* bias,
                       void* stream) {
    return run_impl(h, A, B, C, D, bias, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, stream);
}

gemm_status_t gemm_run_ex(gemm_handle_t h, const void* A, const void* B, const void* C, void* D, const float* bias,
                          float* row_sum, float* col_sum, float* abs_max, void* stream) {
    return run_impl(h, A, B, C, D, bias, row_sum, col_sum, abs_max, nullptr, nullptr, nullptr, stream);
}

gemm_status_t gemm_grouped_run(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
                               const float* bias, const int64_t* group_rows, void* stream) {
    if (!group_rows) return GEMM_ERR_INVALID_ARG;
    return run_impl(h, A, B, C, D, bias, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, stream, group_rows);
}

gemm_status_t gemm_grouped_run_args(gemm_handle_t h, const gemm_args_t* a, const int64_t* group_rows, void* stream) {
    if (!a || !group_rows) return GEMM_ERR_INVALID_ARG;
    return run_impl(h, a->A, a->B, a->C, a->D, a->bias, a->row_sum, a->col_sum, a->abs_max, a->sfa, a->sfb, a->sfd,
                    stream, group_rows);
}

gemm_status_t gemm_run_args(gemm_handle_t h, const gemm_args_t* a, void* stream) {
    if (!a) return GEMM_ERR_INVALID_ARG;
    return run_impl(h, a->A, a->B, a->C, a->D, a->bias, a->row_sum, a->col_sum, a->abs_max, a->sfa, a->sfb, a->sfd,
                    stream);
}

gemm_status_t gemm_check(gemm_handle_t h) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    if (h->launched && cudaStreamSynchronize(h->last_stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    uint32_t word = 0;
    if (cudaMemcpy(&word, h->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (word) {
        cudaMemset(h->status, 0, sizeof(uint32_t));
        if (h->ws || h->red_ws) h->ws_dirty = true;
        return (word & kStatusTimeout) ? GEMM_ERR_TIMEOUT : GEMM_ERR_BOUNDS;
    }
    return GEMM_OK;
}

gemm_status_t gemm_set_stamps(gemm_handle_t h, void* stamps) {
#ifdef GEMM_STAMPS
    if (!h) return GEMM_ERR_INVALID_ARG;
    h->plan.kp.stamps = static_cast<unsigned long long*>(stamps);
    return GEMM_OK;
#else
    (void)h;
    (void)stamps;
    return GEMM_ERR_UNSUPPORTED;
#endif
}

int32_t gemm_build_flags(void) {
    int32_t f = 0;
#ifdef GEMM_DEBUG
    f |= 1;
#endif
#ifdef GEMM_STAMPS
    f |= 2;
#endif
    return f;
}

gemm_status_t gemm_set_schedule(gemm_handle_t h, int32_t mode) {
    if (!h || mode < GEMM_SCHED_AUTO || mode > GEMM_SCHED_DYNAMIC) return GEMM_ERR_INVALID_ARG;
    if (h->plan.kp.groups > 0 && mode != GEMM_SCHED_AUTO && mode != GEMM_SCHED_DATA_PARALLEL)
        return GEMM_ERR_UNSUPPORTED;          // grouped: whole tiles only
    if (h->launched && cudaStreamSynchronize(h->last_stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return apply_schedule(h, mode);
}

gemm_status_t gemm_get_schedule(gemm_handle_t h, int32_t* workers, int64_t* dp_tiles, int64_t* sk_iters,
                                int32_t* sk_ranges) {
    if (!h) return GEMM_ERR_INVALID_ARG;
    if (workers) *workers = h->workers;
    if (dp_tiles) *dp_tiles = h->plan.kp.dp_tiles;
    if (sk_iters) *sk_iters = h->plan.kp.sk_iters;
    if (sk_ranges) *sk_ranges = h->plan.kp.sk_ranges;
    return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_handle_t h) {
    if (!h) return GEMM_OK;
    if (h->launched) cudaStreamSynchronize(h->last_stream);
    if (h->status) cudaFree(h->status);
    if (h->ws) cudaFree(h->ws);
    if (h->red_ws) cudaFree(h->red_ws);
    cudaGetLastError();
    delete h;
    return GEMM_OK;
}

gemm_status_t gemm_set_debug(gemm_handle_t h, int32_t inject_fault, uint32_t timeout_ms) {
    if (!h || (inject_fault != 0 && inject_fault != 1)) return GEMM_ERR_INVALID_ARG;
    h->plan.kp.inject = inject_fault;
    if (timeout_ms) h->plan.kp.timeout_ns = (uint64_t)timeout_ms * 1000000ull;
    return GEMM_OK;
}

uint64_t gemm_launch_count(gemm_handle_t h) { return h ? h->launches : 0; }

const char* gemm_status_str(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "ok";
        case GEMM_ERR_INVALID_ARG: return "invalid argument";
        case GEMM_ERR_UNSUPPORTED: return "unsupported combination";
        case GEMM_ERR_MISALIGNED: return "misaligned pointer, leading dimension or batch stride";
        case GEMM_ERR_CUDA: return "CUDA error";
        case GEMM_ERR_TIMEOUT: return "an in-kernel wait ran out of time";
        case GEMM_ERR_NO_DEVICE: return "no sm_103 GPU available";
        case GEMM_ERR_BOUNDS: return "an index check of the diagnostic build failed";
        default: return "unknown status";
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// One-shot plan-and-launch into a caller-provided status word, with every
// host object on the stack: used by the allocation-free entry point
// (noalloc.cu).  Nothing here allocates host or device memory.
// ---------------------------------------------------------------------------
namespace gemm_sm103 {

gemm_status_t run_unallocated(const gemm_desc_t* desc, const void* A, const void* B, const void* C, void* D,
                              const float* bias, uint32_t* status, int sm_count, cudaStream_t stream,
                              VariantCache* cache, bool* launched) {
    *launched = false;
    Plan P;
    const gemm_status_t s = validate_and_plan(desc, &P);
    if (s != GEMM_OK) return s;
    if (P.d.reduce) return GEMM_ERR_UNSUPPORTED;     // reductions need a handle's workspace
    if (P.kp.block_scaled || P.kp.out_f8) return GEMM_ERR_UNSUPPORTED;   // no scale-factor arguments here
    const gemm_desc_t& d = P.d;
    if (d.M == 0 || d.N == 0) return GEMM_OK;
    if (!D || (d.K > 0 && (!A || !B)) || (P.has_c && !C) || (d.bias != GEMM_BIAS_NONE && !bias))
        return GEMM_ERR_INVALID_ARG;
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al16(D) || (A && !al16(A)) || (B && !al16(B)) || (P.has_c && !al16(C))) return GEMM_ERR_MISALIGNED;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return GEMM_ERR_MISALIGNED;

    const void* a_ptr = A ? A : D;
    const void* b_ptr = B ? B : D;
    const bool swap = P.info.swapped;
    const void* ka = swap ? b_ptr : a_ptr;
    const void* kb = swap ? a_ptr : b_ptr;
    const uint32_t kel = kStageKBytes / P.a_bytes;
    const uint32_t epi_cols = 128u / P.out_bytes;
    LaunchArgs la;
    bool ok = encode_map(&la.tmA, P.a, d.dtype_a, ka, kel, P.kp.a_kmajor ? kTileM : kel, P.kp.a_batched);
    ok = ok && encode_map(&la.tmB, P.b, d.dtype_a, kb, kel,
                          P.kp.b_kmajor ? (uint32_t)(P.tile_n / P.cta_group) : kel, P.kp.b_batched);
    ok = ok && encode_map(&la.tmD, P.cd, d.dtype_d, D, epi_cols, kEpiRows, d.batch > 1);
    if (P.has_c) {
        gl::Layout lc = logical_layout(GEMM_OP_N, d.order_c, d.M, d.N, d.ldc, d.batch, d.stride_c);
        if (swap) lc = transpose2(lc);
        ok = ok && encode_map(&la.tmC, lc, d.dtype_c, C, epi_cols, kEpiRows, P.kp.c_batched);
    } else {
        la.tmC = la.tmD;
    }
    la.tmSA = la.tmA;          // block scaling is refused above
    la.tmSB = la.tmA;
    if (!ok) return GEMM_ERR_CUDA;
    const int slot = VariantCache::slot(P.cta_group, P.tile_n, P.out_bytes);
    if (!cache->prepared[slot].load(std::memory_order_acquire)) {
        if (prepare_kernel(P.cta_group, P.tile_n, P.out_bytes, P.kp.block_scaled) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        cache->prepared[slot].store(1, std::memory_order_release);
    }
    int clusters = cache->clusters_plus1[slot].load(std::memory_order_acquire) - 1;
    if (clusters < 0) {
        clusters = max_active_clusters(P.cta_group, P.tile_n, P.out_bytes, P.kp.block_scaled);
        cache->clusters_plus1[slot].store(clusters + 1, std::memory_order_release);
    }
    la.p = P.kp;
    la.p.bias = bias;
    la.p.d_ptr = D;
    la.p.status = status;
    la.cta_group = P.cta_group;
    la.tile_n = P.tile_n;
    la.out_bytes = P.out_bytes;
    la.block_scaled = P.kp.block_scaled;
    la.grid = grid_for(P, sm_count, clusters);
    la.stream = stream;
    if (la.grid < 1) return GEMM_OK;
    // every check has passed: clear the status word the previous call left
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), stream) != cudaSuccess || launch(la) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    *launched = true;
    return GEMM_OK;
}

}  // namespace gemm_sm103
