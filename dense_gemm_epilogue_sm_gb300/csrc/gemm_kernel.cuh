// gemm_kernel.cuh - persistent, warp-specialised fused-epilogue GEMM for
// sm_103a (GB300): TMA -> shared-memory ring -> tcgen05.mma (fp32
// accumulator in TMEM) -> TMEM loads -> fused alpha/beta/bias/activation ->
// TMA (or direct) store.
//
// Template parameters: CG = 1: one CTA computes a 128 x BN tile with tcgen05
// cta_group::1; CG = 2: a cluster of two CTAs computes a 256 x BN tile with
// cta_group::2 MMAs issued by the even CTA (the leader), each CTA loading its
// own 128 rows of A and BN/2 rows of B, the leader's full[s] barrier counting
// both CTAs' bytes, commits multicast to both CTAs, and each CTA's epilogue
// reading the 128 accumulator rows in its own TMEM and signalling the
// leader's acc_empty barrier.  BN: 128 or 256 tile columns.  OB: output
// element bytes (1 = block-scaled e4m3 / e2m1 output with its factors, stored
// directly).  BS: block-scaled operands (0 none, 1 MXFP8, 2 NVFP4).
//
// Structure (the roles of "Technical Documentation: NVIDIA/cutlass",
// "Blackwell Warp-specialized Persistent Kernel", re-split for this kernel):
//   warp 0      one lane issues TMA loads of A and B tiles (and their scale
//               factors) into a STAGES-deep ring; full[s] counts the bytes,
//               empty[g] is released by the MMA's commit for a group of
//               stages;
//   warp 1      owns the TMEM allocation; one lane issues tcgen05.mma into a
//               TMEM accumulator (two, double buffered, except for 256-wide
//               block-scaled tiles, whose factor columns leave room for one);
//   warps 2..5  the epilogue: each warp owns one 32-lane TMEM quadrant
//               (rows 32q..32q+31 of the 128-row tile), loads the source C
//               subtile by TMA, applies the fusion in registers, stages D in
//               swizzled shared memory and stores it by TMA;
//   warp 6      block-scaled kernels only: one lane copies each stage's
//               scale factors into TMEM once the stage has landed and
//               signals factors_ready[s], which the MMA thread waits on.
// Work: a persistent walk over (tile, K-block range) units shared by all
// roles: whole tiles in a grouped raster order given as a layout
// (raster_full / raster_tail), after the static scheduler of "Blackwell
// Cluster Launch Control", "Static Persistent Kernel"; optionally the last
// wave cut in K (split tail) or stream-K ranges with an fp32 fix-up; or
// tiles taken on the fly through cluster launch control; or the tiles of a
// grouped GEMM, counted from device row offsets.
//
// Every mbarrier wait is bounded: on expiry the waiting thread sets the
// kernel's status word and a shared abort flag, all roles leave their loops,
// outstanding TMA loads are awaited (bounded), the MMA pipe is drained, and
// TMEM is freed before the CTA exits.  Nothing traps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <type_traits>

#include "gemm_internal.h"
#include "gemm_variants.h"
#include "ptx.cuh"

namespace gemm_sm103 {


// Diagnostic timestamps (built with -DGEMM_STAMPS, with a buffer set on the
// handle): %globaltimer at eight points of each CTA, slot i of CTA b at
// stamps[8 b + i]:
//   0 entry, 1 set-up done (barriers, TMEM, tensor maps), 2 first loads
//   issued, 3 first stage's data in (the MMA thread), 4 first accumulator
//   committed, 5 the epilogue sees it, 6 the epilogue's last store complete,
//   7 before TMEM is freed.  Compiled out otherwise.
//   (6: the last stores have read their staging buffers.)
#ifdef GEMM_STAMPS
// The timer is read through a volatile shared-memory round trip, so that the
// read cannot move across the barriers and waits around the stamp point.
__device__ __forceinline__ void gemm_stamp(const KernelParams& p, int i) {
    __shared__ volatile unsigned long long order;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    order = t;
    if (p.stamps) p.stamps[(size_t)blockIdx.x * 8 + i] = order;
}
#define GEMM_STAMP(p, i) gemm_stamp((p), (i))
#else
#define GEMM_STAMP(p, i) \
    do {                 \
    } while (0)
#endif

// Diagnostic index checks (built with -DGEMM_DEBUG): every plain global store
// and every TMA store is first checked against the extents of its buffer; a
// failed check records kStatusBounds in the status word (gemm_check then
// returns GEMM_ERR_BOUNDS) and the access is skipped.  Compiled out (always
// true) otherwise.
#ifdef GEMM_DEBUG
__device__ __forceinline__ bool debug_in_bounds(const KernelParams& p, bool ok) {
    if (!ok) atomicOr(p.status, kStatusBounds);
    return ok;
}
#define GEMM_IN_BOUNDS(p, cond) debug_in_bounds((p), (cond))
#else
#define GEMM_IN_BOUNDS(p, cond) true
#endif

// TMEM accumulators per CTA: two, so the epilogue of one tile overlaps the
// main loop of the next (512 columns for BN = 256).
constexpr int kPairAccBufs = 2;

// Dynamic schedule: responses of cluster launch control kept for the roles
// that have not read them yet.
constexpr int kClcSlots = 4;

// BS: block-scaled operands.  1: MXFP8, e4m3 with one ue8m0 scale factor per
// 32 K elements; 2: NVFP4, e2m1 (two per byte) with one ue4m3 factor per 16.
// Each stage then also holds the 512-byte scale-factor blocks of its A rows
// and B rows (one per 128 rows for MXFP8, whose 128-element stage has four
// factors a row; four for NVFP4, whose 256-element stage has sixteen), which
// the copier warp (factor_copier) copies into TMEM columns after the
// accumulators.
// TMEM accumulators: two, except for block-scaled 256-wide tiles, whose
// 256-column accumulator leaves room for one only beside the scale factors.
__host__ __device__ constexpr int acc_bufs(int cg, int bn, int bs) {
    return (bs && bn == 256) ? 1 : (cg == 2 ? kPairAccBufs : 2);
}

template <int CG, int BN, int OB, int BS = 0>
struct Cfg {
    static constexpr int kAccBufs = acc_bufs(CG, BN, BS);
    static constexpr int kBRows = BN / CG;                          // rows of B this CTA loads
    static constexpr int kStages = BS == 2 ? ((CG == 2 && BN == 128) ? 6 : 5)
                                   : BS ? (CG == 2 ? 6 : 5) : ((CG == 1 && BN == 256) ? 4 : 6);
    static constexpr int kABytes = kTileM * kStageKBytes;           // 16 KiB
    static constexpr int kBBytes = kBRows * kStageKBytes;
    // scale-factor blocks of A's 128 rows and the tile's BN columns, per K
    // stage; the stage keeps 1024-byte alignment
    static constexpr int kSfK = BS == 2 ? 4 : 1;                    // blocks per 128 rows and stage
    static constexpr int kSfTxBytes = BS ? kSfK * (512 + 512 * (BN / 128)) : 0;
    static constexpr int kSfBytes = (kSfTxBytes + 1023) / 1024 * 1024;
    static constexpr int kSfCols = BS ? kSfK * (4 + 4 * (BN / 128)) : 0;   // TMEM columns of one stage's factors
    static constexpr int kStageBytes = kABytes + kBBytes + kSfBytes;   // this CTA's share of a stage
    static constexpr int kTxBytes = kABytes + kBBytes + kSfTxBytes;    // bytes one stage's copies bring
    // 64 (16-bit D), 32 (fp32 D), or 64 (e4m3 D with MX factors, stored directly)
    static constexpr int kEpiCols = OB == 1 ? 64 : 128 / OB;
    static constexpr int kSubtiles = BN / kEpiCols;
    static constexpr int kSfCol0 = kAccBufs * BN;                   // first TMEM column of the scale factors
    static constexpr int kTmemCols = BS ? 512 : kAccBufs * BN;
    static_assert(!BS || kSfCol0 + kSfCols * kStages <= 512, "TMEM");
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static constexpr int kRingBytes = kStages * kStageBytes;
    // epilogue staging buffers per warp: two (a store drains while the next
    // subtile fills), one where the ring needs the room (MXFP8 256-wide)
    static constexpr int kEpiBufs = (BS == 1 && BN == 256) ? 1 : 2;
    static constexpr int kEpiBytes = kEpiWarps * kEpiBufs * kEpiBufBytes;
    // Stages are released to the producer in groups: every tcgen05.commit
    // costs the tensor front end cycles that MMAs cannot use, so one commit
    // frees kGroup stages.
    static constexpr int kGroup = (kStages % 2 == 0 && kStages >= 6) ? 2 : 1;
    static constexpr int kGroups = kStages / kGroup;
    // block-scaled kernels: one more warp, which copies each stage's factors
    // into TMEM and signals the MMA thread on a barrier of its own per stage
    static constexpr int kBlockThreads = kThreads + (BS ? 32 : 0);
    static constexpr int kNumBars = 2 * kStages + 4 + 2 * kEpiWarps + 1 + 2 * kClcSlots + (BS ? kStages : 0);
    static constexpr int kSmemBytes =
        1024 /*alignment slack*/ + kRingBytes + kEpiBytes + kClcSlots * 16 + kNumBars * 8 + 16;
    static_assert(kSmemBytes <= 232448, "227 KB of shared memory per CTA");
};

// Index of factors_ready[0] in the barrier block (block-scaled kernels): after
// full[], empty[], the accumulator, C-load and drain barriers and the
// dynamic-schedule ring.
__host__ __device__ constexpr int factor_bar_index(int stages) { return 2 * stages + 4 + 2 * kEpiWarps + 1 + 2 * kClcSlots; }

// A stage's scale-factor slot: shared memory holds A's blocks of the stage,
// then each 128 columns' blocks of B (512 bytes each); TMEM holds A's block j
// at column 4 j of the slot and B's block j of columns 128 jb .. 128 jb + 127
// at 4 kBlocks + 4 (kNB j + jb).
template <int BN, int BS>
struct SfGeom {
    static constexpr uint32_t kNB = BN / 128;                       // 128-column blocks of the tile
    static constexpr uint32_t kBlocks = BS == 2 ? 4u : 1u;          // blocks per 128 rows and stage
    static constexpr uint32_t kCols = 4u * kBlocks * (1u + kNB);    // TMEM columns of one slot
    static constexpr uint32_t kBytes = (512u * kBlocks * (1u + kNB) + 1023u) / 1024u * 1024u;
};
static_assert(SfGeom<256, 1>::kCols == (uint32_t)Cfg<2, 256, 2, 1>::kSfCols &&
                  SfGeom<256, 2>::kCols == (uint32_t)Cfg<2, 256, 2, 2>::kSfCols &&
                  SfGeom<128, 2>::kBytes == (uint32_t)Cfg<1, 128, 2, 2>::kSfBytes &&
                  SfGeom<256, 1>::kBytes == (uint32_t)Cfg<2, 256, 2, 1>::kSfBytes,
              "one factor-slot geometry");


// ------------------------------------------------------------------------
// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile
// (tcgen05 "matrix descriptor": start address, leading- and stride-dimension
// byte offsets, all >> 4; version 1 at bit 46; swizzle mode 2 = 128B at bits
// 61-63).  K-major: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO);
// LBO unused.  MN-major: 128-byte rows along M/N, one row per K index;
// 8-row K groups 1024 bytes apart (SBO), 128-byte-wide M/N chunks LBO apart.
// ------------------------------------------------------------------------
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Bounded wait on phase `parity` of `bar`.  Gives up when another role has
// aborted or after p.timeout_ns; on timeout records `role` in the status word
// and raises the abort flag.  Waiting threads sleep in try_wait (suspend
// hint) rather than re-polling: polling threads slow the barrier and tensor
// front end that the MMA issuer depends on.
// `peer_abort` (0 outside a CTA pair) is the peer CTA's abort flag as a
// shared::cluster address: a timeout raises it too, so the peer stops
// waiting for work that will not come.
constexpr uint32_t kSleepHintNs = 200000;
static __device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, const KernelParams& p,
                                      volatile uint32_t* abort_flag, uint32_t role, uint32_t peer_abort) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1u;
            if (peer_abort) ptx::st_cluster_u32(peer_abort, 1u);
            atomicOr(p.status, kStatusTimeout | role);
            return false;
        }
    }
}

// The same bounded wait, polling instead of sleeping: the load thread waits
// for free stages this way, so a refill starts the moment the MMA releases
// its stages (measured: +1.2 % fused bf16 8192^3, +2 % bf16 4096^3, +0.7 %
// on the 65536 x 256 x 4096 workload over waiting in try_wait).  The timer
// and the abort flag are read every 64 polls.
static __device__ __noinline__ bool poll_bar(uint32_t bar, uint32_t parity, const KernelParams& p,
                                      volatile uint32_t* abort_flag, uint32_t role, uint32_t peer_abort) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_test_wait(bar, parity)) return true;
        if ((n & 63u) == 0u) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > p.timeout_ns) {
                *abort_flag = 1u;
                if (peer_abort) ptx::st_cluster_u32(peer_abort, 1u);
                atomicOr(p.status, kStatusTimeout | role);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag (used to drain in-flight copies
// and MMAs before the CTA releases its resources).
static __device__ __noinline__ bool drain_bar(uint32_t bar, uint32_t parity, const KernelParams& p) {
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            atomicOr(p.status, kStatusTimeout | kStatusRoleDrain);
            return false;
        }
    }
}

// A flattened raster layout evaluated at c in 32-bit arithmetic (tile counts
// fit in int32), its modes unrolled so that every shape and stride is read
// from the parameter bank at a fixed offset: a loop indexed at run time
// turned each tile's lookup into a chain of dependent parameter loads and
// 64-bit divisions, about a microsecond at a CTA's first tile.
__device__ __forceinline__ int raster_eval(const gl::FlatLayout& f, int c) {
    int idx = 0;
#pragma unroll
    for (int i = 0; i < gl::FlatLayout::kMaxModes; ++i) {
        if (i + 1 >= f.rank) {
            idx += c * (int)f.stride[i];
            break;
        }
        const int s = (int)f.shape[i];
        const int q = c / s;
        idx += (c - q * s) * (int)f.stride[i];
        c = q;
    }
    return idx;
}

__device__ __forceinline__ void tile_coords(const KernelParams& p, int tile, int& mb, int& nb, int& l) {
    l = tile / p.tiles_per_batch;
    const int t = tile - l * p.tiles_per_batch;
    const int idx = t < p.raster_full_count ? raster_eval(p.raster_full, t)
                                            : raster_eval(p.raster_tail, t - p.raster_full_count) + p.raster_tail_offset;
    mb = idx % p.tiles_m;
    nb = idx / p.tiles_m;
}

// Where a tile sits: M and N block, batch (group) index, and the tile's row
// range in A, C and D (rows [m_base, m_end) for a grouped GEMM, [0, M)
// otherwise).
struct TilePos {
    int mb, nb, l;
    int m_base, m_end;
    int cd_l;        // batch index of C and D (0 when grouped: one matrix)
    int sf_base;     // first 128-row scale-factor block of A's rows (grouped: the group's)
};

// Group offsets as the kernel reads them: each clamped to [0, M], and group
// g covers [e_(g-1), e_g) with e_g the running maximum of the clamped
// offsets 0..g+1 (e_(-1) the first offset), so groups never overlap and
// every access stays inside A, C and D whatever offsets the caller passes.
__device__ __forceinline__ int clamp_row(const KernelParams& p, int i) {
    const int64_t a = __ldg(p.group_rows + i);
    return (int)(a < 0 ? 0 : (a > p.M ? (int64_t)p.M : a));
}

__device__ __forceinline__ int group_tiles(const KernelParams& p, int r0, int r1, int tile_rows) {
    return (r1 - r0 + tile_rows - 1) / tile_rows * p.tiles_n;
}

// Tiles of every group (grouped GEMM), counted by one warp at the start:
// 32 groups at a time, the running maximum by a warp scan.
__device__ __forceinline__ int grouped_tile_count(const KernelParams& p, int tile_rows, int lane) {
    int carry = clamp_row(p, 0);
    int n = 0;
    for (int c = 0; c < p.groups; c += 32) {
        const int g = c + lane;
        int e = g < p.groups ? clamp_row(p, g + 1) : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, e, off);
            if (lane >= off) e = max(e, o);
        }
        e = max(e, carry);
        int st = __shfl_up_sync(0xffffffffu, e, 1);
        if (lane == 0) st = carry;
        if (g < p.groups) n += group_tiles(p, st, e, tile_rows);
        carry = __shfl_sync(0xffffffffu, e, 31);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
    return n;
}

// A role's walk over the groups: tiles come in increasing order, so the
// group of the next tile is found by moving forward from the last one.
// Block-scaled A keeps each group's factors in whole 128-row blocks, one
// group after another: sf_base counts the blocks of the groups before.
struct GroupWalk {
    int g, base, tiles, r0, r1, sf_base;
};

__device__ __forceinline__ GroupWalk group_walk_make(const KernelParams& p, int tile_rows) {
    GroupWalk w{0, 0, 0, 0, 0, 0};
    if (p.groups > 0) {
        w.r0 = clamp_row(p, 0);
        w.r1 = max(w.r0, clamp_row(p, 1));
        w.tiles = group_tiles(p, w.r0, w.r1, tile_rows);
    }
    return w;
}

__device__ __forceinline__ void tile_pos(const KernelParams& p, GroupWalk& w, int tile, int tile_rows, TilePos& t) {
    if (p.groups == 0) {
        tile_coords(p, tile, t.mb, t.nb, t.l);
        t.m_base = 0;
        t.m_end = p.M;
        t.cd_l = t.l;
        t.sf_base = 0;
        return;
    }
    while (tile >= w.base + w.tiles && w.g + 1 < p.groups) {
        w.base += w.tiles;
        w.sf_base += (w.r1 - w.r0 + 127) / 128;
        ++w.g;
        w.r0 = w.r1;
        w.r1 = max(w.r1, clamp_row(p, w.g + 1));
        w.tiles = group_tiles(p, w.r0, w.r1, tile_rows);
    }
    const int local = tile - w.base;
    const int tm = (w.r1 - w.r0 + tile_rows - 1) / tile_rows;
    t.mb = tm > 0 ? local % tm : 0;
    t.nb = tm > 0 ? local / tm : 0;
    t.l = w.g;
    t.m_base = w.r0;
    t.m_end = w.r1;
    t.cd_l = 0;
    t.sf_base = w.sf_base;
}

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// ---------------------------------------------------------------- work ---
// The sequence of work units (tile, K blocks [kb0, kb1)) of one worker (a CTA,
// or a CTA pair).  Every role of the worker walks the same sequence.  First
// the whole tiles w, w + workers, ... below dp_tiles; then the worker's range
// of the split iterations (K blocks of the tiles from dp_tiles on, tile by
// tile), cut at tile boundaries.  Range r goes to worker workers - 1 - r, so
// the owner of a cut tile (the worker that ran its first K block) waits only
// for workers of lower index, which were launched no later than itself.
struct Sched {
    int tile, step, dp_end, num_kb;
    int64_t it, it_end;
};

__device__ __forceinline__ int64_t sk_range_start(int64_t sk_iters, int64_t r, int ranges) {
    return sk_iters * r / ranges;
}

__device__ __forceinline__ Sched sched_make(const KernelParams& p, int worker, int workers, int dp_tiles) {
    Sched s;
    s.tile = worker;
    s.step = workers;
    s.dp_end = dp_tiles;
    s.num_kb = p.num_kb;
    const int64_t r = workers - 1 - worker;
    if (r < p.sk_ranges) {
        s.it = sk_range_start(p.sk_iters, r, p.sk_ranges);
        s.it_end = sk_range_start(p.sk_iters, r + 1, p.sk_ranges);
    } else {
        s.it = s.it_end = 0;
    }
    return s;
}

__device__ __forceinline__ bool sched_next(Sched& s, int& tile, int& kb0, int& kb1) {
    if (s.tile < s.dp_end) {
        tile = s.tile;
        kb0 = 0;
        kb1 = s.num_kb;
        s.tile += s.step;
        return true;
    }
    if (s.it < s.it_end) {
        const int64_t t = s.it / s.num_kb;
        kb0 = (int)(s.it - t * s.num_kb);
        const int64_t left = s.it_end - s.it;
        kb1 = left < (int64_t)(s.num_kb - kb0) ? kb0 + (int)left : s.num_kb;
        tile = s.dp_end + (int)t;
        s.it += kb1 - kb0;
        return true;
    }
    return false;
}

// Dynamic schedule ("Blackwell Cluster Launch Control": a launch holds one
// cluster per tile; a running cluster that finishes a tile cancels the
// launch of a cluster that has not started and takes its tile, so SMs that
// another kernel holds do not leave their tiles behind).  The load thread of
// the pair's leader issues one request at a time, at the start of each tile,
// and none after a response that cancelled nothing.  The response goes to
// slot n % kClcSlots of every CTA of the cluster; each role (load thread,
// MMA thread, epilogue warps, in both CTAs) reads response n when it
// finishes its n-th tile and then arrives on the leader's empty[slot], which
// the issuer waits on before the slot's next use.
struct Work {
    Sched s;
    bool dyn, producer, first;
    uint32_t n;                   // responses read so far
    uint32_t armed;               // requests this CTA expects (load thread only)
    uint32_t resp0, full0, empty0;   // response slot 0 and its full / empty barriers
    uint32_t rank;
    int cg;
};

__device__ __forceinline__ Work work_make(const KernelParams& p, int worker, int workers, bool producer,
                                          uint32_t resp0, uint32_t full0, uint32_t empty0, uint32_t rank, int cg,
                                          int dp_tiles) {
    Work w;
    w.s = sched_make(p, worker, workers, dp_tiles);
    w.dyn = p.clc != 0;
    w.producer = producer;
    w.first = true;
    w.n = 0;
    w.armed = 0;
    w.resp0 = resp0;
    w.full0 = full0;
    w.empty0 = empty0;
    w.rank = rank;
    w.cg = cg;
    return w;
}

// Request n: this CTA expects 16 bytes on full[slot]; the leader waits for
// the slot's previous response to be read everywhere, then asks.
static __device__ __noinline__ bool clc_request(uint32_t n, uint32_t resp0, uint32_t full0, uint32_t empty0, uint32_t rank,
                                         int cg, const KernelParams& p, volatile uint32_t* abort_flag,
                                         uint32_t peer_abort) {
    const uint32_t slot = n % kClcSlots;
    ptx::mbar_arrive_expect_tx(full0 + 8u * slot, 16);
    if (rank != 0) return true;
    if (n >= kClcSlots &&
        !wait_bar(empty0 + 8u * slot, ((n / kClcSlots) - 1u) & 1u, p, abort_flag, kStatusRoleLoad, peer_abort))
        return false;
    if (cg == 2)
        ptx::clc_try_cancel_mc(resp0 + 16u * slot, full0 + 8u * slot);
    else
        ptx::clc_try_cancel(resp0 + 16u * slot, full0 + 8u * slot);
    return true;
}

// The next work unit of this role.  `arrive`: this thread releases the
// response slot for its role (one thread per role and CTA).
__device__ __forceinline__ bool work_next(Work& w, const KernelParams& p, int& tile, int& kb0, int& kb1,
                                          volatile uint32_t* abort_flag, uint32_t role, uint32_t peer_abort,
                                          bool arrive) {
    if (!w.dyn) return sched_next(w.s, tile, kb0, kb1);
    kb0 = 0;
    kb1 = p.num_kb;
    if (w.first) {
        w.first = false;
        if (*abort_flag) return false;    // the launch already failed: do no work
        tile = w.s.tile;                  // this cluster's own tile
        if (w.producer) {
            w.armed = 1;
            if (!clc_request(0, w.resp0, w.full0, w.empty0, w.rank, w.cg, p, abort_flag, peer_abort)) return false;
        }
        return true;
    }
    const uint32_t slot = w.n % kClcSlots;
    if (!wait_bar(w.full0 + 8u * slot, (w.n / kClcSlots) & 1u, p, abort_flag, role, peer_abort)) return false;
    uint32_t x;
    const bool cancelled = ptx::clc_query(w.resp0 + 16u * slot, x);
    if (arrive) {
        if (w.rank == 0)
            ptx::mbar_arrive(w.empty0 + 8u * slot);
        else
            ptx::mbar_arrive_cluster(w.empty0 + 8u * slot, 0);
    }
    ++w.n;
    if (!cancelled) return false;
    tile = (int)(x / (uint32_t)w.cg);
    if (w.producer) {
        w.armed = w.n + 1;
        if (!clc_request(w.n, w.resp0, w.full0, w.empty0, w.rank, w.cg, p, abort_flag, peer_abort)) return false;
    }
    return true;
}

// Before the load thread leaves: a response that is still on its way must
// land before the CTA's shared memory is released (abort paths only; a
// normal end has read every response).
__device__ __forceinline__ void work_drain(const Work& w, const KernelParams& p) {
    if (!w.dyn || !w.producer || w.armed <= w.n) return;
    const uint32_t last = w.armed - 1;
    drain_bar(w.full0 + 8u * (last % kClcSlots), (last / kClcSlots) & 1u, p);
}

// Partial-sum slot of `worker`, CTA `rank`, epilogue warp `q`: the warp's 32
// accumulator rows, stored so that each warp-wide 16-byte access is one
// contiguous 512-byte run: [subtile][4-column group][lane] float4.
template <int BN>
__device__ __forceinline__ float4* part_slot(const KernelParams& p, int worker, int cg, uint32_t rank, int q) {
    return reinterpret_cast<float4*>(p.sk_part) + ((size_t)(worker * cg + (int)rank) * kEpiWarps + q) * (kEpiRows * BN / 4);
}

__device__ __forceinline__ uint32_t* part_flag(const KernelParams& p, int worker, int cg, uint32_t rank, int q) {
    return p.sk_flags + ((size_t)(worker * cg + (int)rank) * kEpiWarps + q);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* a) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(uint32_t* a, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// Bounded wait (all lanes of a warp) for another worker's partial sum.
static __device__ __noinline__ bool wait_part(const uint32_t* flag, const KernelParams& p, volatile uint32_t* abort_flag,
                                       uint32_t peer_abort) {
    if (ld_acquire(flag)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        __nanosleep(256);
        if (ld_acquire(flag)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1u;
            if (peer_abort) ptx::st_cluster_u32(peer_abort, 1u);
            atomicOr(p.status, kStatusTimeout | kStatusRoleFixup);
            return false;
        }
    }
}

// Column sums of one 16-byte chunk over the warp's 32 rows: lane i holds
// row i's V values.  Halving exchanges (lanes 16, 8, ... apart) leave each
// lane the sum of one column over the lanes that share its high bits; the
// remaining steps sum across the rest.  Returns that column sum; `j` is its
// column within the chunk.  Lanes whose low log2(32/V) bits are zero hold
// distinct columns.  Fixed order: the sums are the same on every run.
template <int V>
__device__ __forceinline__ float chunk_col_sum(float (&r)[V], int lane, int& j) {
    j = 0;
    int off = 16;
#pragma unroll
    for (int width = V; width > 1; width >>= 1, off >>= 1) {
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < width / 2; ++i) {
            const float send = hi ? r[i] : r[width / 2 + i];
            const float keep = hi ? r[width / 2 + i] : r[i];
            r[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        if (hi) j += width / 2;
    }
#pragma unroll
    for (; off >= 1; off >>= 1) r[0] += __shfl_xor_sync(0xffffffffu, r[0], off);
    return r[0];
}

__device__ __forceinline__ void unpack2(uint32_t w, bool f16, float& lo, float& hi) {
    if (f16) {
        const __half2 h = *reinterpret_cast<const __half2*>(&w);
        const float2 f = __half22float2(h);
        lo = f.x;
        hi = f.y;
    } else {
        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w);
        const float2 f = __bfloat1622float2(h);
        lo = f.x;
        hi = f.y;
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool f16) {
    uint32_t w;
    if (f16) {
        const __half2 h = __floats2half2_rn(lo, hi);
        w = *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        w = *reinterpret_cast<const uint32_t*>(&h);
    }
    return w;
}

// One staged subtile of the plain epilogue: the warp's 32 rows by 128 / OB
// columns, t = alpha*acc (+ beta*C, C read from the staging slot the TMA load
// filled) (+ the column or row bias) (ReLU), rounded once to the output type
// and written back into the same swizzled 128-byte rows (16-byte chunk c of
// row r at chunk c ^ (r % 8)).  The operations and their order are those of
// the general chunk loop, so both give the same bits; this form has no
// per-chunk branches and far less code, which measured 4 to 5 times faster
// per subtile.  BIAS 1 (column bias): lane i holds the bias of columns i and
// 32 + i of the subtile (0 past N) and each column's value is broadcast from
// its lane; BIAS 2: row_bias is the bias of the lane's row.
template <int OB, bool HAS_C, int BIAS, bool RELU>
__device__ __forceinline__ void stage_subtile(const uint32_t (&acc)[128 / OB], uint8_t* row_base, int lane,
                                              float alpha, float beta, float b_lo, float b_hi, float row_bias,
                                              bool f16) {
    constexpr int VPC = 16 / OB;                        // values per 16-byte chunk
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint4* slot = reinterpret_cast<uint4*>(row_base + ((ch ^ (lane & 7)) << 4));
        float v[VPC];
#pragma unroll
        for (int i = 0; i < VPC; ++i) v[i] = alpha * __uint_as_float(acc[ch * VPC + i]);
        if constexpr (HAS_C) {
            const uint4 craw = *slot;
            const uint32_t w[4] = {craw.x, craw.y, craw.z, craw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if constexpr (OB == 4) {
                    v[i] = fmaf(beta, __uint_as_float(w[i]), v[i]);
                } else {
                    float lo, hi;
                    unpack2(w[i], f16, lo, hi);
                    v[2 * i] = fmaf(beta, lo, v[2 * i]);
                    v[2 * i + 1] = fmaf(beta, hi, v[2 * i + 1]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < VPC; ++i) {
            if constexpr (BIAS == 1) {
                constexpr int kLanes = 32;
                const int j = ch * VPC + i;
                v[i] += __shfl_sync(0xffffffffu, j < kLanes ? b_lo : b_hi, j % kLanes);
            } else if constexpr (BIAS == 2) {
                v[i] += row_bias;
            }
            if constexpr (RELU) v[i] = fmaxf(v[i], 0.f);
        }
        if constexpr (OB == 4)
            *slot = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                               __float_as_uint(v[3]));
        else
            *slot = make_uint4(pack2(v[0], v[1], f16), pack2(v[2], v[3], f16), pack2(v[4], v[5], f16),
                               pack2(v[6], v[7], f16));
    }
}

// The values t = alpha*acc (+ the column or row bias) (ReLU) of N whole
// columns j0 .. j0 + N - 1 of a subtile (all inside D), for the block-scaled
// outputs; the same operations in the same order as their general loop, with
// no per-element tests.  BIAS 1: lane i holds the bias of subtile columns i
// and 32 + i, broadcast by shuffle.
template <int N, int BIAS, bool RELU>
__device__ __forceinline__ void block_values(const uint32_t* acc, int j0, float alpha, float b_lo, float b_hi,
                                             float row_bias, float (&v)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        float x = alpha * __uint_as_float(acc[i]);
        if constexpr (BIAS == 1) {
            constexpr int kLanes = 32;
            const int j = j0 + i;
            x += __shfl_sync(0xffffffffu, j < kLanes ? b_lo : b_hi, j % kLanes);
        } else if constexpr (BIAS == 2) {
            x += row_bias;
        }
        if constexpr (RELU) x = fmaxf(x, 0.f);
        v[i] = x;
    }
}

// block_values for a bias mode and activation known at run time
template <int N>
__device__ __forceinline__ void block_values_for(int bias_mode, bool relu, const uint32_t* acc, int j0, float alpha,
                                                 float b_lo, float b_hi, float row_bias, float (&v)[N]) {
    switch (bias_mode * 2 + (relu ? 1 : 0)) {
        case 0: block_values<N, 0, false>(acc, j0, alpha, b_lo, b_hi, row_bias, v); break;
        case 1: block_values<N, 0, true>(acc, j0, alpha, b_lo, b_hi, row_bias, v); break;
        case 2: block_values<N, 1, false>(acc, j0, alpha, b_lo, b_hi, row_bias, v); break;
        case 3: block_values<N, 1, true>(acc, j0, alpha, b_lo, b_hi, row_bias, v); break;
        case 4: block_values<N, 2, false>(acc, j0, alpha, b_lo, b_hi, row_bias, v); break;
        default: block_values<N, 2, true>(acc, j0, alpha, b_lo, b_hi, row_bias, v); break;
    }
}

// tcgen05 instruction descriptor (kind::f16 / kind::f8f6f4, dense): D fp32
// (bits 4-5 = 1), A and B type (bits 7-9, 10-12: f16 0 / bf16 1 for kind::f16,
// e4m3 0 for kind::f8f6f4), A / B MN-major (bits 15, 16), N >> 3 (bits
// 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_for(int cg, int bn, bool f8, uint32_t bf16, uint32_t a_mn,
                                                 uint32_t b_mn) {
    return (1u << 4) | ((f8 ? 0u : bf16) << 7) | ((f8 ? 0u : bf16) << 10) | (a_mn << 15) | (b_mn << 16) |
           ((uint32_t)(bn >> 3) << 17) | ((uint32_t)((128 * cg) >> 4) << 24);
}

// Instruction descriptor for kind::mxf8f6f4 with block scaling: scale-factor
// byte of B (bits 4-5), A and B e4m3 (type 0, bits 7-9, 10-12), A / B
// MN-major (15, 16), N >> 3 (17-22), ue8m0 scale factors (bit 23), M >> 4
// (24-28), scale-factor byte of A (29-30).  The bytes select which of the
// four factors in a TMEM word (four 32-element K blocks) an MMA uses.
__host__ __device__ constexpr uint32_t idesc_mx(int cg, int bn, uint32_t a_mn, uint32_t b_mn, uint32_t sf_byte) {
    return (sf_byte << 4) | (a_mn << 15) | (b_mn << 16) | ((uint32_t)(bn >> 3) << 17) | (1u << 23) |
           ((uint32_t)((128 * cg) >> 4) << 24) | (sf_byte << 29);
}

// Instruction descriptor for kind::mxf4nvf4 with 16-element scale vectors
// (scale_vec::4X): A and B e2m1 (type 1 of this kind, bits 7-9, 10-12), both
// K-major, N >> 3 (17-22), ue4m3 scale factors (bit 23 clear), M >> 4
// (24-28).  Each MMA (K = 64) reads all four factor bytes of its TMEM words,
// so the factor byte selectors stay 0.
__host__ __device__ constexpr uint32_t idesc_nv(int cg, int bn) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)((128 * cg) >> 4) << 24);
}

// Shared-memory descriptor of a 512-byte scale-factor block read as 32 rows
// of 16 bytes, no swizzle: 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t sf_desc(uint32_t addr) {
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// ------------------------------------------------------- NVFP4 output ---
// Round-to-nearest-even of exact quotients onto the e4m3 and e2m1 grids,
// decided by comparisons rather than by a rounded division: x / y lies
// above a midpoint m of the grid exactly when x > m * y, and with m * y'
// exact in fp32 (a midpoint has at most 5 significant bits) the sign of
// fmaf(m y', g, -x) is the sign of the exact m * y' * g - x (the product is
// not rounded inside the FMA, the one rounding keeps sign and zero).  So the
// codes are those of the real quotients of the fp32 values, ties to the even
// code, whatever rounding a division would have added.

// Value of a non-negative e4m3 code (0 .. 0x7E).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const uint32_t fe = c >> 3, fm = c & 7u;
    return fe ? __uint_as_float(((fe + 120u) << 23) | (fm << 20)) : (float)fm * 0.001953125f;   // m * 2^-9
}

// ue4m3 factor of an NVFP4 output block: e4m3(amax / (6 g)), nearest even,
// saturating at 448 (code 0x7E).  amax finite and >= 0, g normal and > 0,
// inv6g a rounded 1 / (6 g).  The candidate amax * inv6g is within one code
// of the exact result (its error is a few 2^-24 of the quotient, the grid's
// spacing at least 2^-3 of it, and past 448 every code saturates); the
// midpoints on either side settle it.
__device__ __forceinline__ uint32_t nv_factor_code(float amax, float g, float inv6g) {
    uint32_t c = ptx::pack4_e4m3(__fmul_rn(amax, inv6g), 0.f, 0.f, 0.f) & 0xFFu;
    if (c > 0u) {
        const float lo6 = 3.0f * (e4m3_value(c - 1u) + e4m3_value(c));        // 6 x the lower midpoint, exact
        const float s = __fmaf_rn(lo6, g, -amax);
        if (s > 0.f || (s == 0.f && (c & 1u))) return c - 1u;
    }
    if (c < 0x7Eu) {
        const float hi6 = 3.0f * (e4m3_value(c) + e4m3_value(c + 1u));
        const float s = __fmaf_rn(hi6, g, -amax);
        if (s < 0.f || (s == 0.f && (c & 1u))) return c + 1u;
    }
    return c;
}

// e2m1 codes of 16 values under factor value f > 0 and global scale g:
// e2m1(v / (f g)), nearest even, saturating at 6, sign in bit 3; packed two
// per byte, the lower index in the low nibble.  The magnitude code is the
// number of midpoints (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) below |v| / (f g),
// a midpoint that |v| / (f g) equals counting when the code below it is odd
// (ties to even); three comparisons find it, one per bit, and every midpoint
// compared at one level has the same parity.
__device__ __forceinline__ uint2 nv_element_codes(const float (&v)[16], float f, float g) {
    const float t0 = 0.25f * f, t1 = 0.75f * f, t2 = 1.25f * f, t3 = 1.75f * f;
    const float t4 = 2.5f * f, t5 = 3.5f * f, t6 = 5.0f * f;     // exact: at most 7 significant bits
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = fabsf(v[i]);
        const bool b2 = __fmaf_rn(t3, g, -a) <= 0.f;                       // at or past 1.75: code >= 4
        const bool b1 = __fmaf_rn(b2 ? t5 : t1, g, -a) <= 0.f;            // past 3.5 / 0.75 (odd below)
        const float tl = b2 ? (b1 ? t6 : t4) : (b1 ? t2 : t0);
        const bool b0 = __fmaf_rn(tl, g, -a) < 0.f;                        // past 5, 2.5, 1.25, 0.25 (even below)
        const uint32_t mag = a > 0.f ? (b2 ? 4u : 0u) | (b1 ? 2u : 0u) | (b0 ? 1u : 0u) : 0u;
        const uint32_t code = mag | (__float_as_uint(v[i]) >> 28 & 8u);
        w[i >> 3] |= code << ((i & 7) * 4);
    }
    return make_uint2(w[0], w[1]);
}

// The same codes, fast: x = v * r with r a rounded 1 / (f g) is within
// 4 * 2^-24 of the exact quotient (relative), so rounding x nudged down and
// up by 2^-20 gives the same e2m1 codes exactly when no rounding midpoint
// lies within that band, and then they are the codes of the exact quotient
// too.  A block where any code differs (a quotient at or next to a midpoint)
// is decided by the comparisons above.  f g below 2^-100 (where r would lose
// precision or overflow) always takes the comparisons.
__device__ __forceinline__ uint2 nv_element_codes_fast(const float (&v)[16], float f, float g) {
    const float fg = __fmul_rn(f, g);
    if (fg < 7.88860905e-31f) return nv_element_codes(v, f, g);
    const float r = __frcp_rn(fg);
    const float r_lo = __fmul_rn(r, 1.0f - 9.5367431640625e-07f), r_hi = __fmul_rn(r, 1.0f + 9.5367431640625e-07f);
    float lo[16], hi[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        lo[i] = __fmul_rn(v[i], r_lo);
        hi[i] = __fmul_rn(v[i], r_hi);
    }
    const uint2 a = make_uint2(ptx::pack8_e2m1(lo), ptx::pack8_e2m1(lo + 8));
    const uint2 b = make_uint2(ptx::pack8_e2m1(hi), ptx::pack8_e2m1(hi + 8));
    if (a.x == b.x && a.y == b.y) return a;
    return nv_element_codes(v, f, g);
}

// What the MMA issuer needs from the kernel.
template <int CG, int BN, int S>
struct MmaCtx {
    const KernelParams& p;
    uint32_t ring;          // shared address of stage 0
    uint32_t a_bytes;       // A tile bytes at the front of a stage
    uint32_t stage_bytes;
    uint32_t bar0;          // barrier block
    uint32_t tmem_base;
    int first_tile, tile_step;
    volatile uint32_t* abort_flag;
    uint32_t peer_abort;
    uint32_t resp0, clc_full0, clc_empty0;   // dynamic schedule ring
    int dp_tiles;           // whole tiles of the launch (counted in the kernel when grouped)
};

// The MMA issuer (one thread of the pair leader).  A tcgen05.mma blocks its
// issuing thread until the tensor core takes it (the queue is about one
// instruction deep), so any work between two MMAs is tensor-pipe idle time:
// the loop asks for the next stage's barrier (non-blocking) once the current
// stage's MMAs are queued, so the question comes as late as it can and is
// answered "ready" more often than right after the first MMA (bf16 4096^3
// +1.9 %); it builds descriptors by adding offsets to a precomputed base and
// carries the instruction descriptor as an immediate.
//
// Every scalar the loop reads is copied into a register first.  The tcgen05
// and mbarrier wrappers clobber "memory", so a value read through `m` or `p`
// (local and kernel-parameter memory behind a reference) would be re-loaded
// after every MMA, a chain of dependent loads between two MMAs.
//
// BS: block-scaled MMAs.  Each stage's scale-factor blocks sit in TMEM (one
// slot of columns per stage after the accumulators), put there by the copier
// (factor_copier) before this thread sees the stage as ready.  MXFP8 (BS = 1):
// one block each for A and for every 128 columns of B, 4 columns apiece; MMA
// j (32 elements of K) reads factor byte j of each word.  NVFP4 (BS = 2): four
// blocks each, and MMA j (64 elements of K) reads the whole words of block j.
template <int CG, int BN, int S, int G, bool F8, uint32_t IDESC, int BS = 0>
__device__ __noinline__ void mma_role(const MmaCtx<CG, BN, S>& m) {
    const KernelParams& p = m.p;                 // slow paths (wait_bar) only
    const int first_tile = m.first_tile, tile_step = m.tile_step;
    const uint32_t bar0 = m.bar0, ring = m.ring, a_bytes = m.a_bytes, stage_bytes = m.stage_bytes;
    const uint32_t tmem_base = m.tmem_base, peer_abort = m.peer_abort;
    volatile uint32_t* const abort_flag = m.abort_flag;
    constexpr int kAccBufs = acc_bufs(CG, BN, BS);
    // block-scaled: a stage is ready once the copier has put its factors in
    // TMEM (after its data landed); otherwise once its data landed
    auto full_bar = [=](int s) { return bar0 + 8u * ((BS ? factor_bar_index(S) : 0) + s); };
    auto empty_bar = [=](int s) { return bar0 + 8u * (S + s); };
    auto accf_bar = [=](int b) { return bar0 + 8u * (2 * S + b); };
    auto acce_bar = [=](int b) { return bar0 + 8u * (2 * S + 2 + b); };
    const uint32_t drain = bar0 + 8u * (2 * S + 4 + 2 * kEpiWarps);
    constexpr bool a_mn = (IDESC >> 15) & 1u, b_mn = (IDESC >> 16) & 1u;
    constexpr int eb = F8 ? 1 : 2;
    constexpr int kel = kStageKBytes / eb;
    // per-K-step advance of the descriptors' start address, in 16-byte units
    constexpr uint32_t a_step = (a_mn ? (kKStepBytes / eb) * 128u : kKStepBytes) >> 4;
    constexpr uint32_t b_step = (b_mn ? (kKStepBytes / eb) * 128u : kKStepBytes) >> 4;
    // shared addresses stay below 2^18, so offsets added to the 14-bit
    // start-address field never carry into the other fields
    const uint64_t a_base = smem_desc(ring, a_mn ? (uint32_t)(kel * 128) : 16u, 1024u);
    const uint64_t b_base = smem_desc(ring + a_bytes, b_mn ? (uint32_t)(kel * 128) : 16u, 1024u);
    // One commit releases a whole group of G stages (empty[] is indexed by
    // group); the commit covers every earlier MMA of this thread.
    auto release = [=](int g) {
        if constexpr (CG == 2)
            ptx::mma_commit_mc(empty_bar(g), 0x3);
        else
            ptx::mma_commit(empty_bar(g));
    };
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool issued = false;
    bool ready = ptx::mbar_test_wait(full_bar(0), 0);
    Work wk = work_make(p, first_tile, tile_step, false, m.resp0, m.clc_full0, m.clc_empty0, 0u, CG, m.dp_tiles);
    int tile, kb0, kb1;
    for (; work_next(wk, p, tile, kb0, kb1, abort_flag, kStatusRoleMma, peer_abort, true); ++it) {
        const int buf = it % kAccBufs;
        const uint32_t acc_par = (uint32_t)(it / kAccBufs) & 1u;
        if (!wait_bar(acce_bar(buf), acc_par ^ 1u, p, abort_flag, kStatusRoleMma, peer_abort)) break;
        ptx::tc_fence_after();   // the epilogue's reads of this accumulator come first
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        bool stop = false;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!ready && !wait_bar(full_bar(stage), phase, p, abort_flag, kStatusRoleMma, peer_abort)) {
                stop = true;
                break;
            }
            if (!issued) GEMM_STAMP(p, 3);
            const int next = stage + 1 == S ? 0 : stage + 1;
            const uint32_t next_phase = stage + 1 == S ? phase ^ 1u : phase;
            const uint64_t soff = (uint64_t)((stage * stage_bytes) >> 4);
            const uint64_t ad = a_base + soff, bd = b_base + soff;
            const uint32_t first = kb != kb0;
            if constexpr (BS == 2) {
                using SG = SfGeom<BN, BS>;
                constexpr uint32_t kNB = SG::kNB;
                const uint32_t sfa = tmem_base + (uint32_t)(kAccBufs * BN) + SG::kCols * (uint32_t)stage;
                const uint32_t sfb = sfa + 4u * SG::kBlocks;
                // (NVFP4's short stages: asking after the first MMA measures better)
                ptx::mma_nv<CG, IDESC>(d_tmem, ad, bd, sfa, sfb, first);
                ready = ptx::mbar_test_wait(full_bar(next), next_phase);
                ptx::mma_nv<CG, IDESC>(d_tmem, ad + a_step, bd + b_step, sfa + 4u, sfb + 4u * kNB, 1u);
                ptx::mma_nv<CG, IDESC>(d_tmem, ad + 2 * a_step, bd + 2 * b_step, sfa + 8u, sfb + 8u * kNB, 1u);
                ptx::mma_nv<CG, IDESC>(d_tmem, ad + 3 * a_step, bd + 3 * b_step, sfa + 12u, sfb + 12u * kNB, 1u);
            } else if constexpr (BS == 1) {
                using SG = SfGeom<BN, BS>;
                const uint32_t sfa = tmem_base + (uint32_t)(kAccBufs * BN) + SG::kCols * (uint32_t)stage;
                const uint32_t sfb = sfa + 4u * SG::kBlocks;
                ptx::mma_mx<CG, IDESC>(d_tmem, ad, bd, sfa, sfb, first);
                ptx::mma_mx<CG, IDESC | (1u << 4) | (1u << 29)>(d_tmem, ad + a_step, bd + b_step, sfa, sfb, 1u);
                ptx::mma_mx<CG, IDESC | (2u << 4) | (2u << 29)>(d_tmem, ad + 2 * a_step, bd + 2 * b_step, sfa, sfb, 1u);
                ptx::mma_mx<CG, IDESC | (3u << 4) | (3u << 29)>(d_tmem, ad + 3 * a_step, bd + 3 * b_step, sfa, sfb, 1u);
                ready = ptx::mbar_test_wait(full_bar(next), next_phase);
            } else {
#pragma unroll
                for (int j = 0; j < kStageKBytes / kKStepBytes; ++j) {
                    ptx::mma_imm<CG, F8, IDESC>(d_tmem, ad + j * a_step, bd + j * b_step, j ? 1u : first);
                    if (j == kStageKBytes / kKStepBytes - 1) ready = ptx::mbar_test_wait(full_bar(next), next_phase);
                }
            }
            issued = true;
            if (stage % G == G - 1) release(stage / G);   // the group's last stage
            stage = next;
            phase = next_phase;
        }
        if (stop) break;
        if (kb1 > kb0) {                         // accumulator complete
            if constexpr (CG == 2)
                ptx::mma_commit_mc(accf_bar(buf), 0x3);
            else
                ptx::mma_commit(accf_bar(buf));
            if (it == 0) GEMM_STAMP(p, 4);
        } else {                                  // K == 0: nothing accumulated
            ptx::mbar_arrive(accf_bar(buf));
            if constexpr (CG == 2) ptx::mbar_arrive_cluster(accf_bar(buf), 1);
        }
    }
    // A group left partly issued is released too, so a producer waiting to
    // drain its copies is not left waiting.
    if (issued && stage % G != 0) release(stage / G);
    // Drain: every MMA issued above must finish before TMEM is freed.
    if (issued) {
        if constexpr (CG == 2)
            ptx::mma_commit_cg2(drain);
        else
            ptx::mma_commit(drain);
        drain_bar(drain, 0, p);
    }
}

// The scale-factor copier of a block-scaled kernel (one thread of the pair
// leader, warp 6).  It walks the same work units as the MMA thread; for each
// stage it waits until the stage's data has landed (full[s]), copies the
// stage's factor blocks into the stage's TMEM slot with tcgen05.cp
// (cta_group::2: each CTA's blocks into its own TMEM) and commits them to
// factors_ready[s], the barrier the MMA thread waits on.  Issued from the MMA
// thread, the copies ran in its issue order between MMAs, about 40 % of an
// NVFP4 stage's tensor time (twelve copies per stage); from this thread they
// overlap the MMAs (NVFP4 8192^3 3242 -> 3974 TFLOP/s, MXFP8 unchanged).
// A slot is rewritten only after full[s] fires for the stage's next fill,
// which follows the MMA thread's release of that stage, so no copy lands
// under an MMA still reading the slot.  Before it leaves, the copier waits
// for its last commit, so no copy is in flight when TMEM is freed.
template <int CG, int BN, int S, int BS>
__device__ __noinline__ void factor_copier(const MmaCtx<CG, BN, S>& m) {
    using G = SfGeom<BN, BS>;
    const KernelParams& p = m.p;
    const uint32_t bar0 = m.bar0, ring = m.ring, stage_bytes = m.stage_bytes, peer_abort = m.peer_abort;
    const uint32_t slot0 = m.tmem_base + (uint32_t)(acc_bufs(CG, BN, BS) * BN);
    const uint32_t ready0 = bar0 + 8u * factor_bar_index(S);
    volatile uint32_t* const abort_flag = m.abort_flag;
    Work wk = work_make(p, m.first_tile, m.tile_step, false, m.resp0, m.clc_full0, m.clc_empty0, 0u, CG, m.dp_tiles);
    int stage = 0, last = -1;
    uint32_t phase = 0, last_phase = 0;
    int tile, kb0, kb1;
    bool stop = false;
    while (!stop && work_next(wk, p, tile, kb0, kb1, abort_flag, kStatusRoleCopy, peer_abort, true)) {
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!ptx::mbar_try_wait(bar0 + 8u * stage, phase) &&
                !wait_bar(bar0 + 8u * stage, phase, p, abort_flag, kStatusRoleCopy, peer_abort)) {
                stop = true;
                break;
            }
            const uint32_t sfs = ring + (uint32_t)stage * stage_bytes + stage_bytes - G::kBytes;
            const uint32_t sfa = slot0 + G::kCols * (uint32_t)stage, sfb = sfa + 4u * G::kBlocks;
#pragma unroll
            for (uint32_t j = 0; j < G::kBlocks; ++j) {
                ptx::tmem_cp_32x128b_x4<CG>(sfa + 4u * j, sf_desc(sfs + 512u * j));
#pragma unroll
                for (uint32_t jb = 0; jb < G::kNB; ++jb)
                    ptx::tmem_cp_32x128b_x4<CG>(sfb + 4u * (G::kNB * j + jb),
                                                sf_desc(sfs + 512u * G::kBlocks * (1u + jb) + 512u * j));
            }
            if constexpr (CG == 2)
                ptx::mma_commit_cg2(ready0 + 8u * stage);
            else
                ptx::mma_commit(ready0 + 8u * stage);
            last = stage;
            last_phase = phase;
            phase = stage + 1 == S ? phase ^ 1u : phase;
            stage = stage + 1 == S ? 0 : stage + 1;
        }
    }
    if (last >= 0) drain_bar(ready0 + 8u * last, last_phase, p);
    ptx::tc_fence_before();
}

template <int CG, int BN, int OB, int BS = 0>
__global__ void __launch_bounds__(Cfg<CG, BN, OB, BS>::kBlockThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                const __grid_constant__ KernelParams p) {
    using C = Cfg<CG, BN, OB, BS>;
    constexpr int S = C::kStages;
    constexpr int kTileRows = kTileM * CG;               // output rows per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint8_t* epi = ring + C::kRingBytes;
    uint8_t* clc_resp = epi + C::kEpiBytes;             // kClcSlots x 16 bytes
    uint64_t* bars = reinterpret_cast<uint64_t*>(clc_resp + kClcSlots * 16);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
    auto cfull_bar = [&](int i) { return bar0 + 8u * (2 * S + 4 + i); };
    const uint32_t drain = bar0 + 8u * (2 * S + 4 + 2 * kEpiWarps);
    const uint32_t clc_full0 = drain + 8u, clc_empty0 = drain + 8u * (1 + kClcSlots);
    const uint32_t resp0 = ptx::smem_addr(clc_resp);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA pair bookkeeping (CG == 2): rank 0 is the leader that issues MMAs.
    const uint32_t rank = CG == 2 ? ptx::cluster_ctarank() : 0u;
    const int first_tile = CG == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int tile_step = CG == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const uint32_t peer_abort = CG == 2 ? ptx::mapa(ptx::smem_addr(tmem_slot + 1), rank ^ 1u) : 0u;

    if (threadIdx.x == 0) {
        GEMM_STAMP(p, 0);
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf_bar(b), 1);
            ptx::mbar_init(acce_bar(b), kEpiWarps * CG);   // every epilogue warp of the pair
        }
        for (int i = 0; i < 2 * kEpiWarps; ++i) ptx::mbar_init(cfull_bar(i), 1);
        ptx::mbar_init(drain, 1);
        if constexpr (BS != 0)
            for (int s = 0; s < S; ++s) ptx::mbar_init(bar0 + 8u * (factor_bar_index(S) + s), 1);
        // A dynamic launch starts clusters that nobody cancelled once others
        // leave; after a recorded error they do no work (no chain of timeouts).
        *abort_flag = p.clc && *reinterpret_cast<volatile uint32_t*>(p.status) != 0u ? 1u : 0u;
        for (int i = 0; i < kClcSlots; ++i) {
            ptx::mbar_init(clc_full0 + 8u * i, 1);
            // readers of a response: load thread, MMA thread (leader), the
            // factor copier (leader, block-scaled) and the four epilogue
            // warps of each CTA
            ptx::mbar_init(clc_empty0 + 8u * i, (CG == 2 ? 2 * (1 + kEpiWarps) + 1 : 2 + kEpiWarps) + (BS ? 1 : 0));
        }
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmD);
        if (p.has_c) ptx::prefetch_tensormap(&tmC);
        if constexpr (BS) {
            ptx::prefetch_tensormap(&tmSA);
            ptx::prefetch_tensormap(&tmSB);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    // grouped GEMM: the launch's tiles, from the group offsets in device memory
    if (warp == 2 && p.groups > 0) {
        const int n = grouped_tile_count(p, kTileRows, lane);
        if (lane == 0) tmem_slot[2] = (uint32_t)n;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) ptx::cluster_sync();   // the peer's barriers exist before anyone signals them
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int dp_tiles = p.groups > 0 ? (int)tmem_slot[2] : p.dp_tiles;
    if (threadIdx.x == 0) GEMM_STAMP(p, 1);

    if (warp == 0) {
        // ------------------------------------------------------ TMA loads --
        if (lane == 0) {
            const int eb = p.elem_bytes;
            const int kel = kStageKBytes / eb;          // K elements per stage
            const int mn_box = kStageKBytes / eb;       // M/N elements per 128-byte row (MN-major)
            // Latest fill of each stage (single CTA: drained on full[s]) or of
            // each release group (pair: drained on empty[g], which a later
            // fill of any stage of the group moves on).
            // (bit masks, so they stay in registers)
            uint32_t pend = 0u, pend_parity = 0u;
            auto pend_slot = [&](int st) { return CG == 2 ? st / C::kGroup : st; };
            int stage = 0;
            uint32_t phase = 0;
            bool skip_first = p.inject != 0 && rank == 0;
            Work wk = work_make(p, first_tile, tile_step, true, resp0, clc_full0, clc_empty0, rank, CG, dp_tiles);
            GroupWalk gw = group_walk_make(p, kTileRows);
            int tile, kb0, kb1;
            while (work_next(wk, p, tile, kb0, kb1, abort_flag, kStatusRoleLoad, peer_abort, true)) {
                TilePos tp;
                tile_pos(p, gw, tile, kTileRows, tp);
                const int mb = tp.mb, nb = tp.nb, l = tp.l;
                const int la = p.a_batched ? l : 0, lb = p.b_batched ? l : 0;
                const int m0 = tp.m_base + mb * kTileRows + (int)rank * kTileM;
                // 128-row factor block of this CTA's A rows (a group's own blocks when grouped)
                [[maybe_unused]] const int a_sfblk = tp.sf_base + (m0 - tp.m_base) / 128;
                const int n0 = nb * BN + (int)rank * C::kBRows;
                bool stop = false;
                for (int kb = kb0; kb < kb1; ++kb) {
                    // a group of stages is released together: wait at its first stage
                    if (stage % C::kGroup == 0 && !ptx::mbar_test_wait(empty_bar(stage / C::kGroup), phase ^ 1u) &&
                        !poll_bar(empty_bar(stage / C::kGroup), phase ^ 1u, p, abort_flag, kStatusRoleLoad, peer_abort)) {
                        stop = true;
                        break;
                    }
                    if (skip_first) {
                        skip_first = false;       // test hook: this stage is never filled
                    } else {
                        // the pair's leader counts both CTAs' bytes
                        const uint32_t fb = CG == 2 ? ptx::mapa(full_bar(stage), 0) : full_bar(stage);
                        if (rank == 0) ptx::mbar_arrive_expect_tx(full_bar(stage), C::kTxBytes * CG);
                        const uint32_t sa = ptx::smem_addr(ring + stage * C::kStageBytes);
                        const uint32_t sb = sa + C::kABytes;
                        const int k0 = kb * kel;
                        auto load = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2) {
                            if constexpr (CG == 2)
                                ptx::tma_load_3d_cg2(dst, map, c0, c1, c2, fb);
                            else
                                ptx::tma_load_3d(dst, map, c0, c1, c2, fb);
                        };
                        if (p.a_kmajor) {
                            load(sa, &tmA, k0, m0, la);
                        } else {
                            for (int c = 0; c < kTileM / mn_box; ++c) load(sa + c * (kel * 128), &tmA, m0 + c * mn_box, k0, la);
                        }
                        if (p.b_kmajor) {
                            load(sb, &tmB, k0, n0, lb);
                        } else {
                            for (int c = 0; c < C::kBRows / mn_box; ++c)
                                load(sb + c * (kel * 128), &tmB, n0 + c * mn_box, k0, lb);
                        }
                        if constexpr (BS == 2) {
                            // Four 512-byte blocks per 128 rows and K stage, one box of
                            // eight 256-byte rows at (K block 4 kb, 128-row block); B's
                            // box spans the tile's BN / 128 row blocks (one copy)
                            const uint32_t sf = sb + C::kBBytes;
                            load(sf, &tmSA, 0, kb * 8, la * p.sf_mblocks + a_sfblk);
                            load(sf + 2048, &tmSB, 0, kb * 8, lb * p.sf_nblocks + nb * BN / 128);
                        } else if constexpr (BS == 1) {
                            // One 512-byte scale-factor block per 128 rows and K stage:
                            // block (rows / 128) * num_kb + kb of the batch's tensor, read
                            // as 2 rows of 256 bytes.  Each CTA takes its own A rows'
                            // block and the blocks of the tile's whole N range, the
                            // latter in one copy through a 4-D view (K block kb of
                            // BN / 128 adjacent 128-column blocks): every TMA
                            // instruction costs the copy engine time apart from its
                            // bytes (three copies per stage instead of four: MXFP8
                            // 8192^3 2705 -> 2852 TFLOP/s).  A block past N multiplies
                            // zero-filled B columns only.
                            const uint32_t sf = sb + C::kBBytes;
                            const int blk_a = (la * p.sf_mblocks + a_sfblk) * p.num_kb + kb;
                            load(sf, &tmSA, 0, blk_a * 2, 0);
                            if constexpr (CG == 2)
                                ptx::tma_load_4d_cg2(sf + 512, &tmSB, 0, 0, kb, lb * p.sf_nblocks + nb * BN / 128, fb);
                            else
                                ptx::tma_load_4d(sf + 512, &tmSB, 0, 0, kb, lb * p.sf_nblocks + nb * BN / 128, fb);
                        }
                        const uint32_t bit = 1u << pend_slot(stage);
                        if (!pend) GEMM_STAMP(p, 2);
                        pend |= bit;
                        pend_parity = phase ? (pend_parity | bit) : (pend_parity & ~bit);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (stop) break;
            }
            // Every issued copy must land before the CTA may exit.  In a pair
            // the copies complete on the leader's barrier, so each CTA waits
            // for the MMA to have consumed its stages instead.
            for (int s = 0; s < S; ++s)
                if ((pend >> s) & 1u) {
                    const uint32_t par = (pend_parity >> s) & 1u;
                    bool ok_drain;
                    if constexpr (CG == 2)
                        ok_drain = drain_bar(empty_bar(s), par, p);   // s indexes a group here
                    else
                        ok_drain = drain_bar(full_bar(s), par, p);
                    if (!ok_drain) break;   // already past the time bound: stop waiting
                }
            work_drain(wk, p);
        }
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA -----
        if (lane == 0 && rank == 0) {
            MmaCtx<CG, BN, S> m{p,          ptx::smem_addr(ring), C::kABytes, C::kStageBytes, bar0,
                                tmem_base,  first_tile,           tile_step,   abort_flag,       peer_abort,
                                resp0,      clc_full0,            clc_empty0,  dp_tiles};
            if constexpr (BS == 2) {
                mma_role<CG, BN, S, C::kGroup, true, idesc_nv(CG, BN), 2>(m);   // K-major only
            } else if constexpr (BS == 1) {
                switch (p.mma_variant & 3) {     // A / B MN-major
#define GEMM_MX_CASE(v)                                                                      \
    case v:                                                                                  \
        mma_role<CG, BN, S, C::kGroup, true, idesc_mx(CG, BN, ((v) >> 1) & 1, (v) & 1, 0), 1>(m); \
        break;
                    GEMM_MX_CASE(0) GEMM_MX_CASE(1) GEMM_MX_CASE(2) GEMM_MX_CASE(3)
#undef GEMM_MX_CASE
                    default: break;
                }
            } else {
                switch (p.mma_variant) {     // one loop per tcgen05 instruction descriptor
#define GEMM_MMA_CASE(v)                                                         \
    case v:                                                                      \
        mma_role<CG, BN, S, C::kGroup, (v) >= 8, idesc_for(CG, BN, (v) >= 8, ((v) >> 2) & 1, \
                                               ((v) >> 1) & 1, (v) & 1)>(m);     \
        break;
                    GEMM_MMA_CASE(0) GEMM_MMA_CASE(1) GEMM_MMA_CASE(2) GEMM_MMA_CASE(3)
                    GEMM_MMA_CASE(4) GEMM_MMA_CASE(5) GEMM_MMA_CASE(6) GEMM_MMA_CASE(7)
                    GEMM_MMA_CASE(8) GEMM_MMA_CASE(9) GEMM_MMA_CASE(10) GEMM_MMA_CASE(11)
#undef GEMM_MMA_CASE
                    default: break;
                }
            }
        }
    } else if (warp == 2 + kEpiWarps) {
        // ------------------------------------------ scale-factor copies ----
        if constexpr (BS != 0) {
            if (lane == 0 && rank == 0) {
                MmaCtx<CG, BN, S> m{p,          ptx::smem_addr(ring), C::kABytes, C::kStageBytes, bar0,
                                    tmem_base,  first_tile,           tile_step,   abort_flag,       peer_abort,
                                    resp0,      clc_full0,            clc_empty0,  dp_tiles};
                factor_copier<CG, BN, S, BS>(m);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue -----
        constexpr int VPC = 16 / OB;                    // output values per 16-byte chunk
        const int ew = warp - 2;                        // staging-buffer owner
        const int q = warp & 3;                         // TMEM lane quadrant this warp may read
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const bool f16_out = p.out_f16 != 0;
        // Compiled twice: EXT adds GELU, the reductions and grouped row
        // ranges, so the plain epilogue carries none of their code.
        auto epilogue = [&](auto ext_tag) {
            constexpr bool EXT = decltype(ext_tag)::value;
            // The scalars of the inner loops, held in registers: read through
            // `p` they would be reloaded from the parameter space after every
            // store to the staging buffer (a generic pointer the compiler
            // cannot tell apart from `p`), several dependent loads per chunk.
            [[maybe_unused]] const float e_alpha = p.alpha, e_beta = p.beta, e_scale_d = p.scale_d;
            [[maybe_unused]] const int e_N = p.N, e_M = p.M, e_bias_mode = p.bias_mode, e_act = p.act, e_out_f8 = p.out_f8;
            [[maybe_unused]] const int e_has_c = p.has_c, e_d_ragged = p.d_ragged, e_num_kb = p.num_kb;
            const int64_t e_ldd = p.ldd, e_d_bstride = p.d_bstride;
            [[maybe_unused]] uint32_t c_phase[2] = {0u, 0u};
            [[maybe_unused]] int sub_count = 0;
            int it = 0;
            bool ok = true;
            const int workers = tile_step;
            // this warp's 32 rows of accumulator `b`, columns [32*..)
            auto load_acc = [&](int b, int sub, uint32_t (&acc)[C::kEpiCols]) {
                const uint32_t taddr = tmem_base + lane_off + (uint32_t)(b * BN + sub * C::kEpiCols);
                ptx::tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&acc[0]));
                if constexpr (C::kEpiCols == 64)
                    ptx::tmem_ld_32x32b_x32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&acc[32]));
                ptx::tmem_ld_wait();
            };
            // This warp is done reading accumulator `b`: tell the MMA issuer.
            auto release_acc = [&](int b) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (CG == 2) {
                        if (rank == 0)
                            ptx::mbar_arrive(acce_bar(b));
                        else
                            ptx::mbar_arrive_cluster(acce_bar(b), 0);
                    } else {
                        ptx::mbar_arrive(acce_bar(b));
                    }
                }
            };
            // The workers whose stream-K ranges hold the later K blocks of a cut
            // tile: ranges r_next, r_next + 1, ... that start before t_end.
            auto for_each_part = [&](int64_t r_next, int64_t t_end, auto&& fn) {
                for (int64_t j = r_next; j < p.sk_ranges; ++j) {
                    const int64_t js = sk_range_start(p.sk_iters, j, p.sk_ranges);
                    if (js >= t_end) break;
                    if (sk_range_start(p.sk_iters, j + 1, p.sk_ranges) == js) continue;     // empty range
                    if (!fn(workers - 1 - (int)j)) return false;
                }
                return true;
            };
            Work wk = work_make(p, first_tile, tile_step, false, resp0, clc_full0, clc_empty0, rank, CG, dp_tiles);
            GroupWalk gw = group_walk_make(p, kTileRows);
            int tile, kb0, kb1;
            for (; ok; ++it) {
                if (!__all_sync(0xffffffffu, work_next(wk, p, tile, kb0, kb1, abort_flag, kStatusRoleEpi, peer_abort,
                                                       lane == 0)))
                    break;
                const int buf = it % C::kAccBufs;
                const uint32_t acc_par = (uint32_t)(it / C::kAccBufs) & 1u;
                // (groups are served by the EXT epilogue only, so the plain one
                // keeps its whole-matrix row range)
                TilePos tp;
                if constexpr (EXT) {
                    tile_pos(p, gw, tile, kTileRows, tp);
                } else {
                    tile_coords(p, tile, tp.mb, tp.nb, tp.l);
                    tp.m_base = 0;
                    tp.m_end = e_M;
                    tp.cd_l = tp.l;
                    tp.sf_base = 0;
                }
                const int mb = tp.mb, nb = tp.nb, l = tp.l;
                const int m_end = tp.m_end;        // rows past it belong to no output of this tile
                const int dl = tp.cd_l;            // batch index of D
                ok = __all_sync(0xffffffffu, wait_bar(accf_bar(buf), acc_par, p, abort_flag, kStatusRoleEpi, peer_abort));
                if (!ok) break;
                if (it == 0 && ew == 0 && lane == 0) GEMM_STAMP(p, 5);
                ptx::tc_fence_after();
                if (kb0 > 0) {
                    // Stream-K: this tile's first K blocks belong to another worker,
                    // its owner, which finishes the tile; hand it the raw sums.
                    float4* slot = part_slot<BN>(p, first_tile, CG, rank, q) + lane;
    #pragma unroll 1
                    for (int sub = 0; sub < C::kSubtiles; ++sub) {
                        uint32_t acc[C::kEpiCols];
                        load_acc(buf, sub, acc);
    #pragma unroll
                        for (int c = 0; c < C::kEpiCols / 4; ++c)
                            __stcg(slot + (sub * (C::kEpiCols / 4) + c) * 32,
                                   make_float4(__uint_as_float(acc[4 * c]), __uint_as_float(acc[4 * c + 1]),
                                               __uint_as_float(acc[4 * c + 2]), __uint_as_float(acc[4 * c + 3])));
                    }
                    release_acc(buf);
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) st_release(part_flag(p, first_tile, CG, rank, q), 1u);
                    continue;
                }
                // A tile cut short (kb1 < num_kb, stream-K region only): its later
                // K blocks come from the next workers' partial sums.
                const bool cut = kb1 < e_num_kb;
                const int64_t t_end = cut ? (int64_t)(tile - p.dp_tiles + 1) * e_num_kb : 0;
                const int64_t r_next = workers - first_tile;        // this worker's range index + 1
                if (cut) {
                    ok = for_each_part(r_next, t_end, [&](int w) {
                        return wait_part(part_flag(p, w, CG, rank, q), p, abort_flag, peer_abort);
                    });
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                [[maybe_unused]] const bool reducing = EXT && (p.red_rows | p.red_cols | p.red_amax) != 0;
                float row_acc = 0.f;          // sum of t over this tile's columns of row `row`
                uint32_t amax_bits = 0u;      // max |t| as fp32 bits (NaN sorts above inf)
                const int row0 = tp.m_base + mb * kTileRows + (int)rank * kTileM + q * kEpiRows;
                const int row = row0 + lane;
                float row_bias = 0.f;
                if (e_bias_mode == 2 && row < m_end) row_bias = p.bias[(int64_t)l * p.bias_stride + row];
                const float* bias_l = e_bias_mode == 1 ? p.bias + (int64_t)l * p.bias_stride : nullptr;
                [[maybe_unused]] const int lc = p.c_batched ? l : 0;
                // With a single accumulator the MMA waits for the whole
                // epilogue, so it is released right after its last subtile's
                // TMEM load, before that subtile's math and stores.  With two
                // the MMA works on the other one meanwhile and the release
                // stays at the end of the tile.
                const int n_end = nb * BN + BN < e_N ? nb * BN + BN : e_N;
                [[maybe_unused]] const int last_sub = (row0 < m_end && n_end > nb * BN) ? (n_end - 1 - nb * BN) / C::kEpiCols : -1;
                bool released = false;
                auto early_release = [&](int sub) {
                    if constexpr (C::kAccBufs == 1) {
                        if (sub == last_sub) {
                            release_acc(buf);
                            released = true;
                        }
                    }
                };
    #pragma unroll 1
                for (int sub = 0; sub < C::kSubtiles; ++sub) {
                    const int col0 = nb * BN + sub * C::kEpiCols;
                    if (row0 >= m_end || col0 >= e_N) continue;     // nothing of this subtile is in range
                    // the subtile's column bias, fetched once (lane i: columns i and
                    // 32 + i, 0 past N) for the plain epilogue's compile-time forms
                    float b_lo = 0.f, b_hi = 0.f;
                    if (!EXT && e_bias_mode == 1) {
                        if (col0 + lane < e_N) b_lo = __ldg(bias_l + col0 + lane);
                        if (C::kEpiCols > 32 && col0 + 32 + lane < e_N) b_hi = __ldg(bias_l + col0 + 32 + lane);
                    }
                    if constexpr (OB == 1) {
                        // MX output: e4m3 elements and one ue8m0 factor per 32
                        // columns of a row (no C; checked on the host).
                        uint32_t acc[C::kEpiCols];
                        if (e_num_kb > 0) {
                            load_acc(buf, sub, acc);
                        } else {
#pragma unroll
                            for (int i = 0; i < C::kEpiCols; ++i) acc[i] = 0u;
                        }
                        early_release(sub);
                        if (cut) {
                            for_each_part(r_next, t_end, [&](int w) {
                                const float4* ps = part_slot<BN>(p, w, CG, rank, q) + sub * (C::kEpiCols / 4) * 32 + lane;
#pragma unroll
                                for (int c = 0; c < C::kEpiCols / 4; ++c) {
                                    const float4 v4 = __ldcg(ps + c * 32);
                                    acc[4 * c] = __float_as_uint(__uint_as_float(acc[4 * c]) + v4.x);
                                    acc[4 * c + 1] = __float_as_uint(__uint_as_float(acc[4 * c + 1]) + v4.y);
                                    acc[4 * c + 2] = __float_as_uint(__uint_as_float(acc[4 * c + 2]) + v4.z);
                                    acc[4 * c + 3] = __float_as_uint(__uint_as_float(acc[4 * c + 3]) + v4.w);
                                }
                                return true;
                            });
                        }
                        if (e_out_f8 == 2) {
                            // NVFP4 output: e2m1 elements and one ue4m3 factor per 16
                            // columns of a row under the global scale g = scale_d:
                            // factor = e4m3(amax / (6 g)), elements e2m1(t / (factor g)),
                            // both the nearest-even codes of the exact quotients
                            const float inv6g = __frcp_rn(__fmul_rn(6.0f, e_scale_d));
#pragma unroll
                            for (int h = 0; h < C::kEpiCols / 16; ++h) {
                                const int c0 = col0 + h * 16;
                                if (c0 >= e_N) break;             // the block lies past the row's end
                                float v[16];
                                if (!EXT && c0 + 16 <= e_N) {
                                    block_values_for<16>(e_bias_mode, e_act == 1, acc + h * 16, h * 16, e_alpha, b_lo,
                                                         b_hi, row_bias, v);
                                } else {
#pragma unroll
                                    for (int i = 0; i < 16; ++i) {
                                        float x = e_alpha * __uint_as_float(acc[h * 16 + i]);
                                        if (e_bias_mode == 1)
                                            x += (c0 + i < e_N) ? __ldg(bias_l + c0 + i) : 0.f;
                                        else if (e_bias_mode == 2)
                                            x += row_bias;
                                        if (e_act == 1)
                                            x = fmaxf(x, 0.f);
                                        else if (EXT && e_act == 2)
                                            x = 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
                                        v[i] = (c0 + i < e_N) ? x : 0.f;   // columns past N join no block
                                    }
                                }
                                uint32_t amax = 0u;
#pragma unroll
                                for (int i = 0; i < 16; ++i) amax = max(amax, __float_as_uint(fabsf(v[i])));
                                uint32_t code = 0x7Fu;            // NaN / inf in the block
                                uint2 out = make_uint2(0u, 0u);
                                if (amax < 0x7F800000u) {
                                    code = nv_factor_code(__uint_as_float(amax), e_scale_d, inv6g);
                                    if (code != 0u) out = nv_element_codes_fast(v, e4m3_value(code), e_scale_d);
                                }
                                if (row < m_end && GEMM_IN_BOUNDS(p, row >= 0 && row < e_M && c0 >= 0 && c0 < e_N &&
                                                                         dl >= 0 && dl < p.L)) {
                                    uint8_t* drow = static_cast<uint8_t*>(p.d_ptr) + (int64_t)dl * e_d_bstride +
                                                    (int64_t)row * e_ldd;          // bytes: two elements each
                                    if (c0 + 16 <= e_N) {
                                        *reinterpret_cast<uint2*>(drow + c0 / 2) = out;
                                    } else {
                                        for (int i = 0; i < 8 && c0 + 2 * i < e_N; ++i)
                                            drow[c0 / 2 + i] = (uint8_t)((i < 4 ? out.x : out.y) >> ((i & 3) * 8));
                                    }
                                    const int f = c0 / 16;
                                    p.sfd[(int64_t)dl * p.sfd_bstride + ((int64_t)(row / 128) * p.sfd_kb4 + f / 4) * 512 +
                                          (row % 32) * 16 + ((row % 128) / 32) * 4 + f % 4] = (uint8_t)code;
                                }
                            }
                            continue;
                        }
#pragma unroll
                        for (int h = 0; h < C::kEpiCols / 32; ++h) {
                            const int c0 = col0 + h * 32;
                            if (c0 >= e_N) break;                 // the block lies past the row's end
                            float v[32];
                            if (!EXT && c0 + 32 <= e_N) {
                                block_values_for<32>(e_bias_mode, e_act == 1, acc + h * 32, h * 32, e_alpha, b_lo, b_hi,
                                                     row_bias, v);
                            } else {
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    float x = e_alpha * __uint_as_float(acc[h * 32 + i]);
                                    if (e_bias_mode == 1)
                                        x += (c0 + i < e_N) ? __ldg(bias_l + c0 + i) : 0.f;
                                    else if (e_bias_mode == 2)
                                        x += row_bias;
                                    if (e_act == 1)
                                        x = fmaxf(x, 0.f);
                                    else if (EXT && e_act == 2)
                                        x = 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
                                    v[i] = (c0 + i < e_N) ? x : 0.f;   // columns past N join no block
                                }
                            }
                            // factor: the OCP MX shared exponent floor(log2 amax) - 8,
                            // read off amax's biased fp32 exponent; 255 for NaN / inf
                            uint32_t amax = 0u;
#pragma unroll
                            for (int i = 0; i < 32; ++i) amax = max(amax, __float_as_uint(fabsf(v[i])));
                            const int be = (int)(amax >> 23);
                            const uint32_t code = amax >= 0x7F800000u ? 255u : (be > 8 ? (uint32_t)(be - 8) : 0u);
                            const float sc = __uint_as_float((254u - (code > 254u ? 254u : code)) << 23);   // 2^(127-code)
                            uint32_t w[8];
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                w[k] = code == 255u ? 0x7F7F7F7Fu
                                                    : ptx::pack4_e4m3(v[4 * k] * sc, v[4 * k + 1] * sc, v[4 * k + 2] * sc,
                                                                      v[4 * k + 3] * sc);
                            if (row < m_end && GEMM_IN_BOUNDS(p, row >= 0 && row < e_M && c0 >= 0 && c0 < e_N &&
                                                                     dl >= 0 && dl < p.L)) {
                                uint8_t* drow = static_cast<uint8_t*>(p.d_ptr) + (int64_t)dl * e_d_bstride +
                                                (int64_t)row * e_ldd;
                                if (c0 + 32 <= e_N) {
                                    *reinterpret_cast<uint4*>(drow + c0) = make_uint4(w[0], w[1], w[2], w[3]);
                                    *reinterpret_cast<uint4*>(drow + c0 + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                                } else {
                                    for (int i = 0; i < 32 && c0 + i < e_N; ++i)
                                        drow[c0 + i] = (uint8_t)(w[i >> 2] >> ((i & 3) * 8));
                                }
                                const int f = c0 / 32;
                                p.sfd[(int64_t)dl * p.sfd_bstride + ((int64_t)(row / 128) * p.sfd_kb4 + f / 4) * 512 +
                                      (row % 32) * 16 + ((row % 128) / 32) * 4 + f % 4] = (uint8_t)code;
                            }
                        }
                    } else {
                        // the subtile holding a ragged row end, or a group's last rows
                        // short of the end of D, is stored element by element
                        const bool direct = (e_d_ragged && col0 + C::kEpiCols > e_N) ||
                                            (EXT && row0 + kEpiRows > m_end && m_end < e_M);
                        // staged tiles of the plain epilogue take stage_subtile
                        const bool quick = !EXT && !direct && e_act != 2;
                        const int sbi = sub_count % C::kEpiBufs;
                        ++sub_count;
                        uint8_t* sbuf = epi + (ew * C::kEpiBufs + sbi) * kEpiBufBytes;
                        const uint32_t sbuf_a = ptx::smem_addr(sbuf);
                        if (lane == 0) ptx::bulk_wait_read<C::kEpiBufs - 1>();   // the store that last used sbuf has read it
                        __syncwarp();
                        if (e_has_c) {
                            const uint32_t cb = cfull_bar(ew * 2 + sbi);
                            if (lane == 0) {
                                ptx::mbar_arrive_expect_tx(cb, kEpiBufBytes);
                                ptx::tma_load_3d(sbuf_a, &tmC, col0, row0, lc, cb);
                            }
                            ok = __all_sync(0xffffffffu, wait_bar(cb, c_phase[sbi], p, abort_flag, kStatusRoleEpi, peer_abort));
                            c_phase[sbi] ^= 1u;
                            if (!ok) break;
                        }
                        uint32_t acc[C::kEpiCols];
                        if (e_num_kb > 0) {
                            load_acc(buf, sub, acc);
                        } else {
        #pragma unroll
                            for (int i = 0; i < C::kEpiCols; ++i) acc[i] = 0u;
                        }
                        early_release(sub);
                        if (cut) {
                            for_each_part(r_next, t_end, [&](int w) {
                                const float4* ps = part_slot<BN>(p, w, CG, rank, q) + sub * (C::kEpiCols / 4) * 32 + lane;
        #pragma unroll
                                for (int c = 0; c < C::kEpiCols / 4; ++c) {
                                    const float4 v4 = __ldcg(ps + c * 32);
                                    acc[4 * c] = __float_as_uint(__uint_as_float(acc[4 * c]) + v4.x);
                                    acc[4 * c + 1] = __float_as_uint(__uint_as_float(acc[4 * c + 1]) + v4.y);
                                    acc[4 * c + 2] = __float_as_uint(__uint_as_float(acc[4 * c + 2]) + v4.z);
                                    acc[4 * c + 3] = __float_as_uint(__uint_as_float(acc[4 * c + 3]) + v4.w);
                                }
                                return true;
                            });
                        }
                        // Row `lane` of the 32-row slab; 128-byte rows, 16-byte chunk c
                        // stored at chunk c ^ (row % 8) (the TMA 128B swizzle).
                        uint8_t* row_base = sbuf + lane * 128;
                        if (quick) {
                            // one of the twelve forms: C or not, no / column / row
                            // bias, ReLU or not
                            const int form = (e_has_c ? 6 : 0) + e_bias_mode * 2 + (e_act == 1 ? 1 : 0);
                            auto stage = [&](auto has_c, auto bias, auto relu) {
                                stage_subtile<OB, decltype(has_c)::value, decltype(bias)::value,
                                              decltype(relu)::value>(acc, row_base, lane, e_alpha, e_beta, b_lo, b_hi,
                                                                     row_bias, f16_out);
                            };
                            using T = std::true_type;
                            using F = std::false_type;
                            using B0 = std::integral_constant<int, 0>;
                            using B1 = std::integral_constant<int, 1>;
                            using B2 = std::integral_constant<int, 2>;
                            switch (form) {
                                case 0: stage(F{}, B0{}, F{}); break;
                                case 1: stage(F{}, B0{}, T{}); break;
                                case 2: stage(F{}, B1{}, F{}); break;
                                case 3: stage(F{}, B1{}, T{}); break;
                                case 4: stage(F{}, B2{}, F{}); break;
                                case 5: stage(F{}, B2{}, T{}); break;
                                case 6: stage(T{}, B0{}, F{}); break;
                                case 7: stage(T{}, B0{}, T{}); break;
                                case 8: stage(T{}, B1{}, F{}); break;
                                case 9: stage(T{}, B1{}, T{}); break;
                                case 10: stage(T{}, B2{}, F{}); break;
                                default: stage(T{}, B2{}, T{}); break;
                            }
                        }
        #pragma unroll
                        for (int ch = 0; ch < 8 && !quick; ++ch) {
                            uint4* slot = reinterpret_cast<uint4*>(row_base + ((ch ^ (lane & 7)) << 4));
                            float v[VPC];
        #pragma unroll
                            for (int i = 0; i < VPC; ++i) v[i] = e_alpha * __uint_as_float(acc[ch * VPC + i]);
                            if (e_has_c) {
                                const uint4 craw = *slot;
                                const uint32_t w[4] = {craw.x, craw.y, craw.z, craw.w};
                                if constexpr (OB == 4) {
        #pragma unroll
                                    for (int i = 0; i < 4; ++i) v[i] = fmaf(e_beta, __uint_as_float(w[i]), v[i]);
                                } else {
        #pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        float lo, hi;
                                        unpack2(w[i], f16_out, lo, hi);
                                        v[2 * i] = fmaf(e_beta, lo, v[2 * i]);
                                        v[2 * i + 1] = fmaf(e_beta, hi, v[2 * i + 1]);
                                    }
                                }
                            }
                            if (e_bias_mode == 1) {
                                const int cb0 = col0 + ch * VPC;
        #pragma unroll
                                for (int i = 0; i < VPC; ++i) v[i] += (cb0 + i < e_N) ? __ldg(bias_l + cb0 + i) : 0.f;
                            } else if (e_bias_mode == 2) {
        #pragma unroll
                                for (int i = 0; i < VPC; ++i) v[i] += row_bias;
                            }
                            if (e_act == 1) {
        #pragma unroll
                                for (int i = 0; i < VPC; ++i) v[i] = fmaxf(v[i], 0.f);
                            } else if (EXT && e_act == 2) {
        #pragma unroll
                                for (int i = 0; i < VPC; ++i) v[i] = 0.5f * v[i] * (1.f + erff(v[i] * 0.70710678118654752f));
                            }
                            if (reducing) {
                                // elements outside D count as 0
                                const int c0 = col0 + ch * VPC;
                                float r[VPC];
        #pragma unroll
                                for (int i = 0; i < VPC; ++i) r[i] = (row < m_end && c0 + i < e_N) ? v[i] : 0.f;
                                if (p.red_rows) {
        #pragma unroll
                                    for (int i = 0; i < VPC; ++i) row_acc += r[i];
                                }
                                if (p.red_amax) {
        #pragma unroll
                                    for (int i = 0; i < VPC; ++i) amax_bits = max(amax_bits, __float_as_uint(fabsf(r[i])));
                                }
                                if (p.red_cols) {
                                    int j;
                                    const float cs = chunk_col_sum<VPC>(r, lane, j);
                                    if ((lane & (32 / VPC - 1)) == 0 && c0 + j < e_N &&
                                        GEMM_IN_BOUNDS(p, l >= 0 && l < p.L && row0 >= 0 && row0 < e_M && c0 + j >= 0))
                                        p.red_col_ws[((int64_t)l * ((e_M + 31) / 32) + row0 / 32) * e_N + c0 + j] = cs;
                                }
                            }
                            uint4 out;
                            if constexpr (OB == 4) {
                                out = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                                                 __float_as_uint(v[3]));
                            } else {
                                out = make_uint4(pack2(v[0], v[1], f16_out), pack2(v[2], v[3], f16_out),
                                                 pack2(v[4], v[5], f16_out), pack2(v[6], v[7], f16_out));
                            }
                            if (!direct) {
                                *slot = out;
                            } else if (row < m_end && GEMM_IN_BOUNDS(p, row >= 0 && row < e_M && col0 >= 0 &&
                                                                          col0 < e_N && dl >= 0 && dl < p.L)) {
                                const int c0 = col0 + ch * VPC;
                                const uint32_t w[4] = {out.x, out.y, out.z, out.w};
                                uint8_t* drow = static_cast<uint8_t*>(p.d_ptr) +
                                                ((int64_t)dl * e_d_bstride + (int64_t)row * e_ldd) * OB;
        #pragma unroll
                                for (int i = 0; i < VPC; ++i) {
                                    if (c0 + i >= e_N) break;
                                    if constexpr (OB == 4)
                                        *reinterpret_cast<uint32_t*>(drow + (int64_t)(c0 + i) * 4) = w[i];
                                    else
                                        *reinterpret_cast<uint16_t*>(drow + (int64_t)(c0 + i) * 2) =
                                            (uint16_t)(w[i >> 1] >> ((i & 1) * 16));
                                }
                            }
                        }
                        if (!direct) {
                            ptx::fence_async_shared();
                            __syncwarp();
                            if (lane == 0 && GEMM_IN_BOUNDS(p, col0 >= 0 && col0 < e_N && row0 >= 0 && row0 < e_M &&
                                                                   dl >= 0 && dl < p.L)) {
                                ptx::tma_store_3d(&tmD, sbuf_a, col0, row0, dl);
                                ptx::bulk_commit();
                            }
                        }
                    }
                }
                if (!ok) break;
                if (!released) release_acc(buf);
                if (EXT && p.red_rows && row < m_end &&
                    GEMM_IN_BOUNDS(p, l >= 0 && l < p.L && nb >= 0 && nb < p.tiles_n && row >= 0 && row < e_M))
                    p.red_row_ws[((int64_t)l * p.tiles_n + nb) * e_M + row] = row_acc;
                if (EXT && p.red_amax) {
    #pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, off));
                    if (lane == 0 && amax_bits) atomicMax(p.red_amax_ws + l, amax_bits);
                }
                // the partial sums are consumed: clear their flags for the next launch
                if (cut && lane == 0)
                    for_each_part(r_next, t_end, [&](int w) {
                        *part_flag(p, w, CG, rank, q) = 0u;
                        return true;
                    });
            }
        };
        if (p.act == 2 || p.red_rows || p.red_cols || p.red_amax || p.groups > 0)
            epilogue(BoolTag<true>{});
        else
            epilogue(BoolTag<false>{});
        // the last stores have read their staging buffers (their global writes
        // complete before the grid does)
        if (lane == 0) ptx::bulk_wait_read<0>();
        if (ew == 0 && lane == 0) GEMM_STAMP(p, 6);
        ptx::tc_fence_before();
    }

    __syncthreads();
    if constexpr (CG == 2) ptx::cluster_sync();   // no CTA leaves while its peer may still touch its memory
    if (threadIdx.x == 0) GEMM_STAMP(p, 7);
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<CG>(tmem_base, C::kTmemCols);
    }
}


// The host-side operations of one kernel variant (declared in
// gemm_variants.h; instantiated in gemm_ob1.cu, gemm_ob2.cu, gemm_ob4.cu).
template <int CG, int BN, int OB, int BS>
static cudaLaunchConfig_t variant_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(Cfg<CG, BN, OB, BS>::kBlockThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<CG, BN, OB, BS>::kSmemBytes;
    cfg.stream = stream;
    attr->id = cudaLaunchAttributeClusterDimension;
    attr->val.clusterDim.x = CG;
    attr->val.clusterDim.y = 1;
    attr->val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CG == 2 ? 1 : 0;      // CTA pairs are launched as clusters of two
    return cfg;
}

template <int CG, int BN, int OB, int BS>
size_t Variant<CG, BN, OB, BS>::smem() {
    return Cfg<CG, BN, OB, BS>::kSmemBytes;
}

template <int CG, int BN, int OB, int BS>
cudaError_t Variant<CG, BN, OB, BS>::prepare() {
    return cudaFuncSetAttribute(gemm_kernel<CG, BN, OB, BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<CG, BN, OB, BS>::kSmemBytes);
}

template <int CG, int BN, int OB, int BS>
cudaError_t Variant<CG, BN, OB, BS>::launch(const LaunchArgs& a) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = variant_config<CG, BN, OB, BS>(a.grid, a.stream, &attr);
    return cudaLaunchKernelEx(&cfg, gemm_kernel<CG, BN, OB, BS>, a.tmA, a.tmB, a.tmC, a.tmD, a.tmSA, a.tmSB, a.p);
}

template <int CG, int BN, int OB, int BS>
int Variant<CG, BN, OB, BS>::max_clusters() {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = variant_config<CG, BN, OB, BS>(CG * 64, nullptr, &attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<CG, BN, OB, BS>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}


}  // namespace gemm_sm103
