// Block-scaled FP8 (mx) grouped GEMM on tcgen05 tensor cores (sm_103a), and
// its C ABI (include/a2av_gmm_mx.h).
//
// "aclnnAlltoAllvGroupedMatMul", Formula: gmmY = permuteOut x gmmWeight and
// mmY = mmX x mmWeight, with every operand in the mx quantisation of the
// "aclnnQuantReduceScatter" page's Constraints: FLOAT8_E4M3FN / FLOAT8_E5M2
// codes with one FLOAT8_E8M0 scale per 32 elements along K.  The tensor cores
// apply the scales themselves (tcgen05.mma kind::mxf8f6f4 with block_scale):
// an MMA of K = 32 takes one E8M0 scale per A row and per B column from TMEM.
//
// Tiles: 128 rows x 128 columns per CTA (cta_group::1), or 256 x 256 on a
// CTA pair (cta_group::2); K in stages of 256 codes: two 128-byte swizzle
// rows per operand row (two 16 KB sub-tiles), eight MMAs.  Per CTA:
//   warp 0     one thread issues a stage's TMA loads: the A rows (read in
//              place from ataOut, or from the prep kernel's staging copy),
//              the K-major weight columns, one 4-D load of both sub-tiles per
//              operand, and before them the stage's scale atoms (below),
//              which complete on a barrier of their own.
//   warp 1     one thread issues the MMAs of a stage once its codes have
//              landed and its scale atoms are in TMEM.
//   warps 10-11 one thread each copies a stage's scale atoms from shared
//              memory into TMEM (tcgen05.cp .32x128b.warpx4) as soon as they
//              land, warp 10 A's and warp 11 B's, then commits to the
//              stage's full barrier, which the codes' bytes and the
//              producer's arrival also complete (three arrivals): the MMA
//              thread waits once per stage, and the copies do not sit in its
//              issue stream.
//   warps 2-9  epilogue, two warps per TMEM lane quarter, each draining half
//              of the columns: TMEM -> registers -> bf16 (nearest even) ->
//              global, rows past the group's end and columns past N masked.
//              A warp loads all its columns, releases the accumulator, and
//              only then converts and stores them.
// Scale atoms: the prep kernel rewrites every operand's E8M0 scales as
// 512-byte atoms, one per 128-row (or 128-column) block and per 4 K blocks
// of 32 codes: 32 rows of 16 bytes, row l holding the four scale bytes of
// block rows l, 32 + l, 64 + l and 96 + l.  tcgen05.cp .32x128b.warpx4 turns
// an atom into the layout the MMA reads: row 32c + l at lane l, column
// base + c, the same in every lane quarter.
// TMEM: the accumulators (single: two of 128 columns, so the epilogue of one
// tile overlaps the main loop of the next; pair: one of 256), then per stage
// eight A-scale and eight (single) or sixteen (pair) B-scale columns.  Every
// wait is bounded: on timeout the CTA sets kStatusTimeout and winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "a2av_gmm_mx.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace a2av {

namespace {

constexpr int MX_BM = 128;       // A rows per CTA
constexpr int MX_BNC = 128;      // weight columns per CTA
constexpr int MX_KCHUNK = 128;   // codes (bytes) in one 128-byte swizzle row
constexpr int MX_CH = 2;         // K chunks per stage
constexpr int MX_BK = MX_KCHUNK * MX_CH;
constexpr int MX_STAGES = 3;
constexpr int kMxEpiWarps = 8;  // two per TMEM lane quarter, each draining half of the columns
constexpr int MX_THREADS = (4 + kMxEpiWarps) * 32;
constexpr int kMxMmaWarp = 1;
constexpr int kMxEpiWarp0 = 2;
constexpr int kMxScaleWarp = kMxEpiWarp0 + kMxEpiWarps;  // copies each stage's A scale atoms into TMEM
constexpr int kMxScaleWarpB = kMxScaleWarp + 1;          // and this one its B scale atoms
constexpr int MX_ATOM_ROWS = 128;     // rows (columns) of a block that one scale atom covers
constexpr uint32_t MX_ATOM_BYTES = 512;  // 32 rows of 16 bytes
constexpr uint32_t kMxAtomLine = 128;    // atoms move as 128-byte lines: 8 atom rows each
constexpr int kMxAtomLineRows = 8;
constexpr int MX_QUAD = 128;          // codes along K per atom: four E8M0 blocks of 32
constexpr uint32_t MX_SUB_BYTES = MX_BM * MX_KCHUNK;      // 16 KB: 128 rows x one chunk
constexpr uint32_t MX_TILE_BYTES = MX_SUB_BYTES * MX_CH;  // one operand's stage; B is the same size
constexpr uint32_t kMxTmemCols = 512;
constexpr uint32_t kMxSfCol0 = 256;  // after the accumulators (2 x 128 single, 1 x 256 pair)
constexpr uint64_t kMxWaitLimitNs = 2000000000ull;

// Tile shapes.  Single: one CTA, 128 x 128 tiles, two accumulators.  Pair:
// a cluster of two CTAs, 256 x 256 tiles (cta_group::2); each CTA stages its
// own 128 A rows and 128 of the weight columns and holds its 128 rows of the
// accumulator, one buffer of 256 columns (two would fill TMEM).
template <bool PAIR>
struct MxShape {
    static constexpr int kCtas = PAIR ? 2 : 1;
    static constexpr int TILE_M = MX_BM * kCtas;
    static constexpr int TILE_N = MX_BNC * kCtas;
    static constexpr int kAccBufs = PAIR ? 1 : 2;
    static constexpr uint32_t kAccCols = TILE_N;
    // Scale words per stage: 2 (eight MMAs, four per word); each word is 32
    // lanes x (rows / 32) columns.  A: this CTA's 128 rows; B: all TILE_N columns.
    static constexpr uint32_t kSfaCols = MX_CH * 4;
    static constexpr uint32_t kSfbCols = MX_CH * (TILE_N / 32);
    static constexpr uint32_t kSfStride = kSfaCols + kSfbCols;
    // Scale atoms of one stage in shared memory: A, the stage's MX_CH quads
    // of this CTA's 128 rows; B, the same quads of each 128-column block of
    // the tile.
    static constexpr uint32_t kSfaBytes = MX_CH * MX_ATOM_BYTES;
    static constexpr uint32_t kSfbBytes = MX_CH * kCtas * MX_ATOM_BYTES;
    static constexpr uint32_t kSfStageBytes = kSfaBytes + kSfbBytes;
};

template <bool PAIR>
__host__ __device__ constexpr uint32_t sfa_col(int s) { return kMxSfCol0 + MxShape<PAIR>::kSfStride * s; }
template <bool PAIR>
__host__ __device__ constexpr uint32_t sfb_col(int s) { return sfa_col<PAIR>(s) + MxShape<PAIR>::kSfaCols; }
static_assert(MxShape<false>::kAccBufs * MxShape<false>::kAccCols <= kMxSfCol0, "accumulators below the scales");
static_assert(MxShape<true>::kAccBufs * MxShape<true>::kAccCols <= kMxSfCol0, "accumulators below the scales");
static_assert(sfb_col<true>(MX_STAGES - 1) + MxShape<true>::kSfbCols <= kMxTmemCols, "scales fit TMEM");
static_assert(sfb_col<false>(MX_STAGES - 1) + MxShape<false>::kSfbCols <= kMxTmemCols, "scales fit TMEM");

struct MxLaunch {
    const int32_t *recvCounts;
    int32_t W, e, A;
    int32_t H1, N1, BS, H2, N2;
    void *gmmY;
    void *mmY;
    int32_t *status;
    int32_t write_status;
    int32_t after_permute;  // launched beside the prep kernel: wait for it before the first load
    int32_t qtype;  // 0 E4M3FN, 1 E5M2 (both operands)
    int32_t pair;
    int32_t grid;
    // Code maps, all 4-D {128 codes, rows, K / 128 chunks, groups}, box
    // 128 x 128 x 2 x 1: one load is a stage's two 16 KB sub-tiles.
    CUtensorMap tmA;   // expert-major codes [A, H1]
    CUtensorMap tmB;   // weight codes [e, N1, H1]
    CUtensorMap tmX;   // mmX codes [BS, H2]
    CUtensorMap tmMW;  // mmWeight codes [N2, H2]
    // Scale atoms (written by the prep kernel) as 128-byte lines, four
    // per atom, no swizzle.  A: 2-D {128, lines}, atom (half, quad) at line
    // 4 (half * quads + quad), box 128 x 4 MX_CH (a stage's quads).  B: 3-D
    // {128, 4 column blocks, groups * quads}, atom (group, quad, block) at
    // line 4 block of plane group * quads + quad, box 128 x 4 kCtas x 2.
    CUtensorMap tmSFA;  // routed A: halves of the expert groups (128 rows from each group's start)
    CUtensorMap tmSFX;  // mmX: halves of the BS rows
    CUtensorMap tmSFB;  // gmmWeight: 128-column blocks of each expert
    CUtensorMap tmSFW;  // mmWeight: 128-column blocks
    // Outputs for the epilogue's TMA stores: 32 x 32 boxes, 64-byte swizzle.
    CUtensorMap tmY_routed;  // gmmY [A, N1] bf16
    CUtensorMap tmY_shared;  // mmY [BS, N2] bf16
    // Halves of a tile (this CTA's 128 rows) whose rows of the group lie in
    // one (source, expert) segment are read in place from ataOut; the permute
    // kernel staged only the others (see half_in_one_segment).
    int32_t direct_halves;
    CUtensorMap tmA_direct;  // ataOut codes [A, H1]
};

// Where this CTA's 128 A rows of a routed tile come from: in place from
// ataOut (a run of one segment), or from the expert-major staging copy.
__device__ __forceinline__ bool mx_direct_row(const MxLaunch &p, const SegmentTable &seg, int row0, int rows, int y,
                                              int32_t *src) {
    if (!p.direct_halves) return false;
    const int g_end = row0 + rows;
    if (y >= g_end || !half_in_one_segment(seg, p.W, p.e, y, g_end)) return false;
    *src = source_row(seg, p.W, p.e, y);
    return true;
}

struct MxGroup {
    int32_t row0;  // first A row (routed: expert-major row)
    int32_t rows;
    int32_t tiles_n;
    int32_t tile_start;
    int32_t half0;  // routed: this group's first 128-row half among all groups' (its scale atoms)
};

struct MxControl {
    uint64_t full[MX_STAGES];    // a stage's codes landed and its atoms are in TMEM (pair: in the even CTA)
    uint64_t sffull[MX_STAGES];  // a stage's scale atoms landed (pair: both CTAs'; in the even CTA)
    uint64_t empty[MX_STAGES];  // the copies and MMAs reading a stage completed
    uint64_t tfull[2];
    uint64_t tempty[2];           // epilogue drained the accumulator (pair: both CTAs; in the even CTA)
    uint32_t tmem_base;
    int32_t abort;
    int32_t total_tiles;
    MxGroup g[kMaxExperts + 2];  // routed, shared, sentinel
    SegmentTable seg;
};

// Epilogue staging: each epilogue warp turns a 32 x 32 block of bf16 results
// around in 2 KB of shared memory (see the epilogue), after the control block.
constexpr uint32_t kMxEpiStageBytes = 32 * 64;
// 1024-aligned: the TMA's 64-byte swizzle pattern repeats every 512 bytes.
__host__ __device__ constexpr size_t mx_epi_offset() { return (sizeof(MxControl) + 1023) / 1024 * 1024; }

template <bool PAIR>
constexpr size_t mx_smem_bytes() {
    return 1024 + MX_STAGES * (2 * MX_TILE_BYTES + MxShape<PAIR>::kSfStageBytes) + mx_epi_offset() +
           kMxEpiWarps * kMxEpiStageBytes;
}
static_assert(mx_smem_bytes<true>() <= 232448 && mx_smem_bytes<false>() <= 232448, "shared memory per CTA");

struct MxTile {
    int g, m, n;
};

__device__ __forceinline__ MxTile mx_decode_tile(const MxControl &c, int t) {
    int g = 0;
    while (t >= c.g[g + 1].tile_start) ++g;
    const int local = t - c.g[g].tile_start;
    return {g, local / c.g[g].tiles_n, local % c.g[g].tiles_n};
}

// Bounded wait on an mbarrier phase; false when it gave up (or another role
// did), with the abort flag and the status word set.  CLUSTER: acquire at
// cluster scope (arrivals come from the peer CTA too).
template <bool CLUSTER = false>
__device__ __noinline__ bool mx_wait(int32_t *abort_flag, uint64_t *bar, uint32_t parity, int32_t *status) {
    const uint32_t b = smem_u32(bar);
    auto try_once = [&]() -> bool {
        if constexpr (CLUSTER) {
            uint32_t ok;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(ok)
                : "r"(b), "r"(parity)
                : "memory");
            return ok != 0;
        } else {
            return mbar_try_wait(b, parity);
        }
    };
    if (try_once()) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (try_once()) return true;
        if (*reinterpret_cast<volatile int32_t *>(abort_flag)) return false;
        if (global_timer_ns() - t0 > kMxWaitLimitNs) {
            *reinterpret_cast<volatile int32_t *>(abort_flag) = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Instruction descriptor of kind::mxf8f6f4: A and B formats (0 E4M3, 1 E5M2),
// both K-major, shape M x N, E8M0 scales; the scale byte of each operand is
// chosen per MMA (bits 29-30 for A, 4-5 for B).
__host__ __device__ constexpr uint32_t mx_idesc(uint32_t qtype, uint32_t M, uint32_t N) {
    return (qtype << 7) | (qtype << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

__device__ __forceinline__ uint32_t mx_sf_ids(uint32_t i) { return (i << 29) | (i << 4); }

template <bool PAIR>
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    if constexpr (PAIR) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
    }
}

// One arrival on `bar` (pair: on the barrier at that offset in both CTAs)
// when this thread's earlier tcgen05 operations have completed.
template <bool PAIR>
__device__ __forceinline__ void mx_commit(uint32_t bar) {
    if constexpr (PAIR) {
        const uint16_t both = 3;
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
            " [%0], %1;" ::"r"(bar),
            "h"(both)
            : "memory");
    } else {
        mma_commit(bar);
    }
}

// Arrival on this CTA's barrier once the calling thread's earlier tcgen05
// operations have completed.
template <bool PAIR>
__device__ __forceinline__ void mx_commit_own(uint32_t bar) {
    if constexpr (PAIR) {
        const uint16_t own = 1;  // the even CTA, the only caller
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
            " [%0], %1;" ::"r"(bar),
            "h"(own)
            : "memory");
    } else {
        mma_commit(bar);
    }
}

__device__ __forceinline__ uint32_t mx_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mx_map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void mx_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// An arrival on a barrier of the even CTA (own CTA when single): an epilogue
// warp handing the accumulator back.  The odd CTA arrives through the
// barrier's cluster address with the default (CTA-scope release) semantics:
// what it hands over is TMEM, whose reads are ordered by tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync before the arrival and by the MMA
// thread's tcgen05.fence::after_thread_sync after its wait.  A cluster-scope
// release arrival measured about 1400 cycles in this kernel.
template <bool PAIR>
__device__ __forceinline__ void mx_arrive_leader(uint32_t own_addr, uint32_t rank) {
    if (PAIR && rank != 0)
        asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(mx_map_to_rank(own_addr, 0)) : "memory");
    else
        mbar_arrive(own_addr);
}

// Copy of one scale atom (32 rows of 16 bytes in shared memory, no swizzle:
// 8-row core matrices 128 bytes apart) into TMEM columns [col, col + 4) of
// lanes 0-31, replicated into every lane quarter (.warpx4).  Pair: the same
// offsets in both CTAs, each from its own shared memory into its own TMEM.
template <bool PAIR>
__device__ __forceinline__ void mx_sf_copy(uint32_t taddr, uint32_t smem_addr) {
    const uint64_t desc = smem_desc(smem_addr, 128, 128, 0);
    if constexpr (PAIR)
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// TMA 3-D load; PAIR: the barrier is the even CTA's (cta_group::2).
template <bool PAIR>
__device__ __forceinline__ void tma_load_3d_mx(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y,
                                               int32_t z) {
    if constexpr (PAIR) {
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
            " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z)
            : "memory");
    } else {
        tma_load_3d(dst, tmap, bar, x, y, z);
    }
}

// TMA 4-D load; PAIR: the barrier is the even CTA's (cta_group::2).
template <bool PAIR>
__device__ __forceinline__ void tma_load_4d_mx(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y,
                                               int32_t z, int32_t w) {
    if constexpr (PAIR) {
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
            " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
            : "memory");
    } else {
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
            : "memory");
    }
}

template <bool PAIR>
__device__ __forceinline__ void mx_tmem_alloc(uint32_t dst_smem) {
    if constexpr (PAIR) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(kMxTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        tmem_alloc(dst_smem, kMxTmemCols);
        tmem_relinquish();
    }
}

template <bool PAIR>
__device__ __forceinline__ void mx_tmem_free(uint32_t taddr) {
    if constexpr (PAIR)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kMxTmemCols)
                     : "memory");
    else
        tmem_dealloc(taddr, kMxTmemCols);
}

__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t *>(&v);
}

template <bool PAIR>
__global__ void __launch_bounds__(MX_THREADS, 1) grouped_gemm_mx_kernel(const __grid_constant__ MxLaunch p) {
    using S = MxShape<PAIR>;
    constexpr int TILE_M = S::TILE_M;
    constexpr int TILE_N = S::TILE_N;
    constexpr int kCtas = S::kCtas;
    constexpr int NB = TILE_N / 32;  // B scale columns per word
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t a_smem = base;
    const uint32_t b_smem = base + MX_STAGES * MX_TILE_BYTES;
    const uint32_t sf_smem = base + 2 * MX_STAGES * MX_TILE_BYTES;  // per stage: A atoms, then B atoms
    MxControl &C = *reinterpret_cast<MxControl *>(base_ptr + 2 * MX_STAGES * MX_TILE_BYTES +
                                                  MX_STAGES * S::kSfStageBytes);
    const uint32_t epi0 = base + 2 * MX_STAGES * MX_TILE_BYTES + MX_STAGES * S::kSfStageBytes + mx_epi_offset();

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int e = p.e;
    const uint32_t rank = PAIR ? mx_cluster_rank() : 0;  // 0: this CTA issues the MMAs
    const int unit = blockIdx.x / kCtas;
    const int nunits = gridDim.x / kCtas;

    // ---- prologue: plan (warp 0), barriers + TMEM (MMA warp), map prefetch (warp 2)
    if (warp == 0) {
        const bool good = build_segment_table(p.recvCounts, p.W, e, p.A, C.seg, lane);
        const int tn1 = (p.N1 + TILE_N - 1) / TILE_N;
        int row0 = 0, rows = 0, tiles = 0, halves = 0;
        if (lane < e) {
            row0 = C.seg.dst[lane * p.W];
            rows = C.seg.dst[(lane + 1) * p.W] - row0;
            tiles = good ? ((rows + TILE_M - 1) / TILE_M) * tn1 : 0;
            halves = (rows + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS;
        }
        int inc = tiles, hinc = halves;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            const int hv = __shfl_up_sync(0xffffffffu, hinc, off);
            if (lane >= off) {
                inc += v;
                hinc += hv;
            }
        }
        if (lane < e) C.g[lane] = MxGroup{row0, rows, tn1, inc - tiles, hinc - halves};
        const int routed_total = __shfl_sync(0xffffffffu, inc, 31);
        if (lane == 0) {
            int ng = e, total = routed_total;
            if (p.BS > 0) {
                const int tn2 = (p.N2 + TILE_N - 1) / TILE_N;
                C.g[e] = MxGroup{0, p.BS, tn2, total, 0};
                total += good ? ((p.BS + TILE_M - 1) / TILE_M) * tn2 : 0;
                ng = e + 1;
            }
            C.g[ng] = MxGroup{0, 0, 1, total, 0};
            C.total_tiles = total;
            C.abort = 0;
            if (blockIdx.x == 0) {
                if (p.write_status) *p.status = good ? 0 : kStatusBadCounts;
                else if (!good) atomicOr(p.status, kStatusBadCounts);
            }
        }
    } else if (warp == kMxMmaWarp) {
        if (lane == 0) {
            for (int s = 0; s < MX_STAGES; ++s) {
                mbar_init(smem_u32(&C.full[s]), 3);  // the producer's arrival and both copiers' commits
                mbar_init(smem_u32(&C.sffull[s]), 1);
                mbar_init(smem_u32(&C.empty[s]), 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(smem_u32(&C.tfull[a]), 1);
                mbar_init(smem_u32(&C.tempty[a]), kMxEpiWarps * kCtas);
            }
            fence_barrier_init();
        }
        __syncwarp();
        mx_tmem_alloc<PAIR>(smem_u32(&C.tmem_base));
    } else if (warp == 2) {
        if (lane == 0) {
            if (p.A > 0) {
                prefetch_tensormap(&p.tmA);
                prefetch_tensormap(&p.tmB);
                prefetch_tensormap(&p.tmSFA);
                prefetch_tensormap(&p.tmSFB);
                prefetch_tensormap(&p.tmY_routed);
                if (p.direct_halves) prefetch_tensormap(&p.tmA_direct);
            }
            if (p.BS > 0) {
                prefetch_tensormap(&p.tmX);
                prefetch_tensormap(&p.tmMW);
                prefetch_tensormap(&p.tmSFX);
                prefetch_tensormap(&p.tmSFW);
                prefetch_tensormap(&p.tmY_shared);
            }
        }
    }
    tc_fence_before_sync();
    if constexpr (PAIR) mx_cluster_sync();
    else __syncthreads();
    tc_fence_after_sync();

    const int total = C.total_tiles;

    if (warp == 0) {
        // =========================================================== TMA producer
        if (lane == 0) {
            // Every tile's scale atoms come from the prep kernel: wait for
            // that grid before the first load.
            if (p.after_permute) asm volatile("griddepcontrol.wait;" ::: "memory");
            uint32_t it = 0;
            bool ok = true;
            for (int t = unit; t < total && ok; t += nunits) {
                const MxTile w = mx_decode_tile(C, t);
                const bool shared = w.g >= e;
                const int K = shared ? p.H2 : p.H1;
                const int nq = K / MX_QUAD;  // scale atoms per 128-row block
                const CUtensorMap *ta = shared ? &p.tmX : &p.tmA;
                const CUtensorMap *tb = shared ? &p.tmMW : &p.tmB;
                const CUtensorMap *tsa = shared ? &p.tmSFX : &p.tmSFA;
                const CUtensorMap *tsb = shared ? &p.tmSFW : &p.tmSFB;
                int ya = C.g[w.g].row0 + w.m * TILE_M + static_cast<int>(rank) * MX_BM;
                int32_t src = 0;
                if (!shared && mx_direct_row(p, C.seg, C.g[w.g].row0, C.g[w.g].rows, ya, &src)) {
                    ta = &p.tmA_direct;
                    ya = src;
                }
                // This CTA's 128-row half: its atoms' first row; the tile's
                // first 128-column block.
                const int half = (shared ? 0 : C.g[w.g].half0) + w.m * kCtas + static_cast<int>(rank);
                const int cb0 = w.n * kCtas;
                const int xn = w.n * TILE_N + static_cast<int>(rank) * MX_BNC;
                const int z = shared ? 0 : w.g;
                for (int kb = 0; kb < K / MX_BK; ++kb, ++it) {
                    const int s = it % MX_STAGES;
                    if (!mx_wait(&C.abort, &C.empty[s], ((it / MX_STAGES) & 1) ^ 1, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_own = smem_u32(&C.full[s]);
                    const uint32_t fb = PAIR ? mx_map_to_rank(fb_own, 0) : fb_own;  // the MMA CTA's barrier
                    const uint32_t sb_own = smem_u32(&C.sffull[s]);
                    const uint32_t sb = PAIR ? mx_map_to_rank(sb_own, 0) : sb_own;
                    if (rank == 0) {
                        mbar_arrive_expect_tx(sb_own, kCtas * S::kSfStageBytes);
                        mbar_arrive_expect_tx(fb_own, kCtas * 2 * MX_TILE_BYTES);
                    }
                    // Scale atoms of quads 2kb and 2kb + 1 first, on their own
                    // barrier: this half's, then each of the tile's column
                    // blocks'.  They land while the stage's 64 KB of codes
                    // are still streaming in, so the copier warps have them
                    // in TMEM by the time the codes are complete.
                    const uint32_t sf_st = sf_smem + s * S::kSfStageBytes;
                    constexpr int kLines = 32 / kMxAtomLineRows;  // 128-byte lines per atom
                    tma_load_3d_mx<PAIR>(sf_st, tsa, sb, 0, kLines * (half * nq + MX_CH * kb), 0);
                    tma_load_3d_mx<PAIR>(sf_st + S::kSfaBytes, tsb, sb, 0, kLines * cb0, z * nq + MX_CH * kb);
                    // {chunk column, row, chunk, group}: both chunks of the stage.
                    tma_load_4d_mx<PAIR>(a_smem + s * MX_TILE_BYTES, ta, fb, 0, ya, kb * MX_CH, 0);
                    tma_load_4d_mx<PAIR>(b_smem + s * MX_TILE_BYTES, tb, fb, 0, xn, kb * MX_CH, z);
                }
            }
            // Wait until the MMAs released every stage that was filled.
            for (int i = 0; i < MX_STAGES && ok; ++i, ++it)
                ok = mx_wait(&C.abort, &C.empty[it % MX_STAGES], ((it / MX_STAGES) & 1) ^ 1, p.status);
        }
    } else if (warp == kMxMmaWarp) {
        // =========================================================== MMA issuer
        if (lane == 0 && rank == 0) {
            const uint32_t idesc0 = mx_idesc(static_cast<uint32_t>(p.qtype), TILE_M, TILE_N);
            // Both operands K-major with a 128-byte swizzle: 128-byte rows,
            // 8-row groups 1024 B apart; an MMA's K step of 32 codes is 32
            // bytes along the row (2 in the 16-byte address field), and the
            // second chunk of a stage starts 16 KB further on.  Pair: both
            // CTAs hold their halves of A and B at the same offsets.
            const uint64_t a_desc0 = smem_desc(a_smem, 16, 1024, kSwizzle128B);
            const uint64_t b_desc0 = smem_desc(b_smem, 16, 1024, kSwizzle128B);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int t = unit; t < total && ok; t += nunits, ++tl) {
                const MxTile w = mx_decode_tile(C, t);
                const int K = w.g >= e ? p.H2 : p.H1;
                const int acc = S::kAccBufs == 2 ? (tl & 1) : 0;
                const uint32_t use = S::kAccBufs == 2 ? (tl >> 1) : tl;  // uses of this buffer so far
                if (!mx_wait<PAIR>(&C.abort, &C.tempty[acc], (use & 1) ^ 1, p.status)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = C.tmem_base + acc * S::kAccCols;
                for (int kb = 0; kb < K / MX_BK; ++kb, ++it) {
                    const int s = it % MX_STAGES;
                    const uint32_t par = (it / MX_STAGES) & 1;
                    // Codes arrive by TMA (async proxy), as the MMAs read them:
                    // the barrier phase orders the two.  The same phase needs
                    // both copier warps' commits, so the stage's atoms are in
                    // TMEM too.
                    if (!mx_wait(&C.abort, &C.full[s], par, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint64_t ad = a_desc0 + ((s * MX_TILE_BYTES) >> 4);
                    const uint64_t bd = b_desc0 + ((s * MX_TILE_BYTES) >> 4);
                    const uint32_t sfa = C.tmem_base + sfa_col<PAIR>(s);
                    const uint32_t sfb = C.tmem_base + sfb_col<PAIR>(s);
#pragma unroll
                    for (int kk = 0; kk < MX_BK / 32; ++kk) {
                        const uint32_t off = ((kk >> 2) * MX_SUB_BYTES + (kk & 3) * 32) >> 4;
                        const uint32_t j = kk >> 2;  // scale word of this MMA
                        mma_mx<PAIR>(d_tmem, ad + off, bd + off, idesc0 | mx_sf_ids(kk & 3), sfa + 4 * j,
                                     sfb + NB * j, (kb | kk) != 0);
                    }
                    mx_commit<PAIR>(smem_u32(&C.empty[s]));
                }
                if (ok) mx_commit<PAIR>(smem_u32(&C.tfull[acc]));
            }
        }
    } else if (warp == kMxScaleWarp || warp == kMxScaleWarpB) {
        // =========================================================== scale atoms into TMEM
        const bool copy_a = warp == kMxScaleWarp;
        if (lane == 0 && rank == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = unit; t < total && ok; t += nunits) {
                const MxTile w = mx_decode_tile(C, t);
                const int K = w.g >= e ? p.H2 : p.H1;
                for (int kb = 0; kb < K / MX_BK; ++kb, ++it) {
                    const int s = it % MX_STAGES;
                    if (!mx_wait(&C.abort, &C.sffull[s], (it / MX_STAGES) & 1, p.status)) {
                        ok = false;
                        break;
                    }
                    // Scale word j (MMAs 4j .. 4j + 3): A's atom to 4 columns;
                    // B's atom of column block i to columns 4i .. 4i + 3 of
                    // the word's NB.  The TMEM columns of stage s are free:
                    // the producer refilled this stage only after the MMAs
                    // that last read them completed.
                    const uint32_t sfa = C.tmem_base + sfa_col<PAIR>(s);
                    const uint32_t sfb = C.tmem_base + sfb_col<PAIR>(s);
                    const uint32_t sf_st = sf_smem + s * S::kSfStageBytes;
                    if (copy_a) {
#pragma unroll
                        for (int j = 0; j < MX_CH; ++j) mx_sf_copy<PAIR>(sfa + 4 * j, sf_st + j * MX_ATOM_BYTES);
                    } else {
#pragma unroll
                        for (int j = 0; j < MX_CH; ++j)
#pragma unroll
                            for (int i = 0; i < kCtas; ++i)
                                mx_sf_copy<PAIR>(sfb + NB * j + 4 * i,
                                                 sf_st + S::kSfaBytes + (j * kCtas + i) * MX_ATOM_BYTES);
                    }
                    mx_commit_own<PAIR>(smem_u32(&C.full[s]));
                }
            }
        }
    } else {
        // =========================================================== epilogue
        const int q = warp & 3;
        constexpr int kChunks = TILE_N / 32 / 2;              // 32-column chunks per warp
        const int c0 = ((warp - kMxEpiWarp0) / 4) * kChunks;  // first chunk of this warp's half
        uint32_t tl = 0;
        for (int t = unit; t < total; t += nunits, ++tl) {
            const MxTile w = mx_decode_tile(C, t);
            const bool shared = w.g >= e;
            const int acc = S::kAccBufs == 2 ? (tl & 1) : 0;
            const uint32_t use = S::kAccBufs == 2 ? (tl >> 1) : tl;
            if (!mx_wait(&C.abort, &C.tfull[acc], use & 1, p.status)) break;
            __syncwarp();  // lanes leave the wait independently; tcgen05.ld needs the whole warp
            tc_fence_after_sync();
            const int N = shared ? p.N2 : p.N1;
            const int row = w.m * TILE_M + static_cast<int>(rank) * MX_BM + q * 32 + lane;
            const bool valid = row < C.g[w.g].rows;
            const int n0 = w.n * TILE_N;
            uint16_t *const out_base = static_cast<uint16_t *>(shared ? p.mmY : p.gmmY);
            const uint32_t t_base = C.tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * S::kAccCols;
            // All of this warp's columns come out of TMEM first (the loads are
            // asynchronous, one wait for all), then the accumulator is
            // released, and only then converted and stored: with one
            // accumulator (pair tiles) the next tile's MMAs wait for this.
            uint32_t v[kChunks][32];
#pragma unroll
            for (int i = 0; i < kChunks; ++i) tmem_ld_32x32b_x32(t_base + (c0 + i) * 32, v[i]);
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mx_arrive_leader<PAIR>(smem_u32(&C.tempty[acc]), rank);
            // Each 32 x 32 block is turned around in this warp's 2 KB of
            // shared memory (64-byte rows, the 16-byte chunk index XORed with
            // (row / 2) % 4: no bank conflicts either way), then stored as 8
            // rows of 64 contiguous bytes per instruction.  After the turn,
            // lane l stores row 8k + l / 4 of the warp's 32, at column
            // 8 (l % 4) of the block.
            const uint32_t valid_mask = __ballot_sync(0xffffffffu, valid);
            const int row0w = row - lane;
            const uint32_t stage = epi0 + static_cast<uint32_t>(warp - kMxEpiWarp0) * kMxEpiStageBytes;
            const CUtensorMap *tmy = shared ? &p.tmY_shared : &p.tmY_routed;
            const int orow0 = shared ? row0w : C.g[w.g].row0 + row0w;
#pragma unroll
            for (int i = 0; i < kChunks; ++i) {
                // The previous block's TMA store (if any) has read the buffer.
                if (lane == 0) bulk_wait_read_0();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t *r = v[i] + j * 8;
                    uint4 pk;
                    pk.x = pack_bf16(r[0], r[1]);
                    pk.y = pack_bf16(r[2], r[3]);
                    pk.z = pack_bf16(r[4], r[5]);
                    pk.w = pack_bf16(r[6], r[7]);
                    st_shared_v4(stage + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), pk);
                }
                const int blk_col = n0 + (c0 + i) * 32;
                if (valid_mask == 0xffffffffu && blk_col < N) {
                    // 32 whole rows of the group: one TMA store (columns past N
                    // are clipped by the map).
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(tmy, stage, blk_col, orow0);
                        bulk_commit_group();
                    }
                } else {
                    __syncwarp();
                    const int j = lane & 3;
                    const int col = (c0 + i) * 32 + j * 8;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int rr = 8 * k + (lane >> 2);
                        const uint4 val = ld_shared_v4(stage + rr * 64 + ((j ^ ((rr >> 1) & 3)) << 4));
                        if (((valid_mask >> rr) & 1u) && n0 + col < N) {
                            const int grow = row0w + rr;
                            const size_t orow = static_cast<size_t>(shared ? grow : C.g[w.g].row0 + grow);
                            st_stream_v4(out_base + orow * N + n0 + col, val);
                        }
                    }
                }
                __syncwarp();  // the next block rewrites the staging area
            }
        }
    }

    if (warp >= kMxEpiWarp0 && warp < kMxEpiWarp0 + kMxEpiWarps && lane == 0)
        bulk_wait_all();  // this warp's TMA stores have landed
    tc_fence_before_sync();
    if constexpr (PAIR) mx_cluster_sync();
    else __syncthreads();
    if (warp == kMxMmaWarp) {
        tc_fence_after_sync();
        mx_tmem_free<PAIR>(C.tmem_base);
    }
}

// ---------------------------------------------------------------- permute and scale atoms
//
// One kernel before the GEMM.  Its warps first do the Permute step for mx
// operands: the expert-major copy of rows' H1 code bytes (and, into
// permuteOut, their H1/32 scale bytes), in 2 KB pieces per warp.  Without
// permuteOut only rows of 128-row halves that straddle a segment boundary are
// copied (the GEMM reads the others in place).  Then its warps write every
// operand's scale atoms (see the top of this file), four atoms of one block
// per warp.
constexpr int kMxPermThreads = 256;
constexpr int kPieceVecs = 4;  // 16-byte vectors per lane in one work item (2 KB per warp)

struct MxPrep {
    const int32_t *recvCounts;
    int32_t W, e, A, H1, N1, BS, H2, N2;
    const uint4 *src_q;    // ataOut codes [A, H1]
    const uint8_t *src_s;  // ataOut scales [A, H1/32]
    uint4 *dst_q;          // expert-major codes: permuteOut or the staging copy
    uint4 *dst_s;          // expert-major scales: permuteOut, or null
    int32_t *status;
    int32_t only_straddling;
    const uint8_t *w_s;   // gmmWeight scales [e, N1, H1/32]
    const uint8_t *x_s;   // mmX scales [BS, H2/32]
    const uint8_t *mw_s;  // mmWeight scales [N2, H2/32]
    uint8_t *sfa, *sfx, *sfb, *sfw;  // atoms: routed A halves, mmX halves, gmmWeight and mmWeight blocks
};

__device__ __forceinline__ uint4 mx_ld_stream(const uint4 *ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

__global__ void __launch_bounds__(kMxPermThreads) mx_prep_kernel(const __grid_constant__ MxPrep p) {
    __shared__ SegmentTable table;
    __shared__ StagedHalves halves;
    __shared__ int32_t half0[kMaxExperts + 1];  // routed: first 128-row half of each expert group
    __shared__ int ok;
    // The first kernel of the call clears the status word before the GEMM
    // behind it can start; every later write to it is an atomicOr.
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            *p.status = 0;
            __threadfence();
        }
        __syncthreads();
    }
    // The GEMM launched after this kernel with programmatic dependent launch
    // may start now: it waits for this grid's completion before it reads
    // anything this kernel writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int W = p.W, e = p.e, H1 = p.H1;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0) {
        const bool good = build_segment_table(p.recvCounts, W, e, p.A, table, lane);
        int nh = 0;
        if (lane < e) nh = (table.dst[(lane + 1) * W] - table.dst[lane * W] + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS;
        int inc = nh;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        if (lane < e) half0[lane] = inc - nh;
        const int all = __shfl_sync(0xffffffffu, inc, 31);
        if (lane == 0) {
            half0[e] = all;
            ok = good;
            if (blockIdx.x == 0 && !good) atomicOr(p.status, kStatusBadCounts);
        }
    }
    __syncthreads();

    if (ok && p.dst_q != nullptr) {
        // Work items are pieces of a code row (kPieceVecs 16-byte vectors per
        // lane, all loaded before any is stored); the first piece of a row
        // also moves its scale row when permuteOut wants it.  One memory round
        // trip per item.
        const int vq = H1 / 16, vs = H1 / 512;  // 16-byte vectors per code row and per scale row
        const int ppr = (vq + 32 * kPieceVecs - 1) / (32 * kPieceVecs);
        const int nwarps = gridDim.x * (kMxPermThreads / 32);
        const int gw = blockIdx.x * (kMxPermThreads / 32) + warp;
        const auto copy_piece = [&](int d, int seg, int piece) {
            const int v0 = piece * 32 * kPieceVecs + lane;
            const size_t srow = static_cast<size_t>(source_row_in(table, W, e, seg, d));
            const uint4 *in = p.src_q + srow * vq;
            uint4 *out = p.dst_q + static_cast<size_t>(d) * vq;
            uint4 r[kPieceVecs];
#pragma unroll
            for (int k = 0; k < kPieceVecs; ++k)
                if (v0 + 32 * k < vq) r[k] = mx_ld_stream(in + v0 + 32 * k);
#pragma unroll
            for (int k = 0; k < kPieceVecs; ++k)
                if (v0 + 32 * k < vq) out[v0 + 32 * k] = r[k];
            if (piece == 0 && p.dst_s != nullptr) {
                const uint4 *ins = reinterpret_cast<const uint4 *>(p.src_s) + srow * vs;
                for (int u = lane; u < vs; u += 32) p.dst_s[static_cast<size_t>(d) * vs + u] = mx_ld_stream(ins + u);
            }
        };
        int listed = -1;
        if (p.only_straddling) {
            list_staged_halves(table, W, e, halves);
            listed = halves.n;
        }
        if (listed >= 0) {
            // Only the rows of the halves the GEMM cannot read in place.
            const int per_half = kHalfRows * ppr;
            for (int i = gw; i < listed * per_half; i += nwarps) {
                const int hi = i / per_half, rem = i - hi * per_half;
                const int r = rem / ppr;
                const int2 span = halves.span[hi];
                const int d = span.x + r;
                if (d < span.y) copy_piece(d, segment_of(table, W, e, d), rem - r * ppr);
            }
        } else {
            const int64_t items = static_cast<int64_t>(p.A) * ppr;
            for (int64_t i = gw; i < items; i += nwarps) {
                const int d = static_cast<int>(i / ppr);
                const int seg = segment_of(table, W, e, d);
                if (p.only_straddling) {
                    // More staged halves than the list holds (not reached: see
                // kMaxStagedHalves): test each row's half.
                    const int j = seg / W;
                    const int g0 = table.dst[j * W], g1 = table.dst[(j + 1) * W];
                    if (half_in_one_segment(table, W, e, g0 + (d - g0) / kHalfRows * kHalfRows, g1)) continue;
                }
                copy_piece(d, seg, static_cast<int>(i - static_cast<int64_t>(d) * ppr));
            }
        }
    }

    // ---- scale atoms: routed A (valid counts only), mmX, gmmWeight, mmWeight
    const int nq1 = H1 / MX_QUAD, nq2 = p.H2 / MX_QUAD;
    const int ncb1 = (p.N1 + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS, ncb2 = (p.N2 + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS;
    const int64_t rows_a = (ok && p.A > 0) ? static_cast<int64_t>(half0[e]) * nq1 * 32 : 0;
    const int64_t rows_x = p.BS > 0 ? static_cast<int64_t>((p.BS + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS) * nq2 * 32 : 0;
    const int64_t rows_b = p.A > 0 ? static_cast<int64_t>(e) * nq1 * ncb1 * 32 : 0;
    const int64_t rows_w = p.BS > 0 ? static_cast<int64_t>(nq2) * ncb2 * 32 : 0;
    // Work items are groups of four atoms: one 128-row (column) block and
    // quads 4k .. 4k + 3 (H is a multiple of 512, so the quads of a row
    // come in fours).  A warp takes an item: lane l loads the 16 bytes of
    // those quads from each of its rows l, 32 + l, 64 + l, 96 + l, and writes
    // row l of each of the four atoms, so one store instruction fills an atom.
    const int64_t items_a = rows_a / 128, items_x = rows_x / 128, items_b = rows_b / 128, items_w = rows_w / 128;
    const int64_t items = items_a + items_x + items_b + items_w;
    const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * (kMxPermThreads / 32) + threadIdx.x / 32;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kMxPermThreads / 32);
    const size_t kb1 = static_cast<size_t>(H1 / 32), kb2 = static_cast<size_t>(p.H2 / 32);
    const int nk1 = nq1 / 4, nk2 = nq2 / 4;
    // Row l of atoms (block, quads 4k .. 4k + 3) from the scale rows row(r):
    // rows at or past `valid` read as 127 (a scale of 1).
    const auto write_atoms = [&](const auto &row, int valid, int k, uint8_t *atoms, int64_t atom0, int64_t step) {
        uint4 w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int r = 32 * c + lane;
            w[c] = r < valid ? *reinterpret_cast<const uint4 *>(row(r) + 16 * k)
                             : make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 v = j == 0 ? make_uint4(w[0].x, w[1].x, w[2].x, w[3].x)
                          : j == 1 ? make_uint4(w[0].y, w[1].y, w[2].y, w[3].y)
                          : j == 2 ? make_uint4(w[0].z, w[1].z, w[2].z, w[3].z)
                                   : make_uint4(w[0].w, w[1].w, w[2].w, w[3].w);
            reinterpret_cast<uint4 *>(atoms + static_cast<size_t>(atom0 + j * step) * MX_ATOM_BYTES)[lane] = v;
        }
    };
    for (int64_t i = gwarp; i < items; i += nwarps) {
        if (i < items_a) {
            const int h = static_cast<int>(i / nk1), k = static_cast<int>(i % nk1);
            int g = 0;
            while (h >= half0[g + 1]) ++g;  // the expert group holding half h
            const int first = table.dst[g * W] + (h - half0[g]) * MX_ATOM_ROWS;
            const int valid = min(MX_ATOM_ROWS, table.dst[(g + 1) * W] - first);
            const auto row = [&](int r) { return p.src_s + static_cast<size_t>(source_row(table, W, e, first + r)) * kb1; };
            write_atoms(row, valid, k, p.sfa, static_cast<int64_t>(h) * nq1 + 4 * k, 1);
        } else if (i < items_a + items_x) {
            const int64_t ix = i - items_a;
            const int h = static_cast<int>(ix / nk2), k = static_cast<int>(ix % nk2);
            const int first = h * MX_ATOM_ROWS;
            const auto row = [&](int r) { return p.x_s + static_cast<size_t>(first + r) * kb2; };
            write_atoms(row, min(MX_ATOM_ROWS, p.BS - first), k, p.sfx, static_cast<int64_t>(h) * nq2 + 4 * k, 1);
        } else if (i < items_a + items_x + items_b) {
            // Atom (z, q, cb) of gmmWeight: plane z * nq1 + q, block cb.
            const int64_t ib = i - items_a - items_x;
            const int cb = static_cast<int>(ib % ncb1);
            const int64_t rest = ib / ncb1;
            const int z = static_cast<int>(rest / nk1), k = static_cast<int>(rest % nk1);
            const int first = cb * MX_ATOM_ROWS;
            const auto row = [&](int r) {
                return p.w_s + (static_cast<size_t>(z) * p.N1 + static_cast<size_t>(first + r)) * kb1;
            };
            write_atoms(row, min(MX_ATOM_ROWS, p.N1 - first), k, p.sfb,
                        (static_cast<int64_t>(z) * nq1 + 4 * k) * ncb1 + cb, ncb1);
        } else {
            const int64_t iw = i - items_a - items_x - items_b;
            const int cb = static_cast<int>(iw % ncb2), k = static_cast<int>(iw / ncb2);
            const int first = cb * MX_ATOM_ROWS;
            const auto row = [&](int r) { return p.mw_s + static_cast<size_t>(first + r) * kb2; };
            write_atoms(row, min(MX_ATOM_ROWS, p.N2 - first), k, p.sfw, static_cast<int64_t>(4 * k) * ncb2 + cb, ncb2);
        }
    }
}

// ---------------------------------------------------------------- host side

constexpr size_t kMxStatusBytes = 256;

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

a2av_status mx_validate(const a2av_gmm_mx_desc *d) {
    if (!d) return A2AV_ERR_NULLPTR;
    if (d->W < 1 || d->e < 1 || d->e > kMaxExperts) return A2AV_ERR_INVALID;
    if (static_cast<int64_t>(d->W) * d->e > kMaxSegments) return A2AV_ERR_INVALID;
    if (d->H1 <= 0 || d->H1 >= 65536 || d->N1 <= 0 || d->N1 >= 65536) return A2AV_ERR_INVALID;
    if (d->A < 0 || d->A > INT32_MAX || d->BS < 0 || d->BS > INT32_MAX) return A2AV_ERR_INVALID;
    if (d->BS > 0 && (d->H2 <= 0 || d->H2 > 12288 || d->N2 <= 0 || d->N2 >= 65536)) return A2AV_ERR_INVALID;
    if (d->qtype != 0 && d->qtype != 1) return A2AV_ERR_INVALID;  // E4M3FN or E5M2
    if (d->tiles != A2AV_TILES_DEFAULT && d->tiles != A2AV_TILES_SINGLE && d->tiles != A2AV_TILES_PAIR)
        return A2AV_ERR_INVALID;
    if (d->H1 % 512 != 0 || d->N1 % 8 != 0) return A2AV_ERR_UNSUPPORTED;
    if (d->BS > 0 && (d->H2 % 512 != 0 || d->N2 % 8 != 0)) return A2AV_ERR_UNSUPPORTED;
    return A2AV_OK;
}

// Workspace after the status word: the staging copy of A's codes (without
// permuteOut), then the scale atoms of routed A (one per 128-row half of each
// expert group and quad of K), of mmX, of gmmWeight and of mmWeight.
struct MxWorkspace {
    size_t staging, sfa, sfx, sfb, sfw, total;
    int64_t sfa_rows;  // 16-byte rows of the routed-A atom buffer (an upper bound on the halves used)
};

MxWorkspace mx_workspace_layout(const a2av_gmm_mx_desc *d) {
    MxWorkspace w{};
    const int64_t A = d->A, BS = d->BS;
    const int64_t nq1 = d->H1 / MX_QUAD, nq2 = BS > 0 ? d->H2 / MX_QUAD : 0;
    const int64_t ncb1 = (d->N1 + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS;
    const int64_t ncb2 = BS > 0 ? (d->N2 + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS : 0;
    size_t off = kMxStatusBytes;
    w.staging = off;
    if (!d->want_permute_out && A > 0) off += align256(static_cast<size_t>(A) * d->H1);
    w.sfa = off;
    w.sfa_rows = A > 0 ? ((A + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS + d->e) * nq1 * 32 : 0;
    off += align256(static_cast<size_t>(w.sfa_rows) * 16);
    w.sfx = off;
    if (BS > 0) off += align256(static_cast<size_t>((BS + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS) * nq2 * MX_ATOM_BYTES);
    w.sfb = off;
    if (A > 0) off += align256(static_cast<size_t>(d->e) * nq1 * ncb1 * MX_ATOM_BYTES);
    w.sfw = off;
    if (BS > 0) off += align256(static_cast<size_t>(nq2) * ncb2 * MX_ATOM_BYTES);
    w.total = off;
    return w;
}

PFN_cuTensorMapEncodeTiled_v12000 mx_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q);
    });
    return fn;
}

// Byte codes [groups][rows][K] seen as 4-D {128 codes, rows, K / 128 chunks,
// groups}; box 128 x 128 x MX_CH x 1, 128-byte swizzle: one load lands a
// stage's K chunks as consecutive 16 KB K-major sub-tiles.  Needs K % 256 == 0.
// bf16 outputs [rows, cols]; box 32 x 32, 64-byte swizzle (the epilogue's
// staging layout).
bool mx_out_map(CUtensorMap *m, void *ptr, int64_t rows, int64_t cols) {
    auto fn = mx_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool mx_codes_map(CUtensorMap *m, const void *ptr, int64_t groups, int64_t rows, int64_t K) {
    auto fn = mx_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {MX_KCHUNK, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K / MX_KCHUNK),
                          static_cast<cuuint64_t>(groups)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(K), MX_KCHUNK, static_cast<cuuint64_t>(K * rows)};
    cuuint32_t box[4] = {MX_KCHUNK, MX_BM, MX_CH, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale atoms, counted in 16-byte atom rows (rows, box_rows: multiples of
// 8), loaded as 128-byte lines: 3-D {128, rows / 8, planes}, box 128 x
// box_rows / 8 x box_planes, no swizzle, so shared memory receives the same
// bytes in the same order with an eighth of the requests; out-of-range rows
// load as zeros.
bool mx_atoms_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t planes, uint32_t box_rows,
                  uint32_t box_planes) {
    auto fn = mx_encode_fn();
    if (!fn || rows % kMxAtomLineRows != 0 || box_rows % kMxAtomLineRows != 0) return false;
    cuuint64_t dims[3] = {kMxAtomLine, static_cast<cuuint64_t>(rows / kMxAtomLineRows),
                          static_cast<cuuint64_t>(planes)};
    cuuint64_t strides[2] = {kMxAtomLine, static_cast<cuuint64_t>(rows * 16)};
    cuuint32_t box[3] = {kMxAtomLine, box_rows / kMxAtomLineRows, box_planes};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int mx_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool mx_aligned16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

// Prep-kernel blocks resident on one SM at once (per device, queried once).
int mx_prep_blocks_per_sm() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mx_prep_kernel, kMxPermThreads, 0) != cudaSuccess)
            return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace

}  // namespace a2av

extern "C" a2av_status a2av_gmm_mx_workspace_size(const a2av_gmm_mx_desc *desc, size_t *bytes) {
    if (!desc || !bytes) return A2AV_ERR_NULLPTR;
    const a2av_status s = a2av::mx_validate(desc);
    if (s != A2AV_OK) return s;
    *bytes = a2av::mx_workspace_layout(desc).total;
    return A2AV_OK;
}

namespace {

// The call; with gemm_begin / gemm_end, those events are recorded right
// around the GEMM launch, which then follows the prep kernel in plain stream
// order (no programmatic dependent launch), so that they time it alone.
a2av_status mx_run_impl(const a2av_gmm_mx_desc *desc, const void *ataOut_q, const void *ataOut_s,
                        const int32_t *recvCounts, const void *gmmWeight_q, const void *gmmWeight_s,
                        const void *mmX_q, const void *mmX_s, const void *mmWeight_q, const void *mmWeight_s,
                        void *permuteOut_q, void *permuteOut_s, void *gmmY, void *mmY, void *workspace,
                        size_t workspace_bytes, a2av_stream_t stream_handle, cudaEvent_t gemm_begin,
                        cudaEvent_t gemm_end) {
    using namespace a2av;
    const a2av_status vs = mx_validate(desc);
    if (vs != A2AV_OK) return vs;
    const a2av_gmm_mx_desc &d = *desc;
    const bool routed = d.A > 0, shared = d.BS > 0;
    if (!recvCounts || !gmmWeight_q || !gmmWeight_s || !workspace) return A2AV_ERR_NULLPTR;
    if (routed && (!ataOut_q || !ataOut_s || !gmmY)) return A2AV_ERR_NULLPTR;
    if (routed && d.want_permute_out && (!permuteOut_q || !permuteOut_s)) return A2AV_ERR_NULLPTR;
    if (shared && (!mmX_q || !mmX_s || !mmWeight_q || !mmWeight_s || !mmY)) return A2AV_ERR_NULLPTR;
    const void *ptrs[] = {ataOut_q, ataOut_s, gmmWeight_q, gmmWeight_s, mmX_q, mmX_s, mmWeight_q, mmWeight_s,
                          gmmY, mmY, d.want_permute_out ? permuteOut_q : nullptr,
                          d.want_permute_out ? permuteOut_s : nullptr};
    for (const void *q : ptrs)
        if (!mx_aligned16(q)) return A2AV_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(recvCounts) & 3u) != 0) return A2AV_ERR_UNSUPPORTED;
    size_t need = 0;
    a2av_gmm_mx_workspace_size(desc, &need);
    if (workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return A2AV_ERR_WORKSPACE;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    const int sms = mx_sm_count();
    if (sms <= 0) return A2AV_ERR_CUDA;
    int32_t *status = static_cast<int32_t *>(workspace);

    MxLaunch g;
    std::memset(&g, 0, sizeof g);
    g.recvCounts = recvCounts;
    g.W = d.W;
    g.e = d.e;
    g.A = static_cast<int32_t>(d.A);
    g.H1 = static_cast<int32_t>(d.H1);
    g.N1 = static_cast<int32_t>(d.N1);
    g.BS = shared ? static_cast<int32_t>(d.BS) : 0;
    g.H2 = shared ? static_cast<int32_t>(d.H2) : 0;
    g.N2 = shared ? static_cast<int32_t>(d.N2) : 0;
    g.gmmY = gmmY;
    g.mmY = mmY;
    if (routed && !mx_out_map(&g.tmY_routed, gmmY, d.A, d.N1)) return A2AV_ERR_CUDA;
    if (shared && !mx_out_map(&g.tmY_shared, mmY, d.BS, d.N2)) return A2AV_ERR_CUDA;
    g.status = status;
    g.qtype = d.qtype;
    const bool pair = d.tiles != A2AV_TILES_SINGLE;
    const uint32_t ctas = pair ? 2 : 1;
    const MxWorkspace ws = mx_workspace_layout(&d);
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    const int64_t nq1 = d.H1 / MX_QUAD, ncb1 = (d.N1 + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS;
    if (!mx_codes_map(&g.tmB, gmmWeight_q, d.e, d.N1, d.H1)) return A2AV_ERR_CUDA;
    if (routed) {
        // Atoms as 16-byte rows: routed A, 2-D in effect (one plane), a
        // stage's MX_CH quads per load; gmmWeight, plane z * nq1 + quad, the
        // tile's column blocks and the stage's quads per load.
        if (!mx_atoms_map(&g.tmSFA, wsb + ws.sfa, ws.sfa_rows, 1, 32 * MX_CH, 1)) return A2AV_ERR_CUDA;
        if (!mx_atoms_map(&g.tmSFB, wsb + ws.sfb, ncb1 * 32, d.e * nq1, 32 * ctas, MX_CH)) return A2AV_ERR_CUDA;
    }
    if (shared) {
        const int64_t nq2 = d.H2 / MX_QUAD, ncb2 = (d.N2 + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS;
        const int64_t nh2 = (d.BS + MX_ATOM_ROWS - 1) / MX_ATOM_ROWS;
        if (!mx_codes_map(&g.tmX, mmX_q, 1, d.BS, d.H2)) return A2AV_ERR_CUDA;
        if (!mx_codes_map(&g.tmMW, mmWeight_q, 1, d.N2, d.H2)) return A2AV_ERR_CUDA;
        if (!mx_atoms_map(&g.tmSFX, wsb + ws.sfx, nh2 * nq2 * 32, 1, 32 * MX_CH, 1)) return A2AV_ERR_CUDA;
        if (!mx_atoms_map(&g.tmSFW, wsb + ws.sfw, ncb2 * 32, nq2, 32 * ctas, MX_CH)) return A2AV_ERR_CUDA;
    }
    // The prep kernel: expert-major codes (into permuteOut, or only the
    // halves that straddle a segment boundary into the staging copy), and
    // every operand's scale atoms.
    MxPrep pp;
    std::memset(&pp, 0, sizeof pp);
    pp.recvCounts = recvCounts;
    pp.W = d.W;
    pp.e = d.e;
    pp.A = static_cast<int32_t>(d.A);
    pp.H1 = static_cast<int32_t>(d.H1);
    pp.N1 = static_cast<int32_t>(d.N1);
    pp.BS = g.BS;
    pp.H2 = g.H2;
    pp.N2 = g.N2;
    pp.status = status;
    pp.src_q = static_cast<const uint4 *>(ataOut_q);
    pp.src_s = static_cast<const uint8_t *>(ataOut_s);
    pp.w_s = static_cast<const uint8_t *>(gmmWeight_s);
    pp.x_s = static_cast<const uint8_t *>(mmX_s);
    pp.mw_s = static_cast<const uint8_t *>(mmWeight_s);
    pp.sfa = wsb + ws.sfa;
    pp.sfx = wsb + ws.sfx;
    pp.sfb = wsb + ws.sfb;
    pp.sfw = wsb + ws.sfw;
    if (routed) {
        uint8_t *dq = static_cast<uint8_t *>(permuteOut_q);
        if (!d.want_permute_out) {
            dq = wsb + ws.staging;
            // Only the 128-row halves that straddle a segment boundary are
            // staged; the GEMM reads the others from ataOut.
            if (!mx_codes_map(&g.tmA_direct, ataOut_q, 1, d.A, d.H1)) return A2AV_ERR_CUDA;
            g.direct_halves = 1;
        }
        pp.dst_q = reinterpret_cast<uint4 *>(dq);
        pp.dst_s = d.want_permute_out ? static_cast<uint4 *>(permuteOut_s) : nullptr;
        pp.only_straddling = d.want_permute_out ? 0 : 1;
        if (!mx_codes_map(&g.tmA, dq, 1, d.A, d.H1)) return A2AV_ERR_CUDA;
    }
    bool prep_ran = false;
    if (routed || shared) {
        // Blocks for a warp per row of A, or a thread per atom row, at most
        // as many as are resident at once (registers allow five per SM), so
        // that no block waits for a second wave.
        const int64_t atom_rows = ws.sfa_rows + static_cast<int64_t>(ws.total - ws.sfx) / 16;
        const int64_t want = std::max<int64_t>((d.A + kMxPermThreads / 32 - 1) / (kMxPermThreads / 32),
                                               (atom_rows + kMxPermThreads - 1) / kMxPermThreads);
        const int per_sm = mx_prep_blocks_per_sm();
        if (per_sm <= 0) return A2AV_ERR_CUDA;
        const int blocks =
            static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(sms) * per_sm)));
        mx_prep_kernel<<<blocks, kMxPermThreads, 0, stream>>>(pp);
        if (cudaGetLastError() != cudaSuccess) return A2AV_ERR_CUDA;
        prep_ran = true;
    }
    g.write_status = prep_ran ? 0 : 1;
    g.after_permute = (prep_ran && !gemm_begin) ? 1 : 0;

    // Persistent grid: one CTA (pair: cluster of two) per SM (pair), never
    // more than there can be tiles.
    g.pair = pair ? 1 : 0;
    const int64_t tm = pair ? 2 * MX_BM : MX_BM, tn = pair ? 2 * MX_BNC : MX_BNC;
    const int64_t tiles = ((d.A + tm - 1) / tm + d.e) * ((d.N1 + tn - 1) / tn) +
                          (shared ? ((d.BS + tm - 1) / tm) * ((d.N2 + tn - 1) / tn) : 0);
    const int64_t units = std::max<int64_t>(1, std::min<int64_t>(pair ? sms / 2 : sms, tiles));
    g.grid = static_cast<int32_t>(units * (pair ? 2 : 1));
    const size_t smem = pair ? mx_smem_bytes<true>() : mx_smem_bytes<false>();
    auto kern = pair ? grouped_gemm_mx_kernel<true> : grouped_gemm_mx_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return A2AV_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.grid, 1, 1);
    cfg.blockDim = dim3(MX_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 0;
    if (pair) {
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = 2;
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    if (g.after_permute) {  // start beside the prep kernel; the producer waits for it before its first load
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    if (gemm_begin && cudaEventRecord(gemm_begin, stream) != cudaSuccess) return A2AV_ERR_CUDA;
    if (cudaLaunchKernelEx(&cfg, kern, g) != cudaSuccess) return A2AV_ERR_CUDA;
    if (gemm_end && cudaEventRecord(gemm_end, stream) != cudaSuccess) return A2AV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? A2AV_OK : A2AV_ERR_CUDA;
}

}  // namespace

extern "C" {

a2av_status a2av_gmm_mx_run(const a2av_gmm_mx_desc *desc, const void *ataOut_q, const void *ataOut_s,
                            const int32_t *recvCounts, const void *gmmWeight_q, const void *gmmWeight_s,
                            const void *mmX_q, const void *mmX_s, const void *mmWeight_q, const void *mmWeight_s,
                            void *permuteOut_q, void *permuteOut_s, void *gmmY, void *mmY, void *workspace,
                            size_t workspace_bytes, a2av_stream_t stream) {
    return mx_run_impl(desc, ataOut_q, ataOut_s, recvCounts, gmmWeight_q, gmmWeight_s, mmX_q, mmX_s, mmWeight_q,
                       mmWeight_s, permuteOut_q, permuteOut_s, gmmY, mmY, workspace, workspace_bytes, stream,
                       nullptr, nullptr);
}

a2av_status a2av_gmm_mx_run_profiled(const a2av_gmm_mx_desc *desc, const void *ataOut_q, const void *ataOut_s,
                                     const int32_t *recvCounts, const void *gmmWeight_q,
                                     const void *gmmWeight_s, const void *mmX_q, const void *mmX_s,
                                     const void *mmWeight_q, const void *mmWeight_s, void *permuteOut_q,
                                     void *permuteOut_s, void *gmmY, void *mmY, void *workspace,
                                     size_t workspace_bytes, a2av_stream_t stream, void *gemm_begin_event,
                                     void *gemm_end_event) {
    if (!gemm_begin_event || !gemm_end_event) return A2AV_ERR_NULLPTR;
    return mx_run_impl(desc, ataOut_q, ataOut_s, recvCounts, gmmWeight_q, gmmWeight_s, mmX_q, mmX_s, mmWeight_q,
                       mmWeight_s, permuteOut_q, permuteOut_s, gmmY, mmY, workspace, workspace_bytes, stream,
                       static_cast<cudaEvent_t>(gemm_begin_event), static_cast<cudaEvent_t>(gemm_end_event));
}

}  // extern "C"
