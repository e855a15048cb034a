// Persistent ragged grouped GEMM on tcgen05 tensor cores (sm_103a).
//
// "aclnnAlltoAllvGroupedMatMul", Formula: gmmY = permuteOut x gmmWeight
// (routed experts, one [H1, N1] weight per local expert) and
// mmY = mmX x mmWeight (shared expert).  The page fuses the two ("parallel
// fusion with the MatMul for shared experts"); here the shared product is one
// more group in the same persistent launch.
//
// Tiles: TILE_M rows x bn columns (bn <= 256, chosen per group on the host),
// K in steps of 64 16-bit elements (one 128-byte swizzle row).  Two tile
// shapes share the code:
//   single   one CTA computes a 128-row tile (tcgen05 cta_group::1);
//   pair     a cluster of two CTAs computes a 256-row tile with one
//            cta_group::2 MMA: each CTA stages its own 128 A rows and half of
//            the bn weight columns, so each CTA moves half the weight bytes
//            per FLOP.  The even CTA issues the MMAs; both hold half of the
//            accumulator rows in their own TMEM.
// Per CTA:
//   warp 0     producer.  Split path: one thread issues TMA loads of the
//              expert-major A rows and the weight columns.  Fused path: the
//              permute happens in the operand load: the CTA's 128 A rows are
//              read from their arrival places in ataOut, as one TMA box per
//              aligned block of rows that lies in one (source, expert)
//              segment and a TMA row gather (tile::gather4) for each 4-row
//              group that straddles a segment boundary, all landing in the
//              128-byte-swizzled layout the tensor core reads.
//   warps 1-3  fused path with permuteOut wanted: copy the rows of every
//              first-column tile from ataOut to permuteOut, independently of
//              the shared-memory pipeline.
//   warp 4     one thread issues tcgen05.mma (K=16 each) into TMEM.
//   warps 5-8  epilogue: TMEM -> registers -> bf16/fp16 (nearest even) ->
//              global, rows past the group's end masked.
// TMEM holds two 128-lane x 256-column fp32 accumulators so the epilogue of
// one tile overlaps the main loop of the next.  Every wait is bounded: on
// timeout the CTA records kStatusTimeout in the status word and winds down.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace a2av {

namespace {

constexpr int BM = 128;      // rows per CTA
constexpr int KCHUNK = 64;   // K elements in one 128-byte swizzle row
constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kThreads = 9 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;

// CH = 64-wide K chunks per pipeline stage (1 or 2).  With CH = 2 each stage
// holds 128 of K in the same bytes-in-flight budget as twice as many CH = 1
// stages, and is still one TMA load per operand: half the TMA instructions
// per FLOP, the issue rate being what bounds the main loop.
template <bool PAIR, int CH>
struct Shape {
    static constexpr int kCtas = PAIR ? 2 : 1;
    static constexpr int TILE_M = BM * kCtas;
    static constexpr int BK = KCHUNK * CH;                    // K per stage
    static constexpr uint32_t A_SUB_BYTES = BM * KCHUNK * 2;  // 16 KB: 128 rows x one chunk
    static constexpr uint32_t A_STAGE_BYTES = A_SUB_BYTES * CH;
    static constexpr uint32_t B_ATOM_BYTES = BK * 64 * 2;     // BK K-rows x 64 N columns
    // Weight columns one CTA stages: bn (<= 256) or bn / 2 (<= 128).
    static constexpr uint32_t B_STAGE_BYTES = (PAIR ? 2 : 4) * B_ATOM_BYTES;
    static constexpr int STAGES = (PAIR ? 6 : 4) / CH;
};

struct GroupInfo {
    int32_t row0;        // first A-operand row (routed: expert-major row)
    int32_t rows;
    int32_t tiles_n;
    int32_t tile_start;  // first linear tile of this group
};

// Arrival-driven start: the routed row tiles (each with all its column tiles)
// are taken in the order of the latest source their rows come from, so the
// units work on tiles whose rows have arrived while later sources are still
// landing.  Up to kMaxOrder row tiles; beyond that, group order.
constexpr int kMaxOrder = 2048;

template <int STAGES>
struct Control {
    uint64_t full[STAGES];     // A and B of a stage landed (pair: in both CTAs; used in the even CTA)
    uint64_t empty[STAGES];    // the MMAs reading a stage have completed
    uint64_t tfull[2];         // accumulator ready for the epilogue
    uint64_t tempty[2];        // epilogue drained the accumulator (pair: both CTAs, used in the even CTA)
    uint32_t tmem_base;
    int32_t abort;
    int32_t ngroups;
    int32_t total_tiles;
    int32_t routed_tiles;
    GroupInfo g[kMaxExperts + 2];  // routed, shared, sentinel
    SegmentTable seg;
    int32_t order_n;               // row tiles in `order` (0: group order)
    uint16_t order[kMaxOrder];     // routed row tiles by latest source (arrival-driven start)
};

// Epilogue staging: each epilogue warp turns its 32 rows x 32 columns of
// 16-bit results around in 2 KB of shared memory (two such buffers per warp,
// alternating), in the TMA's 64-byte swizzle; a block whose 32 rows are all
// in the group then goes out as one TMA store, any other as masked stores of
// 8 rows of 64 contiguous bytes.
constexpr uint32_t kEpiStageBytes = 2 * 32 * 64;
constexpr uint32_t kEpiBufBytes = 32 * 64;
constexpr int kEpiWarps = 4;

template <int STAGES>
__host__ __device__ constexpr size_t epi_stage_offset() {
    return (sizeof(Control<STAGES>) + 1023) / 1024 * 1024;  // the swizzle pattern repeats every 512 bytes
}

template <bool PAIR, int CH>
constexpr size_t smem_bytes() {
    using S = Shape<PAIR, CH>;
    return 1024 + S::STAGES * (S::A_STAGE_BYTES + S::B_STAGE_BYTES) + epi_stage_offset<S::STAGES>() +
           kEpiWarps * kEpiStageBytes;
}
static_assert(smem_bytes<true, 2>() <= 232448 && smem_bytes<true, 1>() <= 232448 &&
                  smem_bytes<false, 1>() <= 232448 && smem_bytes<false, 2>() <= 232448,
              "shared memory per CTA");

struct Tile {
    int g, m, n;
};

template <typename C>
__device__ __forceinline__ Tile decode_tile(const C &c, int t) {
    int g = 0;
    while (t >= c.g[g + 1].tile_start) ++g;
    const int local = t - c.g[g].tile_start;
    const int tn = c.g[g].tiles_n;
    return {g, local / tn, local % tn};
}

// Bounded wait on an mbarrier phase.  False: gave up (or another role did);
// the abort flag and the status word are set.  CLUSTER: acquire at cluster
// scope (the arrivals come from the peer CTA too).
template <bool CLUSTER = false>
__device__ __noinline__ bool wait_phase(int32_t *abort_flag, uint64_t *bar, uint32_t parity, int32_t *status,
                                        uint64_t limit_ns) {
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
        if (global_timer_ns() - t0 > limit_ns) {
            *reinterpret_cast<volatile int32_t *>(abort_flag) = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Arrival-driven start: bounded wait, by the whole warp, until sources
// w0 .. w1 have all arrived (arrived[w] == tag).  The flags are written by
// whatever moved the rows (a copy engine, a peer GPU, the host) after the
// rows themselves, so they are read at system scope, relaxed and all in
// flight at once, then ordered by one acquire fence; the rows are read next
// by TMA, hence the proxy fence.  On expiry the status word gets
// kStatusArrivalTimeout and the caller winds the kernel down.
__device__ __noinline__ bool wait_arrivals(int32_t *abort_flag, const uint64_t *arrived, int w0, int w1,
                                           uint64_t tag, int32_t *status, uint64_t limit_ns) {
    const int lane = threadIdx.x & 31;
    const auto all_arrived = [&]() {
        bool mine = true;
        for (int w = w0 + lane; w <= w1; w += 32) {
            uint64_t v;
            asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(arrived + w) : "memory");
            mine &= v == tag;
        }
        return __all_sync(0xffffffffu, mine);
    };
    if (!all_arrived()) {
        const uint64_t t0 = global_timer_ns();
        uint32_t pause = 256;  // backs off to 4 us: many CTAs poll while the rows stream in
        while (true) {
            bool done = false;
            for (int i = 0; i < 8 && !done; ++i) {
                __nanosleep(pause);
                pause = min(2u * pause, 4096u);
                done = all_arrived();
            }
            if (done) break;
            const bool give_up = *reinterpret_cast<volatile int32_t *>(abort_flag) ||
                                 global_timer_ns() - t0 > limit_ns;
            if (__any_sync(0xffffffffu, give_up)) {
                if (lane == 0) atomicOr(status, kStatusArrivalTimeout);
                return false;
            }
        }
    }
    asm volatile("fence.acq_rel.sys;\n\tfence.proxy.async.global;" ::: "memory");
    return true;
}

// Sources whose rows a routed tile half reads: expert-major rows
// [first, min(first + 128, group end)) of one expert lie in segments
// j * W + w0 .. j * W + w1.
__device__ __forceinline__ int2 sources_of_rows(const SegmentTable &t, int W, int e, int32_t first, int32_t g_end) {
    const int last = min(first + kHalfRows, g_end) - 1;
    return make_int2(segment_of(t, W, e, first) % W, segment_of(t, W, e, last) % W);
}

// ---- cluster (CTA pair) helpers

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// ---- TMA loads; PAIR: the barrier may live in the peer CTA (cta_group::2).

template <bool PAIR>
__device__ __forceinline__ void tma_2d(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y) {
    if constexpr (PAIR) {
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
            " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y)
            : "memory");
    } else {
        tma_load_2d(dst, tmap, bar, x, y);
    }
}

template <bool PAIR>
__device__ __forceinline__ void tma_3d(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y,
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

template <bool PAIR>
__device__ __forceinline__ void tma_4d(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y,
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

// Four rows (r0..r3, any order) of a 2-D tensor whose map has a one-row box;
// they land as a 4-row box at dst in the map's swizzled layout.
template <bool PAIR>
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t r0,
                                            int32_t r1, int32_t r2, int32_t r3) {
    if constexpr (PAIR) {
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
            ".cta_group::2 [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
            : "memory");
    } else {
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
            : "memory");
    }
}

// ---- tcgen05 for either tile shape

template <bool PAIR>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                    uint32_t accumulate) {
    if constexpr (PAIR) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        mma_f16(d_tmem, a_desc, b_desc, idesc, accumulate);
    }
}

// One arrival on `bar` (pair: on the barrier at that offset in both CTAs)
// when this thread's earlier tcgen05 operations have completed.
template <bool PAIR>
__device__ __forceinline__ void commit(uint32_t bar) {
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

template <bool PAIR>
__device__ __forceinline__ void tmem_alloc_all(uint32_t dst_smem) {
    if constexpr (PAIR) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        tmem_alloc(dst_smem, kTmemCols);
        tmem_relinquish();
    }
}

template <bool PAIR>
__device__ __forceinline__ void tmem_free_all(uint32_t taddr) {
    if constexpr (PAIR) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols)
                     : "memory");
    } else {
        tmem_dealloc(taddr, kTmemCols);
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) {
    const float a = __uint_as_float(lo), b = __uint_as_float(hi);
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    } else {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
}

// B_FIRST: each stage's weight load goes out before its A load (the host
// picks it when the weights are the operand a wave of units touches more of).
template <bool BF16, bool GATHER, bool PAIR, int CH, bool B_FIRST = false>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmLaunch p) {
    static_assert(CH == 1 || !GATHER, "row gathers use one-chunk stages");
    static_assert(!B_FIRST || (CH == 2 && !GATHER), "weights first only on two-chunk TMA stages");
    using S = Shape<PAIR, CH>;
    constexpr int BK = S::BK;
    constexpr uint32_t A_STAGE_BYTES = S::A_STAGE_BYTES;
    constexpr uint32_t B_ATOM_BYTES = S::B_ATOM_BYTES;
    constexpr int STAGES = S::STAGES;
    constexpr int TILE_M = S::TILE_M;
    constexpr int kCtas = S::kCtas;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t a_smem = base;
    const uint32_t b_smem = base + STAGES * A_STAGE_BYTES;
    Control<STAGES> &C =
        *reinterpret_cast<Control<STAGES> *>(base_ptr + STAGES * (A_STAGE_BYTES + S::B_STAGE_BYTES));
    const uint32_t epi0 = base + STAGES * (A_STAGE_BYTES + S::B_STAGE_BYTES) + epi_stage_offset<STAGES>();

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int e = p.e;
    const uint32_t rank = PAIR ? cluster_rank() : 0;  // 0: this CTA issues the MMAs
    const int unit = blockIdx.x / kCtas;                // CTA (pair) index in the persistent grid
    const int nunits = gridDim.x / kCtas;

    // ---- prologue: plan (warp 0), barriers (warp 1), TMEM (MMA warp)
    if (warp == 0) {
        const bool good = build_segment_table(p.recvCounts, p.W, e, p.A, C.seg, lane);
        const int tn1 = (p.N1 + p.bn1 - 1) / p.bn1;
        int row0 = 0, rows = 0, tiles = 0;
        if (lane < e) {
            row0 = C.seg.dst[lane * p.W];
            rows = C.seg.dst[(lane + 1) * p.W] - row0;
            tiles = good ? ((rows + TILE_M - 1) / TILE_M) * tn1 : 0;
        }
        int inc = tiles;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        if (lane < e) C.g[lane] = GroupInfo{row0, rows, tn1, inc - tiles};
        const int routed_total = __shfl_sync(0xffffffffu, inc, 31);
        if (lane == 0) {
            int ng = e, total = routed_total;
            if (p.BS > 0) {
                const int tn2 = (p.N2 + p.bn2 - 1) / p.bn2;
                C.g[e] = GroupInfo{0, p.BS, tn2, total};
                total += good ? ((p.BS + TILE_M - 1) / TILE_M) * tn2 : 0;
                ng = e + 1;
            }
            C.g[ng] = GroupInfo{0, 0, 1, total};
            C.ngroups = ng;
            C.total_tiles = total;
            C.routed_tiles = routed_total;
            C.abort = 0;
            C.order_n = 0;
            if (blockIdx.x == 0) {
                if (p.write_status) *p.status = good ? 0 : kStatusBadCounts;
                else if (!good) atomicOr(p.status, kStatusBadCounts);
            }
        }
        __syncwarp();
        const int total_m = tn1 > 0 ? routed_total / tn1 : 0;  // routed row tiles
        if (p.arrived != nullptr && good && total_m > 0 && total_m <= kMaxOrder) {
            // Stable counting sort of the row tiles by the latest source of
            // their rows (C.seg.tmp is free after the scan: the histogram).
            int32_t *base = C.seg.tmp;
            for (int w = lane; w < p.W; w += 32) base[w] = 0;
            __syncwarp();
            // key: the source of the tile's last row that belongs to its group
            const auto key_of = [&](int mt) {
                int g = 0;
                while (mt >= C.g[g + 1].tile_start / tn1) ++g;
                const int m = mt - C.g[g].tile_start / tn1;
                const int g_end = C.g[g].row0 + C.g[g].rows;
                const int last = min(C.g[g].row0 + (m + 1) * TILE_M, g_end) - 1;
                return segment_of(C.seg, p.W, e, last) % p.W;
            };
            for (int mt0 = 0; mt0 < total_m; mt0 += 32) {
                const int mt = mt0 + lane;
                const int k = mt < total_m ? key_of(mt) : p.W;  // p.W: no tile
                const uint32_t same = __match_any_sync(0xffffffffu, k);
                if (k < p.W && (same & ((1u << lane) - 1u)) == 0) base[k] += __popc(same);
                __syncwarp();
            }
            // exclusive prefix over the sources (base[] -> first slot of each key)
            int run = 0;
            for (int w0 = 0; w0 < p.W; w0 += 32) {
                const int w = w0 + lane;
                const int c = w < p.W ? base[w] : 0;
                int inc = c;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, inc, off);
                    if (lane >= off) inc += v;
                }
                if (w < p.W) base[w] = run + inc - c;
                run += __shfl_sync(0xffffffffu, inc, 31);
                __syncwarp();
            }
            for (int mt0 = 0; mt0 < total_m; mt0 += 32) {
                const int mt = mt0 + lane;
                const int k = mt < total_m ? key_of(mt) : p.W;
                const uint32_t same = __match_any_sync(0xffffffffu, k);
                const uint32_t before = same & ((1u << lane) - 1u);
                if (k < p.W) C.order[base[k] + __popc(before)] = static_cast<uint16_t>(mt);
                __syncwarp();
                if (k < p.W && before == 0) base[k] += __popc(same);
                __syncwarp();
            }
            if (lane == 0) C.order_n = total_m;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(smem_u32(&C.full[s]), 1);
                mbar_init(smem_u32(&C.empty[s]), 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(smem_u32(&C.tfull[a]), 1);
                mbar_init(smem_u32(&C.tempty[a]), 4 * kCtas);
            }
            fence_barrier_init();
        }
    } else if (warp == 2) {
        if (lane == 0) {
            if (p.A > 0) {
                prefetch_tensormap(&p.tmA_routed);
                prefetch_tensormap(&p.tmY_routed);
            }
            if (p.direct_halves) prefetch_tensormap(&p.tmA_direct);
            prefetch_tensormap(p.b4_routed ? &p.tmB4_routed : &p.tmB_routed);
            if (p.BS > 0) {
                prefetch_tensormap(&p.tmA_shared);
                prefetch_tensormap(p.b4_shared ? &p.tmB4_shared : &p.tmB_shared);
                prefetch_tensormap(&p.tmY_shared);
            }
        }
    } else if (warp == kMmaWarp) {
        tmem_alloc_all<PAIR>(smem_u32(&C.tmem_base));
    }
    tc_fence_before_sync();
    if constexpr (PAIR) cluster_sync_all();
    else __syncthreads();
    tc_fence_after_sync();

    const int total = C.total_tiles;
    const uint32_t full0 = smem_u32(&C.full[0]);
    // Tile order: routed groups, then the shared expert.  With shared_first
    // the shared tiles are rotated to the front (they read no exchanged
    // rows, so they run while the routed rows are still arriving).
    const int rot = (p.shared_first && total > C.routed_tiles) ? C.routed_tiles : 0;
    const int tn_routed = (p.N1 + p.bn1 - 1) / p.bn1;
    const auto tile_at = [&](int t) {
        int u = t + rot;
        if (u >= total) u -= total;
        if (u < C.routed_tiles && C.order_n > 0) {  // arrival order of the routed row tiles
            const int mt = C.order[u / tn_routed];
            int g = 0;
            while (mt >= C.g[g + 1].tile_start / tn_routed) ++g;
            return Tile{g, mt - C.g[g].tile_start / tn_routed, u % tn_routed};
        }
        return decode_tile(C, u);
    };

    if (warp < kProducerWarps) {
        // =========================================================== producers
        if (warp == 0) {
            uint32_t it = 0;  // stages issued
            bool ok = true;
            bool staged_ready = !p.after_permute;  // the permute kernel's rows are visible
            for (int t = unit; t < total && ok; t += nunits) {
                const Tile w = tile_at(t);
                const bool shared = w.g >= e;
                const CUtensorMap *tb = shared ? &p.tmB_shared : &p.tmB_routed;
                const CUtensorMap *tb4 = shared ? &p.tmB4_shared : &p.tmB4_routed;
                const bool b4 = shared ? p.b4_shared : p.b4_routed;
                const int K = shared ? p.H2 : p.H1;
                const int bn = shared ? p.bn2 : p.bn1;
                const int bnc = bn / kCtas;           // weight columns this CTA stages
                const int nb = (bnc + 63) / 64;
                const int y = C.g[w.g].row0 + w.m * TILE_M + rank * BM;  // this CTA's first row
                const int xn = w.n * bn + rank * bnc;
                const int z = shared ? 0 : w.g;
                const uint32_t bytes = kCtas * (A_STAGE_BYTES + nb * B_ATOM_BYTES);
                const int kblocks = (K + BK - 1) / BK;
                // Fused path: lane l owns tile rows 4l .. 4l+3 (expert-major rows
                // y + 4l + k; they may run past the group, and those results
                // are masked).  Rows of one segment come from consecutive
                // ataOut rows, so an aligned block of 8 .. 128 tile rows that
                // lies in one segment is one ordinary TMA box; only 4-row
                // groups that straddle a segment boundary (or the end of A)
                // use a row gather.  box_level: 0 = gather4 of this lane's
                // rows, k >= 1 = this lane loads the box of 4 << k rows it
                // starts, -1 = another lane's box covers these rows.
                // Split path: a half whose rows of this group lie in one segment
                // is read straight from ataOut; the permute kernel staged only
                // the halves that straddle a segment boundary.
                bool direct = false;
                int32_t direct_row = 0;
                if (!GATHER && !shared && p.direct_halves) {
                    const int g_end = C.g[w.g].row0 + C.g[w.g].rows;
                    if (y < g_end && half_in_one_segment(C.seg, p.W, e, y, g_end)) {
                        direct = true;
                        direct_row = source_row(C.seg, p.W, e, y);
                        // The half's rows of this group are one run of ataOut.
                        if (!in_bounds(direct_row >= 0 && direct_row + min(BM, g_end - y) <= p.A, p.status))
                            direct = false;
                    }
                }
                if (GATHER && !shared && p.arrived != nullptr) {
                    // Arrival-driven start: this half's rows must have
                    // arrived from every source they come from.  (Rows past
                    // the group's end are loaded too, but their products
                    // are discarded.)
                    const int g_end = C.g[w.g].row0 + C.g[w.g].rows;
                    if (y < g_end) {
                        const int2 ws = sources_of_rows(C.seg, p.W, e, y, g_end);
                        if (!wait_arrivals(&C.abort, p.arrived, ws.x, ws.y, p.arrival_tag, p.status,
                                           p.wait_limit_ns)) {
                            // Give up: first let the MMAs release every stage
                            // already filled (no copy left in flight), then
                            // make every role wind down.
                            if (lane == 0) {
                                for (int i = 0; i < STAGES; ++i, ++it)
                                    if (!wait_phase(&C.abort, &C.empty[it % STAGES], ((it / STAGES) & 1) ^ 1,
                                                    p.status, p.wait_limit_ns))
                                        break;
                                *reinterpret_cast<volatile int32_t *>(&C.abort) = 1;
                            }
                            ok = false;
                            break;
                        }
                    }
                }
                int32_t src[4] = {0, 0, 0, 0};
                int box_level = 0;
                if (GATHER && !shared) {
                    const int nseg = p.W * e;  // sentinel segment: past the last row
                    int seg_first = nseg, seg_last = nseg;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int d = y + 4 * lane + k;
                        const int sg = d < p.A ? segment_of(C.seg, p.W, e, d) : nseg;
                        src[k] = sg < nseg ? source_row_in(C.seg, p.W, e, sg, d) : p.A - 1;
                        if (!in_bounds(src[k] >= 0 && src[k] < p.A, p.status)) src[k] = p.A - 1;
                        if (k == 0) seg_first = sg;
                        if (k == 3) seg_last = sg;
                    }
                    int best = 0;
#pragma unroll
                    for (int k = 1; k <= 5; ++k) {
                        const int g0 = lane & ~((1 << k) - 1);
                        const int sf = __shfl_sync(0xffffffffu, seg_first, g0);
                        const int sl = __shfl_sync(0xffffffffu, seg_last, g0 + (1 << k) - 1);
                        if (sf == sl && sf < nseg) best = k;
                    }
                    box_level = best == 0 ? 0 : ((lane & ((1 << best) - 1)) == 0 ? best : -1);
                }
                if (!GATHER && !shared && !direct && !staged_ready) {
                    // This tile reads rows the permute kernel stages: wait for
                    // that grid (the tiles before needed none of its output).
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    staged_ready = true;
                }
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    bool free_slot = true;
                    if (lane == 0)
                        free_slot = wait_phase(&C.abort, &C.empty[s], ((it / STAGES) & 1) ^ 1, p.status, p.wait_limit_ns);
                    if (!__shfl_sync(0xffffffffu, free_slot, 0)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_own = full0 + s * sizeof(uint64_t);
                    const uint32_t fb = PAIR ? map_to_rank(fb_own, 0) : fb_own;  // the MMA CTA's barrier
                    const uint32_t a_st = a_smem + s * A_STAGE_BYTES;
                    if (lane == 0 && rank == 0) mbar_arrive_expect_tx(fb_own, bytes);
                    __syncwarp();
                    // The stage's weight columns: all its atoms in one load
                    // when the 4-D view applies.
                    auto load_b = [&]() {
                        if (b4)
                            tma_4d<PAIR>(b_smem + s * S::B_STAGE_BYTES, tb4, fb, 0, kb * BK, xn / 64, z);
                        else
                            for (int c = 0; c < nb; ++c)
                                tma_3d<PAIR>(b_smem + s * S::B_STAGE_BYTES + c * B_ATOM_BYTES, tb, fb,
                                             xn + c * 64, kb * BK, z);
                    };
                    if (B_FIRST && lane == 0) load_b();
                    if (GATHER && !shared) {
                        if (box_level == 0)
                            tma_gather4<PAIR>(a_st + lane * 512, &p.tmA_routed, fb, kb * BK, src[0], src[1],
                                              src[2], src[3]);
                        else if (box_level > 0)
                            tma_2d<PAIR>(a_st + lane * 512, &p.tmA_box[box_level - 1], fb, kb * BK, src[0]);
                    } else if (lane == 0) {
                        const CUtensorMap *ta = direct ? &p.tmA_direct : shared ? &p.tmA_shared : &p.tmA_routed;
                        const int ya = direct ? direct_row : shared ? w.m * TILE_M + static_cast<int>(rank) * BM : y;
                        if constexpr (CH == 1)
                            tma_2d<PAIR>(a_st, ta, fb, kb * BK, ya);
                        else  // 3-D view {64 columns, rows, K chunks}: CH chunks in one load
                            tma_3d<PAIR>(a_st, ta, fb, 0, ya, kb * CH);
                    }
                    if (!B_FIRST && lane == 0) load_b();
                }
            }
            // Tail: wait until the MMAs released every stage we filled.
            if (lane == 0)
                for (int i = 0; i < STAGES && ok; ++i, ++it)
                    ok = wait_phase(&C.abort, &C.empty[it % STAGES], ((it / STAGES) & 1) ^ 1, p.status, p.wait_limit_ns);
        } else if (GATHER && p.permuteOut != nullptr) {
            // Warps 1-3 write permuteOut for this CTA's rows of the tiles of
            // the first column, straight from ataOut (16-byte vectors, 4 in
            // flight per lane), independent of the shared-memory pipeline.
            const int cw = warp - 1;  // 0..2
            const int vpr = p.H1 / 8;
            const uint4 *ata = static_cast<const uint4 *>(p.ataOut);
            uint4 *perm = static_cast<uint4 *>(p.permuteOut);
            for (int t = unit; t < total; t += nunits) {
                const Tile w = tile_at(t);
                if (w.g >= e || w.n != 0) continue;
                const int first = w.m * TILE_M + static_cast<int>(rank) * BM;  // row within the group
                const int r_end = min(BM, C.g[w.g].rows - first);
                const int y = C.g[w.g].row0 + first;
                if (p.arrived != nullptr && r_end > 0) {
                    const int2 ws = sources_of_rows(C.seg, p.W, e, y, C.g[w.g].row0 + C.g[w.g].rows);
                    // (On expiry the producer, waiting for the same rows,
                    // winds the kernel down.)
                    if (!wait_arrivals(&C.abort, p.arrived, ws.x, ws.y, p.arrival_tag, p.status, p.wait_limit_ns))
                        break;
                }
                for (int r = cw; r < r_end; r += kProducerWarps - 1) {
                    const int d = y + r;
                    const uint4 *in = ata + static_cast<size_t>(source_row(C.seg, p.W, e, d)) * vpr;
                    uint4 *out = perm + static_cast<size_t>(d) * vpr;
                    int v = lane;
                    for (; v + 96 < vpr; v += 128) {
                        const uint4 a = in[v], b = in[v + 32], c = in[v + 64], f = in[v + 96];
                        out[v] = a;
                        out[v + 32] = b;
                        out[v + 64] = c;
                        out[v + 96] = f;
                    }
                    for (; v < vpr; v += 32) out[v] = in[v];
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // =========================================================== MMA issuer
        if (lane == 0 && rank == 0) {
            const uint32_t idesc1 = instr_desc_f16(BF16, TILE_M, p.bn1);
            const uint32_t idesc2 = instr_desc_f16(BF16, TILE_M, p.bn2 > 0 ? p.bn2 : 16);
            // A: K-major, 128-byte swizzle, 8-row groups 1024 B apart; a K
            //    step of 16 elements is 32 bytes along the row.
            // B: N-major, 128-byte swizzle; 64-column atoms 8 KB apart
            //    (leading offset), 8-row K groups 1024 B apart (stride
            //    offset); a K step of 16 rows is 2 KB.
            // Pair: both CTAs hold their operand halves at the same offsets.
            const uint64_t a_desc0 = smem_desc(a_smem, 16, 1024, kSwizzle128B);
            const uint64_t b_desc0 = smem_desc(b_smem, B_ATOM_BYTES, 1024, kSwizzle128B);
            const uint32_t empty0 = smem_u32(&C.empty[0]);
            uint32_t it = 0, tl = 0;  // stages consumed, tiles done
            bool ok = true;
            for (int t = unit; t < total && ok; t += nunits, ++tl) {
                const Tile w = tile_at(t);
                const bool shared = w.g >= e;
                const int K = shared ? p.H2 : p.H1;
                const uint32_t idesc = shared ? idesc2 : idesc1;
                const int kblocks = (K + BK - 1) / BK;
                const int acc = tl & 1;
                if (!wait_phase<PAIR>(&C.abort, &C.tempty[acc], ((tl >> 1) & 1) ^ 1, p.status, p.wait_limit_ns)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = C.tmem_base + acc * kAccCols;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t par = (it / STAGES) & 1;
                    // Operands arrive by TMA (async proxy), as the MMA reads
                    // them: the barrier phase alone orders the two, and no
                    // tcgen05 fence is needed here.
                    if (!mbar_try_wait(full0 + s * sizeof(uint64_t), par) &&
                        !wait_phase(&C.abort, &C.full[s], par, p.status, p.wait_limit_ns)) {
                        ok = false;
                        break;
                    }
                    // Descriptor start addresses are in 16-byte units, so a
                    // stage or K step is a plain add to the base descriptor.
                    const uint64_t ad0 = a_desc0 + ((s * A_STAGE_BYTES) >> 4);
                    const uint64_t bd0 = b_desc0 + ((s * S::B_STAGE_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // A: chunk kk / 4 (16 KB apart), 32 bytes per K step of 16 within it.
                        const uint32_t a_off = ((kk >> 2) * S::A_SUB_BYTES + (kk & 3) * 32) >> 4;
                        mma<PAIR>(d_tmem, ad0 + a_off, bd0 + 128 * kk, idesc, (kb | kk) != 0);
                    }
                    commit<PAIR>(empty0 + s * sizeof(uint64_t));
                }
                if (ok) commit<PAIR>(smem_u32(&C.tfull[acc]));
            }
        }
    } else {
        // =========================================================== epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        const uint32_t tempty0 = smem_u32(&C.tempty[0]);
        uint32_t tl = 0;
        uint32_t nblk = 0;  // blocks staged so far: the buffer alternates across tiles too
        for (int t = unit; t < total; t += nunits, ++tl) {
            const Tile w = tile_at(t);
            const bool shared = w.g >= e;
            const int acc = tl & 1;
            if (!wait_phase(&C.abort, &C.tfull[acc], (tl >> 1) & 1, p.status, p.wait_limit_ns)) break;
            __syncwarp();  // lanes leave the wait independently; tcgen05.ld needs the whole warp
            tc_fence_after_sync();
            const int N = shared ? p.N2 : p.N1;
            const int bn = shared ? p.bn2 : p.bn1;
            const int row = w.m * TILE_M + static_cast<int>(rank) * BM + q * 32 + lane;
            const bool valid = row < C.g[w.g].rows &&
                               in_bounds(static_cast<int64_t>(shared ? row : C.g[w.g].row0 + row) <
                                             static_cast<int64_t>(shared ? p.BS : p.A),
                                         p.status);
            const int n0 = w.n * bn;
            uint16_t *const out_base = static_cast<uint16_t *>(shared ? p.mmY : p.gmmY);
            const uint32_t t_base = C.tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
            const int nchunks = (bn + 31) / 32;
            // This warp's 32 rows: lane l holds row0w + l of the tile's group.
            // After the turn-around, lane l stores row row0w + 8k + l / 4,
            // 16 bytes at column 8 (l % 4) of the chunk, for k = 0 .. 3.
            const int row0w = row - lane;
            bool ok_k[4];
            uint16_t *out_k[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int rr = row0w + 8 * k + (lane >> 2);
                ok_k[k] = __shfl_sync(0xffffffffu, valid, 8 * k + (lane >> 2));
                const size_t orow = static_cast<size_t>(shared ? rr : C.g[w.g].row0 + rr);
                out_k[k] = out_base + orow * N + n0;
            }
            // 64-byte rows; the 16-byte chunk index is XORed with (row / 2) % 4
            // (the TMA's 64-byte swizzle), so that both the row-wise writes and
            // the column-wise reads touch eight distinct 16-byte slots of each
            // 128 bytes.
            const uint32_t stage = epi0 + static_cast<uint32_t>(warp - kMmaWarp - 1) * kEpiStageBytes;
            const bool all_rows = __all_sync(0xffffffffu, valid);
            const CUtensorMap *tmy = shared ? &p.tmY_shared : &p.tmY_routed;
            const int orow0 = shared ? row0w : C.g[w.g].row0 + row0w;
            for (int c = 0; c < nchunks; ++c) {
                const uint32_t buf = stage + (nblk++ & 1u) * kEpiBufBytes;
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c * 32, r);
                // Every block commits one bulk group (empty unless it went out by
                // TMA), so this wait leaves only the previous block's store
                // pending: the store that read this buffer two blocks ago is done.
                if (lane == 0) bulk_wait_read_1();
                __syncwarp();
                tmem_ld_wait();
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 pk;
                    pk.x = pack2<BF16>(r[v * 8 + 0], r[v * 8 + 1]);
                    pk.y = pack2<BF16>(r[v * 8 + 2], r[v * 8 + 3]);
                    pk.z = pack2<BF16>(r[v * 8 + 4], r[v * 8 + 5]);
                    pk.w = pack2<BF16>(r[v * 8 + 6], r[v * 8 + 7]);
                    st_shared_v4(buf + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4), pk);
                }
                // A block of whole rows inside this tile's columns goes out as
                // one TMA store (columns past N are clipped by the map);
                // anything else by masked stores.
                if (all_rows && (c + 1) * 32 <= bn && n0 + c * 32 < N) {
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(tmy, buf, n0 + c * 32, orow0);
                        bulk_commit_group();
                    }
                } else {
                    // An empty group, so that "all but the most recent group"
                    // above always means "all but the previous block's".
                    if (lane == 0) bulk_commit_group();
                    __syncwarp();
                    const int v = lane & 3;
                    const int col = c * 32 + v * 8;
                    const bool col_ok = col < bn && n0 + col < N;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int rr = 8 * k + (lane >> 2);
                        const uint4 val = ld_shared_v4(buf + rr * 64 + ((v ^ ((rr >> 1) & 3)) << 4));
                        if (ok_k[k] && col_ok) st_stream_v4(out_k[k] + col, val);
                    }
                }
                __syncwarp();  // the buffer is rewritten two blocks later
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                const uint32_t te = tempty0 + acc * sizeof(uint64_t);
                if constexpr (PAIR) mbar_arrive_cluster(map_to_rank(te, 0));
                else mbar_arrive(te);
            }
        }
        if (lane == 0) bulk_wait_all();  // this warp's TMA stores have landed
    }

    tc_fence_before_sync();
    if constexpr (PAIR) cluster_sync_all();
    else __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_free_all<PAIR>(C.tmem_base);
    }
}

template <bool BF16, bool GATHER, bool PAIR, int CH, bool B_FIRST = false>
cudaError_t launch_variant(const GemmLaunch &p, cudaStream_t stream) {
    auto kern = grouped_gemm_kernel<BF16, GATHER, PAIR, CH, B_FIRST>;
    constexpr size_t smem = smem_bytes<PAIR, CH>();
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (PAIR) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = Shape<PAIR, CH>::kCtas;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (p.after_permute) {  // start beside the permute kernel; the producer waits where it must
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    err = cudaLaunchKernelEx(&cfg, kern, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

template <bool BF16, bool GATHER, bool PAIR>
int max_units_for() {
    auto kern = grouped_gemm_kernel<BF16, GATHER, PAIR, 1>;
    constexpr size_t smem = smem_bytes<PAIR, 1>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 1024, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = Shape<PAIR, 1>::kCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace

size_t grouped_gemm_smem_bytes(int pair) { return pair ? smem_bytes<true, 1>() : smem_bytes<false, 1>(); }

int grouped_gemm_max_coresident(int pair) {
    // Clusters (pair) or CTAs (single) that fit on the device at once.
    return pair ? max_units_for<true, true, true>() : max_units_for<true, true, false>();
}

cudaError_t launch_grouped_gemm(const GemmLaunch &p, cudaStream_t stream) {
    const bool pair = p.pair != 0;
    if (p.kchunks == 2) {  // two-chunk stages: CTA pairs, TMA-fed A (no row gathers)
        if (!pair || p.gather) return cudaErrorInvalidValue;
        if (p.b_first)
            return p.bf16 ? launch_variant<true, false, true, 2, true>(p, stream)
                          : launch_variant<false, false, true, 2, true>(p, stream);
        return p.bf16 ? launch_variant<true, false, true, 2>(p, stream)
                      : launch_variant<false, false, true, 2>(p, stream);
    }
#define A2AV_LAUNCH(B, G)                                                                          \
    (pair ? launch_variant<B, G, true, 1>(p, stream) : launch_variant<B, G, false, 1>(p, stream))
    if (p.bf16) return p.gather ? A2AV_LAUNCH(true, true) : A2AV_LAUNCH(true, false);
    return p.gather ? A2AV_LAUNCH(false, true) : A2AV_LAUNCH(false, false);
#undef A2AV_LAUNCH
}

}  // namespace a2av
