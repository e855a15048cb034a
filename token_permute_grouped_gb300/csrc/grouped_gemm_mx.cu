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
// Tiles: 128 rows x 128 columns per CTA (cta_group::1); K in stages of 256
// codes: two 128-byte swizzle rows per operand row (two 16 KB sub-tiles),
// eight MMAs.  Per CTA:
//   warp 0     one thread issues a stage's TMA loads: 128 expert-major A rows
//              (staged by the permute kernel) and 128 K-major weight columns,
//              one 4-D load of both sub-tiles per operand.
//   warp 1     one thread issues the MMAs.
//   warps 2-5  scales: lane l loads the E8M0 scales of tile rows and tile
//              columns l, 32 + l, 64 + l, 96 + l, 16 bytes (two stages) at a
//              time, and writes each stage's two 32-bit words per row (byte i
//              of word j for MMA 4j + i) into TMEM with tcgen05.st: per word,
//              32 lanes x 4 columns, the layout the MMA reads, in the warp's
//              own lane quarter (each quarter holds a copy).
//   warps 6-9  epilogue: TMEM -> registers -> bf16 (nearest even) -> global,
//              rows past the group's end and columns past N masked.
// TMEM: two 128-column fp32 accumulators (the epilogue of one tile overlaps
// the main loop of the next), then per stage eight A-scale and eight B-scale
// columns.  Every wait is bounded: on timeout the CTA sets kStatusTimeout and
// winds down.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "a2av_gmm_mx.h"
#include "kernels.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace a2av {

namespace {

constexpr int MX_BM = 128;  // rows per tile
constexpr int MX_BN = 128;  // columns per tile
constexpr int MX_KCHUNK = 128;  // codes (bytes) in one 128-byte swizzle row
constexpr int MX_CH = 2;         // K chunks per stage
constexpr int MX_BK = MX_KCHUNK * MX_CH;
constexpr int MX_STAGES = 3;
constexpr int MX_THREADS = 10 * 32;
constexpr int kMxMmaWarp = 1;
constexpr int kMxScaleWarp0 = 2;
constexpr int kMxEpiWarp0 = 6;
constexpr uint32_t MX_SUB_BYTES = MX_BM * MX_KCHUNK;   // 16 KB: 128 rows x one chunk
constexpr uint32_t MX_TILE_BYTES = MX_SUB_BYTES * MX_CH;  // one operand's stage; B is the same size
constexpr uint32_t kMxTmemCols = 512;
constexpr uint32_t kMxAccCols = 128;
constexpr uint32_t kMxSfCol0 = 2 * kMxAccCols;
constexpr uint64_t kMxWaitLimitNs = 2000000000ull;

// Per stage: A scales in 4 columns per word (2 words), then B scales likewise.
__host__ __device__ constexpr uint32_t sfa_col(int s) { return kMxSfCol0 + 16u * s; }
__host__ __device__ constexpr uint32_t sfb_col(int s) { return kMxSfCol0 + 16u * s + 8u; }
static_assert(sfb_col(MX_STAGES - 1) + 8 <= kMxTmemCols, "scale columns must fit the TMEM allocation");

struct MxLaunch {
    const int32_t *recvCounts;
    int32_t W, e, A;
    int32_t H1, N1, BS, H2, N2;
    const uint8_t *a_s;   // [A, H1/32] expert-major scales (staged, or permuteOut_s)
    const uint8_t *w_s;   // [e, N1, H1/32]
    const uint8_t *x_s;   // [BS, H2/32]
    const uint8_t *mw_s;  // [N2, H2/32]
    void *gmmY;
    void *mmY;
    int32_t *status;
    int32_t write_status;
    int32_t qtype;  // 0 E4M3FN, 1 E5M2 (both operands)
    int32_t grid;
    // Code maps, all 4-D {128 codes, rows, K / 128 chunks, groups}, box
    // 128 x 128 x 2 x 1: one load is a stage's two 16 KB sub-tiles.
    CUtensorMap tmA;   // expert-major codes [A, H1]
    CUtensorMap tmB;   // weight codes [e, N1, H1]
    CUtensorMap tmX;   // mmX codes [BS, H2]
    CUtensorMap tmMW;  // mmWeight codes [N2, H2]
};

struct MxGroup {
    int32_t row0;  // first A row (routed: expert-major row)
    int32_t rows;
    int32_t tiles_n;
    int32_t tile_start;
};

struct MxControl {
    uint64_t full[MX_STAGES];     // a stage's codes landed
    uint64_t empty[MX_STAGES];    // the MMAs reading a stage (codes and scale columns) completed
    uint64_t sf_full[MX_STAGES];  // the stage's scale words are in TMEM (one arrival per scale warp)
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint32_t tmem_base;
    int32_t abort;
    int32_t total_tiles;
    MxGroup g[kMaxExperts + 2];  // routed, shared, sentinel
    SegmentTable seg;
};

constexpr size_t mx_smem_bytes() { return 1024 + MX_STAGES * 2 * MX_TILE_BYTES + sizeof(MxControl); }

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
// did), with the abort flag and the status word set.
__device__ __noinline__ bool mx_wait(int32_t *abort_flag, uint64_t *bar, uint32_t parity, int32_t *status) {
    const uint32_t b = smem_u32(bar);
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(b, parity)) return true;
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

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Thread i of the warp writes eight 32-bit words to lane (quarter base + i),
// columns [col, col + 8).
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tma_load_4d_mx(uint32_t dst, const void *tmap, uint32_t bar, int32_t x, int32_t y,
                                               int32_t z, int32_t w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__global__ void __launch_bounds__(MX_THREADS, 1) grouped_gemm_mx_kernel(const __grid_constant__ MxLaunch p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t a_smem = base;
    const uint32_t b_smem = base + MX_STAGES * MX_TILE_BYTES;
    MxControl &C = *reinterpret_cast<MxControl *>(base_ptr + 2 * MX_STAGES * MX_TILE_BYTES);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int e = p.e;

    // ---- prologue: plan (warp 0), barriers + TMEM (MMA warp), map prefetch (warp 2)
    if (warp == 0) {
        const bool good = build_segment_table(p.recvCounts, p.W, e, p.A, C.seg, lane);
        const int tn1 = (p.N1 + MX_BN - 1) / MX_BN;
        int row0 = 0, rows = 0, tiles = 0;
        if (lane < e) {
            row0 = C.seg.dst[lane * p.W];
            rows = C.seg.dst[(lane + 1) * p.W] - row0;
            tiles = good ? ((rows + MX_BM - 1) / MX_BM) * tn1 : 0;
        }
        int inc = tiles;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += v;
        }
        if (lane < e) C.g[lane] = MxGroup{row0, rows, tn1, inc - tiles};
        const int routed_total = __shfl_sync(0xffffffffu, inc, 31);
        if (lane == 0) {
            int ng = e, total = routed_total;
            if (p.BS > 0) {
                const int tn2 = (p.N2 + MX_BN - 1) / MX_BN;
                C.g[e] = MxGroup{0, p.BS, tn2, total};
                total += good ? ((p.BS + MX_BM - 1) / MX_BM) * tn2 : 0;
                ng = e + 1;
            }
            C.g[ng] = MxGroup{0, 0, 1, total};
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
                mbar_init(smem_u32(&C.full[s]), 1);
                mbar_init(smem_u32(&C.empty[s]), 1);
                mbar_init(smem_u32(&C.sf_full[s]), 4);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(smem_u32(&C.tfull[a]), 1);
                mbar_init(smem_u32(&C.tempty[a]), 4);
            }
            fence_barrier_init();
        }
        __syncwarp();
        tmem_alloc(smem_u32(&C.tmem_base), kMxTmemCols);
        tmem_relinquish();
    } else if (warp == 2) {
        if (lane == 0) {
            if (p.A > 0) {
                prefetch_tensormap(&p.tmA);
                prefetch_tensormap(&p.tmB);
            }
            if (p.BS > 0) {
                prefetch_tensormap(&p.tmX);
                prefetch_tensormap(&p.tmMW);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    const int total = C.total_tiles;
    const int stride = gridDim.x;

    if (warp == 0) {
        // =========================================================== TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += stride) {
                const MxTile w = mx_decode_tile(C, t);
                const bool shared = w.g >= e;
                const int K = shared ? p.H2 : p.H1;
                const CUtensorMap *ta = shared ? &p.tmX : &p.tmA;
                const CUtensorMap *tb = shared ? &p.tmMW : &p.tmB;
                const int ya = C.g[w.g].row0 + w.m * MX_BM;
                const int xn = w.n * MX_BN;
                const int z = shared ? 0 : w.g;
                for (int kb = 0; kb < K / MX_BK; ++kb, ++it) {
                    const int s = it % MX_STAGES;
                    if (!mx_wait(&C.abort, &C.empty[s], ((it / MX_STAGES) & 1) ^ 1, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&C.full[s]);
                    mbar_arrive_expect_tx(fb, 2 * MX_TILE_BYTES);
                    // {chunk column, row, chunk, group}: both chunks of the stage.
                    tma_load_4d_mx(a_smem + s * MX_TILE_BYTES, ta, fb, 0, ya, kb * MX_CH, 0);
                    tma_load_4d_mx(b_smem + s * MX_TILE_BYTES, tb, fb, 0, xn, kb * MX_CH, z);
                }
            }
            // Wait until the MMAs released every stage that was filled.
            for (int i = 0; i < MX_STAGES && ok; ++i, ++it)
                ok = mx_wait(&C.abort, &C.empty[it % MX_STAGES], ((it / MX_STAGES) & 1) ^ 1, p.status);
        }
    } else if (warp == kMxMmaWarp) {
        // =========================================================== MMA issuer
        if (lane == 0) {
            const uint32_t idesc0 = mx_idesc(static_cast<uint32_t>(p.qtype), MX_BM, MX_BN);
            // Both operands K-major with a 128-byte swizzle: 128-byte rows,
            // 8-row groups 1024 B apart; an MMA's K step of 32 codes is 32
            // bytes along the row (2 in the 16-byte address field), and the
            // second chunk of a stage starts 16 KB further on.
            const uint64_t a_desc0 = smem_desc(a_smem, 16, 1024, kSwizzle128B);
            const uint64_t b_desc0 = smem_desc(b_smem, 16, 1024, kSwizzle128B);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += stride, ++tl) {
                const MxTile w = mx_decode_tile(C, t);
                const int K = w.g >= e ? p.H2 : p.H1;
                const int acc = tl & 1;
                if (!mx_wait(&C.abort, &C.tempty[acc], ((tl >> 1) & 1) ^ 1, p.status)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = C.tmem_base + acc * kMxAccCols;
                for (int kb = 0; kb < K / MX_BK; ++kb, ++it) {
                    const int s = it % MX_STAGES;
                    const uint32_t par = (it / MX_STAGES) & 1;
                    if (!mx_wait(&C.abort, &C.full[s], par, p.status) ||
                        !mx_wait(&C.abort, &C.sf_full[s], par, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();  // the scale words came by tcgen05.st from other threads
                    const uint64_t ad = a_desc0 + ((s * MX_TILE_BYTES) >> 4);
                    const uint64_t bd = b_desc0 + ((s * MX_TILE_BYTES) >> 4);
                    const uint32_t sfa = C.tmem_base + sfa_col(s);
                    const uint32_t sfb = C.tmem_base + sfb_col(s);
#pragma unroll
                    for (int kk = 0; kk < MX_BK / 32; ++kk) {
                        const uint32_t off = ((kk >> 2) * MX_SUB_BYTES + (kk & 3) * 32) >> 4;
                        const uint32_t word = (kk >> 2) * 4;  // scale column group of this MMA
                        mma_mx(d_tmem, ad + off, bd + off, idesc0 | mx_sf_ids(kk & 3), sfa + word, sfb + word,
                               (kb | kk) != 0);
                    }
                    mma_commit(smem_u32(&C.empty[s]));
                }
                if (ok) mma_commit(smem_u32(&C.tfull[acc]));
            }
        }
    } else if (warp >= kMxScaleWarp0 && warp < kMxEpiWarp0) {
        // =========================================================== scale writers
        // The MMA reads the 128 scale bytes of a K block as 32 lanes x 4
        // columns: row (B: column) 32c + l at lane l, column base + c, and
        // each 32-lane quarter of TMEM holds the same copy.  A warp reaches
        // only its own quarter, so every scale warp writes the whole tile.
        const int q = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += stride) {
            const MxTile w = mx_decode_tile(C, t);
            const bool shared = w.g >= e;
            const int K = shared ? p.H2 : p.H1;
            const int N = shared ? p.N2 : p.N1;
            const int kblocks = K / MX_BK;
            const int64_t srow = K / 32;  // scale bytes per row
            const uint8_t *sa[4];
            const uint8_t *sb[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = 32 * c + lane;
                const int64_t arow = static_cast<int64_t>(C.g[w.g].row0) + w.m * MX_BM + r;
                const int64_t bcol = static_cast<int64_t>(w.n) * MX_BN + r;
                sa[c] = arow < (shared ? p.BS : p.A) ? (shared ? p.x_s : p.a_s) + arow * srow : nullptr;
                sb[c] = bcol < N ? (shared ? p.mw_s + bcol * srow : p.w_s + (static_cast<int64_t>(w.g) * N + bcol) * srow)
                                 : nullptr;
            }
            // Scales of two stages (16 bytes per row) at a time, one chunk ahead.
            const uint4 zero = make_uint4(0, 0, 0, 0);
            uint4 ca[4], cb[4], na[4], nb[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                ca[c] = sa[c] ? __ldg(reinterpret_cast<const uint4 *>(sa[c])) : zero;
                cb[c] = sb[c] ? __ldg(reinterpret_cast<const uint4 *>(sb[c])) : zero;
                na[c] = nb[c] = zero;
            }
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                if ((kb & 1) == 0) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (kb > 0) {
                            ca[c] = na[c];
                            cb[c] = nb[c];
                        }
                        if (kb + 2 < kblocks) {  // a stage's 8 scale bytes per row; 16 bytes cover two
                            na[c] = sa[c] ? __ldg(reinterpret_cast<const uint4 *>(sa[c] + (kb + 2) * 8)) : zero;
                            nb[c] = sb[c] ? __ldg(reinterpret_cast<const uint4 *>(sb[c] + (kb + 2) * 8)) : zero;
                        }
                    }
                }
                const int s = it % MX_STAGES;
                bool free_slot = true;
                if (lane == 0) free_slot = mx_wait(&C.abort, &C.empty[s], ((it / MX_STAGES) & 1) ^ 1, p.status);
                if (!__shfl_sync(0xffffffffu, free_slot, 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // Column 4j + c: word j of this stage for row (column) 32c + lane.
                const int j0 = (kb & 1) * 2;
                uint32_t wa[8], wb[8];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        wa[4 * j + c] = word_of(ca[c], j0 + j);
                        wb[4 * j + c] = word_of(cb[c], j0 + j);
                    }
                tmem_st_32x32b_x8(C.tmem_base + lane_base + sfa_col(s), wa);
                tmem_st_32x32b_x8(C.tmem_base + lane_base + sfb_col(s), wb);
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&C.sf_full[s]));
            }
        }
    } else {
        // =========================================================== epilogue
        const int q = warp & 3;
        uint32_t tl = 0;
        for (int t = blockIdx.x; t < total; t += stride, ++tl) {
            const MxTile w = mx_decode_tile(C, t);
            const bool shared = w.g >= e;
            const int acc = tl & 1;
            if (!mx_wait(&C.abort, &C.tfull[acc], (tl >> 1) & 1, p.status)) break;
            __syncwarp();  // lanes leave the wait independently; tcgen05.ld needs the whole warp
            tc_fence_after_sync();
            const int N = shared ? p.N2 : p.N1;
            const int row = w.m * MX_BM + q * 32 + lane;
            const bool valid = row < C.g[w.g].rows;
            const int n0 = w.n * MX_BN;
            const size_t out_row = static_cast<size_t>(shared ? row : C.g[w.g].row0 + row);
            uint16_t *out = static_cast<uint16_t *>(shared ? p.mmY : p.gmmY) + out_row * N + n0;
            const uint32_t t_base = C.tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kMxAccCols;
            for (int c = 0; c < MX_BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(t_base + c * 32, v);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int col = c * 32 + j * 8;
                        if (n0 + col < N) {
                            uint4 pk;
                            pk.x = pack_bf16(v[j * 8 + 0], v[j * 8 + 1]);
                            pk.y = pack_bf16(v[j * 8 + 2], v[j * 8 + 3]);
                            pk.z = pack_bf16(v[j * 8 + 4], v[j * 8 + 5]);
                            pk.w = pack_bf16(v[j * 8 + 6], v[j * 8 + 7]);
                            *reinterpret_cast<uint4 *>(out + col) = pk;
                        }
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&C.tempty[acc]));
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMxMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(C.tmem_base, kMxTmemCols);
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
    if (d->H1 % 512 != 0 || d->N1 % 8 != 0) return A2AV_ERR_UNSUPPORTED;
    if (d->BS > 0 && (d->H2 % 512 != 0 || d->N2 % 8 != 0)) return A2AV_ERR_UNSUPPORTED;
    return A2AV_OK;
}

size_t mx_staging_bytes(const a2av_gmm_mx_desc *d) {
    if (d->want_permute_out || d->A == 0) return 0;
    return align256(static_cast<size_t>(d->A) * d->H1) + align256(static_cast<size_t>(d->A) * d->H1 / 32);
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

int mx_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool mx_aligned16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace

}  // namespace a2av

extern "C" {

a2av_status a2av_gmm_mx_workspace_size(const a2av_gmm_mx_desc *desc, size_t *bytes) {
    if (!desc || !bytes) return A2AV_ERR_NULLPTR;
    const a2av_status s = a2av::mx_validate(desc);
    if (s != A2AV_OK) return s;
    *bytes = a2av::kMxStatusBytes + a2av::mx_staging_bytes(desc);
    return A2AV_OK;
}

a2av_status a2av_gmm_mx_run(const a2av_gmm_mx_desc *desc, const void *ataOut_q, const void *ataOut_s,
                            const int32_t *recvCounts, const void *gmmWeight_q, const void *gmmWeight_s,
                            const void *mmX_q, const void *mmX_s, const void *mmWeight_q, const void *mmWeight_s,
                            void *permuteOut_q, void *permuteOut_s, void *gmmY, void *mmY, void *workspace,
                            size_t workspace_bytes, a2av_stream_t stream_handle) {
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
    g.w_s = static_cast<const uint8_t *>(gmmWeight_s);
    g.x_s = static_cast<const uint8_t *>(mmX_s);
    g.mw_s = static_cast<const uint8_t *>(mmWeight_s);
    g.gmmY = gmmY;
    g.mmY = mmY;
    g.status = status;
    g.qtype = d.qtype;
    if (!mx_codes_map(&g.tmB, gmmWeight_q, d.e, d.N1, d.H1)) return A2AV_ERR_CUDA;
    if (shared) {
        if (!mx_codes_map(&g.tmX, mmX_q, 1, d.BS, d.H2)) return A2AV_ERR_CUDA;
        if (!mx_codes_map(&g.tmMW, mmWeight_q, 1, d.N2, d.H2)) return A2AV_ERR_CUDA;
    }
    bool permute_ran = false;
    if (routed) {
        // Expert-major codes and scales: into permuteOut, or into the staging area.
        uint8_t *dq = static_cast<uint8_t *>(permuteOut_q);
        uint8_t *ds = static_cast<uint8_t *>(permuteOut_s);
        if (!d.want_permute_out) {
            dq = static_cast<uint8_t *>(workspace) + kMxStatusBytes;
            ds = dq + align256(static_cast<size_t>(d.A) * d.H1);
        }
        // The row permute moves 16-byte vectors of rows given in 2-byte
        // elements: a code row is H1 / 2 of them, a scale row H1 / 64.
        PermuteLaunch pq{recvCounts, d.W, d.e, static_cast<int32_t>(d.A), static_cast<int32_t>(d.H1 / 2),
                         ataOut_q, dq, status, 1, 0};
        PermuteLaunch ps{recvCounts, d.W, d.e, static_cast<int32_t>(d.A), static_cast<int32_t>(d.H1 / 64),
                         ataOut_s, ds, status, 0, 0};
        if (launch_permute(pq, sms, stream) != cudaSuccess) return A2AV_ERR_CUDA;
        if (launch_permute(ps, sms, stream) != cudaSuccess) return A2AV_ERR_CUDA;
        permute_ran = true;
        if (!mx_codes_map(&g.tmA, dq, 1, d.A, d.H1)) return A2AV_ERR_CUDA;
        g.a_s = ds;
    }
    g.write_status = permute_ran ? 0 : 1;

    const int64_t tiles = ((d.A + MX_BM - 1) / MX_BM + d.e) * ((d.N1 + MX_BN - 1) / MX_BN) +
                          (shared ? ((d.BS + MX_BM - 1) / MX_BM) * ((d.N2 + MX_BN - 1) / MX_BN) : 0);
    g.grid = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(sms, tiles)));
    constexpr size_t smem = mx_smem_bytes();
    if (cudaFuncSetAttribute(grouped_gemm_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return A2AV_ERR_CUDA;
    grouped_gemm_mx_kernel<<<g.grid, MX_THREADS, smem, stream>>>(g);
    return cudaGetLastError() == cudaSuccess ? A2AV_OK : A2AV_ERR_CUDA;
}

}  // extern "C"
