// Persistent ragged grouped GEMM on tcgen05 tensor cores (sm_103a).
//
// "aclnnAlltoAllvGroupedMatMul", Formula: gmmY = permuteOut x gmmWeight
// (routed experts, one [H1, N1] weight per local expert) and
// mmY = mmX x mmWeight (shared expert).  The page fuses the two ("parallel
// fusion with the MatMul for shared experts"); here the shared product is one
// more group in the same persistent launch.
//
// Tiles: 128 rows x bn columns (bn <= 256, chosen per group on the host),
// K in steps of 64 16-bit elements (one 128-byte swizzle row).  Per CTA:
//   warps 0-3  producers.  Split path: one thread issues TMA loads of the
//              expert-major A tile and the weight tile.  Fused path: the 128
//              threads gather A rows straight from ataOut with cp.async
//              (the permute happens in the operand load), written in the
//              128-byte-swizzled layout the tensor core reads; weights by TMA.
//              When permuteOut is wanted, each gathered A tile of the first
//              column tile is also stored to permuteOut by a TMA store.
//   warp 4     one thread issues tcgen05.mma (M=128, N=bn, K=16) into TMEM.
//   warps 5-8  epilogue: TMEM -> registers -> bf16/fp16 (nearest even) ->
//              global, rows past the group's end masked.
// TMEM holds two 128 x 256 fp32 accumulators so the epilogue of one tile
// overlaps the main loop of the next.  Every wait is bounded: on timeout the
// CTA records kStatusTimeout in the status word and winds down.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace a2av {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN_MAX = 256;
constexpr int STAGES = 4;
constexpr uint32_t A_STAGE_BYTES = BM * BK * 2;                  // 16 KB
constexpr uint32_t B_ATOM_BYTES = BK * 64 * 2;                   // 64 K-rows x 64 N: 8 KB
constexpr uint32_t B_STAGE_BYTES = (BN_MAX / 64) * B_ATOM_BYTES;  // 32 KB
constexpr int kProducerWarps = 4;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kMmaWarp = 4;
constexpr int kThreads = 9 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr int kGatherLag = 3;  // cp.async groups kept in flight per producer thread
constexpr uint64_t kWaitLimitNs = 2000000000ull;

static_assert(kGatherLag < STAGES, "gather lag must leave a free stage");

struct GroupInfo {
    int32_t row0;        // first A-operand row (routed: expert-major row)
    int32_t rows;
    int32_t tiles_n;
    int32_t tile_start;  // first linear tile of this group
};

struct Control {
    uint64_t full[STAGES];     // A and B of a stage are in shared memory
    uint64_t empty[STAGES];    // the MMAs reading a stage have completed
    uint64_t written[STAGES];  // fused path: every producer thread's rows landed
    uint64_t tfull[2];         // accumulator ready for the epilogue
    uint64_t tempty[2];        // epilogue drained the accumulator
    uint32_t tmem_base;
    int32_t abort;
    int32_t ngroups;
    int32_t total_tiles;
    int32_t store_x[STAGES];   // fused path: permuteOut tile coordinates per stage
    int32_t store_y[STAGES];
    GroupInfo g[kMaxExperts + 2];  // routed, shared, sentinel
    SegmentTable seg;
};

constexpr size_t kSmemBytes = 1024 + STAGES * (A_STAGE_BYTES + B_STAGE_BYTES) + sizeof(Control);

struct Tile {
    int g, m, n;
};

__device__ __forceinline__ Tile decode_tile(const Control &c, int t) {
    int g = 0;
    while (t >= c.g[g + 1].tile_start) ++g;
    const int local = t - c.g[g].tile_start;
    const int tn = c.g[g].tiles_n;
    return {g, local / tn, local % tn};
}

// Bounded wait on an mbarrier phase.  False: gave up (or another role did);
// the abort flag and the status word are set.
__device__ __noinline__ bool wait_phase(Control &c, uint64_t *bar, uint32_t parity, int32_t *status) {
    const uint32_t b = smem_u32(bar);
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(b, parity)) return true;
        if (*reinterpret_cast<volatile int32_t *>(&c.abort)) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *reinterpret_cast<volatile int32_t *>(&c.abort) = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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

template <bool BF16, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmLaunch p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t a_smem = base;
    const uint32_t b_smem = base + STAGES * A_STAGE_BYTES;
    Control &C = *reinterpret_cast<Control *>(base_ptr + STAGES * (A_STAGE_BYTES + B_STAGE_BYTES));

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int e = p.e;

    // ---- prologue: plan (warp 0), TMEM (MMA warp), barriers (warp 1)
    if (warp == 0) {
        const bool good = build_segment_table(p.recvCounts, p.W, e, p.A, C.seg, lane);
        const int tn1 = (p.N1 + p.bn1 - 1) / p.bn1;
        int row0 = 0, rows = 0, tiles = 0;
        if (lane < e) {
            row0 = C.seg.dst[lane * p.W];
            rows = C.seg.dst[(lane + 1) * p.W] - row0;
            tiles = good ? ((rows + BM - 1) / BM) * tn1 : 0;
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
                total += good ? ((p.BS + BM - 1) / BM) * tn2 : 0;
                ng = e + 1;
            }
            C.g[ng] = GroupInfo{0, 0, 1, total};
            C.ngroups = ng;
            C.total_tiles = total;
            C.abort = 0;
            if (blockIdx.x == 0) {
                if (p.write_status) *p.status = good ? 0 : kStatusBadCounts;
                else if (!good) atomicOr(p.status, kStatusBadCounts);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(smem_u32(&C.full[s]), 1);
                mbar_init(smem_u32(&C.empty[s]), 1);
                mbar_init(smem_u32(&C.written[s]), kProducerThreads);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(smem_u32(&C.tfull[a]), 1);
                mbar_init(smem_u32(&C.tempty[a]), 4);
            }
            fence_barrier_init();
        }
    } else if (warp == 2) {
        if (lane == 0) {
            if (!GATHER) prefetch_tensormap(&p.tmA_routed);
            prefetch_tensormap(&p.tmB_routed);
            if (p.BS > 0) {
                prefetch_tensormap(&p.tmA_shared);
                prefetch_tensormap(&p.tmB_shared);
            }
        }
    } else if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&C.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    const int total = C.total_tiles;

    if (warp < kProducerWarps) {
        // =========================================================== producers
        if (!GATHER) {
            if (threadIdx.x == 0) {
                uint32_t it = 0;  // stages issued
                bool ok = true;
                for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                    const Tile w = decode_tile(C, t);
                    const bool shared = w.g >= e;
                    const CUtensorMap *ta = shared ? &p.tmA_shared : &p.tmA_routed;
                    const CUtensorMap *tb = shared ? &p.tmB_shared : &p.tmB_routed;
                    const int K = shared ? p.H2 : p.H1;
                    const int bn = shared ? p.bn2 : p.bn1;
                    const int nb = (bn + 63) / 64;
                    const int y = C.g[w.g].row0 + w.m * BM;
                    const int xn = w.n * bn;
                    const int z = shared ? 0 : w.g;
                    const uint32_t bytes = A_STAGE_BYTES + nb * B_ATOM_BYTES;
                    const int kblocks = (K + BK - 1) / BK;
                    for (int kb = 0; kb < kblocks; ++kb, ++it) {
                        const int s = it % STAGES;
                        if (!wait_phase(C, &C.empty[s], ((it / STAGES) & 1) ^ 1, p.status)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_u32(&C.full[s]);
                        mbar_arrive_expect_tx(fb, bytes);
                        tma_load_2d(a_smem + s * A_STAGE_BYTES, ta, fb, kb * BK, y);
                        for (int c = 0; c < nb; ++c)
                            tma_load_3d(b_smem + s * B_STAGE_BYTES + c * B_ATOM_BYTES, tb, fb, xn + c * 64,
                                        kb * BK, z);
                    }
                }
                // Tail: wait until the MMAs released every stage we filled.
                for (int i = 0; i < STAGES && ok; ++i, ++it)
                    ok = wait_phase(C, &C.empty[it % STAGES], ((it / STAGES) & 1) ^ 1, p.status);
            }
        } else {
            const int ptid = threadIdx.x;     // 0..127
            const int chunk = lane & 7;       // 16-byte chunk of the 128-byte row slice
            const int rsub = warp * 32 + (lane >> 3);  // rows rsub + 4 * i, i < 8
            const uint16_t *ata = static_cast<const uint16_t *>(p.ataOut);
            const bool want_perm = p.permuteOut != nullptr;
            uint32_t issued = 0, completed = 0;
            uint32_t store_bits = 0;  // stages whose A tile goes to permuteOut
            bool ok = true;

            auto complete_oldest = [&]() -> bool {
                const int s = completed % STAGES;
                const uint32_t par = (completed / STAGES) & 1;
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&C.written[s]));
                bool good = true;
                if (ptid == 0) {
                    good = wait_phase(C, &C.written[s], par, p.status);
                    if (good) {
                        if ((store_bits >> s) & 1) {
                            tma_store_2d(&p.tmA_routed, a_smem + s * A_STAGE_BYTES, C.store_x[s],
                                         C.store_y[s]);
                            bulk_wait_read_all();
                        }
                        mbar_arrive(smem_u32(&C.full[s]));
                    }
                }
                ++completed;
                return good;
            };

            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile w = decode_tile(C, t);
                const bool shared = w.g >= e;
                const int K = shared ? p.H2 : p.H1;
                const int bn = shared ? p.bn2 : p.bn1;
                const int nb = (bn + 63) / 64;
                const int xn = w.n * bn;
                const int y = C.g[w.g].row0 + w.m * BM;
                const int kblocks = (K + BK - 1) / BK;
                const bool store = want_perm && !shared && w.n == 0;
                // Source row of each of this thread's 8 rows (nullptr: zero fill).
                const uint16_t *src[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = rsub + 4 * i;
                    if (!shared) {
                        const int d = y + r;  // expert-major row; may run into the next group
                        src[i] = d < p.A ? ata + static_cast<size_t>(source_row(C.seg, p.W, e, d)) * p.H1
                                         : nullptr;
                    } else {
                        src[i] = nullptr;  // shared rows arrive by TMA
                    }
                }
                for (int kb = 0; kb < kblocks; ++kb, ++issued) {
                    const int s = issued % STAGES;
                    if (!wait_phase(C, &C.empty[s], ((issued / STAGES) & 1) ^ 1, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_st = a_smem + s * A_STAGE_BYTES;
                    if (ptid == 0) {
                        const uint32_t fb = smem_u32(&C.full[s]);
                        const CUtensorMap *tb = shared ? &p.tmB_shared : &p.tmB_routed;
                        const int z = shared ? 0 : w.g;
                        asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(fb),
                                     "r"(nb * B_ATOM_BYTES + (shared ? A_STAGE_BYTES : 0u))
                                     : "memory");
                        if (shared) tma_load_2d(a_st, &p.tmA_shared, fb, kb * BK, y);
                        for (int c = 0; c < nb; ++c)
                            tma_load_3d(b_smem + s * B_STAGE_BYTES + c * B_ATOM_BYTES, tb, fb, xn + c * 64,
                                        kb * BK, z);
                        C.store_x[s] = kb * BK;
                        C.store_y[s] = y;
                    }
                    if (!shared) {
                        const int col = kb * BK + chunk * 8;
                        const bool col_ok = col < K;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int r = rsub + 4 * i;
                            const uint32_t dst = a_st + r * 128 + ((chunk ^ (r & 7)) << 4);
                            const bool live = col_ok && src[i] != nullptr;
                            cp_async_16_zfill(dst, live ? src[i] + col : ata, live ? 16u : 0u);
                        }
                    }
                    cp_async_commit();
                    store_bits = (store_bits & ~(1u << s)) | ((store ? 1u : 0u) << s);
                    if (issued + 1 - completed > kGatherLag) {
                        cp_async_wait<kGatherLag>();
                        if (!complete_oldest()) {
                            ok = false;
                            break;
                        }
                    }
                }
            }
            cp_async_wait<0>();
            while (ok && completed < issued) ok = complete_oldest();
            if (ptid == 0) {
                bulk_wait_all();
                for (int i = 0; i < STAGES && ok; ++i, ++issued)
                    ok = wait_phase(C, &C.empty[issued % STAGES], ((issued / STAGES) & 1) ^ 1, p.status);
            }
        }
    } else if (warp == kMmaWarp) {
        // =========================================================== MMA issuer
        if (lane == 0) {
            const uint32_t idesc1 = instr_desc_f16(BF16, BM, p.bn1);
            const uint32_t idesc2 = instr_desc_f16(BF16, BM, p.bn2 > 0 ? p.bn2 : 16);
            uint32_t it = 0, tl = 0;  // stages consumed, tiles done
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tl) {
                const Tile w = decode_tile(C, t);
                const bool shared = w.g >= e;
                const int K = shared ? p.H2 : p.H1;
                const uint32_t idesc = shared ? idesc2 : idesc1;
                const int kblocks = (K + BK - 1) / BK;
                const int acc = tl & 1;
                if (!wait_phase(C, &C.tempty[acc], ((tl >> 1) & 1) ^ 1, p.status)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = C.tmem_base + acc * kAccCols;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!wait_phase(C, &C.full[s], (it / STAGES) & 1, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a0 = a_smem + s * A_STAGE_BYTES;
                    const uint32_t b0 = b_smem + s * B_STAGE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // A: K-major, 128-byte swizzle, 8-row groups 1024 B apart;
                        //    a K step of 16 elements is 32 bytes along the row.
                        // B: N-major, 128-byte swizzle; 64-column atoms 8 KB apart
                        //    (leading offset), 8-row K groups 1024 B apart
                        //    (stride offset); a K step of 16 rows is 2 KB.
                        const uint64_t ad = smem_desc(a0 + kk * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(b0 + kk * 2048, B_ATOM_BYTES, 1024, kSwizzle128B);
                        mma_f16(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                    }
                    mma_commit(smem_u32(&C.empty[s]));
                }
                if (ok) mma_commit(smem_u32(&C.tfull[acc]));
            }
        }
    } else {
        // =========================================================== epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        uint32_t tl = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tl) {
            const Tile w = decode_tile(C, t);
            const bool shared = w.g >= e;
            const int acc = tl & 1;
            if (!wait_phase(C, &C.tfull[acc], (tl >> 1) & 1, p.status)) break;
            __syncwarp();  // lanes leave the wait independently; tcgen05.ld needs the whole warp
            tc_fence_after_sync();
            const int N = shared ? p.N2 : p.N1;
            const int bn = shared ? p.bn2 : p.bn1;
            const int row = w.m * BM + q * 32 + lane;
            const bool valid = row < C.g[w.g].rows;
            const int n0 = w.n * bn;
            const size_t out_row = static_cast<size_t>(shared ? row : C.g[w.g].row0 + row);
            uint16_t *out = static_cast<uint16_t *>(shared ? p.mmY : p.gmmY) + out_row * N + n0;
            const uint32_t t_base = C.tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
            const int nchunks = (bn + 31) / 32;
            for (int c = 0; c < nchunks; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + c * 32, r);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int col = c * 32 + v * 8;
                        if (col < bn && n0 + col < N) {
                            uint4 pk;
                            pk.x = pack2<BF16>(r[v * 8 + 0], r[v * 8 + 1]);
                            pk.y = pack2<BF16>(r[v * 8 + 2], r[v * 8 + 3]);
                            pk.z = pack2<BF16>(r[v * 8 + 4], r[v * 8 + 5]);
                            pk.w = pack2<BF16>(r[v * 8 + 6], r[v * 8 + 7]);
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
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(C.tmem_base, kTmemCols);
    }
}

template <bool BF16, bool GATHER>
cudaError_t launch_variant(const GemmLaunch &p, cudaStream_t stream) {
    auto kern = grouped_gemm_kernel<BF16, GATHER>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSmemBytes));
    if (err != cudaSuccess) return err;
    kern<<<p.grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t grouped_gemm_smem_bytes() { return kSmemBytes; }

cudaError_t launch_grouped_gemm(const GemmLaunch &p, cudaStream_t stream) {
    if (p.bf16) return p.gather ? launch_variant<true, true>(p, stream) : launch_variant<true, false>(p, stream);
    return p.gather ? launch_variant<false, true>(p, stream) : launch_variant<false, false>(p, stream);
}

}  // namespace a2av
