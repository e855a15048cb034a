// C ABI of the library (declared in include/a2av_gmm.h).
//
// Two-phase call of the "aclnnAlltoAllvGroupedMatMul" page: phase 1 checks the
// parameters and sizes the workspace ("The first-phase API implements input
// parameter verification"), phase 2 runs on a stream.  Limits come from the
// page's "Shape variables" list.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "a2av_gmm.h"
#include "kernels.h"
#include "plan.cuh"

// Scratch for a2av_gmm_run_static_scratch: callers that cannot allocate get
// this array instead of a workspace.  One per device, alive until exit.
static __device__ __align__(256) uint8_t g_static_scratch[A2AV_STATIC_SCRATCH_BYTES];

namespace {

constexpr size_t kStatusBytes = 256;  // status word, padded to keep what follows aligned
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bound on every device-side wait
constexpr int kMaxDevices = 64;
constexpr int kBM = 128;

bool mult8(int64_t v) { return v % 8 == 0; }

a2av_status validate(const a2av_gmm_desc *d) {
    if (!d) return A2AV_ERR_NULLPTR;
    if (d->W < 1 || d->e < 1 || d->e > a2av::kMaxExperts) return A2AV_ERR_INVALID;
    if (static_cast<int64_t>(d->W) * d->e > a2av::kMaxSegments) return A2AV_ERR_INVALID;
    if (d->H1 <= 0 || d->H1 >= 65536 || d->N1 <= 0 || d->N1 >= 65536) return A2AV_ERR_INVALID;
    if (d->A < 0 || d->A > INT32_MAX) return A2AV_ERR_INVALID;
    if (d->BS < 0 || d->BS > INT32_MAX) return A2AV_ERR_INVALID;
    if (d->BS > 0) {
        if (d->H2 <= 0 || d->H2 > 12288 || d->N2 <= 0 || d->N2 >= 65536) return A2AV_ERR_INVALID;
    }
    if (d->dtype != A2AV_BF16 && d->dtype != A2AV_FP16) return A2AV_ERR_INVALID;
    if (d->path < A2AV_PATH_DEFAULT || d->path > A2AV_PATH_SPLIT_RUNS) return A2AV_ERR_INVALID;
    if (d->tiles < A2AV_TILES_DEFAULT || d->tiles > A2AV_TILES_PAIR_K64) return A2AV_ERR_INVALID;
    if (!mult8(d->H1) || !mult8(d->N1)) return A2AV_ERR_UNSUPPORTED;
    if (d->BS > 0 && (!mult8(d->H2) || !mult8(d->N2))) return A2AV_ERR_UNSUPPORTED;
    return A2AV_OK;
}

// Default: SPLIT_RUNS.  The permute kernel stages only the 128-row halves of
// a tile that straddle a (source, expert) segment boundary, and the GEMM
// reads every other half in place from ataOut; which halves those are is
// decided on the device, from recvCounts, so no host-side threshold on the
// shapes is involved.  Measured on GB300 it matches or beats staging every
// row (SPLIT) on all the workloads, by 16 % on the 262K-row one, and the
// one-kernel row-gathering FUSED path everywhere.
int resolve_path(const a2av_gmm_desc *d) {
    if (d->path != A2AV_PATH_DEFAULT) return d->path;
    return A2AV_PATH_SPLIT_RUNS;
}

bool use_split(const a2av_gmm_desc *d) { return resolve_path(d) != A2AV_PATH_FUSED; }

bool use_pair(const a2av_gmm_desc *d) { return d->tiles != A2AV_TILES_SINGLE; }

// Clusters (pair) or CTAs (single) of the GEMM that fit on the device at once.
int coresident_units(bool pair) {
    static int cache[kMaxDevices][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int &c = cache[dev][pair ? 1 : 0];
    if (c == 0) c = a2av::grouped_gemm_max_coresident(pair ? 1 : 0);
    return c;
}

// Bytes of the expert-major staging buffer the split path needs when the
// caller does not ask for permuteOut.
size_t staging_bytes(const a2av_gmm_desc *d) {
    if (!use_split(d) || d->want_permute_out || d->A == 0) return 0;
    const size_t b = static_cast<size_t>(d->A) * d->H1 * 2;
    return (b + 255) / 256 * 256;
}

// Tile width.  When N is a multiple of 64 the width is a whole number of
// 64-column atoms per CTA, so a stage's weight columns are one TMA load (the
// TMA issue rate, not bandwidth, bounds the main loop): up to 256, the last
// tile zero-filled past N.  Otherwise the fewest column tiles of at most 256,
// each the narrowest multiple of 16 that covers N.
int pick_bn(int64_t N, int ctas) {
    const int64_t atom = 64 * ctas;
    if (N % 64 == 0) return static_cast<int>(std::min<int64_t>(256, (N + atom - 1) / atom * atom));
    const int64_t tiles = (N + 255) / 256;
    int64_t bn = (N + tiles - 1) / tiles;
    bn = (bn + 15) / 16 * 16;
    return static_cast<int>(std::max<int64_t>(bn, 16));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

CUtensorMapDataType tmap_type(int32_t dtype) {
    return dtype == A2AV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// [rows, cols] row-major; box = 64 columns x box_rows rows, 128-byte swizzle.
// box_rows = 128 for tile loads, 1 for row gathers (tile::gather4).
bool make_rows_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int32_t dtype,
                   uint32_t box_rows = kBM) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, tmap_type(dtype), 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, cols] row-major output; box = 32 columns x 32 rows, 64-byte
// swizzle: the layout in which an epilogue warp turns a block around in
// shared memory before the TMA store.
bool make_out_map(CUtensorMap *m, void *ptr, int64_t rows, int64_t cols, int32_t dtype) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, tmap_type(dtype), 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// [groups, K, N] row-major weights; box = 64 columns (N) x 64 rows (K) x 1.
bool make_weight_map(CUtensorMap *m, const void *ptr, int64_t groups, int64_t K, int64_t N, int32_t dtype) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K),
                          static_cast<cuuint64_t>(groups)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(N * 2), static_cast<cuuint64_t>(K * N * 2)};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, tmap_type(dtype), 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, cols] seen as 3-D {64 columns, rows, cols / 64 chunks}; box = 64
// columns x 128 rows x 2 chunks: one load brings 128 of K as two 16 KB
// K-major swizzled sub-tiles.  Needs cols % 128 == 0.
bool make_rows_map_chunks(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, int32_t dtype) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols * 2), 128};
    cuuint32_t box[3] = {64, kBM, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, tmap_type(dtype), 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same weights seen as 4-D: [groups][N / 64 atoms][K][64 columns], box =
// 64 columns x kbox K rows x `atoms` atoms.  One load then fills a stage's
// weight columns in the layout of consecutive 64-column atoms (kbox * 128 B
// apart), the same bytes as `atoms` loads of the 3-D map.  Needs N % 64 == 0.
bool make_weight_map_atoms(CUtensorMap *m, const void *ptr, int64_t groups, int64_t K, int64_t N,
                           int32_t dtype, uint32_t atoms, uint32_t kbox) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N / 64),
                          static_cast<cuuint64_t>(groups)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(N * 2), 128, static_cast<cuuint64_t>(K * N * 2)};
    cuuint32_t box[4] = {64, kbox, atoms, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, tmap_type(dtype), 4, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= kMaxDevices) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of g_static_scratch in the current device's context.  In
// host code the symbol name is only a host-side stand-in, never a device
// address, so it must go through cudaGetSymbolAddress.  The lookup is a
// host-side query that allocates nothing; it is repeated on every call
// rather than cached, because a context torn down and created again (after
// cudaDeviceReset, for one) loads the module afresh and the array may then
// sit at another address.
void *static_scratch_address() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
    return p;
}

}  // namespace

extern "C" {

a2av_status a2av_gmm_workspace_size(const a2av_gmm_desc *desc, size_t *bytes) {
    if (!desc || !bytes) return A2AV_ERR_NULLPTR;
    const a2av_status s = validate(desc);
    if (s != A2AV_OK) return s;
    *bytes = kStatusBytes + staging_bytes(desc);
    return A2AV_OK;
}

int32_t a2av_gmm_launch_count(const a2av_gmm_desc *desc) {
    if (validate(desc) != A2AV_OK) return 0;
    return (use_split(desc) && desc->A > 0) ? 2 : 1;
}

}  // extern "C"

namespace {

// The body of a2av_gmm_run.  With gemm_begin / gemm_end set, those events
// are recorded on the stream right before and right after the GEMM launch
// (which then starts after the permute kernel in plain stream order).
a2av_status run_impl(const a2av_gmm_desc *desc, const void *ataOut, const int32_t *recvCounts,
                     const void *gmmWeight, const void *mmX, const void *mmWeight, void *permuteOut, void *gmmY,
                     void *mmY, void *workspace, size_t workspace_bytes, a2av_stream_t stream_handle,
                     cudaEvent_t gemm_begin, cudaEvent_t gemm_end, const uint64_t *arrived = nullptr,
                     uint64_t arrival_tag = 0, uint64_t wait_limit_ns = kWaitLimitNs) {
    const a2av_status vs = validate(desc);
    if (vs != A2AV_OK) return vs;
    const a2av_gmm_desc &d = *desc;
    const bool has_routed = d.A > 0;
    const bool has_shared = d.BS > 0;
    if (!recvCounts || !gmmWeight || !workspace) return A2AV_ERR_NULLPTR;
    if (has_routed && (!ataOut || !gmmY)) return A2AV_ERR_NULLPTR;
    if (has_routed && d.want_permute_out && !permuteOut) return A2AV_ERR_NULLPTR;
    if (has_shared && (!mmX || !mmWeight || !mmY)) return A2AV_ERR_NULLPTR;
    const void *ptrs[] = {ataOut, gmmWeight, mmX, mmWeight, gmmY, mmY,
                          d.want_permute_out ? permuteOut : nullptr};
    for (const void *q : ptrs)
        if (!aligned16(q)) return A2AV_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(recvCounts) & 3u) != 0) return A2AV_ERR_UNSUPPORTED;
    size_t need = 0;
    a2av_gmm_workspace_size(desc, &need);
    if (workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return A2AV_ERR_WORKSPACE;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    const int sms = sm_count();
    if (sms <= 0) return A2AV_ERR_CUDA;
    int32_t *status = static_cast<int32_t *>(workspace);
    void *perm_out = d.want_permute_out ? permuteOut : nullptr;
    const bool split = use_split(&d);

    a2av::GemmLaunch g;
    std::memset(&g, 0, sizeof g);
    g.recvCounts = recvCounts;
    g.W = d.W;
    g.e = d.e;
    g.A = static_cast<int32_t>(d.A);
    g.H1 = static_cast<int32_t>(d.H1);
    g.N1 = static_cast<int32_t>(d.N1);
    g.bn1 = pick_bn(d.N1, use_pair(&d) ? 2 : 1);
    g.BS = has_shared ? static_cast<int32_t>(d.BS) : 0;
    g.H2 = has_shared ? static_cast<int32_t>(d.H2) : 0;
    g.N2 = has_shared ? static_cast<int32_t>(d.N2) : 0;
    g.bn2 = has_shared ? pick_bn(d.N2, use_pair(&d) ? 2 : 1) : 0;
    g.gmmY = gmmY;
    g.mmY = mmY;
    if (has_routed && !make_out_map(&g.tmY_routed, gmmY, d.A, d.N1, d.dtype)) return A2AV_ERR_CUDA;
    if (has_shared && !make_out_map(&g.tmY_shared, mmY, d.BS, d.N2, d.dtype)) return A2AV_ERR_CUDA;
    g.status = status;
    g.bf16 = d.dtype == A2AV_BF16;
    g.gather = split ? 0 : 1;
    g.ataOut = ataOut;
    g.permuteOut = split ? nullptr : perm_out;

    // One-load weight stages where the columns come in whole 64-wide atoms;
    // two-chunk (128-deep) stages on CTA pairs where, in addition, both K's
    // are multiples of 128 and A is TMA-fed (not row-gathered).
    const int cta_cols = use_pair(&d) ? 2 : 1;
    const bool b4r = d.N1 % 64 == 0 && (g.bn1 / cta_cols) % 64 == 0;
    const bool b4s = has_shared && d.N2 % 64 == 0 && (g.bn2 / cta_cols) % 64 == 0;
    const bool wide = use_pair(&d) && d.tiles != A2AV_TILES_PAIR_K64 && split && b4r &&
                      (!has_shared || b4s) && d.H1 % 128 == 0 && (!has_shared || d.H2 % 128 == 0);
    g.kchunks = wide ? 2 : 1;
    const uint32_t kbox = wide ? 128 : 64;
    auto rows_map = [&](CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols) {
        return wide ? make_rows_map_chunks(m, ptr, rows, cols, d.dtype) : make_rows_map(m, ptr, rows, cols, d.dtype);
    };
    if (!make_weight_map(&g.tmB_routed, gmmWeight, d.e, d.H1, d.N1, d.dtype)) return A2AV_ERR_CUDA;
    if (has_shared) {
        if (!rows_map(&g.tmA_shared, mmX, d.BS, d.H2)) return A2AV_ERR_CUDA;
        if (!make_weight_map(&g.tmB_shared, mmWeight, 1, d.H2, d.N2, d.dtype)) return A2AV_ERR_CUDA;
    }
    if (b4r) {
        if (!make_weight_map_atoms(&g.tmB4_routed, gmmWeight, d.e, d.H1, d.N1, d.dtype, g.bn1 / cta_cols / 64,
                                   kbox))
            return A2AV_ERR_CUDA;
        g.b4_routed = 1;
    }
    if (b4s) {
        if (!make_weight_map_atoms(&g.tmB4_shared, mmWeight, 1, d.H2, d.N2, d.dtype, g.bn2 / cta_cols / 64, kbox))
            return A2AV_ERR_CUDA;
        g.b4_shared = 1;
    }

    bool permute_ran = false;
    if (has_routed) {
        if (split) {
            // Expert-major rows go to permuteOut, or to the staging area.
            void *dst = perm_out ? perm_out : static_cast<uint8_t *>(workspace) + kStatusBytes;
            // SPLIT_RUNS without permuteOut: only the 128-row halves that
            // straddle a segment boundary are staged; the GEMM reads the rest
            // in place.
            const int32_t partial = (!perm_out && resolve_path(&d) == A2AV_PATH_SPLIT_RUNS) ? 1 : 0;
            // Eight permute blocks per SM (all resident at once).  The GEMM
            // is launched beside it (programmatic dependent launch) and waits
            // only before staged rows; in practice its CTAs find SMs as the
            // permute blocks retire.
            a2av::PermuteLaunch pl{recvCounts, d.W, d.e, static_cast<int32_t>(d.A),
                                   static_cast<int32_t>(d.H1), ataOut, dst, status, 1, partial, 8};
            g.after_permute = 1;
            if (a2av::launch_permute(pl, sms, stream) != cudaSuccess) return A2AV_ERR_CUDA;
            permute_ran = true;
            if (!rows_map(&g.tmA_routed, dst, d.A, d.H1)) return A2AV_ERR_CUDA;
            if (partial) {
                if (!rows_map(&g.tmA_direct, ataOut, d.A, d.H1)) return A2AV_ERR_CUDA;
                g.direct_halves = 1;
            }
        } else {
            // Maps over ataOut in arrival order: a one-row box for row gathers,
            // and 8 .. 128-row boxes for runs of rows from one segment.
            if (!make_rows_map(&g.tmA_routed, ataOut, d.A, d.H1, d.dtype, 1)) return A2AV_ERR_CUDA;
            for (int k = 0; k < 5; ++k)
                if (!make_rows_map(&g.tmA_box[k], ataOut, d.A, d.H1, d.dtype, 8u << k)) return A2AV_ERR_CUDA;
        }
    }
    g.write_status = permute_ran ? 0 : 1;
    g.wait_limit_ns = wait_limit_ns;
    g.arrived = arrived;
    g.arrival_tag = arrival_tag;
    g.shared_first = arrived != nullptr ? 1 : 0;

    // Persistent grid: as many CTAs (pair: clusters of two) as fit on the
    // device at once, never more than there can be tiles.
    const bool pair = use_pair(&d);
    const int64_t tile_m = pair ? 2 * kBM : kBM;
    const int64_t tn1 = (d.N1 + g.bn1 - 1) / g.bn1;
    int64_t tiles = ((d.A + tile_m - 1) / tile_m + d.e) * tn1;
    if (has_shared) tiles += ((d.BS + tile_m - 1) / tile_m) * ((d.N2 + g.bn2 - 1) / g.bn2);
    int units = coresident_units(pair);
    if (units <= 0) units = pair ? sms / 2 : sms;
    g.pair = pair ? 1 : 0;
    const int64_t n_units = std::max<int64_t>(1, std::min<int64_t>(units, tiles));
    g.grid = static_cast<int32_t>(n_units * (pair ? 2 : 1));
    // Which operand of a stage to request first: the one a wave of units
    // touches more of, as it is the likelier to come from DRAM rather than
    // L2.  With tn column tiles per group, a wave covers about n_units / tn
    // row tiles of a group's A and all tn of its column tiles, so the
    // weights are the larger footprint when tn * tn > n_units.  Weights
    // first only when that holds for every group with tiles.
    {
        const int64_t tn2 = has_shared ? (d.N2 + g.bn2 - 1) / g.bn2 : 0;
        const bool routed_b = d.A == 0 || tn1 * tn1 > n_units;
        const bool shared_b = !has_shared || tn2 * tn2 > n_units;
        g.b_first = (g.kchunks == 2 && routed_b && shared_b && (d.A > 0 || has_shared)) ? 1 : 0;
    }
    if (gemm_begin) {
        g.after_permute = 0;  // an event between the kernels: plain stream order
        if (cudaEventRecord(gemm_begin, stream) != cudaSuccess) return A2AV_ERR_CUDA;
    }
    if (a2av::launch_grouped_gemm(g, stream) != cudaSuccess) return A2AV_ERR_CUDA;
    if (gemm_end && cudaEventRecord(gemm_end, stream) != cudaSuccess) return A2AV_ERR_CUDA;
    return A2AV_OK;
}

}  // namespace

extern "C" {

a2av_status a2av_gmm_run(const a2av_gmm_desc *desc, const void *ataOut, const int32_t *recvCounts,
                         const void *gmmWeight, const void *mmX, const void *mmWeight, void *permuteOut,
                         void *gmmY, void *mmY, void *workspace, size_t workspace_bytes,
                         a2av_stream_t stream) {
    return run_impl(desc, ataOut, recvCounts, gmmWeight, mmX, mmWeight, permuteOut, gmmY, mmY, workspace,
                    workspace_bytes, stream, nullptr, nullptr);
}

a2av_status a2av_gmm_run_profiled(const a2av_gmm_desc *desc, const void *ataOut, const int32_t *recvCounts,
                                  const void *gmmWeight, const void *mmX, const void *mmWeight,
                                  void *permuteOut, void *gmmY, void *mmY, void *workspace,
                                  size_t workspace_bytes, a2av_stream_t stream, void *gemm_begin_event,
                                  void *gemm_end_event) {
    if (!gemm_begin_event || !gemm_end_event) return A2AV_ERR_NULLPTR;
    return run_impl(desc, ataOut, recvCounts, gmmWeight, mmX, mmWeight, permuteOut, gmmY, mmY, workspace,
                    workspace_bytes, stream, static_cast<cudaEvent_t>(gemm_begin_event),
                    static_cast<cudaEvent_t>(gemm_end_event));
}

a2av_status a2av_gmm_run_arrivals(const a2av_gmm_desc *desc, const void *ataOut, const int32_t *recvCounts,
                                  const void *gmmWeight, const void *mmX, const void *mmWeight,
                                  void *permuteOut, void *gmmY, void *mmY, const uint64_t *arrived,
                                  uint64_t arrival_tag, uint64_t wait_limit_ns, void *workspace,
                                  size_t workspace_bytes, a2av_stream_t stream) {
    if (!desc || (desc->A > 0 && !arrived)) return A2AV_ERR_NULLPTR;
    if (desc->path != A2AV_PATH_DEFAULT && desc->path != A2AV_PATH_FUSED) return A2AV_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(arrived) & 7u) != 0) return A2AV_ERR_UNSUPPORTED;
    a2av_gmm_desc d = *desc;
    d.path = A2AV_PATH_FUSED;  // the GEMM reads each row where it arrived
    return run_impl(&d, ataOut, recvCounts, gmmWeight, mmX, mmWeight, permuteOut, gmmY, mmY, workspace,
                    workspace_bytes, stream, nullptr, nullptr, desc->A > 0 ? arrived : nullptr, arrival_tag,
                    wait_limit_ns > 0 ? wait_limit_ns : kWaitLimitNs);
}

a2av_status a2av_gmm_run_static_scratch(const a2av_gmm_desc *desc, const void *ataOut,
                                        const int32_t *recvCounts, const void *gmmWeight, const void *mmX,
                                        const void *mmWeight, void *permuteOut, void *gmmY, void *mmY,
                                        a2av_stream_t stream) {
    size_t need = 0;
    const a2av_status s = a2av_gmm_workspace_size(desc, &need);
    if (s != A2AV_OK) return s;
    if (need > A2AV_STATIC_SCRATCH_BYTES) return A2AV_ERR_SCRATCH_LIMIT;
    void *scratch = static_scratch_address();
    if (!scratch) return A2AV_ERR_CUDA;
    return a2av_gmm_run(desc, ataOut, recvCounts, gmmWeight, mmX, mmWeight, permuteOut, gmmY, mmY, scratch,
                        A2AV_STATIC_SCRATCH_BYTES, stream);
}

a2av_status a2av_amp_update_scale(float *scale, int32_t *growth_tracker, const float *found_inf,
                                  float growth_factor, float backoff_factor, int32_t growth_interval,
                                  a2av_stream_t stream) {
    if (!scale || !growth_tracker || !found_inf) return A2AV_ERR_NULLPTR;
    if (growth_interval < 1) return A2AV_ERR_INVALID;
    if (a2av::launch_amp_update_scale(scale, growth_tracker, found_inf, growth_factor, backoff_factor,
                                      growth_interval, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return A2AV_ERR_CUDA;
    return A2AV_OK;
}

a2av_status a2av_found_nonfinite(const void *x, int64_t n, int32_t dtype, float *found_inf,
                                 a2av_stream_t stream) {
    if (!found_inf || (n > 0 && !x)) return A2AV_ERR_NULLPTR;
    if (n < 0 || dtype < A2AV_BF16 || dtype > A2AV_FP32) return A2AV_ERR_INVALID;
    if (n == 0) return A2AV_OK;
    if (!aligned16(x)) return A2AV_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms <= 0) return A2AV_ERR_CUDA;
    const int64_t bytes = n * (dtype == A2AV_FP32 ? 4 : 2);
    if (a2av::launch_nonfinite_scan(x, bytes, dtype, found_inf, sms, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return A2AV_ERR_CUDA;
    return A2AV_OK;
}

a2av_status a2av_gmm_read_device_status(const void *workspace, a2av_stream_t stream, int32_t *code) {
    if (!workspace) return A2AV_ERR_NULLPTR;
    int32_t word = 0;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return A2AV_ERR_CUDA;
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return A2AV_ERR_CUDA;
    if (code) *code = word;
    if (word & a2av::kStatusArrivalTimeout) return A2AV_ERR_ARRIVAL_TIMEOUT;
    if (word & a2av::kStatusTimeout) return A2AV_ERR_CUDA;
    if (word & (a2av::kStatusBadCounts | a2av::kStatusBoundsCheck)) return A2AV_ERR_DEVICE_CHECK;
    return A2AV_OK;
}

const char *a2av_gmm_status_string(a2av_status status) {
    switch (status) {
        case A2AV_OK: return "ok";
        case A2AV_ERR_NULLPTR: return "a required pointer is NULL";
        case A2AV_ERR_INVALID: return "shape, range or dtype outside the operator's limits";
        case A2AV_ERR_UNSUPPORTED: return "not supported by this library (alignment)";
        case A2AV_ERR_WORKSPACE: return "workspace too small or misaligned";
        case A2AV_ERR_CUDA: return "CUDA call failed, or a kernel gave up waiting";
        case A2AV_ERR_DEVICE_CHECK: return "recvCounts negative or not summing to A";
        case A2AV_ERR_SCRATCH_LIMIT: return "needs more scratch than the static scratch array holds";
        case A2AV_ERR_ARRIVAL_TIMEOUT: return "a source's rows did not arrive within the wait limit";
    }
    return "unknown status";
}

}  // extern "C"
