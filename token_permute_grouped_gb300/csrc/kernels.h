// Host-side launch descriptions of the CUDA kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace a2av {

// Row gather ataOut (rank-major) -> dst (expert-major).
struct PermuteLaunch {
    const int32_t *recvCounts;
    int32_t W, e;
    int32_t A;
    int32_t H1;           // elements per row (multiple of 8)
    const void *ataOut;   // [A, H1]
    void *dst;            // [A, H1]
    int32_t *status;      // device status word
    int32_t write_status; // 1: this kernel stores the word (first kernel of a call)
    int32_t only_straddling;  // 1: copy only 128-row halves that straddle a segment boundary
    int32_t blocks_per_sm;    // grid cap per SM (0: as many as are resident at once); a GEMM
                              // that starts while this kernel runs needs room beside it
};

cudaError_t launch_permute(const PermuteLaunch &p, int num_sms, cudaStream_t stream);

// Persistent grouped GEMM over e routed groups (+ one shared group).
struct GemmLaunch {
    const int32_t *recvCounts;
    int32_t W, e;
    int32_t A;
    int32_t H1, N1, bn1;  // routed: K, N, tile width
    int32_t BS, H2, N2, bn2;  // shared: rows, K, N, tile width (BS = 0: none)
    void *gmmY;
    void *mmY;
    int32_t *status;
    int32_t write_status;
    int32_t bf16;         // 1: bf16, 0: fp16
    int32_t gather;       // 1: A rows gathered from ataOut (fused permute)
    const void *ataOut;   // for gather
    void *permuteOut;     // for gather: rows copied by warps 1-3 (may be NULL)
    int32_t pair;         // 1: 256-row tiles on CTA pairs (cta_group::2), 0: 128-row tiles
    int32_t kchunks;      // 64-wide K chunks per stage: 1, or 2 (pair, TMA-fed A, maps below in 3-D/4-D)
    int32_t grid;         // persistent CTAs (pair: an even number, two per cluster)
    int32_t b_first;      // two-chunk stages: issue each stage's weight load before its A load
    CUtensorMap tmA_routed;   // split: expert-major A, 128-row box; fused: ataOut, 1-row box (gather)
    CUtensorMap tmA_box[5];   // fused: ataOut with 8, 16, 32, 64, 128-row boxes (contiguous runs)
    CUtensorMap tmB_routed;   // gmmWeight [e, H1, N1]
    CUtensorMap tmA_shared;   // mmX [BS, H2]
    CUtensorMap tmB_shared;   // mmWeight as [1, H2, N2]
    CUtensorMap tmA_direct;   // split path: ataOut, 128-row box, for halves read in place
    int32_t direct_halves;    // 1: halves inside one segment are read from ataOut directly
    CUtensorMap tmB4_routed;  // gmmWeight as 64-column atoms: one load per stage (when b4_routed)
    CUtensorMap tmB4_shared;  // mmWeight likewise (when b4_shared)
    CUtensorMap tmY_routed;   // gmmY [A, N1], box 32 x 32, 64-byte swizzle (epilogue stores)
    CUtensorMap tmY_shared;   // mmY [BS, N2], likewise
    int32_t b4_routed, b4_shared;
    int32_t after_permute;    // 1: launched to overlap the permute kernel before it (programmatic
                              // dependent launch); the producer waits for it before staged loads
    uint64_t wait_limit_ns;   // bound on every pipeline wait; on expiry the kernel records
                              // kStatusTimeout and winds down
    // Arrival-driven start (fused path): the rows of source w in ataOut may
    // be read once arrived[w] == arrival_tag; every tile that reads a
    // source's rows waits for its flag first.  NULL: everything has arrived.
    const uint64_t *arrived;
    uint64_t arrival_tag;
    int32_t shared_first;     // 1: shared-expert tiles first (they read no exchanged rows)
};

cudaError_t launch_grouped_gemm(const GemmLaunch &p, cudaStream_t stream);

// Dynamic loss scaling (amp.cu).
cudaError_t launch_amp_update_scale(float *scale, int32_t *tracker, const float *found_inf, float growth,
                                    float backoff, int32_t interval, cudaStream_t stream);
cudaError_t launch_nonfinite_scan(const void *x, int64_t bytes, int dtype, float *found_inf, int num_sms,
                                  cudaStream_t stream);
size_t grouped_gemm_smem_bytes(int pair);
int grouped_gemm_max_coresident(int pair);  // CTAs (single) or clusters (pair) resident at once

}  // namespace a2av
