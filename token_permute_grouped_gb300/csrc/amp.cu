// Dynamic loss scaling for mixed-precision training: the scale update of the
// "aclnnAmpUpdateScale" page, and the scan for inf/NaN that feeds its
// found_inf input.
//
// Page "aclnnAmpUpdateScale", Formula and notes:
//   found_inf != 0                      -> scale * backoff, tracker = 0
//   else tracker + 1 == growth_interval -> grown = scale * growth; scale =
//                                          grown if finite, else unchanged;
//                                          tracker = 0
//   else                                -> tracker + 1
// ("Inf/NaN priority": found_inf != 0 wins over the tracker; "overflow
// protection": a non-finite grown scale keeps the old scale.)
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace a2av {

namespace {

__global__ void amp_update_scale_kernel(float *scale, int32_t *tracker, const float *found_inf, float growth,
                                        float backoff, int32_t interval) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    const float found = *found_inf;
    float s = *scale;
    int32_t t = *tracker;
    if (found != 0.0f) {  // a NaN found_inf compares unequal to 0: backoff
        s = __fmul_rn(s, backoff);
        t = 0;
    } else if (t + 1 == interval) {
        const float grown = __fmul_rn(s, growth);
        if (isfinite(grown)) s = grown;
        t = 0;
    } else {
        t = t + 1;
    }
    *scale = s;
    *tracker = t;
}

// Exponent field all ones: inf or NaN.
__device__ __forceinline__ bool half_word_nonfinite(uint32_t h, uint32_t exp_mask) {
    return (h & exp_mask) == exp_mask;
}

__device__ __forceinline__ bool vec_nonfinite(const uint4 v, int dtype) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    bool bad = false;
    if (dtype == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) bad |= (w[i] & 0x7F800000u) == 0x7F800000u;
    } else {
        const uint32_t m = dtype == 0 ? 0x7F80u : 0x7C00u;
#pragma unroll
        for (int i = 0; i < 4; ++i) bad |= half_word_nonfinite(w[i] & 0xFFFFu, m) | half_word_nonfinite(w[i] >> 16, m);
    }
    return bad;
}

constexpr int kScanThreads = 256;

// found_inf = 1.0 when any element is inf or NaN; left as it was otherwise.
__global__ void __launch_bounds__(kScanThreads)
    nonfinite_scan_kernel(const uint4 *__restrict__ x, int64_t nvec, const uint8_t *__restrict__ tail,
                          int tail_bytes, int dtype, float *found_inf) {
    bool bad = false;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < nvec; i += 4 * stride) {  // four 16-byte loads in flight
        const uint4 a = __ldg(x + i), b = __ldg(x + i + stride), c = __ldg(x + i + 2 * stride),
                    d = __ldg(x + i + 3 * stride);
        bad |= vec_nonfinite(a, dtype) | vec_nonfinite(b, dtype) | vec_nonfinite(c, dtype) |
               vec_nonfinite(d, dtype);
    }
    for (; i < nvec; i += stride) bad |= vec_nonfinite(__ldg(x + i), dtype);
    if (blockIdx.x == 0 && threadIdx.x == 0) {  // the last < 16 bytes, element by element
        const int esize = dtype == 2 ? 4 : 2;
        for (int b = 0; b + esize <= tail_bytes; b += esize) {
            uint32_t word = tail[b] | (static_cast<uint32_t>(tail[b + 1]) << 8);
            if (esize == 4)
                word |= (static_cast<uint32_t>(tail[b + 2]) << 16) | (static_cast<uint32_t>(tail[b + 3]) << 24);
            bad |= esize == 4 ? (word & 0x7F800000u) == 0x7F800000u
                              : half_word_nonfinite(word, dtype == 0 ? 0x7F80u : 0x7C00u);
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) *found_inf = 1.0f;
}

}  // namespace

cudaError_t launch_amp_update_scale(float *scale, int32_t *tracker, const float *found_inf, float growth,
                                    float backoff, int32_t interval, cudaStream_t stream) {
    amp_update_scale_kernel<<<1, 32, 0, stream>>>(scale, tracker, found_inf, growth, backoff, interval);
    return cudaGetLastError();
}

cudaError_t launch_nonfinite_scan(const void *x, int64_t bytes, int dtype, float *found_inf, int num_sms,
                                  cudaStream_t stream) {
    const int64_t nvec = bytes / 16;
    const int tail = static_cast<int>(bytes - nvec * 16);
    int64_t blocks = (nvec + kScanThreads - 1) / kScanThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * (2048 / kScanThreads);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    nonfinite_scan_kernel<<<static_cast<int>(blocks), kScanThreads, 0, stream>>>(
        static_cast<const uint4 *>(x), nvec, static_cast<const uint8_t *>(x) + nvec * 16, tail, dtype, found_inf);
    return cudaGetLastError();
}

}  // namespace a2av
