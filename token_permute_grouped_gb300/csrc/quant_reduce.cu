// Dequantising reduce over the ranks' data ("aclnnQuantReduceScatter" page).
//
// "Formula": output = Reduce(AllToAllScales * AllToAllData), the Reduce over
// the data received from the different ranks.  After the AllToAll this rank
// holds, from each source rank w, data[w] [rows, H] (8-bit) and its scales:
//   out[i][h] = sum over w of value(data[w][i][h]) * scale(w, i, h)
// "Constraints": mx quantisation = FLOAT8_E4M3FN / FLOAT8_E5M2 data with
// FLOAT8_E8M0 scales, one per 32 elements along H; pertoken-pergroup = INT8 /
// FLOAT8 data with float scales, one per 128 elements along H.
//
// A thread owns units of 16 consecutive outputs of a row: per unit, one
// 16-byte load per rank and one scale per rank (16 elements never straddle a
// 32-element group).  Codes are widened exactly to float32 and accumulated by
// float32 fused multiply-adds, ranks in ascending order (one rounding per
// rank); the sum is rounded once to the output type.  HBM-bound: per output,
// W code bytes, W/32 scale bytes (one E8M0 byte per 32 codes, or one float
// per 128), and 2 output bytes (bf16).
//
// Decoding costs a few instructions per code, not a bit-field walk:
//   E5M2   is the upper byte of an fp16 of the same value (same sign, 5-bit
//          exponent with bias 15, top two fraction bits), so one byte permute
//          makes two fp16 lanes, then a half-to-float conversion;
//   E4M3FN goes through the cvt.rn.f16x2.e4m3x2 conversion (exact: every
//          E4M3FN value, subnormals and NaN included, is an fp16 value);
//   INT8   b + 128 (b xor 0x80) is placed in the low byte of the float 2^23,
//          whose unit in the last place is 1; subtracting 2^23 + 128 is exact.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "a2av_quant_reduce.h"
#include "ptx.cuh"

namespace a2av {

namespace {

constexpr int kQrThreads = 256;
constexpr int kLoadsInFlight = 8;  // 16-byte code loads per thread per step, for any W

struct QuantReduceLaunch {
    int32_t W;
    int64_t rows, H;
    int32_t qtype, mode, out_dtype;  // a2av_qtype, a2av_qmode, a2av_dtype
    const void *data;                // [W, rows, H] codes
    const void *scales;              // [W, rows, H/32] E8M0 or [W, rows, H/128] float
    void *out;                       // [rows, H]
};

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Two fp16 lanes of a 32-bit word to float32 (exact).
__device__ __forceinline__ void f16x2_to_f32(uint32_t h, float &lo, float &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
}

// The four codes of a word (byte k is element k) as float32.
template <int QT>
__device__ __forceinline__ void decode_word(uint32_t w, float (&v)[4]) {
    if constexpr (QT == A2AV_Q_E5M2) {
        f16x2_to_f32(__byte_perm(w, 0u, 0x1404), v[0], v[1]);  // bytes 0, 1 to the high byte of each lane
        f16x2_to_f32(__byte_perm(w, 0u, 0x3424), v[2], v[3]);
    } else if constexpr (QT == A2AV_Q_E4M3FN) {
        uint32_t lo, hi;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t"
            "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
        f16x2_to_f32(lo, v[0], v[1]);
        f16x2_to_f32(hi, v[2], v[3]);
    } else {
        const uint32_t x = w ^ 0x80808080u;  // b + 128 in each byte
#pragma unroll
        for (int k = 0; k < 4; ++k)
            v[k] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7650 + k)) - 8388736.0f;  // 2^23 + 128
    }
}

// E8M0 scale code: 2^(e - 127); 0xFF is NaN.
__device__ __forceinline__ float e8m0_to_float(uint32_t e) {
    if (e == 255) return __uint_as_float(0x7FC00000u);
    if (e == 0) return __uint_as_float(0x00400000u);  // 2^-127, a float subnormal
    return __uint_as_float(e << 23);
}

// Two float32 lanes in one 64-bit register, and their fused multiply-add
// (fma.rn.f32x2: each lane is one fma.rn.f32, so results equal the scalar
// form, in half the instructions).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ void f32x2_split(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// One unit: sum over the W ranks of 16 decoded codes times their scales, then
// the 16 results (rounded to the output type) stored at out + off.
template <int W, int QT, int OUT>
__device__ __forceinline__ void reduce_unit(const uint4 (&q)[W], const float (&sc)[W], void *out, int64_t off) {
    uint64_t acc2[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc2[k] = 0;  // +0.0f in both lanes
#pragma unroll
    for (int w = 0; w < W; ++w) {
        const uint32_t word[4] = {q[w].x, q[w].y, q[w].z, q[w].w};
        const uint64_t s2 = f32x2(sc[w], sc[w]);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            float v[4];
            decode_word<QT>(word[t], v);
            acc2[2 * t] = fma_f32x2(f32x2(v[0], v[1]), s2, acc2[2 * t]);
            acc2[2 * t + 1] = fma_f32x2(f32x2(v[2], v[3]), s2, acc2[2 * t + 1]);
        }
    }
    float acc[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) f32x2_split(acc2[k], acc[2 * k], acc[2 * k + 1]);
    if constexpr (OUT == A2AV_FP32) {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + off);
#pragma unroll
        for (int t = 0; t < 4; ++t) o[t] = make_float4(acc[4 * t], acc[4 * t + 1], acc[4 * t + 2], acc[4 * t + 3]);
    } else {
        uint32_t packed[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if constexpr (OUT == A2AV_BF16) {
                __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * t], acc[2 * t + 1]);
                packed[t] = *reinterpret_cast<uint32_t *>(&b);
            } else {
                __half2 b = __floats2half2_rn(acc[2 * t], acc[2 * t + 1]);
                packed[t] = *reinterpret_cast<uint32_t *>(&b);
            }
        }
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + off);
        o[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        o[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
}

// Units from u_begin on, loaded straight from global memory (any alignment
// of the scale planes; also the tail the staged kernel leaves).
template <int W, int QT, int MODE, int OUT>
__global__ void __launch_bounds__(kQrThreads)
    quant_reduce_kernel(int64_t rows, int64_t H, const uint8_t *__restrict__ data, const void *__restrict__ scales,
                        void *__restrict__ out, int64_t u_begin) {
    constexpr int U = kLoadsInFlight / W;  // units per thread per step
    constexpr int64_t kGroup = MODE == A2AV_QMODE_MX ? 32 : 128;
    const int64_t vpr = H / 16;      // units per row
    const int64_t ngr = H / kGroup;  // scale groups per row
    const int64_t plane = rows * H, splane = rows * ngr;
    // Unit u = i * vpr + c (row i, 16-column chunk c).  Units of one step are
    // spaced by the block size, so each load instruction is coalesced; a step
    // advances every unit by `stride`, kept as (row, chunk) increments.
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kQrThreads * U;
    const int64_t dq = stride / vpr, dr = stride % vpr;
    int64_t ri[U], ci[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
        const int64_t u = u_begin + (static_cast<int64_t>(blockIdx.x) * U + j) * kQrThreads + threadIdx.x;
        ri[j] = u / vpr;
        ci[j] = u % vpr;
    }
    while (ri[0] < rows) {
        uint4 q[U][W];
        float sc[U][W];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            if (ri[j] < rows) {
                const int64_t off = ri[j] * H + ci[j] * 16;
                const int64_t soff = ri[j] * ngr + ci[j] * 16 / kGroup;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    q[j][w] = ld_stream(data + w * plane + off);
                    if constexpr (MODE == A2AV_QMODE_MX)
                        sc[j][w] = e8m0_to_float(__ldg(static_cast<const uint8_t *>(scales) + w * splane + soff));
                    else
                        sc[j][w] = __ldg(static_cast<const float *>(scales) + w * splane + soff);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            if (ri[j] < rows) reduce_unit<W, QT, OUT>(q[j], sc[j], out, ri[j] * H + ci[j] * 16);
            ci[j] += dr;
            if (ci[j] >= vpr) {
                ci[j] -= vpr;
                ri[j] += 1;
            }
            ri[j] += dq;
        }
    }
}

// ---- staged kernel: chunks of 256 units (4096 outputs), brought into shared
// memory by one-dimensional bulk copies (cp.async.bulk): per rank one copy of
// 4096 codes and one of the chunk's 128 scale bytes (E8M0 per 32, or float
// per 128: 4096 / 32 bytes either way).  A producer warp keeps a ring of
// stages full; 256 consumer threads each reduce one unit per chunk from shared
// memory.  All three arrays are contiguous, so unit u of the flattened
// [rows, H] output is codes u*16.. of each rank and scale byte (u*16 / group
// in elements) of each rank's scale plane.
constexpr int kQbConsumers = 256;
constexpr int kQbThreads = kQbConsumers + 32;
constexpr int kQbChunk = kQbConsumers;  // units per chunk
constexpr uint32_t kQbCodeBytes = kQbChunk * 16;
constexpr uint32_t kQbScaleBytes = kQbChunk * 16 / 32;
constexpr uint64_t kQbWaitLimitNs = 2000000000ull;
constexpr uint32_t kQbHeader = 256;  // barriers and the abort flag, before the ring

template <int W>
struct Qb {
    static constexpr uint32_t kStageBytes = W * (kQbCodeBytes + kQbScaleBytes);
    static constexpr int kStages = W == 8 ? 3 : W == 4 ? 6 : 12;  // about 100 KB per CTA, two CTAs per SM
    static constexpr size_t kSmem = kQbHeader + kStages * kStageBytes;
};

// Set when a staged-kernel wait gave up (it then stops early); it cannot be
// reached by correct code, since every wait is on this CTA's own copies.
__device__ int32_t g_qr_wait_timeouts = 0;

__device__ __forceinline__ bool qb_wait(uint32_t bar, uint32_t parity, volatile int32_t *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kQbWaitLimitNs) {
            *abort_flag = 1;
            atomicAdd(&g_qr_wait_timeouts, 1);
            return false;
        }
    }
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

template <int W, int QT, int MODE, int OUT>
__global__ void __launch_bounds__(kQbThreads)
    quant_reduce_staged_kernel(int64_t chunks, int64_t plane, int64_t splane_bytes, const uint8_t *__restrict__ data,
                               const uint8_t *__restrict__ scales, void *__restrict__ out) {
    using L = Qb<W>;
    extern __shared__ __align__(128) uint8_t qb_smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(qb_smem);  // [kStages], then empty[kStages]
    uint64_t *empty = full + L::kStages;
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(empty + L::kStages);
    const uint32_t ring = smem_u32(qb_smem) + kQbHeader;
    static_assert(2 * L::kStages * 8 + 4 <= kQbHeader, "barriers fit in front of the ring");
    if (threadIdx.x == 0) {
        for (int st = 0; st < L::kStages; ++st) {
            mbar_init(smem_u32(&full[st]), 1);
            mbar_init(smem_u32(&empty[st]), kQbConsumers / 32);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == kQbConsumers / 32) {
        // ---- producer
        if (lane == 0) {
            uint32_t it = 0;
            for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x, ++it) {
                const int st = it % L::kStages;
                if (!qb_wait(smem_u32(&empty[st]), ((it / L::kStages) & 1) ^ 1, abort_flag)) break;
                const uint32_t fb = smem_u32(&full[st]);
                mbar_arrive_expect_tx(fb, L::kStageBytes);
                const uint32_t dst = ring + st * L::kStageBytes;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    bulk_copy(dst + w * kQbCodeBytes, data + w * plane + c * kQbCodeBytes, kQbCodeBytes, fb);
                    bulk_copy(dst + W * kQbCodeBytes + w * kQbScaleBytes, scales + w * splane_bytes + c * kQbScaleBytes,
                              kQbScaleBytes, fb);
                }
            }
        }
        return;
    }
    // ---- consumers: thread t reduces unit t of each chunk
    const int t = threadIdx.x;
    uint32_t it = 0;
    for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x, ++it) {
        const int st = it % L::kStages;
        bool ready = true;
        if (lane == 0) ready = qb_wait(smem_u32(&full[st]), (it / L::kStages) & 1, abort_flag);
        if (!__shfl_sync(0xffffffffu, ready, 0)) break;
        const uint8_t *stage = qb_smem + kQbHeader + st * L::kStageBytes;
        uint4 q[W];
        float sc[W];
#pragma unroll
        for (int w = 0; w < W; ++w) {
            q[w] = *reinterpret_cast<const uint4 *>(stage + w * kQbCodeBytes + t * 16);
            const uint8_t *sp = stage + W * kQbCodeBytes + w * kQbScaleBytes;
            if constexpr (MODE == A2AV_QMODE_MX) sc[w] = e8m0_to_float(sp[t / 2]);  // 16 codes share a byte per 32
            else sc[w] = reinterpret_cast<const float *>(sp)[t / 8];              // one float per 128
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[st]));  // the stage's bytes are in registers now
        reduce_unit<W, QT, OUT>(q, sc, out, (c * kQbChunk + t) * 16);
    }
}

template <int W, int QT, int MODE, int OUT>
cudaError_t launch_qr(const QuantReduceLaunch &p, int num_sms, cudaStream_t stream) {
    constexpr int U = kLoadsInFlight / W;
    const int64_t units = p.rows * (p.H / 16);
    const int64_t splane_bytes = p.rows * (p.H / 32);  // E8M0 per 32 or float per 128: H / 32 bytes per row
    // Bulk copies need 16-byte aligned sources: the staged kernel takes the
    // full chunks when every rank's scale plane starts on a 16-byte boundary.
    int64_t u_begin = 0;
    if ((reinterpret_cast<uintptr_t>(p.scales) & 15u) == 0 && splane_bytes % 16 == 0 && units >= kQbChunk) {
        using L = Qb<W>;
        auto kern = quant_reduce_staged_kernel<W, QT, MODE, OUT>;
        static bool attr_set = false;  // once per instantiation
        if (!attr_set) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::kSmem)) !=
                cudaSuccess)
                return cudaErrorInvalidValue;
            attr_set = true;
        }
        const int64_t chunks = units / kQbChunk;
        const int64_t blocks = std::min<int64_t>(chunks, 2 * static_cast<int64_t>(num_sms));
        kern<<<static_cast<int>(blocks), kQbThreads, L::kSmem, stream>>>(
            chunks, p.rows * p.H, splane_bytes, static_cast<const uint8_t *>(p.data),
            static_cast<const uint8_t *>(p.scales), p.out);
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        u_begin = chunks * kQbChunk;
        if (u_begin == units) return cudaSuccess;
    }
    static int resident = 0;  // CTAs per SM, from the occupancy calculator, once per instantiation
    if (resident == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_reduce_kernel<W, QT, MODE, OUT>, kQrThreads,
                                                          0) != cudaSuccess || n < 1)
            n = 1;
        resident = n;
    }
    const int64_t per_block = static_cast<int64_t>(kQrThreads) * U;
    int64_t blocks = (units - u_begin + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(num_sms) * resident;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quant_reduce_kernel<W, QT, MODE, OUT><<<static_cast<int>(blocks), kQrThreads, 0, stream>>>(
        p.rows, p.H, static_cast<const uint8_t *>(p.data), p.scales, p.out, u_begin);
    return cudaGetLastError();
}

template <int W, int QT, int MODE>
cudaError_t launch_qr_out(const QuantReduceLaunch &p, int num_sms, cudaStream_t stream) {
    if (p.out_dtype == A2AV_BF16) return launch_qr<W, QT, MODE, A2AV_BF16>(p, num_sms, stream);
    if (p.out_dtype == A2AV_FP16) return launch_qr<W, QT, MODE, A2AV_FP16>(p, num_sms, stream);
    return launch_qr<W, QT, MODE, A2AV_FP32>(p, num_sms, stream);
}

template <int W>
cudaError_t launch_qr_w(const QuantReduceLaunch &p, int num_sms, cudaStream_t stream) {
    if (p.mode == A2AV_QMODE_MX) {  // FLOAT8 data, E8M0 scales per 32
        return p.qtype == A2AV_Q_E4M3FN ? launch_qr_out<W, A2AV_Q_E4M3FN, A2AV_QMODE_MX>(p, num_sms, stream)
                                        : launch_qr_out<W, A2AV_Q_E5M2, A2AV_QMODE_MX>(p, num_sms, stream);
    }
    if (p.qtype == A2AV_Q_E4M3FN) return launch_qr_out<W, A2AV_Q_E4M3FN, A2AV_QMODE_GROUP128>(p, num_sms, stream);
    if (p.qtype == A2AV_Q_E5M2) return launch_qr_out<W, A2AV_Q_E5M2, A2AV_QMODE_GROUP128>(p, num_sms, stream);
    return launch_qr_out<W, A2AV_Q_INT8, A2AV_QMODE_GROUP128>(p, num_sms, stream);
}

cudaError_t launch_quant_reduce(const QuantReduceLaunch &p, int num_sms, cudaStream_t stream) {
    if (p.W == 2) return launch_qr_w<2>(p, num_sms, stream);
    if (p.W == 4) return launch_qr_w<4>(p, num_sms, stream);
    return launch_qr_w<8>(p, num_sms, stream);
}

int qr_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

}  // namespace a2av

extern "C" a2av_status a2av_quant_reduce(int32_t W, int64_t rows, int64_t H, int32_t qtype, int32_t mode,
                                         const void *data, const void *scales, void *out, int32_t out_dtype,
                                         a2av_stream_t stream) {
    if (!data || !scales || !out) return A2AV_ERR_NULLPTR;
    if (W != 2 && W != 4 && W != 8) return A2AV_ERR_INVALID;
    if (rows < 1 || H < 1024 || H > 8192 || H % 128 != 0) return A2AV_ERR_INVALID;
    if (qtype < A2AV_Q_E4M3FN || qtype > A2AV_Q_INT8 || mode < A2AV_QMODE_MX || mode > A2AV_QMODE_GROUP128)
        return A2AV_ERR_INVALID;
    if (mode == A2AV_QMODE_MX && qtype == A2AV_Q_INT8) return A2AV_ERR_INVALID;
    if (out_dtype < A2AV_BF16 || out_dtype > A2AV_FP32) return A2AV_ERR_INVALID;
    if (rows > (int64_t{1} << 40) / H) return A2AV_ERR_INVALID;
    if (!a2av::aligned(data, 16) || !a2av::aligned(out, 16) ||
        (mode == A2AV_QMODE_GROUP128 && !a2av::aligned(scales, 4)))
        return A2AV_ERR_UNSUPPORTED;
    const int sms = a2av::qr_sm_count();
    if (sms <= 0) return A2AV_ERR_CUDA;
    const a2av::QuantReduceLaunch p{W, rows, H, qtype, mode, out_dtype, data, scales, out};
    return a2av::launch_quant_reduce(p, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? A2AV_OK
               : A2AV_ERR_CUDA;
}
