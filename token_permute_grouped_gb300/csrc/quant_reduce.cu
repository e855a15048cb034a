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
// One thread makes 16 consecutive outputs of a row: one 16-byte load per
// rank, one scale per rank (16 elements never straddle a 32-element group),
// fp32 products and sums with ranks in order, then one rounding to the
// output type.  HBM-bound: W * 16 + W * (1 or 4) bytes in, 16 * out bytes out.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "a2av_quant_reduce.h"

namespace a2av {

namespace {

constexpr int kQrThreads = 256;
constexpr int kMaxRanks = 8;

struct QuantReduceLaunch {
    int32_t W;
    int64_t rows, H;
    int32_t qtype, mode, out_dtype;  // a2av_qtype, a2av_qmode, a2av_dtype
    const void *data;                // [W, rows, H] codes
    const void *scales;              // [W, rows, H/32] E8M0 or [W, rows, H/128] float
    void *out;                       // [rows, H]
};

// 8-bit codes to float, from the format definitions.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
    const uint32_t s = (b >> 7) & 1, e = (b >> 3) & 0xf, f = b & 7;
    float v;
    if (e == 15 && f == 7)
        v = __uint_as_float(0x7FC00000u);                       // the only NaN code
    else if (e == 0)
        v = static_cast<float>(f) * 0.001953125f;               // f/8 * 2^-6 = f * 2^-9
    else
        v = __uint_as_float(((e + 120u) << 23) | (f << 20));    // (1 + f/8) * 2^(e-7)
    return s ? -v : v;
}

__device__ __forceinline__ float e5m2_to_float(uint32_t b) {
    const uint32_t s = (b >> 7) & 1, e = (b >> 2) & 0x1f, f = b & 3;
    float v;
    if (e == 31)
        v = f ? __uint_as_float(0x7FC00000u) : __uint_as_float(0x7F800000u);
    else if (e == 0)
        v = static_cast<float>(f) * 1.52587890625e-05f;         // f/4 * 2^-14 = f * 2^-16
    else
        v = __uint_as_float(((e + 112u) << 23) | (f << 21));    // (1 + f/4) * 2^(e-15)
    return s ? -v : v;
}

__device__ __forceinline__ float e8m0_to_float(uint32_t e) {
    if (e == 255) return __uint_as_float(0x7FC00000u);
    if (e == 0) return __uint_as_float(0x00400000u);            // 2^-127, a float subnormal
    return __uint_as_float(e << 23);                            // 2^(e-127)
}

template <int QT>
__device__ __forceinline__ float q_to_float(uint32_t b) {
    if constexpr (QT == 0) return e4m3_to_float(b);
    else if constexpr (QT == 1) return e5m2_to_float(b);
    else return static_cast<float>(static_cast<int8_t>(b));
}

template <int QT, int MODE, int OUT>
__global__ void __launch_bounds__(kQrThreads)
    quant_reduce_kernel(int W, int64_t rows, int64_t H, const uint8_t *__restrict__ data,
                        const void *__restrict__ scales, void *__restrict__ out) {
    const int64_t vpr = H / 16;  // 16-element units per row
    const int64_t units = rows * vpr;
    const int64_t group = MODE == 0 ? 32 : 128;
    const int64_t ngr = H / group;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units; u += stride) {
        const int64_t i = u / vpr, h0 = (u % vpr) * 16;
        uint4 v[kMaxRanks];
        float sc[kMaxRanks];
#pragma unroll
        for (int w = 0; w < kMaxRanks; ++w) {
            if (w < W) {
                const int64_t row = static_cast<int64_t>(w) * rows + i;
                v[w] = __ldg(reinterpret_cast<const uint4 *>(data + row * H + h0));
                if constexpr (MODE == 0)
                    sc[w] = e8m0_to_float(__ldg(static_cast<const uint8_t *>(scales) + row * ngr + h0 / group));
                else
                    sc[w] = __ldg(static_cast<const float *>(scales) + row * ngr + h0 / group);
            }
        }
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
#pragma unroll
        for (int w = 0; w < kMaxRanks; ++w) {
            if (w < W) {
                const uint32_t word[4] = {v[w].x, v[w].y, v[w].z, v[w].w};
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    acc[k] = __fadd_rn(acc[k], __fmul_rn(q_to_float<QT>((word[k >> 2] >> (8 * (k & 3))) & 0xFF), sc[w]));
            }
        }
        if constexpr (OUT == 2) {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + i * H + h0);
#pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        } else {
            uint32_t packed[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if constexpr (OUT == 0) {
                    __nv_bfloat162 t = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
                    packed[q] = *reinterpret_cast<uint32_t *>(&t);
                } else {
                    __half2 t = __floats2half2_rn(acc[2 * q], acc[2 * q + 1]);
                    packed[q] = *reinterpret_cast<uint32_t *>(&t);
                }
            }
            uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + i * H + h0);
            o[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            o[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
    }
}

template <int QT, int MODE, int OUT>
cudaError_t launch_qr(const QuantReduceLaunch &p, int num_sms, cudaStream_t stream) {
    const int64_t units = p.rows * (p.H / 16);
    int64_t blocks = (units + kQrThreads - 1) / kQrThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * (2048 / kQrThreads) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quant_reduce_kernel<QT, MODE, OUT><<<static_cast<int>(blocks), kQrThreads, 0, stream>>>(
        p.W, p.rows, p.H, static_cast<const uint8_t *>(p.data), p.scales, p.out);
    return cudaGetLastError();
}

template <int QT, int MODE>
cudaError_t launch_qr_out(const QuantReduceLaunch &p, int num_sms, cudaStream_t stream) {
    if (p.out_dtype == 0) return launch_qr<QT, MODE, 0>(p, num_sms, stream);
    if (p.out_dtype == 1) return launch_qr<QT, MODE, 1>(p, num_sms, stream);
    return launch_qr<QT, MODE, 2>(p, num_sms, stream);
}

cudaError_t launch_quant_reduce(const QuantReduceLaunch &p, int num_sms, cudaStream_t stream) {
    if (p.mode == 0) {  // mx: FLOAT8 data, E8M0 scales per 32
        return p.qtype == 0 ? launch_qr_out<0, 0>(p, num_sms, stream) : launch_qr_out<1, 0>(p, num_sms, stream);
    }
    if (p.qtype == 0) return launch_qr_out<0, 1>(p, num_sms, stream);
    if (p.qtype == 1) return launch_qr_out<1, 1>(p, num_sms, stream);
    return launch_qr_out<2, 1>(p, num_sms, stream);
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
