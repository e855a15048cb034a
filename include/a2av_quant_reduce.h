/*
 * a2av_quant_reduce — the local half of a quantised reduce-scatter on one GB300.
 *
 * Operation ("aclnnQuantReduceScatter" operator page, "Formula"): each rank's
 * 8-bit x and its scales go through an AllToAll; the ranks' received pieces
 * are then dequantised and summed:
 *
 *     out = Reduce over source ranks w of (scales[w] * data[w])
 *
 * This call is that Reduce on one GPU, after the AllToAll has landed: from
 * each of the W source ranks this rank holds `rows` rows of H codes and their
 * scales, and it writes
 *
 *     out[i][h] = sum_{w = 0 .. W-1} value(data[w][i][h]) * scale(w, i, h)
 *
 * Quantisation modes (page "Constraints"):
 *   A2AV_QMODE_MX        data FLOAT8_E4M3FN or FLOAT8_E5M2, scales
 *                        FLOAT8_E8M0 (2^(s-127)), one per 32 consecutive
 *                        elements of a row (scalesDataSize = BS * H / 32 B)
 *   A2AV_QMODE_GROUP128  data INT8, FLOAT8_E4M3FN or FLOAT8_E5M2, scales
 *                        float32, one per 128 consecutive elements of a row
 *                        (pertoken-pergroup, groupSize = 128)
 * HIFLOAT8 data, also allowed there, is not supported.
 *
 * Limits (page "Constraints"): W (the communicator size) is 2, 4 or 8; H is a
 * multiple of 128 in [1024, 8192]; no empty tensor (rows >= 1).
 *
 * Layouts (row-major, contiguous, device memory):
 *   data    [W, rows, H]          uint8 codes, source rank w's block at w*rows*H;
 *                                 16-byte aligned
 *   scales  [W, rows, H / 32]     uint8 E8M0  (MX), or
 *           [W, rows, H / 128]    float32     (GROUP128, 4-byte aligned)
 *   out     [rows, H]             out_dtype: A2AV_BF16, A2AV_FP16 or A2AV_FP32;
 *                                 16-byte aligned
 * Arithmetic: codes and scales are decoded exactly to float32; the sum over w
 * (ascending w) is formed by float32 fused multiply-adds, rounded to nearest
 * once per rank; the sum is rounded once to out_dtype (nearest even).  NaN codes
 * (E4M3FN S.1111.111, E5M2 exponent 31 with a non-zero fraction, E8M0 0xFF)
 * give NaN; E5M2 infinities propagate.  Results are deterministic.
 *
 * Ownership: the caller owns every buffer; nothing is allocated or kept, and
 * the call only enqueues one kernel on `stream`.  Errors: A2AV_ERR_NULLPTR
 * for a NULL pointer, A2AV_ERR_INVALID for W, rows, H, qtype, mode or
 * out_dtype outside the limits above (including MX with INT8 data),
 * A2AV_ERR_UNSUPPORTED for a misaligned pointer, A2AV_ERR_CUDA if the launch
 * fails.
 */
#ifndef A2AV_QUANT_REDUCE_H
#define A2AV_QUANT_REDUCE_H

#include <stdint.h>

#include "a2av_gmm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { A2AV_Q_E4M3FN = 0, A2AV_Q_E5M2 = 1, A2AV_Q_INT8 = 2 } a2av_qtype;
typedef enum { A2AV_QMODE_MX = 0, A2AV_QMODE_GROUP128 = 1 } a2av_qmode;

a2av_status a2av_quant_reduce(int32_t W, int64_t rows, int64_t H, int32_t qtype, int32_t mode,
                              const void *data, const void *scales, void *out, int32_t out_dtype,
                              a2av_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* A2AV_QUANT_REDUCE_H */
