/*
 * a2av_gmm_mx — Permute + GroupedMatMul (+ shared-expert MatMul) with
 * block-scaled FP8 (mx) operands on one GB300.
 *
 * The operation of a2av_gmm.h ("aclnnAlltoAllvGroupedMatMul" page, "Formula":
 * permuteOut = Permute(ataOut), gmmY = permuteOut x gmmWeight, mmY = mmX x
 * mmWeight) with every operand in the mx quantisation that the
 * "aclnnQuantReduceScatter" page's "Constraints" define: FLOAT8_E4M3FN or
 * FLOAT8_E5M2 codes with one FLOAT8_E8M0 scale (2^(s - 127)) per 32
 * consecutive elements along the contraction dimension:
 *
 *   gmmY[i][n] = sum_k value(a[i][k]) 2^(sa[i][k/32]-127) value(w[n][k]) 2^(sw[n][k/32]-127)
 *
 * computed on the tensor cores' block-scaled FP8 path (tcgen05.mma
 * kind::mxf8f6f4), accumulated in fp32 and rounded once to bf16 (nearest
 * even).
 *
 * Shapes (as in a2av_gmm.h): W ranks, e local experts (1 <= e <= 32,
 * W * e <= 256), A routed rows (sum of recvCounts, 0 allowed), H1 x N1 routed
 * weights, BS x H2 shared-expert input, H2 x N2 shared weight (BS = 0: none).
 * This library needs H1 and H2 to be multiples of 512 (scale rows of H/32
 * bytes start on 16-byte boundaries), N1 and N2 multiples of 8, and the
 * same code format for activations and weights.
 *
 * Layouts (row-major, contiguous, 16-byte aligned, device memory):
 *   ataOut_q  [A, H1]       codes, rank-major (as ataOut in a2av_gmm.h)
 *   ataOut_s  [A, H1/32]    E8M0 scales of those rows, same order
 *   recvCounts [W * e]      int32, entry w * e + j
 *   gmmWeight_q [e, N1, H1] codes: each output column's H1 codes contiguous
 *   gmmWeight_s [e, N1, H1/32]
 *   mmX_q [BS, H2], mmX_s [BS, H2/32], mmWeight_q [N2, H2], mmWeight_s [N2, H2/32]
 *   permuteOut_q [A, H1], permuteOut_s [A, H1/32]   expert-major (optional)
 *   gmmY [A, N1] bf16, mmY [BS, N2] bf16
 *
 * Two phases, as in a2av_gmm.h: a2av_gmm_mx_workspace_size validates the
 * descriptor and sizes the workspace; a2av_gmm_mx_run enqueues the work (it
 * never synchronises or allocates).  The caller owns every buffer.  Errors
 * found on the device (recvCounts inconsistent with A) are recorded in the
 * workspace's status word: read them with a2av_gmm_read_device_status.
 * Status codes: those of a2av_gmm.h (A2AV_ERR_INVALID: a shape or format
 * outside the limits; A2AV_ERR_UNSUPPORTED: a limit of this library or a
 * misaligned pointer; A2AV_ERR_WORKSPACE: workspace too small or not 256-byte
 * aligned).
 */
#ifndef A2AV_GMM_MX_H
#define A2AV_GMM_MX_H

#include <stddef.h>
#include <stdint.h>

#include "a2av_gmm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t W, e;
    int64_t A, H1, N1;
    int64_t BS, H2, N2;
    int32_t qtype;            /* code format of every operand: 0 E4M3FN, 1 E5M2 */
    int32_t want_permute_out; /* 1: write permuteOut_q / permuteOut_s */
    int32_t tiles;            /* a2av_tiles: DEFAULT (= PAIR), SINGLE (128 x 128 tiles on one CTA),
                                 PAIR (256 x 256 tiles on a cluster of two CTAs, cta_group::2) */
} a2av_gmm_mx_desc;

a2av_status a2av_gmm_mx_workspace_size(const a2av_gmm_mx_desc *desc, size_t *bytes);

a2av_status a2av_gmm_mx_run(const a2av_gmm_mx_desc *desc, const void *ataOut_q, const void *ataOut_s,
                            const int32_t *recvCounts, const void *gmmWeight_q, const void *gmmWeight_s,
                            const void *mmX_q, const void *mmX_s, const void *mmWeight_q, const void *mmWeight_s,
                            void *permuteOut_q, void *permuteOut_s, void *gmmY, void *mmY, void *workspace,
                            size_t workspace_bytes, a2av_stream_t stream);

/*
 * Diagnostic form of a2av_gmm_mx_run for measurement, as a2av_gmm_run_profiled
 * is for the bf16 call: the same work, plus two CUDA events (cudaEvent_t,
 * created by the caller) recorded on `stream` right before and right after
 * the grouped-GEMM kernel, which then follows the prep kernel in plain
 * stream order.  Returns A2AV_ERR_NULLPTR when either event is NULL, else as
 * a2av_gmm_mx_run.
 */
a2av_status a2av_gmm_mx_run_profiled(const a2av_gmm_mx_desc *desc, const void *ataOut_q, const void *ataOut_s,
                                     const int32_t *recvCounts, const void *gmmWeight_q,
                                     const void *gmmWeight_s, const void *mmX_q, const void *mmX_s,
                                     const void *mmWeight_q, const void *mmWeight_s, void *permuteOut_q,
                                     void *permuteOut_s, void *gmmY, void *mmY, void *workspace,
                                     size_t workspace_bytes, a2av_stream_t stream, void *gemm_begin_event,
                                     void *gemm_end_event);

#ifdef __cplusplus
}
#endif

#endif /* A2AV_GMM_MX_H */
