/*
 * a2av_gmm — Permute + GroupedMatMul (+ shared-expert MatMul) on one GB300.
 *
 * The receive side of an expert-parallel MoE layer, after the AlltoAllv has
 * landed on this GPU.  Operation ("aclnnAlltoAllvGroupedMatMul" operator
 * page, "API function" and "Formula"):
 *
 *     permuteOut = Permute(ataOut)             routed experts
 *     gmmY       = permuteOut x gmmWeight      one [H1, N1] matrix per expert
 *     mmY        = mmX x mmWeight              shared expert, independent
 *
 * Two-phase call, as on that page ("... is called to obtain the input
 * parameters and compute the required workspace size ... Then ... is called
 * to perform computation"): a2av_gmm_workspace_size() validates the
 * descriptor and sizes the workspace on the host; a2av_gmm_run() enqueues the
 * work on a CUDA stream.  Both return a status code ("Returns": status code;
 * the first phase implements input parameter verification).
 *
 * Shapes and ranges ("Shape variables"):
 *     W   ranks in the expert-parallel domain (sources of ataOut)
 *     e   experts on this rank, 1 <= e <= 32, and W * e <= 256
 *     A   rows received = sum of recvCounts (0 allowed: only mmY is computed)
 *     H1  routed hidden size, 0 < H1 < 65536
 *     N1  routed output width, 0 < N1 < 65536
 *     BS  shared-expert rows (0 = no shared expert)
 *     H2  shared hidden size, 0 < H2 <= 12288 (when BS > 0)
 *     N2  shared output width, 0 < N2 < 65536 (when BS > 0)
 * This library additionally needs H1, N1, H2, N2 to be multiples of 8 (rows
 * start on 16-byte boundaries) and A <= 2^31 - 1.
 *
 * Layouts (all row-major, contiguous, 16-byte aligned, device memory):
 *     ataOut     [A, H1]     rank-major: all rows from source 0 (its rows for
 *                            expert 0, then expert 1, ...), then source 1, ...
 *     recvCounts [W * e]     int32, entry w * e + j = rows from source w for
 *                            local expert j
 *     gmmWeight  [e, H1, N1]
 *     mmX        [BS, H2],  mmWeight [H2, N2],  mmY [BS, N2]
 *     permuteOut [A, H1]     expert-major: rows of expert 0 (source 0 first,
 *                            arrival order kept), then expert 1, ...
 *     gmmY       [A, N1]     row i pairs with row i of permuteOut
 * Element type: bf16 or fp16 for every tensor (same type throughout);
 * products accumulate in fp32 and are rounded to the element type (nearest
 * even).
 *
 * Ownership: the caller owns every buffer, including the workspace.  The
 * library allocates nothing, never synchronises inside a2av_gmm_run, and
 * keeps no pointer after the call returns; the workspace may be reused once
 * the stream has passed the call.  Results are deterministic: the same inputs
 * give bitwise the same outputs ("Deterministic computing").
 *
 * Errors found on the device (recvCounts that do not sum to A, a negative
 * count) cannot be returned by the asynchronous call: the kernels then write
 * no output and record the error in the workspace, where
 * a2av_gmm_read_device_status() finds it.
 */
#ifndef A2AV_GMM_H
#define A2AV_GMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *a2av_stream_t;

typedef enum {
    A2AV_OK = 0,
    A2AV_ERR_NULLPTR = 1,      /* a required pointer is NULL */
    A2AV_ERR_INVALID = 2,      /* shape, range or dtype outside the limits above */
    A2AV_ERR_UNSUPPORTED = 3,  /* allowed by the operator, not by this library (alignment) */
    A2AV_ERR_WORKSPACE = 4,    /* workspace too small or misaligned */
    A2AV_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
    A2AV_ERR_DEVICE_CHECK = 6, /* the device found inconsistent recvCounts */
    A2AV_ERR_SCRATCH_LIMIT = 7, /* a2av_gmm_run_static_scratch: the problem needs more
                                   scratch than the library's static array holds */
    A2AV_ERR_ARRIVAL_TIMEOUT = 8 /* a2av_gmm_run_arrivals: a source's rows did not arrive
                                   within the wait limit (device-detected) */
} a2av_status;

typedef enum { A2AV_BF16 = 0, A2AV_FP16 = 1, A2AV_FP32 = 2 /* a2av_found_nonfinite only */ } a2av_dtype;

/* Execution path.  All give bitwise-identical outputs. */
typedef enum {
    A2AV_PATH_DEFAULT = 0,     /* SPLIT_RUNS: which halves are staged is decided on the
                                  device from recvCounts */
    A2AV_PATH_FUSED = 1,       /* one kernel: the grouped GEMM gathers its A rows from ataOut */
    A2AV_PATH_SPLIT = 2,       /* a permute kernel stages every row expert-major, then the GEMM */
    A2AV_PATH_SPLIT_RUNS = 3   /* the permute kernel stages only the 128-row halves of a GEMM
                                  tile that straddle a run boundary; the GEMM reads the
                                  others in place from ataOut */
} a2av_path;

/* GEMM tile shape.  All give bitwise-identical outputs. */
typedef enum {
    A2AV_TILES_DEFAULT = 0,    /* the faster shape for this library */
    A2AV_TILES_SINGLE = 1,     /* 128-row tiles, one CTA each */
    A2AV_TILES_PAIR = 2,       /* 256-row tiles on a cluster of two CTAs; pipeline stages
                                  128 deep in K where H1, H2 are multiples of 128 and the
                                  weight columns load in whole 64-wide atoms */
    A2AV_TILES_PAIR_K64 = 3    /* 256-row tiles, stages always 64 deep in K */
} a2av_tiles;

typedef struct {
    int32_t W, e;              /* ranks, local experts */
    int64_t A, H1, N1;         /* routed experts */
    int64_t BS, H2, N2;        /* shared expert; BS = 0: none */
    int32_t dtype;             /* a2av_dtype */
    int32_t want_permute_out;  /* nonzero: permuteOut is written */
    int32_t path;              /* a2av_path */
    int32_t tiles;             /* a2av_tiles */
} a2av_gmm_desc;

/*
 * Phase 1 (host only, touches no GPU).  Validates *desc against the limits
 * above and writes the workspace size in bytes to *bytes.
 * Returns A2AV_ERR_NULLPTR if desc or bytes is NULL, A2AV_ERR_INVALID or
 * A2AV_ERR_UNSUPPORTED for a bad descriptor, else A2AV_OK.
 */
a2av_status a2av_gmm_workspace_size(const a2av_gmm_desc *desc, size_t *bytes);

/*
 * Phase 2.  Enqueues the whole hot path on `stream` and returns without
 * waiting.  Pointers are device pointers.  mmX, mmWeight and mmY may be NULL
 * when desc->BS == 0; permuteOut may be NULL unless desc->want_permute_out.
 * ataOut and gmmY may be NULL when desc->A == 0.  workspace must be 256-byte
 * aligned and at least the size phase 1 returned.
 * Returns: the phase-1 codes for the descriptor; A2AV_ERR_NULLPTR for a
 * missing required pointer; A2AV_ERR_UNSUPPORTED for a pointer that is not
 * 16-byte aligned; A2AV_ERR_WORKSPACE; A2AV_ERR_CUDA when a launch fails.
 */
a2av_status a2av_gmm_run(const a2av_gmm_desc *desc, const void *ataOut,
                         const int32_t *recvCounts, const void *gmmWeight,
                         const void *mmX, const void *mmWeight, void *permuteOut,
                         void *gmmY, void *mmY, void *workspace,
                         size_t workspace_bytes, a2av_stream_t stream);

/*
 * Diagnostic form of a2av_gmm_run for measurement: the same work, plus two
 * CUDA events (cudaEvent_t, created by the caller) recorded on `stream`
 * right before and right after the grouped-GEMM kernel, so that the
 * elapsed time between them is that kernel's duration alone.  The GEMM then
 * starts after the permute kernel in plain stream order instead of being
 * launched beside it.  (The operator page has no counterpart.)
 * Returns A2AV_ERR_NULLPTR when either event is NULL, else as a2av_gmm_run.
 */
a2av_status a2av_gmm_run_profiled(const a2av_gmm_desc *desc, const void *ataOut,
                                  const int32_t *recvCounts, const void *gmmWeight,
                                  const void *mmX, const void *mmWeight, void *permuteOut,
                                  void *gmmY, void *mmY, void *workspace,
                                  size_t workspace_bytes, a2av_stream_t stream,
                                  void *gemm_begin_event, void *gemm_end_event);

/*
 * The same computation, started before the AlltoAllv has finished: the
 * overlap of the exchange with the grouped GEMM ("aclnnAlltoAllvGroupedMatMul",
 * API function: AlltoAllv fused with Permute and GroupedMatMul; Formula:
 * ataOut = AlltoAllv(gmmX)).
 *
 * `arrived` is a device array of W 64-bit flags, one per source rank.  The
 * rows source w sends (its e runs of ataOut, rank-major) may be read once
 * arrived[w] == arrival_tag; whatever moves them (a copy engine, a peer GPU's
 * stores, the host) sets the flag after the rows have landed, for example
 * by a copy of the tag ordered after the row copies on the same stream.
 * recvCounts must be final when the call starts.  The kernel computes the
 * shared expert first (it reads no exchanged rows), then each routed tile
 * waits for the flags of the sources its rows come from and gathers those
 * rows straight from ataOut (the fused path; desc->path must be
 * A2AV_PATH_DEFAULT or A2AV_PATH_FUSED).  Flags must be 8-byte aligned; a
 * new call uses a new tag, so flags need no reset between calls.
 *
 * Every wait is bounded by wait_limit_ns (0: 2 s).  A source that has not
 * arrived by then makes the kernel wind down without finishing; the device
 * status then reads A2AV_ERR_ARRIVAL_TIMEOUT (a2av_gmm_read_device_status)
 * and the outputs are incomplete.  Other arguments and return codes are
 * those of a2av_gmm_run.
 */
a2av_status a2av_gmm_run_arrivals(const a2av_gmm_desc *desc, const void *ataOut,
                                  const int32_t *recvCounts, const void *gmmWeight,
                                  const void *mmX, const void *mmWeight, void *permuteOut,
                                  void *gmmY, void *mmY, const uint64_t *arrived,
                                  uint64_t arrival_tag, uint64_t wait_limit_ns,
                                  void *workspace, size_t workspace_bytes, a2av_stream_t stream);

/*
 * Waits for `stream`, then reads the device-side status a2av_gmm_run left in
 * `workspace`: A2AV_OK, or A2AV_ERR_DEVICE_CHECK (recvCounts negative or not
 * summing to A; outputs were not written; or, in a debug build compiled with
 * A2AV_CHECKS, an index found out of range and not used), A2AV_ERR_ARRIVAL_TIMEOUT
 * (a2av_gmm_run_arrivals: a source never arrived), or A2AV_ERR_CUDA (a kernel
 * gave up waiting on one of its own pipeline barriers).  The raw device word is
 * written to *code when code is not NULL.  For tests and diagnostics: it
 * synchronises.
 */
a2av_status a2av_gmm_read_device_status(const void *workspace, a2av_stream_t stream,
                                        int32_t *code);

/*
 * Same computation as a2av_gmm_run, for callers that cannot allocate device
 * memory.  (The operator page has no counterpart: this entry point exists
 * only in this library.)
 *
 * Who needs it: code that is handed only its inputs and outputs and has no
 * way to obtain a workspace, for example an operator plugged into a
 * framework or runtime that owns the whole device memory pool, or a
 * latency-critical loop that must not call cudaMalloc, which can block the
 * host and synchronise the device.
 *
 * Instead of a caller-provided workspace it uses one scratch array that the
 * library defines in device memory: A2AV_STATIC_SCRATCH_BYTES bytes, held on
 * every GPU that loads the library until the process exits.  The fused
 * path needs only its 256-byte status area; the split path without
 * permuteOut also stages A * H1 * 2 bytes there.  A descriptor whose
 * workspace (as a2av_gmm_workspace_size reports it) exceeds the array is
 * rejected with A2AV_ERR_SCRATCH_LIMIT before anything is enqueued.  This
 * call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 *
 * Set-up: every call looks up the array's device address in the current
 * device's context (cudaGetSymbolAddress, a host-side query that allocates
 * nothing), so a context that was torn down and created again (after
 * cudaDeviceReset) gets the array's new address.  The first call on a device
 * may also load the library's kernels into that context; make that first
 * call before any stream capture begins.
 *
 * Sharing: every call on a device uses the same array, and the array keeps
 * the previous call's contents.  The kernels overwrite every scratch byte
 * they later read (the status word is stored afresh at the start of each
 * call), so nothing needs clearing between calls.  Two calls that may run at
 * the same time on the GPU (different streams without ordering between
 * them) race on the array: order them on one stream or with events.  The
 * device status word of this call cannot be read back; on inconsistent
 * recvCounts the outputs are left unwritten, as with a2av_gmm_run.
 *
 * Arguments and other return codes are those of a2av_gmm_run.
 */
#define A2AV_STATIC_SCRATCH_BYTES ((size_t)256 + ((size_t)8 << 20))
a2av_status a2av_gmm_run_static_scratch(const a2av_gmm_desc *desc, const void *ataOut,
                                        const int32_t *recvCounts, const void *gmmWeight,
                                        const void *mmX, const void *mmWeight,
                                        void *permuteOut, void *gmmY, void *mmY,
                                        a2av_stream_t stream);

/*
 * Dynamic loss-scale update ("aclnnAmpUpdateScale" page, "Formula" and its
 * notes), in place on device scalars, enqueued on `stream`:
 *   *found_inf != 0                  -> *scale *= backoff_factor, *tracker = 0
 *   else *tracker + 1 == interval    -> grown = *scale * growth_factor;
 *                                       *scale = grown if finite (else kept);
 *                                       *tracker = 0
 *   else                             -> *tracker += 1
 * scale and found_inf are float32 (the page requires one type for both),
 * growth_tracker int32.  Products are float32, rounded to nearest.
 * Returns A2AV_ERR_NULLPTR for a NULL pointer, A2AV_ERR_INVALID for
 * growth_interval < 1 (the page's range is [1, 2147483647]).
 */
a2av_status a2av_amp_update_scale(float *scale, int32_t *growth_tracker, const float *found_inf,
                                  float growth_factor, float backoff_factor,
                                  int32_t growth_interval, a2av_stream_t stream);

/*
 * Sets *found_inf = 1.0f when any of the n elements of x (device, a2av_dtype:
 * bf16, fp16 or fp32) is inf or NaN, and leaves it unchanged otherwise, so
 * several tensors can be checked into one flag before a2av_amp_update_scale.
 * x must be 16-byte aligned.  Enqueued on `stream`.
 */
a2av_status a2av_found_nonfinite(const void *x, int64_t n, int32_t dtype, float *found_inf,
                                 a2av_stream_t stream);

/* A static, human-readable name for a status code. */
const char *a2av_gmm_status_string(a2av_status status);

/* Kernels a2av_gmm_run launches for this descriptor (0 on a bad descriptor). */
int32_t a2av_gmm_launch_count(const a2av_gmm_desc *desc);

#ifdef __cplusplus
}
#endif

#endif /* A2AV_GMM_H */
