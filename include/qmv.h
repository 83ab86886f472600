/*
 * qmv.h -- C ABI of the weight-only mixed-bit packed matvec library (GB300,
 * sm_103a).
 *
 * y = W . x for weights stored as packed low-bit codes with fp16 scales,
 * fp16 activations and fp32 accumulation, with an optional residual-add +
 * RMSNorm folded into the matvec.  The method follows these pages:
 *   [A19]  "Gemma4 raw-Metal loop on A19 -- findings + the remaining (parked)
 *          levers", section "What moved the needle": int2 codes, 16 per 32-bit
 *          word, exact products, fp32 sums in code order; q/k/v and gate/up
 *          fused into single dispatches; residual-add + RMSNorm folded into
 *          the next matvec's prologue; int8 weights loaded as vectors.
 *   [PLAY] "raw-metal-loop-playbook", prefill-regimes table: chunks of M
 *          tokens read the weights once per M tokens; M = 8/16 tiles keep each
 *          output scalar's K-dot in the M = 1 order; M = 64/128 tiles use the
 *          matrix units and change the order.
 *
 * Conventions (all entry points):
 *   - Every pointer named d_* or described as "device" is a CUDA device
 *     pointer owned by the caller.  The library allocates no device memory:
 *     the scratch some calls need (the tensor-core tiles' split-K partial
 *     tiles, the fused prologue's normalised activations for M >= 2) is a
 *     caller-provided workspace whose size qmv_workspace_bytes() gives.
 *   - fp16 values are IEEE binary16 bit patterns (uint16_t / __half).
 *   - Matrices are row-major with no padding.  Activations are M x K (row m is
 *     column m of the matvec, i.e. token m); outputs are M x N.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on it; nothing synchronises.
 *   - Every call returns a qmv_status.  Arguments are validated on the host;
 *     no call aborts, throws across the ABI or traps on the device.  A failed
 *     launch returns QMV_ERR_CUDA and qmv_last_cuda_error() gives the raw
 *     cudaError_t (thread-local).
 *   - Packs are immutable after qmv_pack_weights, so concurrent calls that
 *     share a pack are safe.
 *
 * Packed layout (the bit order is a reading: the pages give only "16 codes
 * per word"): row n of codes is K*bits/32 little-endian uint32 words; code k
 * sits in word floor(k*bits/32) at bit offset bits*(k mod (32/bits)); the
 * field holds u = v + 2^(bits-1) for the signed code v, so int2 fields
 * 0,1,2,3 decode to -2,-1,0,1.  Scales are fp16 [N][K/group].
 *
 * Accumulation order (QMV_EXACT, every CUDA-core path, any M): for
 * each output scalar, each block of 32 consecutive codes is summed serially
 * in k in fp32 (products are exact); with group 32 the block sum is
 * multiplied by its scale (rounded) and added to the accumulator (rounded),
 * blocks in order; with one scale per row (group == K) the block sums are
 * added serially and the total is multiplied by the scale once.  This is the
 * oracle's order, so QMV_EXACT results are bit-identical to it, and every
 * column of an M-tile is bit-identical to the M = 1 result.
 *
 * QMV_FAST (CUDA-core paths): the same blocks, scales and fold, with the code offset
 * taken out of the per-code work: each block is summed as sum(y*u) over the
 * unsigned fields u (even and odd words in two serial chains, then added)
 * minus 2^(bits-1) times the block's activation sum formed in the same
 * order.  Results are within max |y - ref| <= 1e-3*(1+|ref|) of the oracle
 * (in practice a few fp32 ulps of the block sums), a block of zero codes
 * gives exactly 0, and every column of an M-tile is still bit-identical to
 * the QMV_FAST M = 1 result.  Shapes outside the M = 1 pipeline (K not a
 * multiple of 256) keep the exact order in both modes.
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QMV_API __attribute__((visibility("default")))
#else
#define QMV_API
#endif

typedef struct qmv_pack qmv_pack;   /* opaque host descriptor; owns no device memory */
typedef struct qmv_chain qmv_chain; /* opaque host descriptor of a matvec chain */

typedef enum {
    QMV_OK = 0,
    QMV_ERR_INVALID_ARG = -1,   /* null pointer, bad enum value, M out of range */
    QMV_ERR_UNSUPPORTED = -2,   /* valid but not implemented (e.g. a tile shape) */
    QMV_ERR_ALIGNMENT = -3,     /* a pointer is not aligned as documented */
    QMV_ERR_SHAPE = -4,         /* N/K/bits/group disagree with the pack or layout rules */
    QMV_ERR_CUDA = -5,          /* a CUDA runtime call or launch failed */
    QMV_ERR_TIMEOUT = -6,       /* a bounded device-side wait ran out */
    QMV_ERR_WORKSPACE = -7      /* the call needs a larger workspace (qmv_workspace_bytes) */
} qmv_status;

typedef enum { QMV_F32 = 0, QMV_F16 = 1 } qmv_dtype;      /* output element type */
typedef enum { QMV_FAST = 0, QMV_EXACT = 1 } qmv_mode;    /* accumulation mode */

/*
 * qmv_create_pack -- describe a packed weight matrix.  [A19] int2 item:
 * 16 codes per word; int4 and int8 use the same offset-binary rule.
 *   N, K   output and input features; K*bits/8 must be a multiple of 16
 *          (K % 64 == 0 for int2, K % 32 == 0 for int4 and int8).
 *   bits   2, 4 or 8.
 *   group  32 (one fp16 scale per 32 consecutive k of a row) or K (one
 *          scale per row).
 *   codes_bytes, scales_bytes  (out, nullable) bytes the caller must allocate
 *          for the packed codes (N*K*bits/8) and the scales (N*(K/group)*2).
 * Errors: QMV_ERR_INVALID_ARG (out is NULL, bits/group not allowed),
 * QMV_ERR_SHAPE (N < 1, K not allowed).  Host only; touches no device.
 */
QMV_API int qmv_create_pack(qmv_pack **out, int N, int K, int bits, int group,
                    size_t *codes_bytes, size_t *scales_bytes);

/*
 * qmv_pack_weights -- pack signed codes on the device and bind the pack to
 * the caller's buffers.  [A19] int2 item (16 codes per 32-bit word).
 *   d_codes_in   device int8 [N][K], signed codes in [-2^(bits-1), 2^(bits-1)-1].
 *                A code out of range is masked to its low `bits` bits.
 *   d_scales_in  device fp16 [N][K/group].
 *   d_codes      device, codes_bytes, 16-byte aligned: receives the words.
 *   d_scales     device, scales_bytes, 16-byte aligned: receives a copy of
 *                the scales.
 * The pack keeps d_codes/d_scales; they must outlive every later call that
 * uses the pack.  Errors: INVALID_ARG (NULL), ALIGNMENT, CUDA.
 */
QMV_API int qmv_pack_weights(qmv_pack *p, const int8_t *d_codes_in, const uint16_t *d_scales_in,
                     void *d_codes, void *d_scales, void *stream);

/*
 * qmv_workspace_bytes -- device scratch bytes that a call of qmv_gemv /
 * qmv_chunk_gemm (fused = 0) or qmv_fused_rmsnorm_gemv (fused = 1) with this
 * pack, M, y_dtype and mode needs in its d_workspace:
 *   - M = 1, or K not a multiple of 256: 0.
 *   - M > 32, QMV_FAST, int2, fused = 0 (the tensor-core tiles): fp32
 *     split-K partial tiles when the chosen split needs more than the output
 *     itself, else 0.
 *   - every other M >= 2 (the CUDA-core M-column tiles): the activation
 *     tables, built once per call: per 512 codes, 8960 bytes per 4 columns
 *     (ceil(M/4) * ceil(K/512) * 8960), or 17408 per 8 columns where the
 *     library takes 8-column tiles (M >= 5), fused or not.
 * The size depends only on these arguments and the device's SM count, so one
 * workspace serves every later call with them.  Host only; 0 for invalid
 * arguments.
 */
QMV_API size_t qmv_workspace_bytes(const qmv_pack *p, int M, int y_dtype, int mode, int fused);

/*
 * qmv_gemv -- y = x . W^T for M columns: y[m][n] = sum_g (sum_{k in g}
 * x[m][k] * v[n][k]) * s[n][g] in the order stated at the top of this file.
 * [A19] int2 item (exact products, fp32 in code order); [PLAY] K-order-fixed
 * row for M <= 16 and matrix-unit row for M >= 64.
 *   M            1 .. 4096.  Every M runs the CUDA-core kernels (QMV_EXACT
 *                bit-exact, QMV_FAST within tolerance, each column equal to
 *                the M = 1 result), except M > 32 with QMV_FAST and int2
 *                weights, which runs tcgen05 tensor-core tiles (fp32
 *                accumulate, hardware order, within tolerance).  With K a
 *                multiple of 256 the M >= 2 CUDA-core tiles take all M
 *                columns in one launch; otherwise 32 columns per launch.
 *   N, K, bits, group  must equal the pack's (QMV_ERR_SHAPE otherwise).
 *   x            device fp16 [M][K], 16-byte aligned.
 *   y            device [M][N] of y_dtype (fp32, or fp16 = RNE of the fp32
 *                result), 4-byte aligned.
 *   mode         QMV_FAST or QMV_EXACT.
 *   d_workspace, workspace_bytes  caller scratch, 256-byte aligned, at least
 *                qmv_workspace_bytes(p, M, y_dtype, mode, 0) bytes (may be
 *                NULL, 0 when that is 0).  Its contents on entry do not
 *                matter; calls that share a workspace must not overlap.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, UNSUPPORTED, WORKSPACE, CUDA.
 */
QMV_API int qmv_gemv(const qmv_pack *p, int M, int N, int K, int bits, int group,
             const void *x, void *y, int y_dtype, int mode, void *d_workspace,
             size_t workspace_bytes, void *stream);

/*
 * qmv_fused_rmsnorm_gemv -- residual add + RMSNorm folded into the matvec
 * prologue ([A19] dispatch-count fusion item).  For each column m:
 *   h = fp16(x + residual); ss = sum of h*h (serial in blocks of 32, then
 *   serial over blocks); inv = 1/sqrt(ss/K + eps) (IEEE fp32 ops);
 *   y16 = fp16((h * inv) * gamma); then y = matvec(y16) as qmv_gemv.
 *   x, residual  device fp16 [M][K]; gamma device fp16 [K]; 16-byte aligned.
 *   h_out        nullable device fp16 [M][K]: receives h (the next residual).
 *   M            1 .. 4096; every column runs the CUDA-core kernels (the
 *                fused prologue never takes the tensor-core tiles), each
 *                column equal to the M = 1 result.
 *   d_workspace, workspace_bytes  as qmv_gemv, sized by
 *                qmv_workspace_bytes(p, M, y_dtype, mode, 1).
 * Errors: as qmv_gemv.
 */
QMV_API int qmv_fused_rmsnorm_gemv(const qmv_pack *p, int M, const void *x, const void *residual,
                           const void *gamma, float eps, void *h_out, void *y,
                           int y_dtype, int mode, void *d_workspace, size_t workspace_bytes,
                           void *stream);

/*
 * qmv_chunk_gemm -- a prefill chunk of M tokens against one pack ([PLAY]
 * prefill-regimes table): the same computation as qmv_gemv with the pack's
 * own N, K, bits and group.  M = 4, 8, 16 (and any M <= 32, or any M in
 * QMV_EXACT, or int4/int8) use the K-order-fixed CUDA-core tiles; M = 64,
 * 128 (any M > 32) in QMV_FAST with int2 weights use tcgen05 tensor-core
 * tiles.  d_workspace, workspace_bytes as qmv_gemv.
 */
QMV_API int qmv_chunk_gemm(const qmv_pack *p, int M, const void *x, void *y, int y_dtype,
                   int mode, void *d_workspace, size_t workspace_bytes, void *stream);

/*
 * qmv_gemv_argmax -- the lm_head matvec with the greedy-token step fused into
 * its epilogue ([A19] "The parked levers" table, argmax stage1+2 merge row:
 * one dispatch, first-max tie-break): y = matvec(x) for M = 1 as qmv_gemv
 * (or, with residual != NULL, as qmv_fused_rmsnorm_gemv with gamma, eps and
 * h_out), then the index of the largest fp32 result -- the lowest index among
 * equal maxima; values compare as numbers (-0 equals +0); NaN never wins.
 *   y            nullable: device [N] of y_dtype receives the logits; NULL
 *                skips the store.
 *   d_index      device int32: receives the index (-1 if every value is NaN).
 *   d_value      nullable device fp32: receives the maximum (its value;
 *                a maximum of -0 reads +0).
 *   d_workspace  device, qmv_argmax_workspace_bytes() bytes, 8-byte aligned,
 *                all zero before the first call; every completed call leaves
 *                it zero.  Calls sharing a workspace must not overlap.
 * The index is exact against the oracle in QMV_EXACT mode.  Needs
 * K % 256 == 0 (the M = 1 pipeline); QMV_ERR_UNSUPPORTED otherwise.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, CUDA.
 */
QMV_API size_t qmv_argmax_workspace_bytes(void);
QMV_API int qmv_gemv_argmax(const qmv_pack *p, const void *x, const void *residual,
                            const void *gamma, float eps, void *h_out, void *y, int y_dtype,
                            int mode, int *d_index, float *d_value, void *d_workspace,
                            void *stream);

/*
 * qmv_gemv_gather -- the expert-gather matvec of a mixture-of-experts decode
 * step, with no gathered copy of the weights ([PLAY] ranked-targets table,
 * MoE row: a zero-materialization expert-gather matvec): the pack holds E = N / rows_per_expert experts
 * of rows_per_expert rows each, stacked; for the n_selected expert ids in
 * d_expert_ids, y[j*rows_per_expert + r] = (row r of expert ids[j]) . x, for
 * M = 1, computed exactly as qmv_gemv computes those rows (the row groups of
 * the selected experts are fetched by index inside the kernel).
 *   rows_per_expert  divides N.
 *   d_expert_ids     device int32 [n_selected], 1 <= n_selected <= 256; may be
 *                    written by the kernel launched just before (it is read
 *                    after that kernel completes).  An id outside [0, E)
 *                    yields zero outputs for its rows and sets the device
 *                    error word (8).
 *   x  device fp16 [K];  y  device [n_selected * rows_per_expert] of y_dtype.
 * Needs K % 256 == 0 (the M = 1 pipeline).
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, UNSUPPORTED, CUDA.
 */
QMV_API int qmv_gemv_gather(const qmv_pack *p, int rows_per_expert, const int *d_expert_ids,
                            int n_selected, const void *x, void *y, int y_dtype, int mode,
                            void *stream);

/*
 * qmv_unpack_codes -- decode the packed words back to signed int8 codes
 * [N][K] with the same decode routine the matvec kernels use (a check of
 * that routine; not on the hot path).  d_codes_out: device int8, N*K bytes.
 */
QMV_API int qmv_unpack_codes(const qmv_pack *p, int8_t *d_codes_out, void *stream);

/* qmv_pack_info -- read back a pack's shape (any out pointer may be NULL). */
QMV_API int qmv_pack_info(const qmv_pack *p, int *N, int *K, int *bits, int *group);

/*
 * Saving and reloading packed weights.  A saved pack is its 64-byte header
 * followed by the bytes of d_codes and of d_scales exactly as
 * qmv_pack_weights wrote them (the caller copies them; the library does no
 * file or host I/O).  Header, little-endian:
 *   bytes  0..7   magic "QMVPACK" and a zero byte
 *   bytes  8..11  uint32 layout version (QMV_PACK_VERSION: the packed-word
 *                 layout of qmv_pack_weights; any other version is refused)
 *   bytes 12..15  uint32 header size (64)
 *   bytes 16..31  int32 N, K, bits, group
 *   bytes 32..47  uint64 codes_bytes, scales_bytes
 *   bytes 48..63  zero
 */
#define QMV_PACK_HEADER_BYTES 64
#define QMV_PACK_VERSION 1

/* qmv_pack_header -- write the header of pack p to header_out (64 bytes,
 * host memory).  Errors: INVALID_ARG (p not a pack, header_out NULL).
 * Host only. */
QMV_API int qmv_pack_header(const qmv_pack *p, void *header_out);

/* qmv_create_pack_from_header -- check a saved header and describe its pack,
 * as qmv_create_pack would (codes_bytes, scales_bytes nullable).
 * Errors: INVALID_ARG (NULL, wrong magic or header size, nonzero reserved
 * bytes, bits/group not allowed), UNSUPPORTED (another layout version),
 * SHAPE (shape not allowed, or byte counts that disagree with it).  Host only. */
QMV_API int qmv_create_pack_from_header(qmv_pack **out, const void *header,
                                        size_t *codes_bytes, size_t *scales_bytes);

/* qmv_bind_packed -- bind device buffers that already hold packed words and
 * scales (the output of qmv_pack_weights for this shape, e.g. reloaded from a
 * saved pack), without packing.  d_codes, d_scales: device, 16-byte aligned,
 * codes_bytes and scales_bytes long; the pack keeps them, as with
 * qmv_pack_weights.  Errors: INVALID_ARG (NULL), ALIGNMENT.  Host only. */
QMV_API int qmv_bind_packed(qmv_pack *p, void *d_codes, void *d_scales);

/* qmv_destroy_pack -- free the host descriptor (never the device buffers). */
QMV_API int qmv_destroy_pack(qmv_pack *p);

/*
 * qmv_set_pdl -- programmatic dependent launch of the M = 1 matvec kernels
 * for the calling thread (default off).  When on, a matvec launched right
 * after another kernel in the same stream may start while that kernel is
 * still running: it begins streaming its packed weights at once and waits
 * for the previous kernel to complete (griddepcontrol.wait) before it reads
 * x / residual / gamma or writes any output.  This hides launch latency
 * between the dependent matvecs of a decode layer ([A19] "What moved the
 * needle", dispatch-count item: the per-dispatch tax between kernels).
 * Requirement: the packed weights of a matvec must not be written by the
 * kernel launched just before it in the stream (pack once, then run).
 * Works under stream capture (CUDA graphs).  Always returns QMV_OK.
 */
QMV_API int qmv_set_pdl(int enable);

/* qmv_status_string -- static text for a status code. */
QMV_API const char *qmv_status_string(int status);

/* qmv_last_cuda_error -- the raw cudaError_t behind the calling thread's
 * last QMV_ERR_CUDA (0 if none). */
QMV_API int qmv_last_cuda_error(void);

/*
 * qmv_device_error -- the device error word of the current device: 0, or
 * the code of the first bounded device-side wait that ran out (a kernel that
 * hits one stops, lets its own copies land and returns; its outputs are then
 * incomplete).  Synchronises with the device (reads a device symbol).
 *   out    receives the word.  clear: non-zero resets it to 0.
 * Errors: INVALID_ARG (out NULL), CUDA.
 */
QMV_API int qmv_device_error(int *out, int clear);

/*
 * Chains: a sequence of M = 1 matvecs (plain or with the fused residual-add +
 * RMSNorm prologue) run by one persistent launch -- the whole-layer / multi-
 * stage single dispatch of [A19] "The parked levers" (mega-kernel item),
 * against the per-dispatch tax of "What moved the needle".  Each op computes
 * exactly what the matching qmv_gemv / qmv_fused_rmsnorm_gemv call computes
 * (bit for bit, same mode), in order.  The weight stream runs across op
 * boundaries; a grid-wide barrier is inserted only before an op whose
 * activation reads (x, residual, gamma) overlap the outputs (y, h_out) of an
 * earlier op since the last barrier, or whose outputs overlap the reads or
 * outputs of such an op.  Packed weights must not change while a chain runs.
 * Every op needs K % 256 == 0.
 *
 * qmv_chain_workspace_bytes -- device bytes a chain of up to max_ops ops
 * needs (barrier words + op table); 0 if max_ops < 1.
 */
QMV_API size_t qmv_chain_workspace_bytes(int max_ops);

/*
 * qmv_chain_create -- an empty chain using the caller's device workspace
 * (256-byte aligned, at least qmv_chain_workspace_bytes(max_ops) bytes; it
 * must outlive the chain and must not be shared by two chains that run at
 * the same time).  Host only.
 * Errors: INVALID_ARG (NULL, max_ops < 1, workspace too small), ALIGNMENT.
 */
QMV_API int qmv_chain_create(qmv_chain **out, int max_ops, void *d_workspace,
                             size_t workspace_bytes);

/*
 * qmv_chain_create_no_alloc -- an empty chain whose barrier words and op table
 * live in the library's own scratch array (a file-scope device array, one per
 * device, room for 1024 ops), so neither the caller nor the library allocates
 * device memory for it.  The source pages have no counterpart: it is an interface
 * variant of qmv_chain_create.  The array's address is looked up here, once per
 * device (host bookkeeping behind a lock, so chains may be made and run from
 * several host threads); the chain must run on the device that was current
 * here.  Every run clears the barrier words; a run after another chain used
 * the array re-copies this chain's op table on the run's stream, so runs of
 * such chains queued one after another on one stream are ordered.  Chains
 * made this way share the array: runs of two of them that overlap in time
 * on the GPU (different streams) race, and so would a run overlapping its
 * own earlier run on another stream.
 * Errors: INVALID_ARG (NULL, max_ops < 1), UNSUPPORTED (max_ops > 1024), CUDA.
 */
QMV_API int qmv_chain_create_no_alloc(qmv_chain **out, int max_ops);

/*
 * qmv_chain_add_gemv / qmv_chain_add_fused_rmsnorm_gemv -- append one M = 1
 * matvec with the arguments of qmv_gemv / qmv_fused_rmsnorm_gemv (pointers
 * are recorded, not read, until qmv_chain_run).  Host only.
 * Errors: INVALID_ARG (NULL, chain full, bad enum), ALIGNMENT, UNSUPPORTED
 * (K % 256 != 0, or K too large for the chain's shared memory).
 */
QMV_API int qmv_chain_add_gemv(qmv_chain *c, const qmv_pack *p, const void *x, void *y,
                               int y_dtype, int mode);
QMV_API int qmv_chain_add_fused_rmsnorm_gemv(qmv_chain *c, const qmv_pack *p, const void *x,
                                             const void *residual, const void *gamma, float eps,
                                             void *h_out, void *y, int y_dtype, int mode);

/*
 * qmv_chain_run -- run every op of the chain, in order, as one cooperative
 * launch of one CTA per SM on `stream` (INVALID_ARG for a chain from
 * qmv_chain_create_no_alloc run on another device).  The first run after ops
 * were added copies the op table to the workspace with an asynchronous copy
 * on `stream` (ordered after the work queued there before); a run that needs
 * that copy while `stream` is capturing returns UNSUPPORTED.  Later runs only
 * clear the barrier words (an async memset) and launch.  Two runs of chains
 * that share a workspace must not overlap on the GPU.  A bounded device wait
 * that runs out shows in qmv_device_error.
 * Errors: INVALID_ARG, UNSUPPORTED (kernel does not fit an SM, or a table
 * copy during stream capture), CUDA.
 */
QMV_API int qmv_chain_run(qmv_chain *c, void *stream);

/* qmv_chain_info -- ops, inserted grid barriers, and the kernel's dynamic
 * shared memory (any out pointer may be NULL). */
QMV_API int qmv_chain_info(const qmv_chain *c, int *n_ops, int *n_barriers, int *smem_bytes);

/* qmv_chain_destroy -- free the host descriptor (never the workspace). */
QMV_API int qmv_chain_destroy(qmv_chain *c);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
