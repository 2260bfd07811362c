/*
 * libmgscan: scan primitives of the minGRU family on one NVIDIA GB300 (sm_103a).
 *
 * The operations are the scan primitives named on the mingru-scans pages
 * ("mingru-scans" home page, scan-op speedup table; "Run the benchmarks",
 * Step 2 timing matrix): matrix_affine_scan, matrix_scan and
 * parallel_scan_log, each with a forward and a backward pass.  The pages name
 * them without formulas; the recurrences are the standard ones for those
 * names and are stated at each entry point below.  parallel_scan_log is
 * Heinsen's log-space scan (arXiv:2311.06281, cited in the home page's
 * lineage paragraph).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor arguments are DEVICE pointers to contiguous, row-major fp32
 *   buffers owned by the caller.  The library never allocates, frees, prints
 *   or aborts.  Every pointer passed must be 16-byte aligned.
 * - Time index: outputs hold t = 1..T at positions 0..T-1; the initial state
 *   (h_0 or P_0 = I) is never part of an output.
 * - Block layout for the matrix ops, with d = H*k channels split into H
 *   independent k x k blocks per token:
 *       A, dA, P, grad_P   [B][T][H][k][k]   (A[..][i][j] multiplies h[j]
 *                                              into output row i)
 *       b, h, grad_h, db   [B][T][H][k]
 *       h0, dh0            [B][H][k]
 *   parallel_scan_log layout (D diagonal channels):
 *       log_coeffs, log_values, h, log_h, grad_h, d_log_coeffs,
 *       d_log_values       [B][T][D];   log_h0, d_log_h0   [B][D]
 * - Supported block sizes k: 4, 8, 16 for any H; 1 and 2 when H*k is a
 *   multiple of 4.  Other k return MGS_ERR_UNSUPPORTED.
 *   parallel_scan_log needs D to be a multiple of 4.
 * - B, T, H, D must be >= 0; T == 0 or an empty batch is a successful no-op.
 * - Outputs must not overlap any input or each other (MGS_ERR_INVALID_ARG).
 * - Calls are asynchronous on `stream` (NULL = the legacy default stream).  A
 *   returned MGS_OK means the work was validated and enqueued.  Faults found
 *   on the device (a bounded wait that gave up) are recorded in a per-device
 *   error word and reported by mgs_check().
 * - Workspace: entry points that take `workspace` need a caller-allocated
 *   device buffer of at least mgs_workspace_size(op, ...) bytes, 256-byte
 *   aligned (MGS_ERR_WORKSPACE otherwise).  The size depends only on the op and
 *   shape.  When the size is 0, workspace may be NULL.  Calls that share one
 *   workspace must be ordered on the same stream.
 */
#ifndef MGSCAN_H
#define MGSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mgs_status {
    MGS_OK = 0,
    MGS_ERR_INVALID_ARG = 1, /* null required pointer, negative size, overlap, overflow */
    MGS_ERR_UNSUPPORTED = 2, /* k or D outside the supported set, misaligned pointer   */
    MGS_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned            */
    MGS_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed           */
    MGS_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (see mgs_check)    */
} mgs_status;

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st *mgs_stream_t;

/* Operation ids for mgs_workspace_size. */
enum {
    MGS_OP_MATRIX_AFFINE_SCAN_FWD = 1,
    MGS_OP_MATRIX_AFFINE_SCAN_BWD = 2,
    MGS_OP_MATRIX_SCAN_FWD = 3,
    MGS_OP_MATRIX_SCAN_BWD = 4,
    MGS_OP_PARALLEL_SCAN_LOG_FWD = 5,
    MGS_OP_PARALLEL_SCAN_LOG_BWD = 6,
    MGS_OP_LINEAR_SCAN_FWD = 7,
    MGS_OP_LINEAR_SCAN_BWD = 8,
    MGS_OP_GIVENS_AFFINE_SCAN_FWD = 9,
    MGS_OP_GIVENS_AFFINE_SCAN_BWD = 10,
    MGS_OP_GIVENS_MATRIX_SCAN_FWD = 11,
    MGS_OP_GIVENS_MATRIX_SCAN_BWD = 12,
    MGS_OP_DELTA_SCAN_FWD = 13,
    MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE = 14
};

/* Bytes of device workspace `op` needs for this shape (H_or_D is H for the
 * matrix ops and D for parallel_scan_log; k is ignored for the latter).
 * Returns 0 when no workspace is needed, and also for invalid shapes (the
 * entry point then reports the error).  MGS_OP_PARALLEL_SCAN_LOG_BWD gives the
 * bytes of the recompute mode (h == NULL); with h saved it needs none.
 * MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE is the recompute-mode entry point's. */
size_t mgs_workspace_size(int op, int64_t B, int64_t T, int64_t H_or_D, int k);

/* matrix_affine_scan, forward ("mingru-scans" home page, scan-op table,
 * matrix_affine_scan row; the recurrence behind RotationMinGRU and
 * GivensMinGRU):
 *     h_t = A_t h_{t-1} + b_t,   t = 1..T,   per (batch, head) lane,
 * with h_0 = h0, or zeros when h0 is NULL.
 * In: A [B][T][H][k][k], b [B][T][H][k], h0 [B][H][k] (nullable).
 * Out: h [B][T][H][k]. */
mgs_status mgs_matrix_affine_scan_fwd(const float *A, const float *b, const float *h0, float *h,
                                      int64_t B, int64_t T, int64_t H, int k, void *workspace,
                                      size_t workspace_bytes, mgs_stream_t stream);

/* matrix_affine_scan, backward: gradients of L = sum_t <grad_h_t, h_t> through
 * the forward above.  With lambda_t = dL/dh_t,
 *     lambda_T = grad_h_T,   lambda_t = grad_h_t + A_{t+1}^T lambda_{t+1},
 *     db_t = lambda_t,   dA_t = lambda_t h_{t-1}^T,   dh0 = A_1^T lambda_1.
 * In: A, h0 (nullable: zero initial state), h = the forward output (saved),
 *     grad_h.  b is not needed.
 * Out: dA [B][T][H][k][k], db [B][T][H][k], dh0 [B][H][k] (nullable: not
 *     written). */
mgs_status mgs_matrix_affine_scan_bwd(const float *A, const float *h0, const float *h,
                                      const float *grad_h, float *dA, float *db, float *dh0,
                                      int64_t B, int64_t T, int64_t H, int k, void *workspace,
                                      size_t workspace_bytes, mgs_stream_t stream);

/* matrix_affine_scan, backward in recompute mode: the same gradients as
 * mgs_matrix_affine_scan_bwd without the saved forward output (the pages'
 * scans keep memory down by recomputing the forward in the backward).  The
 * call runs the forward over each lane's sequence keeping only h at the start
 * of every chunk of TS steps (TS = 8 for k = 8) in the workspace, then walks
 * the chunks downwards, recomputing each chunk's h from its checkpoint before
 * taking the adjoint back over it.  Reads A and b twice and grad_h once per
 * step (896 bytes per step at k = 8, against 608 with h saved).  Shapes with
 * few lanes and a long sequence (those where the saved-h backward splits T
 * into chunks, see mgs_workspace_size) instead run the time-chunked forward
 * into the workspace and the saved-h backward on it.
 * In: A, b (the forward's inputs), h0 (nullable: zero initial state), grad_h.
 * Out: dA, db, dh0 (nullable: not written), as mgs_matrix_affine_scan_bwd.
 * Workspace: mgs_workspace_size(MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE, B, T,
 * H, k) bytes (the checkpoints: 1/TS of the size of h, rounded up per group
 * of 32/k heads; for the few-lane shapes h itself and the chunked kernels'
 * workspace), disjoint from every other argument. */
mgs_status mgs_matrix_affine_scan_bwd_recompute(const float *A, const float *b, const float *h0,
                                                const float *grad_h, float *dA, float *db, float *dh0,
                                                int64_t B, int64_t T, int64_t H, int k, void *workspace,
                                                size_t workspace_bytes, mgs_stream_t stream);

/* matrix_scan, forward ("mingru-scans" home page, scan-op table, matrix_scan
 * row): prefix products
 *     P_t = A_t P_{t-1},   P_0 = I,   per (batch, head) lane.
 * In: A [B][T][H][k][k].  Out: P [B][T][H][k][k].
 * Long sequences with few lanes are split into time chunks whose aggregates
 * and carries go through the workspace (see mgs_workspace_size). */
mgs_status mgs_matrix_scan_fwd(const float *A, float *P, int64_t B, int64_t T, int64_t H, int k,
                               void *workspace, size_t workspace_bytes, mgs_stream_t stream);

/* Size of the device scratch array behind mgs_matrix_scan_fwd_noalloc. */
#define MGS_NOALLOC_SCRATCH_BYTES (4u << 20)

/* matrix_scan forward that allocates nothing and takes no workspace.
 * No counterpart on the mingru-scans pages: this entry point exists for callers
 * that hold only their input and output buffers and cannot call cudaMalloc,
 * for instance a host program whose device memory is owned by another
 * runtime's pool allocator (a raw cudaMalloc there fails or fragments the
 * pool), or a latency-bound loop that cannot afford the device-wide
 * synchronisation cudaMalloc/cudaFree imply.
 * Same operation, layouts and results as mgs_matrix_scan_fwd, without the
 * workspace arguments.  When the shape needs scratch (few lanes, long
 * sequence: see mgs_workspace_size with MGS_OP_MATRIX_SCAN_FWD), it uses a
 * file-scope device array of MGS_NOALLOC_SCRATCH_BYTES inside the library
 * instead; every GPU that loads the library holds that array until the
 * process exits.  Shapes needing more
 * scratch than that return MGS_ERR_WORKSPACE and do nothing.
 * The first call on each device looks up the array's device address with that
 * device current; make that first call before any stream capture.  The
 * address is cached per device context: if the context is destroyed and
 * created again (cudaDeviceReset), the next call looks it up again.
 * All calls on a device share the one array, which keeps the previous call's
 * contents; a call writes every part of it that it reads before reading it,
 * so nothing needs to start at zero.  Calls that overlap on the GPU, e.g. on
 * two unordered streams, race on the array: order them. */
mgs_status mgs_matrix_scan_fwd_noalloc(const float *A, float *P, int64_t B, int64_t T, int64_t H,
                                       int k, mgs_stream_t stream);

/* matrix_scan, backward: gradient of L = sum_t <grad_P_t, P_t>_F.  With
 * Lambda_t = dL/dP_t,
 *     Lambda_T = grad_P_T,   Lambda_t = grad_P_t + A_{t+1}^T Lambda_{t+1},
 *     dA_t = Lambda_t P_{t-1}^T   (P_0 = I).
 * In: A, P = the forward output (saved), grad_P.  Out: dA. */
mgs_status mgs_matrix_scan_bwd(const float *A, const float *P, const float *grad_P, float *dA,
                               int64_t B, int64_t T, int64_t H, int k, void *workspace,
                               size_t workspace_bytes, mgs_stream_t stream);

/* parallel_scan_log, forward ("mingru-scans" home page, scan-op table,
 * parallel_scan_log row; Heinsen's log-space scan behind MinGRU and
 * SignedMinGRU), per (batch, channel) lane:
 *     log h_t = log(exp(log_coeffs_t + log h_{t-1}) + exp(log_values_t)),
 *     log h_0 = log_h0 (NULL: h_0 = 0),   h_t = exp(log h_t),
 * i.e. h_t = exp(a*_t + logcumsumexp_{s<=t}(log_values_s - a*_s)) with
 * a*_t = sum_{s<=t} log_coeffs_s, evaluated as a max-shifted log-sum-exp
 * recurrence so no cumulative sum loses precision.  With T <= 32768 and
 * fewer than 2048 groups of 32 channels (B * ceil(D / 32)) the call is one
 * launch that is parallel over time (thread-block clusters), else one warp
 * walks each 128 channels' sequence.
 * In: log_coeffs, log_values [B][T][D], log_h0 [B][D] (nullable).
 * Out: h [B][T][D]; log_h [B][T][D] (nullable: not written). */
mgs_status mgs_parallel_scan_log_fwd(const float *log_coeffs, const float *log_values,
                                     const float *log_h0, float *h, float *log_h, int64_t B,
                                     int64_t T, int64_t D, void *workspace, size_t workspace_bytes,
                                     mgs_stream_t stream);

/* parallel_scan_log, backward: gradients of L = sum_t grad_h_t * h_t.  With
 * a_t = exp(log_coeffs_t) and lambda_t = dL/dh_t,
 *     lambda_T = grad_h_T,   lambda_t = grad_h_t + a_{t+1} lambda_{t+1},
 *     d_log_values_t = lambda_t exp(log_values_t),
 *     d_log_coeffs_t = lambda_t a_t h_{t-1},
 *     d_log_h0 = lambda_1 a_1 h_0.
 * In: log_coeffs, log_values, log_h0 (nullable: h_0 = 0), h = the forward
 *     output (nullable, see below), grad_h.
 * Out: d_log_coeffs, d_log_values [B][T][D]; d_log_h0 [B][D] (nullable; must
 *     be NULL when log_h0 is NULL).
 * With h saved, no workspace is needed.  With h == NULL the forward is
 * recomputed inside the call (the pages' log op recomputes its forward in
 * backward): one forward pass stores log2 h every 16 steps in the workspace,
 * then each 16-step segment's h is rebuilt from its checkpoint as the reverse
 * sweep reaches it.  That needs mgs_workspace_size(MGS_OP_PARALLEL_SCAN_LOG_BWD,
 * B, T, D, 0) = 4 * B * ceil(T / 16) * D bytes, 256-byte aligned (else
 * MGS_ERR_WORKSPACE), reads log_coeffs and log_values twice, and gives the
 * same results as passing the h this library's forward wrote.  On the
 * time-parallel path (the forward's condition above) h is recomputed in
 * registers instead (the gradients then equal the saved-h call's up to
 * rounding) and the workspace, still required at that size, is not
 * touched. */
mgs_status mgs_parallel_scan_log_bwd(const float *log_coeffs, const float *log_values,
                                     const float *log_h0, const float *h, const float *grad_h,
                                     float *d_log_coeffs, float *d_log_values, float *d_log_h0,
                                     int64_t B, int64_t T, int64_t D, void *workspace,
                                     size_t workspace_bytes, mgs_stream_t stream);

/* linear_scan, forward ("mingru-scans" home page, scan-op table, linear_scan
 * row): the diagonal linear recurrence in linear space, per (batch, channel)
 * lane,
 *     h_t = a_t * h_{t-1} + b_t,   h_0 = h0 (zeros when NULL),
 * with signed coefficients allowed (the negative-eigenvalue gates of
 * SignedMinGRU, home page lineage paragraph).  It is matrix_affine_scan with
 * k = 1 and H = D and validates as that op; T <= 1024 with fewer than 2048
 * groups of 32 channels (B * ceil(D / 32)) runs as one time-parallel launch
 * on thread-block clusters that uses no workspace, other shapes on the
 * matrix_affine_scan kernels.  The workspace size is that op's either way.
 * In: a, b [B][T][D], h0 [B][D] (nullable).  Out: h [B][T][D].  D must be a
 * multiple of 4.  Workspace: mgs_workspace_size(MGS_OP_LINEAR_SCAN_FWD, ...). */
mgs_status mgs_linear_scan_fwd(const float *a, const float *b, const float *h0, float *h, int64_t B,
                               int64_t T, int64_t D, void *workspace, size_t workspace_bytes,
                               mgs_stream_t stream);

/* linear_scan, backward: gradients of L = sum_t <grad_h_t, h_t>.  With
 * lambda_t = dL/dh_t,
 *     lambda_T = grad_h_T,   lambda_t = grad_h_t + a_{t+1} lambda_{t+1},
 *     db_t = lambda_t,   da_t = lambda_t h_{t-1},   dh0 = a_1 lambda_1.
 * In: a, h0 (nullable), h = the forward output (saved), grad_h.
 * Out: da, db [B][T][D], dh0 [B][D] (nullable: not written). */
mgs_status mgs_linear_scan_bwd(const float *a, const float *h0, const float *h, const float *grad_h,
                               float *da, float *db, float *dh0, int64_t B, int64_t T, int64_t D,
                               void *workspace, size_t workspace_bytes, mgs_stream_t stream);

/* Givens-mesh scans: matrix_affine_scan and matrix_scan whose k x k
 * transition is GivensMinGRU's brick-wall rotation mesh, given by its angles
 * ("mingru-scans" home page, lineage paragraph: the Clements et al. 2016 mesh
 * of Golub & Van Loan plane rotations; "Run the benchmarks", Step 3: the
 * angle-fused backward).  Only k = 8 is supported (else MGS_ERR_UNSUPPORTED);
 * N = k(k-1)/2 = 28 angles per (batch, step, head).
 *
 * G(theta) = L_k ... L_1: layer l = 1..k rotates the disjoint coordinate pairs
 * (0,1),(2,3),.. (odd l) or (1,2),(3,4),.. (even l), no wrap-around; the
 * angles are consumed layer by layer, pairs ascending, and the rotation of
 * angle th on (p, p+1) maps (x_p, x_{p+1}) to
 * (cos th x_p - sin th x_{p+1}, sin th x_p + cos th x_{p+1}).
 * Neither direction ever forms A_t or dA_t in memory.  With enough (batch,
 * head) lanes, or T < 256, no workspace is needed.  With few lanes and a long
 * sequence (when matrix_affine_scan would split T into chunks, and T >= 256)
 * the serial chain per lane would dominate, so T is split into chunks as in
 * the matrix scans' chunked paths, each chunk's aggregate built from the
 * angles: mgs_workspace_size(MGS_OP_GIVENS_*, B, T, H, 8) is then nonzero -
 * the per-chunk aggregates and carries only, the same bytes as
 * MGS_OP_MATRIX_AFFINE_SCAN_* (affine) or MGS_OP_MATRIX_SCAN_* (matrix) for
 * that shape - and a smaller or misaligned workspace gives
 * MGS_ERR_WORKSPACE.  Without the gate a (the orthogonal case) the call runs
 * the per-lane kernels in extended precision at every shape and leaves the
 * workspace unused.
 *
 * Affine forward:  h_t = G(theta_t) diag(a_t) h_{t-1} + b_t, h_0 = h0 (zeros
 * when NULL); a NULL means A_t = G(theta_t).
 * In: theta [B][T][H][28], a [B][T][H][8] (nullable), b [B][T][H][8],
 *     h0 [B][H][8] (nullable).  Out: h [B][T][H][8]. */
mgs_status mgs_givens_affine_scan_fwd(const float *theta, const float *a, const float *b,
                                      const float *h0, float *h, int64_t B, int64_t T, int64_t H,
                                      int k, void *workspace, size_t workspace_bytes,
                                      mgs_stream_t stream);

/* Affine backward: gradients of L = sum_t <grad_h_t, h_t> with respect to the
 * angles, a, b and h0.  With lambda_t = dL/dh_t (lambda_t = grad_h_t +
 * A_{t+1}^T lambda_{t+1}): db_t = lambda_t; d_theta_t[n] = <lambda_t h_{t-1}^T,
 * dA_t/dtheta_n>; da_t[j] = (G_t^T lambda_t)[j] h_{t-1}[j]; dh0 = A_1^T lambda_1.
 * In: theta, a (nullable, as in the forward), h0 (nullable), h = the forward
 *     output (saved), grad_h.  b is not needed.
 * Out: d_theta [B][T][H][28]; da [B][T][H][8] (nullable; must be NULL when a
 *     is NULL); db [B][T][H][8]; dh0 [B][H][8] (nullable). */
mgs_status mgs_givens_affine_scan_bwd(const float *theta, const float *a, const float *h0,
                                      const float *h, const float *grad_h, float *d_theta, float *da,
                                      float *db, float *dh0, int64_t B, int64_t T, int64_t H, int k,
                                      void *workspace, size_t workspace_bytes, mgs_stream_t stream);

/* Matrix forward: P_t = G(theta_t) P_{t-1}, P_0 = I.
 * In: theta [B][T][H][28].  Out: P [B][T][H][8][8]. */
mgs_status mgs_givens_matrix_scan_fwd(const float *theta, float *P, int64_t B, int64_t T, int64_t H,
                                      int k, void *workspace, size_t workspace_bytes,
                                      mgs_stream_t stream);

/* Matrix backward: gradient of L = sum_t <grad_P_t, P_t>_F with respect to the
 * angles, d_theta_t[n] = <Lambda_t P_{t-1}^T, dA_t/dtheta_n> with Lambda_t =
 * grad_P_t + A_{t+1}^T Lambda_{t+1}.
 * In: theta, P = the forward output (saved), grad_P [B][T][H][8][8].
 * Out: d_theta [B][T][H][28]. */
mgs_status mgs_givens_matrix_scan_bwd(const float *theta, const float *P, const float *grad_P,
                                      float *d_theta, int64_t B, int64_t T, int64_t H, int k,
                                      void *workspace, size_t workspace_bytes, mgs_stream_t stream);

/* Delta rule (DeltaNet), forward ("mingru-scans" home page, lineage
 * paragraph: DeltaMinGRU reimplements DeltaNet, Yang et al. 2024,
 * arXiv:2406.06484, whose chunked WY representation is its parallel forward),
 * per (batch, head) lane with a D x D state S (S[i][j], i the value index):
 *     S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T,   o_t = S_t q_t,
 * S_0 = S0 (zeros when NULL).  Computed chunk by chunk (64 steps) in the WY
 * form: for every chunk at once, W, U (the solve of
 * (I + strict_tril(diag(beta) K K^T)) against diag(beta) [K | V]) and
 * P = tril(Q K^T), folded into the chunk's affine map of the state,
 * S^T <- M S^T + N, O = R S^T + P U with M = I - K^T W, N = K^T U and
 * R = Q - P W; then the state carried through the chunks in order.  Only
 * D = 64 is supported (else MGS_ERR_UNSUPPORTED).
 * In: q, k, v [B][T][H][D]; beta [B][T][H] (4-byte aligned); S0 [B][H][D][D]
 *     (nullable).
 * Out: o [B][T][H][D]; S_T [B][H][D][D] (nullable: not written), the state
 *     after step T (S0, or zeros, when T = 0).
 * Workspace: mgs_workspace_size(MGS_OP_DELTA_SCAN_FWD, B, T, H, 64) bytes
 * (64 KiB per lane and 64-step chunk: R, M, (P U)^T and N^T of every chunk),
 * disjoint from every other argument, else MGS_ERR_INVALID_ARG. */
mgs_status mgs_delta_scan_fwd(const float *q, const float *k, const float *v, const float *beta,
                              const float *S0, float *o, float *S_T, int64_t B, int64_t T, int64_t H,
                              int D, void *workspace, size_t workspace_bytes, mgs_stream_t stream);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns MGS_ERR_TIMEOUT if a kernel's bounded wait gave up since the
 * last check, MGS_ERR_CUDA if the synchronisation failed, else MGS_OK. */
mgs_status mgs_check(mgs_stream_t stream);

/* Sets the limit, in nanoseconds, after which a device-side wait gives up
 * (default 1e9, i.e. one second).  Applies to launches made after the call on
 * any device.  Values below 1000 are raised to 1000. */
void mgs_set_wait_timeout_ns(uint64_t ns);

/* Diagnostic: launches one warp that waits, with the library's bounded wait,
 * on the device flag `*flag` (a device int) until it becomes nonzero.  When
 * nothing sets the flag, the wait gives up after the timeout and the error
 * word records it; mgs_check() then returns MGS_ERR_TIMEOUT.  Used to test
 * failure detection without faulting or hanging the GPU. */
mgs_status mgs_debug_wait_flag(const int *flag, mgs_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *mgs_status_string(mgs_status status);

/* Library version as an integer, major*10000 + minor*100 + patch. */
int mgs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MGSCAN_H */
