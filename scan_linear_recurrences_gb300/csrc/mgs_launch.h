// Internal launcher interface between the C ABI (mgs_api.cu) and the kernel
// translation units.  Not installed; the public interface is include/mgscan.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "mgs_device.cuh"

namespace mgs {

// matrix_affine_scan
size_t mas_workspace_bytes(int64_t B, int64_t T, int64_t H, int K);
cudaError_t launch_mas_fwd(int K, const float *A, const float *b, const float *h0, float *h,
                           int64_t B, int64_t T, int64_t H, void *ws, size_t ws_bytes,
                           const DevCtl &ctl, cudaStream_t s);
cudaError_t launch_mas_bwd(int K, const float *A, const float *h0, const float *h,
                           const float *gh, float *dA, float *db, float *dh0, int64_t B,
                           int64_t T, int64_t H, void *ws, size_t ws_bytes, const DevCtl &ctl,
                           cudaStream_t s);
// recompute-mode backward (h not saved): checkpoints in the workspace
size_t mas_rc_workspace_bytes(int64_t B, int64_t T, int64_t H, int K);
cudaError_t launch_mas_bwd_recompute(int K, const float *A, const float *b, const float *h0, const float *gh,
                                     float *dA, float *db, float *dh0, int64_t B, int64_t T, int64_t H, void *ws,
                                     const DevCtl &ctl, cudaStream_t s);

// linear_scan (matrix_affine_scan with k = 1), time-parallel in one launch
// for few channel groups and T <= 1024; no workspace.  h0 and dh0 may be null.
bool lin_supported(int64_t B, int64_t T, int64_t D);
// the same for parallel_scan_log, T <= 32768
bool psl_cl_supported(int64_t B, int64_t T, int64_t D);
cudaError_t launch_lin_fwd(const float *a, const float *b, const float *h0, float *h, int64_t B, int64_t T,
                           int64_t D, cudaStream_t s);
cudaError_t launch_lin_bwd(const float *a, const float *h0, const float *h, const float *g, float *da, float *db,
                           float *dh0, int64_t B, int64_t T, int64_t D, cudaStream_t s);

// parallel_scan_log with the saved-h backward on the same time-parallel
// kernels (psl_cl_supported decides, D as the channel count); no workspace.
cudaError_t launch_psl_fwd_cl(const float *lc, const float *lv, const float *lh0, float *h, float *logh, int64_t B,
                              int64_t T, int64_t D, cudaStream_t s);
cudaError_t launch_psl_bwd_cl(const float *lc, const float *lv, const float *lh0, const float *h, const float *g,
                              float *dlc, float *dlv, float *dlh0, int64_t B, int64_t T, int64_t D, cudaStream_t s);
// ... and its backward recomputing the forward in registers (h not saved)
cudaError_t launch_psl_bwd_rc_cl(const float *lc, const float *lv, const float *lh0, const float *g, float *dlc,
                                 float *dlv, float *dlh0, int64_t B, int64_t T, int64_t D, cudaStream_t s);

// matrix_scan
size_t ms_workspace_bytes(int64_t B, int64_t T, int64_t H, int K, bool bwd);
cudaError_t launch_ms_fwd(int K, const float *A, float *P, int64_t B, int64_t T, int64_t H,
                          void *ws, size_t ws_bytes, const DevCtl &ctl, cudaStream_t s);
// matrix_scan forward with the library's own static device scratch (see
// mgs_matrix_scan_fwd_noalloc); returns cudaErrorInvalidValue if the shape
// needs more scratch than the array holds.
cudaError_t launch_ms_fwd_static_scratch(int K, const float *A, float *P, int64_t B, int64_t T,
                                         int64_t H, const DevCtl &ctl, cudaStream_t s);
size_t ms_static_scratch_bytes();
cudaError_t launch_ms_bwd(int K, const float *A, const float *P, const float *G, float *dA,
                          int64_t B, int64_t T, int64_t H, void *ws, size_t ws_bytes,
                          const DevCtl &ctl, cudaStream_t s);

// parallel_scan_log
cudaError_t launch_psl_fwd(const float *lc, const float *lv, const float *lh0, float *h,
                           float *logh, int64_t B, int64_t T, int64_t D, const DevCtl &ctl,
                           cudaStream_t s);
size_t psl_recompute_workspace_bytes(int64_t B, int64_t T, int64_t D);
cudaError_t launch_psl_bwd_recompute(const float *lc, const float *lv, const float *lh0, const float *gh,
                                     float *dlc, float *dlv, float *dlh0, void *ws, int64_t B, int64_t T,
                                     int64_t D, const DevCtl &ctl, cudaStream_t s);
cudaError_t launch_psl_bwd(const float *lc, const float *lv, const float *lh0, const float *h,
                           const float *gh, float *dlc, float *dlv, float *dlh0, int64_t B,
                           int64_t T, int64_t D, const DevCtl &ctl, cudaStream_t s);

// Givens-mesh affine and matrix scans (k = 8).  op: 0 affine fwd, 1 affine
// bwd, 2 matrix fwd, 3 matrix bwd; nonzero only for few lanes and long T.
size_t givens_workspace_bytes(int op, int64_t B, int64_t T, int64_t H);
cudaError_t launch_gas_fwd(const float *theta, const float *a, const float *b, const float *h0, float *h,
                           int64_t B, int64_t T, int64_t H, void *ws, size_t ws_bytes, const DevCtl &ctl,
                           cudaStream_t s);
cudaError_t launch_gas_bwd(const float *theta, const float *a, const float *h0, const float *h, const float *gh,
                           float *dth, float *da, float *db, float *dh0, int64_t B, int64_t T, int64_t H,
                           void *ws, size_t ws_bytes, const DevCtl &ctl, cudaStream_t s);
cudaError_t launch_gms_fwd(const float *theta, float *P, int64_t B, int64_t T, int64_t H, void *ws,
                           size_t ws_bytes, const DevCtl &ctl, cudaStream_t s);
cudaError_t launch_gms_bwd(const float *theta, const float *P, const float *G, float *dth, int64_t B, int64_t T,
                           int64_t H, void *ws, size_t ws_bytes, const DevCtl &ctl, cudaStream_t s);

// delta rule forward (head dimension 64); the workspace holds W, U and P of
// every 64-step chunk
size_t delta_workspace_bytes(int64_t B, int64_t T, int64_t H);
cudaError_t launch_delta_fwd(const float *q, const float *k, const float *v, const float *beta, const float *S0,
                             float *o, float *ST, int64_t B, int64_t T, int64_t H, void *ws, const DevCtl &ctl,
                             cudaStream_t s);

// Encodes a tiled fp32 tensor map over `base` (rank 2 or 3).  dims and box are
// innermost first; byte_strides has rank-1 entries (strides of dims 1..).
cudaError_t make_tmap(CUtensorMap *map, const float *base, int rank, const uint64_t *dims,
                      const uint64_t *byte_strides, const uint32_t *box, bool swizzle128 = false);

// Sets the dynamic shared-memory limit of `fn` once per device context.
cudaError_t ensure_smem_attr(const void *fn, int bytes);

// Unique id of the CUDA context current on the calling thread, 0 when none is
// current (or the driver does not report one).
uint64_t current_context_id();

// Device address of a file-scope __device__ variable, looked up with
// cudaGetSymbolAddress once per device context and cached.  A device's
// context can be torn down and created again (cudaDeviceReset), after which
// the variable lives at a new address; the cache is keyed on the context id,
// so a new context gets a fresh lookup rather than a stale address.
struct SymbolAddressCache {
    static constexpr int kMaxDevices = 64;
    std::mutex mu;
    uint64_t ctx[kMaxDevices] = {};
    void *addr[kMaxDevices] = {};
};
cudaError_t cached_symbol_address(SymbolAddressCache &cache, const void *symbol, void **out);

}  // namespace mgs
