// C ABI of libmgscan (declared in include/mgscan.h): argument validation,
// the per-device error word, and dispatch to the kernel launchers.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <map>
#include <set>
#include <utility>

#include <cudaTypedefs.h>

#include "../../include/mgscan.h"
#include "mgs_launch.h"

#define MGS_VERSION_INT 100  // 0.1.0

namespace {

// Error word written by kernels whose bounded waits give up (one per device:
// a __device__ variable exists once in every device context that loads the
// library).  Host code never dereferences its name; it asks the runtime for
// the device address, once per device.
__device__ unsigned g_mgs_error_word = 0;

mgs::SymbolAddressCache g_err_cache;
std::atomic<uint64_t> g_timeout_ns{1000000000ull};

mgs_status current_ctl(mgs::DevCtl *ctl) {
    void *p = nullptr;
    if (mgs::cached_symbol_address(g_err_cache, (const void *)&g_mgs_error_word, &p) != cudaSuccess)
        return MGS_ERR_CUDA;
    ctl->err = static_cast<unsigned *>(p);
    ctl->timeout_ns = g_timeout_ns.load();
    return MGS_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// n = a*b*c*... with overflow detection (all factors >= 0).
bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    if (a == 0 || b == 0) { *out = 0; return true; }
    if (a > INT64_MAX / b) return false;
    *out = a * b;
    return true;
}

struct Range {
    uintptr_t lo, hi;
};
Range rng(const void *p, int64_t count) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + uintptr_t(count) * sizeof(float)};
}
bool overlap(Range x, Range y) { return x.lo < y.hi && y.lo < x.hi; }

// Every output must be disjoint from every input and from the other outputs.
bool disjoint(std::initializer_list<std::pair<const void *, int64_t>> outs,
              std::initializer_list<std::pair<const void *, int64_t>> ins) {
    for (auto o = outs.begin(); o != outs.end(); ++o) {
        if (o->first == nullptr || o->second == 0) continue;
        Range ro = rng(o->first, o->second);
        for (auto &i : ins)
            if (i.first != nullptr && i.second != 0 && overlap(ro, rng(i.first, i.second))) return false;
        for (auto o2 = o + 1; o2 != outs.end(); ++o2)
            if (o2->first != nullptr && o2->second != 0 && overlap(ro, rng(o2->first, o2->second)))
                return false;
    }
    return true;
}

bool k_supported(int k, int64_t H) {
    if (k == 4 || k == 8 || k == 16) return true;
    if (k == 1 || k == 2) return (H * k) % 4 == 0;
    return false;
}

struct BlockSizes {
    int64_t mat, vec, init;  // element counts: [B,T,H,k,k], [B,T,H,k], [B,H,k]
};

// Validates (B, T, H, k) for the matrix ops and computes element counts.
mgs_status block_sizes(int64_t B, int64_t T, int64_t H, int k, BlockSizes *s) {
    if (B < 0 || T < 0 || H < 0 || k <= 0) return MGS_ERR_INVALID_ARG;
    if (!k_supported(k, H)) return MGS_ERR_UNSUPPORTED;
    int64_t bth, bh;
    if (!mul_ok(B, T, &bth) || !mul_ok(bth, H, &bth) || !mul_ok(B, H, &bh)) return MGS_ERR_INVALID_ARG;
    if (!mul_ok(bth, int64_t(k) * k, &s->mat) || !mul_ok(bth, k, &s->vec) || !mul_ok(bh, k, &s->init))
        return MGS_ERR_INVALID_ARG;
    if (s->mat > (INT64_MAX / 8)) return MGS_ERR_INVALID_ARG;
    // tensor-map row coordinates are 32-bit
    if (B * T > INT32_MAX || H > INT32_MAX / 256) return MGS_ERR_UNSUPPORTED;
    return MGS_OK;
}

struct GivensSizes {
    int64_t ang, vec, mat, init;  // element counts: [B,T,H,N], [B,T,H,k], [B,T,H,k,k], [B,H,k]
};

// Validates (B, T, H, k) for the Givens-mesh ops (k = 8 only).
mgs_status givens_sizes(int64_t B, int64_t T, int64_t H, int k, GivensSizes *s) {
    if (B < 0 || T < 0 || H < 0 || k <= 0) return MGS_ERR_INVALID_ARG;
    if (k != 8) return MGS_ERR_UNSUPPORTED;
    int64_t bth, bh;
    if (!mul_ok(B, T, &bth) || !mul_ok(bth, H, &bth) || !mul_ok(B, H, &bh)) return MGS_ERR_INVALID_ARG;
    if (!mul_ok(bth, 64, &s->mat) || !mul_ok(bth, 28, &s->ang) || !mul_ok(bth, 8, &s->vec) ||
        !mul_ok(bh, 8, &s->init))
        return MGS_ERR_INVALID_ARG;
    if (s->mat > (INT64_MAX / 8)) return MGS_ERR_INVALID_ARG;
    if (B * T > INT32_MAX || H > INT32_MAX / 256) return MGS_ERR_UNSUPPORTED;  // 32-bit map coordinates
    return MGS_OK;
}

mgs_status check_ptrs(std::initializer_list<const void *> required,
                      std::initializer_list<const void *> optional) {
    for (const void *p : required)
        if (p == nullptr) return MGS_ERR_INVALID_ARG;
    for (const void *p : required)
        if (!aligned16(p)) return MGS_ERR_UNSUPPORTED;
    for (const void *p : optional)
        if (p != nullptr && !aligned16(p)) return MGS_ERR_UNSUPPORTED;
    return MGS_OK;
}

mgs_status check_ws(size_t need, const void *ws, size_t ws_bytes) {
    if (need == 0) return MGS_OK;
    if (ws == nullptr || ws_bytes < need) return MGS_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MGS_ERR_WORKSPACE;
    return MGS_OK;
}

mgs_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MGS_OK : MGS_ERR_CUDA; }

}  // namespace

namespace mgs {

cudaError_t make_tmap(CUtensorMap *map, const float *base, int rank, const uint64_t *dims,
                      const uint64_t *byte_strides, const uint32_t *box, bool swizzle128) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (encode == nullptr) return cudaErrorNotSupported;
    cuuint64_t gdim[3], gstr[2];
    cuuint32_t bdim[3], estr[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) gstr[i] = byte_strides[i];
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, cuuint32_t(rank), const_cast<float *>(base), gdim,
                        gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

uint64_t current_context_id() {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? uint64_t(id) : 0;
}

cudaError_t cached_symbol_address(SymbolAddressCache &cache, const void *symbol, void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= SymbolAddressCache::kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(cache.mu);
    const uint64_t ctx = current_context_id();
    if (ctx != 0 && cache.ctx[dev] == ctx && cache.addr[dev] != nullptr) {
        *out = cache.addr[dev];
        return cudaSuccess;
    }
    // the lookup also creates and binds the device's primary context when no
    // context is current yet, so the id is read again after it
    void *p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, symbol)) != cudaSuccess) return e;
    cache.ctx[dev] = current_context_id();
    cache.addr[dev] = p;
    *out = p;
    return cudaSuccess;
}

cudaError_t ensure_smem_attr(const void *fn, int bytes) {
    // the limit set for each kernel in each device context; raised (to the
    // opt-in maximum) when a launch needs more than the 48 KB default
    static std::mutex mu;
    static std::map<std::pair<const void *, uint64_t>, int> limit;
    const uint64_t ctx = current_context_id();
    const int want = bytes > 48 * 1024 ? 227 * 1024 : 48 * 1024;
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(fn, ctx);
    auto itr = limit.find(key);
    if (ctx != 0 && itr != limit.end() && itr->second >= want) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e == cudaSuccess && ctx != 0) limit[key] = want;
    return e;
}

}  // namespace mgs

extern "C" {

static mgs_status psl_sizes(int64_t B, int64_t T, int64_t D, int64_t *n, int64_t *n0);

size_t mgs_workspace_size(int op, int64_t B, int64_t T, int64_t H_or_D, int k) {
    BlockSizes s;
    switch (op) {
        case MGS_OP_MATRIX_AFFINE_SCAN_FWD:
        case MGS_OP_MATRIX_AFFINE_SCAN_BWD:
            if (block_sizes(B, T, H_or_D, k, &s) != MGS_OK) return 0;
            return mgs::mas_workspace_bytes(B, T, H_or_D, k);
        case MGS_OP_LINEAR_SCAN_FWD:
        case MGS_OP_LINEAR_SCAN_BWD:
            if (block_sizes(B, T, H_or_D, 1, &s) != MGS_OK) return 0;
            return mgs::mas_workspace_bytes(B, T, H_or_D, 1);
        case MGS_OP_MATRIX_AFFINE_SCAN_BWD_RECOMPUTE:
            if (block_sizes(B, T, H_or_D, k, &s) != MGS_OK || s.vec == 0) return 0;
            return mgs::mas_rc_workspace_bytes(B, T, H_or_D, k);
        case MGS_OP_MATRIX_SCAN_FWD:
        case MGS_OP_MATRIX_SCAN_BWD:
            if (block_sizes(B, T, H_or_D, k, &s) != MGS_OK) return 0;
            return mgs::ms_workspace_bytes(B, T, H_or_D, k, op == MGS_OP_MATRIX_SCAN_BWD);
        case MGS_OP_GIVENS_AFFINE_SCAN_FWD:
        case MGS_OP_GIVENS_AFFINE_SCAN_BWD:
        case MGS_OP_GIVENS_MATRIX_SCAN_FWD:
        case MGS_OP_GIVENS_MATRIX_SCAN_BWD: {
            GivensSizes gs;
            if (givens_sizes(B, T, H_or_D, k, &gs) != MGS_OK || gs.vec == 0) return 0;
            return mgs::givens_workspace_bytes(op - MGS_OP_GIVENS_AFFINE_SCAN_FWD, B, T, H_or_D);
        }
        case MGS_OP_DELTA_SCAN_FWD: {
            int64_t ns;
            if (B < 0 || T < 0 || H_or_D < 0 || k != 64 || !mul_ok(B, T, &ns) || !mul_ok(ns, H_or_D, &ns) ||
                !mul_ok(B, H_or_D, &ns) || !mul_ok(ns, (T + 63) / 64, &ns) || ns > INT64_MAX / (3 * 64 * 64 * 4))
                return 0;
            return mgs::delta_workspace_bytes(B, T, H_or_D);
        }
        case MGS_OP_PARALLEL_SCAN_LOG_BWD: {
            int64_t n, n0;
            if (psl_sizes(B, T, H_or_D, &n, &n0) != MGS_OK || n == 0) return 0;
            return mgs::psl_recompute_workspace_bytes(B, T, H_or_D);
        }
        default:
            return 0;
    }
}

mgs_status mgs_matrix_affine_scan_fwd(const float *A, const float *b, const float *h0, float *h,
                                      int64_t B, int64_t T, int64_t H, int k, void *workspace,
                                      size_t workspace_bytes, mgs_stream_t stream) {
    BlockSizes s;
    mgs_status st = block_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.vec == 0) return MGS_OK;
    if ((st = check_ptrs({A, b, h}, {h0})) != MGS_OK) return st;
    if (!disjoint({{h, s.vec}}, {{A, s.mat}, {b, s.vec}, {h0, h0 ? s.init : 0}})) return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(mgs::mas_workspace_bytes(B, T, H, k), workspace, workspace_bytes)) != MGS_OK) return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    if (k == 1 && mgs::lin_supported(B, T, H))
        return from_cuda(mgs::launch_lin_fwd(A, b, h0, h, B, T, H, reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(mgs::launch_mas_fwd(k, A, b, h0, h, B, T, H, workspace, workspace_bytes, ctl,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_matrix_affine_scan_bwd(const float *A, const float *h0, const float *h,
                                      const float *grad_h, float *dA, float *db, float *dh0,
                                      int64_t B, int64_t T, int64_t H, int k, void *workspace,
                                      size_t workspace_bytes, mgs_stream_t stream) {
    BlockSizes s;
    mgs_status st = block_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.init == 0) return MGS_OK;
    if (s.vec == 0) {
        // T == 0: lambda is empty, the initial-state gradient is zero
        if (dh0 == nullptr) return MGS_OK;
        if ((st = check_ptrs({dh0}, {})) != MGS_OK) return st;
        return from_cuda(cudaMemsetAsync(dh0, 0, size_t(s.init) * sizeof(float),
                                         reinterpret_cast<cudaStream_t>(stream)));
    }
    if ((st = check_ptrs({A, h, grad_h, dA, db}, {h0, dh0})) != MGS_OK) return st;
    if (!disjoint({{dA, s.mat}, {db, s.vec}, {dh0, dh0 ? s.init : 0}},
                  {{A, s.mat}, {h0, h0 ? s.init : 0}, {h, s.vec}, {grad_h, s.vec}}))
        return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(mgs::mas_workspace_bytes(B, T, H, k), workspace, workspace_bytes)) != MGS_OK) return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    if (k == 1 && mgs::lin_supported(B, T, H))
        return from_cuda(mgs::launch_lin_bwd(A, h0, h, grad_h, dA, db, dh0, B, T, H,
                                             reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(mgs::launch_mas_bwd(k, A, h0, h, grad_h, dA, db, dh0, B, T, H, workspace, workspace_bytes,
                                         ctl, reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_matrix_affine_scan_bwd_recompute(const float *A, const float *b, const float *h0,
                                                const float *grad_h, float *dA, float *db, float *dh0,
                                                int64_t B, int64_t T, int64_t H, int k, void *workspace,
                                                size_t workspace_bytes, mgs_stream_t stream) {
    BlockSizes s;
    mgs_status st = block_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.init == 0) return MGS_OK;
    if (s.vec == 0) {
        // T == 0: lambda is empty, the initial-state gradient is zero
        if (dh0 == nullptr) return MGS_OK;
        if ((st = check_ptrs({dh0}, {})) != MGS_OK) return st;
        return from_cuda(cudaMemsetAsync(dh0, 0, size_t(s.init) * sizeof(float),
                                         reinterpret_cast<cudaStream_t>(stream)));
    }
    if ((st = check_ptrs({A, b, grad_h, dA, db}, {h0, dh0})) != MGS_OK) return st;
    if (!disjoint({{dA, s.mat}, {db, s.vec}, {dh0, dh0 ? s.init : 0}},
                  {{A, s.mat}, {b, s.vec}, {h0, h0 ? s.init : 0}, {grad_h, s.vec}}))
        return MGS_ERR_INVALID_ARG;
    const size_t need = mgs::mas_rc_workspace_bytes(B, T, H, k);
    if ((st = check_ws(need, workspace, workspace_bytes)) != MGS_OK) return st;
    if (!disjoint({{static_cast<float *>(workspace), int64_t(need / sizeof(float))}},
                  {{A, s.mat}, {b, s.vec}, {h0, h0 ? s.init : 0}, {grad_h, s.vec}, {dA, s.mat}, {db, s.vec},
                   {dh0, dh0 ? s.init : 0}}))
        return MGS_ERR_INVALID_ARG;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_mas_bwd_recompute(k, A, b, h0, grad_h, dA, db, dh0, B, T, H, workspace, ctl,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_matrix_scan_fwd(const float *A, float *P, int64_t B, int64_t T, int64_t H, int k,
                               void *workspace, size_t workspace_bytes, mgs_stream_t stream) {
    BlockSizes s;
    mgs_status st = block_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.mat == 0) return MGS_OK;
    if ((st = check_ptrs({A, P}, {})) != MGS_OK) return st;
    if (!disjoint({{P, s.mat}}, {{A, s.mat}})) return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(mgs::ms_workspace_bytes(B, T, H, k, false), workspace, workspace_bytes)) != MGS_OK)
        return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_ms_fwd(k, A, P, B, T, H, workspace, workspace_bytes, ctl,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_matrix_scan_fwd_noalloc(const float *A, float *P, int64_t B, int64_t T, int64_t H,
                                       int k, mgs_stream_t stream) {
    BlockSizes s;
    mgs_status st = block_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.mat == 0) return MGS_OK;
    if ((st = check_ptrs({A, P}, {})) != MGS_OK) return st;
    if (!disjoint({{P, s.mat}}, {{A, s.mat}})) return MGS_ERR_INVALID_ARG;
    if (mgs::ms_workspace_bytes(B, T, H, k, false) > mgs::ms_static_scratch_bytes()) return MGS_ERR_WORKSPACE;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_ms_fwd_static_scratch(k, A, P, B, T, H, ctl,
                                                       reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_matrix_scan_bwd(const float *A, const float *P, const float *grad_P, float *dA,
                               int64_t B, int64_t T, int64_t H, int k, void *workspace,
                               size_t workspace_bytes, mgs_stream_t stream) {
    BlockSizes s;
    mgs_status st = block_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.mat == 0) return MGS_OK;
    if ((st = check_ptrs({A, P, grad_P, dA}, {})) != MGS_OK) return st;
    if (!disjoint({{dA, s.mat}}, {{A, s.mat}, {P, s.mat}, {grad_P, s.mat}})) return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(mgs::ms_workspace_bytes(B, T, H, k, true), workspace, workspace_bytes)) != MGS_OK)
        return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_ms_bwd(k, A, P, grad_P, dA, B, T, H, workspace, workspace_bytes, ctl,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

static mgs_status psl_sizes(int64_t B, int64_t T, int64_t D, int64_t *n, int64_t *n0) {
    if (B < 0 || T < 0 || D < 0) return MGS_ERR_INVALID_ARG;
    if (D % 4 != 0) return MGS_ERR_UNSUPPORTED;
    int64_t bt;
    if (!mul_ok(B, T, &bt) || !mul_ok(bt, D, n) || !mul_ok(B, D, n0)) return MGS_ERR_INVALID_ARG;
    if (*n > INT64_MAX / 8) return MGS_ERR_INVALID_ARG;
    if (B * T > INT32_MAX || D > INT32_MAX) return MGS_ERR_UNSUPPORTED;  // 32-bit map coordinates
    return MGS_OK;
}

mgs_status mgs_parallel_scan_log_fwd(const float *log_coeffs, const float *log_values,
                                     const float *log_h0, float *h, float *log_h, int64_t B,
                                     int64_t T, int64_t D, void *workspace, size_t workspace_bytes,
                                     mgs_stream_t stream) {
    int64_t n, n0;
    mgs_status st = psl_sizes(B, T, D, &n, &n0);
    if (st != MGS_OK) return st;
    if (n == 0) return MGS_OK;
    if ((st = check_ptrs({log_coeffs, log_values, h}, {log_h0, log_h})) != MGS_OK) return st;
    if (!disjoint({{h, n}, {log_h, log_h ? n : 0}},
                  {{log_coeffs, n}, {log_values, n}, {log_h0, log_h0 ? n0 : 0}}))
        return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(0, workspace, workspace_bytes)) != MGS_OK) return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    if (mgs::psl_cl_supported(B, T, D))
        return from_cuda(mgs::launch_psl_fwd_cl(log_coeffs, log_values, log_h0, h, log_h, B, T, D,
                                                reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(mgs::launch_psl_fwd(log_coeffs, log_values, log_h0, h, log_h, B, T, D, ctl,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_parallel_scan_log_bwd(const float *log_coeffs, const float *log_values,
                                     const float *log_h0, const float *h, const float *grad_h,
                                     float *d_log_coeffs, float *d_log_values, float *d_log_h0,
                                     int64_t B, int64_t T, int64_t D, void *workspace,
                                     size_t workspace_bytes, mgs_stream_t stream) {
    int64_t n, n0;
    mgs_status st = psl_sizes(B, T, D, &n, &n0);
    if (st != MGS_OK) return st;
    if (d_log_h0 != nullptr && log_h0 == nullptr) return MGS_ERR_INVALID_ARG;
    if (n0 == 0) return MGS_OK;
    if (n == 0) {
        if (d_log_h0 == nullptr) return MGS_OK;
        if ((st = check_ptrs({d_log_h0}, {})) != MGS_OK) return st;
        return from_cuda(cudaMemsetAsync(d_log_h0, 0, size_t(n0) * sizeof(float),
                                         reinterpret_cast<cudaStream_t>(stream)));
    }
    if ((st = check_ptrs({log_coeffs, log_values, grad_h, d_log_coeffs, d_log_values},
                         {log_h0, h, d_log_h0})) != MGS_OK)
        return st;
    if (!disjoint({{d_log_coeffs, n}, {d_log_values, n}, {d_log_h0, d_log_h0 ? n0 : 0}},
                  {{log_coeffs, n}, {log_values, n}, {log_h0, log_h0 ? n0 : 0}, {h, h ? n : 0},
                   {grad_h, n}}))
        return MGS_ERR_INVALID_ARG;
    const size_t need = (h == nullptr) ? mgs::psl_recompute_workspace_bytes(B, T, D) : 0;
    if ((st = check_ws(need, workspace, workspace_bytes)) != MGS_OK) return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    if (h == nullptr && mgs::psl_cl_supported(B, T, D))
        return from_cuda(mgs::launch_psl_bwd_rc_cl(log_coeffs, log_values, log_h0, grad_h, d_log_coeffs,
                                                   d_log_values, d_log_h0, B, T, D,
                                                   reinterpret_cast<cudaStream_t>(stream)));
    if (h == nullptr)
        return from_cuda(mgs::launch_psl_bwd_recompute(log_coeffs, log_values, log_h0, grad_h, d_log_coeffs,
                                                       d_log_values, d_log_h0, workspace, B, T, D, ctl,
                                                       reinterpret_cast<cudaStream_t>(stream)));
    if (mgs::psl_cl_supported(B, T, D))
        return from_cuda(mgs::launch_psl_bwd_cl(log_coeffs, log_values, log_h0, h, grad_h, d_log_coeffs,
                                                d_log_values, d_log_h0, B, T, D,
                                                reinterpret_cast<cudaStream_t>(stream)));
    return from_cuda(mgs::launch_psl_bwd(log_coeffs, log_values, log_h0, h, grad_h, d_log_coeffs,
                                         d_log_values, d_log_h0, B, T, D, ctl,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

// linear_scan is matrix_affine_scan with 1 x 1 blocks: [B][T][D] is
// [B][T][H=D][1][1], so it validates and runs exactly as that op with k = 1.
mgs_status mgs_linear_scan_fwd(const float *a, const float *b, const float *h0, float *h, int64_t B,
                               int64_t T, int64_t D, void *workspace, size_t workspace_bytes,
                               mgs_stream_t stream) {
    if (D >= 0 && D % 4 != 0) return MGS_ERR_UNSUPPORTED;
    return mgs_matrix_affine_scan_fwd(a, b, h0, h, B, T, D, 1, workspace, workspace_bytes, stream);
}

mgs_status mgs_linear_scan_bwd(const float *a, const float *h0, const float *h, const float *grad_h,
                               float *da, float *db, float *dh0, int64_t B, int64_t T, int64_t D,
                               void *workspace, size_t workspace_bytes, mgs_stream_t stream) {
    if (D >= 0 && D % 4 != 0) return MGS_ERR_UNSUPPORTED;
    return mgs_matrix_affine_scan_bwd(a, h0, h, grad_h, da, db, dh0, B, T, D, 1, workspace, workspace_bytes,
                                      stream);
}

mgs_status mgs_givens_affine_scan_fwd(const float *theta, const float *a, const float *b,
                                      const float *h0, float *h, int64_t B, int64_t T, int64_t H,
                                      int k, void *workspace, size_t workspace_bytes,
                                      mgs_stream_t stream) {
    GivensSizes s;
    mgs_status st = givens_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.vec == 0) return MGS_OK;
    if ((st = check_ptrs({theta, b, h}, {a, h0})) != MGS_OK) return st;
    if (!disjoint({{h, s.vec}}, {{theta, s.ang}, {a, a ? s.vec : 0}, {b, s.vec}, {h0, h0 ? s.init : 0}}))
        return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(mgs::givens_workspace_bytes(0, B, T, H), workspace, workspace_bytes)) != MGS_OK) return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_gas_fwd(theta, a, b, h0, h, B, T, H, workspace, workspace_bytes, ctl,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_givens_affine_scan_bwd(const float *theta, const float *a, const float *h0,
                                      const float *h, const float *grad_h, float *d_theta, float *da,
                                      float *db, float *dh0, int64_t B, int64_t T, int64_t H, int k,
                                      void *workspace, size_t workspace_bytes, mgs_stream_t stream) {
    GivensSizes s;
    mgs_status st = givens_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (da != nullptr && a == nullptr) return MGS_ERR_INVALID_ARG;
    if (s.init == 0) return MGS_OK;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (s.vec == 0) {  // T = 0: dh0 = 0
        if (dh0 == nullptr) return MGS_OK;
        if ((st = check_ptrs({dh0}, {})) != MGS_OK) return st;
        return from_cuda(cudaMemsetAsync(dh0, 0, size_t(s.init) * sizeof(float), cs));
    }
    if ((st = check_ptrs({theta, h, grad_h, d_theta, db}, {a, h0, da, dh0})) != MGS_OK) return st;
    if (!disjoint({{d_theta, s.ang}, {da, da ? s.vec : 0}, {db, s.vec}, {dh0, dh0 ? s.init : 0}},
                  {{theta, s.ang}, {a, a ? s.vec : 0}, {h0, h0 ? s.init : 0}, {h, s.vec}, {grad_h, s.vec}}))
        return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(mgs::givens_workspace_bytes(1, B, T, H), workspace, workspace_bytes)) != MGS_OK) return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_gas_bwd(theta, a, h0, h, grad_h, d_theta, da, db, dh0, B, T, H, workspace,
                                         workspace_bytes, ctl, cs));
}

mgs_status mgs_givens_matrix_scan_fwd(const float *theta, float *P, int64_t B, int64_t T, int64_t H,
                                      int k, void *workspace, size_t workspace_bytes,
                                      mgs_stream_t stream) {
    GivensSizes s;
    mgs_status st = givens_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.mat == 0) return MGS_OK;
    if ((st = check_ptrs({theta, P}, {})) != MGS_OK) return st;
    if (!disjoint({{P, s.mat}}, {{theta, s.ang}})) return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(mgs::givens_workspace_bytes(2, B, T, H), workspace, workspace_bytes)) != MGS_OK) return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_gms_fwd(theta, P, B, T, H, workspace, workspace_bytes, ctl,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_givens_matrix_scan_bwd(const float *theta, const float *P, const float *grad_P,
                                      float *d_theta, int64_t B, int64_t T, int64_t H, int k,
                                      void *workspace, size_t workspace_bytes, mgs_stream_t stream) {
    GivensSizes s;
    mgs_status st = givens_sizes(B, T, H, k, &s);
    if (st != MGS_OK) return st;
    if (s.mat == 0) return MGS_OK;
    if ((st = check_ptrs({theta, P, grad_P, d_theta}, {})) != MGS_OK) return st;
    if (!disjoint({{d_theta, s.ang}}, {{theta, s.ang}, {P, s.mat}, {grad_P, s.mat}})) return MGS_ERR_INVALID_ARG;
    if ((st = check_ws(mgs::givens_workspace_bytes(3, B, T, H), workspace, workspace_bytes)) != MGS_OK) return st;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_gms_bwd(theta, P, grad_P, d_theta, B, T, H, workspace, workspace_bytes, ctl,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

mgs_status mgs_delta_scan_fwd(const float *q, const float *k, const float *v, const float *beta,
                              const float *S0, float *o, float *S_T, int64_t B, int64_t T, int64_t H,
                              int D, void *workspace, size_t workspace_bytes, mgs_stream_t stream) {
    if (B < 0 || T < 0 || H < 0 || D <= 0) return MGS_ERR_INVALID_ARG;
    if (D != 64) return MGS_ERR_UNSUPPORTED;
    int64_t nb, n, ns;
    if (!mul_ok(B, T, &nb) || !mul_ok(nb, H, &nb) || !mul_ok(nb, D, &n) || !mul_ok(B, H, &ns) ||
        !mul_ok(ns, int64_t(D) * D, &ns))
        return MGS_ERR_INVALID_ARG;
    if (n > INT64_MAX / 8 || ns > INT64_MAX / 8) return MGS_ERR_INVALID_ARG;
    if (B * T > INT32_MAX || H > INT32_MAX) return MGS_ERR_UNSUPPORTED;  // 32-bit map coordinates
    if (ns == 0) return MGS_OK;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    mgs_status st;
    if (n == 0) {  // T = 0: the final state is the initial one
        if (S_T == nullptr) return MGS_OK;
        if ((st = check_ptrs({S_T}, {S0})) != MGS_OK) return st;
        if (!disjoint({{S_T, ns}}, {{S0, S0 ? ns : 0}})) return MGS_ERR_INVALID_ARG;
        return from_cuda(S0 ? cudaMemcpyAsync(S_T, S0, size_t(ns) * sizeof(float), cudaMemcpyDeviceToDevice, cs)
                            : cudaMemsetAsync(S_T, 0, size_t(ns) * sizeof(float), cs));
    }
    if ((st = check_ptrs({q, k, v, o}, {S0, S_T})) != MGS_OK) return st;
    if (beta == nullptr) return MGS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(beta) & 3u) != 0) return MGS_ERR_UNSUPPORTED;
    if (!disjoint({{o, n}, {S_T, S_T ? ns : 0}},
                  {{q, n}, {k, n}, {v, n}, {beta, nb}, {S0, S0 ? ns : 0}}))
        return MGS_ERR_INVALID_ARG;
    int64_t chunks;
    if (!mul_ok(B * H, (T + 63) / 64, &chunks) || chunks > INT32_MAX / (3 * 64)) return MGS_ERR_UNSUPPORTED;
    const size_t need = mgs::delta_workspace_bytes(B, T, H);
    if ((st = check_ws(need, workspace, workspace_bytes)) != MGS_OK) return st;
    if (!disjoint({{static_cast<float *>(workspace), int64_t(need / sizeof(float))}},
                  {{q, n}, {k, n}, {v, n}, {beta, nb}, {S0, S0 ? ns : 0}, {o, n}, {S_T, S_T ? ns : 0}}))
        return MGS_ERR_INVALID_ARG;
    mgs::DevCtl ctl;
    if ((st = current_ctl(&ctl)) != MGS_OK) return st;
    return from_cuda(mgs::launch_delta_fwd(q, k, v, beta, S0, o, S_T, B, T, H, workspace, ctl, cs));
}

mgs_status mgs_check(mgs_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MGS_ERR_CUDA;
    mgs::DevCtl ctl;
    mgs_status st = current_ctl(&ctl);
    if (st != MGS_OK) return st;
    unsigned word = 0;
    if (cudaMemcpy(&word, ctl.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MGS_ERR_CUDA;
    if (word != 0) {
        if (cudaMemset(ctl.err, 0, sizeof(unsigned)) != cudaSuccess) return MGS_ERR_CUDA;
        return MGS_ERR_TIMEOUT;
    }
    return MGS_OK;
}

void mgs_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns < 1000 ? 1000 : ns); }

const char *mgs_status_string(mgs_status status) {
    switch (status) {
        case MGS_OK: return "MGS_OK";
        case MGS_ERR_INVALID_ARG: return "MGS_ERR_INVALID_ARG";
        case MGS_ERR_UNSUPPORTED: return "MGS_ERR_UNSUPPORTED";
        case MGS_ERR_WORKSPACE: return "MGS_ERR_WORKSPACE";
        case MGS_ERR_CUDA: return "MGS_ERR_CUDA";
        case MGS_ERR_TIMEOUT: return "MGS_ERR_TIMEOUT";
        default: return "MGS_ERR_UNKNOWN";
    }
}

int mgs_version(void) { return MGS_VERSION_INT; }

}  // extern "C"

// ---------------------------------------------------------------- diagnostic wait
namespace {
__global__ void debug_wait_flag_kernel(const int *flag, mgs::DevCtl ctl) {
    if (threadIdx.x != 0) return;
    const uint64_t t0 = mgs::global_ns();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v != 0) return;
        if (mgs::global_ns() - t0 > ctl.timeout_ns) {
            mgs::record_error(ctl, mgs::ERR_FLAG_TIMEOUT);
            return;
        }
        __nanosleep(1000);
    }
}
}  // namespace

extern "C" mgs_status mgs_debug_wait_flag(const int *flag, mgs_stream_t stream) {
    if (flag == nullptr) return MGS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(flag) & 3u) != 0) return MGS_ERR_UNSUPPORTED;
    mgs::DevCtl ctl;
    mgs_status st = current_ctl(&ctl);
    if (st != MGS_OK) return st;
    debug_wait_flag_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(flag, ctl);
    return from_cuda(cudaGetLastError());
}
