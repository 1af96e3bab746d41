// C-ABI entry points of libqgemm: argument validation (host, before any
// launch), dispatch to the kernels, and per-thread error messages.
#include <cuda.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "qg_internal.h"

namespace qg {

namespace {
thread_local char g_err[512] = {0};
}

void set_error(const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

qg_status fail(qg_status st, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

qg_status cuda_fail(cudaError_t e, const char* what)
{
    set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
    return QG_ERR_CUDA;
}

// Per-device attribute caches (any thread may call; the values written are
// the same whoever writes them, and the atomics make the reads well defined).
namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_smem_per_sm[kMaxDevices];
std::atomic<int> g_smem_reserved[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];
}  // namespace

// Dynamic shared memory per CTA that lets at most `cap` CTAs share an SM.
int smem_for_cap(int cap)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
    int per_sm = g_smem_per_sm[dev].load(std::memory_order_acquire);
    int reserved = g_smem_reserved[dev].load(std::memory_order_relaxed);
    if (!per_sm) {
        if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            per_sm <= 0)
            per_sm = 233472;
        if (cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
            reserved < 0)
            reserved = 1024;
        g_smem_reserved[dev].store(reserved, std::memory_order_relaxed);
        g_smem_per_sm[dev].store(per_sm, std::memory_order_release);
    }
    return per_sm / (cap + 1) - reserved + 16;   // (cap + 1) CTAs no longer fit, cap still do
}

int num_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached) {
        const int v = g_sm_count[dev].load(std::memory_order_relaxed);
        if (v) return v;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    if (cached) g_sm_count[dev].store(v, std::memory_order_relaxed);
    return v;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t nnz_of(int64_t N, int64_t K, float frac)
{
    if (frac <= 0.0f) return 0;
    return (int64_t)std::floor((double)frac * (double)N * (double)K);
}

qg_status check_shape(int64_t N, int64_t K, int bits, int group)
{
    if (N <= 0 || K <= 0) return fail(QG_ERR_INVALID_ARG, "N and K must be positive (N=%lld K=%lld)", (long long)N, (long long)K);
    if ((bits < 2 || bits > 6) && bits != 8) return fail(QG_ERR_UNSUPPORTED, "bits must be 2..6 or 8 (got %d)", bits);
    if (group != 32 && group != 64 && group != 128)
        return fail(QG_ERR_UNSUPPORTED, "group must be 32, 64 or 128 (got %d)", group);
    if (K % group) return fail(QG_ERR_INVALID_ARG, "K=%lld is not a multiple of group=%d", (long long)K, group);
    if ((int64_t)N * K > (int64_t)1 << 34) return fail(QG_ERR_INVALID_ARG, "N*K too large");
    return QG_OK;
}

// Validate a weight descriptor for use by a product kernel or as the output
// of a quantizer.
qg_status check_qweight(const qg_qweight* w, const char* who)
{
    if (!w) return fail(QG_ERR_INVALID_ARG, "%s: null weight descriptor", who);
    qg_status st = check_shape(w->N, w->K, w->bits, w->group);
    if (st != QG_OK) return st;
    if (!w->packed) return fail(QG_ERR_INVALID_ARG, "%s: packed is null", who);
    if (!aligned(w->packed, 16)) return fail(QG_ERR_ALIGNMENT, "%s: packed must be 16-byte aligned", who);
    if (w->bits == 2) {
        if (w->scale8) return fail(QG_ERR_INVALID_ARG, "%s: 8-bit scales need bits 3..8 (2 bits use codebooks)", who);
        if (!w->codebook) return fail(QG_ERR_INVALID_ARG, "%s: codebook is null for bits=2", who);
        if (!aligned(w->codebook, 8)) return fail(QG_ERR_ALIGNMENT, "%s: codebook must be 8-byte aligned", who);
    } else if (w->scale8) {
        // 8-bit scales with the fp16 fallback list (scale unused)
        if (!w->zp || !w->scale8_exp || !w->fb_row_ptr)
            return fail(QG_ERR_INVALID_ARG, "%s: zp, scale8_exp or fb_row_ptr null with 8-bit scales", who);
        if (w->fb_cap < 0) return fail(QG_ERR_INVALID_ARG, "%s: fb_cap < 0", who);
        if (w->fb_cap > 0 && (!w->fb_col || !w->fb_val))
            return fail(QG_ERR_INVALID_ARG, "%s: fallback arrays null with fb_cap=%d", who, w->fb_cap);
        if (!aligned(w->scale8_exp, 4) || !aligned(w->fb_row_ptr, 4) || !aligned(w->fb_col, 4) ||
            !aligned(w->fb_val, 2))
            return fail(QG_ERR_ALIGNMENT, "%s: scale8_exp or fallback arrays misaligned", who);
    } else {
        if (!w->scale || !w->zp) return fail(QG_ERR_INVALID_ARG, "%s: scale/zp null for bits=%d", who, w->bits);
        if (!aligned(w->scale, 2)) return fail(QG_ERR_ALIGNMENT, "%s: scale must be 2-byte aligned", who);
    }
    if (w->nnz < 0) return fail(QG_ERR_INVALID_ARG, "%s: nnz < 0", who);
    if (w->nnz > 0) {
        if (!w->out_row_ptr || !w->out_col || !w->out_val)
            return fail(QG_ERR_INVALID_ARG, "%s: outlier arrays null with nnz=%d", who, w->nnz);
        if (!aligned(w->out_row_ptr, 4) || !aligned(w->out_col, 4) || !aligned(w->out_val, 2))
            return fail(QG_ERR_ALIGNMENT, "%s: outlier arrays misaligned", who);
    }
    return QG_OK;
}

// Checks shared by both quantizer entry points (everything but the scratch).
qg_status check_quantize_args(const uint16_t* W, float outlier_frac, const qg_qweight* out, const char* who)
{
    if (!W) return fail(QG_ERR_INVALID_ARG, "%s: W is null", who);
    if (!aligned(W, 16)) return fail(QG_ERR_ALIGNMENT, "%s: W must be 16-byte aligned", who);
    qg_status st = check_qweight(out, who);
    if (st != QG_OK) return st;
    if (!(outlier_frac >= 0.0f && outlier_frac < 1.0f))
        return fail(QG_ERR_INVALID_ARG, "%s: outlier_frac must be in [0, 1)", who);
    const int64_t n = nnz_of(out->N, out->K, outlier_frac);
    if (n != out->nnz)
        return fail(QG_ERR_INVALID_ARG, "%s: nnz=%d but floor(frac*N*K)=%lld", who, out->nnz, (long long)n);
    if (out->nnz > 0 && (int64_t)out->N * out->K > 0xFFFFFFFFll)
        return fail(QG_ERR_INVALID_ARG, "%s: N*K above 2^32 with outliers", who);
    return QG_OK;
}

// Identity of the CUDA context current on this thread (0 if none): caches of
// device addresses are keyed on it, so that a context destroyed and created
// again (cudaDeviceReset) gets its addresses looked up again.
unsigned long long current_context_id()
{
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static std::atomic<GetCurrent> get_current{nullptr};
    static std::atomic<GetId> get_id{nullptr};
    GetCurrent gc = get_current.load(std::memory_order_acquire);
    GetId gi = get_id.load(std::memory_order_acquire);
    if (!gc || !gi) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || !f1)
            return 0;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess || !f2)
            return 0;
        gc = reinterpret_cast<GetCurrent>(f1);
        gi = reinterpret_cast<GetId>(f2);
        get_current.store(gc, std::memory_order_release);
        get_id.store(gi, std::memory_order_release);
    }
    CUcontext ctx = nullptr;
    if (gc(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (gi(ctx, &id) != CUDA_SUCCESS) return 0;
    return id + 1;   // never 0 for a live context
}

// Programmatic dependent launch of the dense products: decode and tensor-core
// kernels (qgemm_set_dependent_launch).
std::atomic<int> g_dependent_launch{1};
bool dependent_launch_enabled() { return g_dependent_launch.load(std::memory_order_relaxed) != 0; }

}  // namespace qg

using namespace qg;

extern "C" {

const char* qgemm_last_error(void) { return g_err; }

qg_status qgemm_set_dependent_launch(int32_t enable)
{
    qg::g_dependent_launch.store(enable ? 1 : 0, std::memory_order_relaxed);
    return QG_OK;
}

qg_status qgemm_device_status(int32_t* status, int32_t reset)
{
    if (!status) return fail(QG_ERR_INVALID_ARG, "qgemm_device_status: status is NULL");
    int v = 0;
    qg_status st = read_device_status(&v, reset);
    if (st != QG_OK) return st;
    *status = v;
    return QG_OK;
}

qg_status qrepack_tiles_size(const qg_qweight* w, size_t* bytes)
{
    if (!bytes) return fail(QG_ERR_INVALID_ARG, "qrepack_tiles_size: bytes is null");
    qg_status st = check_qweight(w, "qrepack_tiles_size");
    if (st != QG_OK) return st;
    *bytes = tiles_bytes(*w);
    return QG_OK;
}

qg_status qrepack_tiles(const qg_qweight* w, void* tiles, size_t tiles_bytes_given, void* stream)
{
    qg_status st = check_qweight(w, "qrepack_tiles");
    if (st != QG_OK) return st;
    if (!tiles) return fail(QG_ERR_INVALID_ARG, "qrepack_tiles: tiles is null");
    if (!aligned(tiles, 128)) return fail(QG_ERR_ALIGNMENT, "qrepack_tiles: tiles must be 128-byte aligned");
    if (tiles_bytes_given < tiles_bytes(*w))
        return fail(QG_ERR_INVALID_ARG, "qrepack_tiles: %zu bytes < %zu", tiles_bytes_given, tiles_bytes(*w));
    if (!aligned(w->packed, 4)) return fail(QG_ERR_ALIGNMENT, "qrepack_tiles: packed misaligned");
    return launch_repack(*w, tiles, static_cast<cudaStream_t>(stream));
}

qg_status qgemm_tiles_workspace_size(int32_t M, const qg_qweight* w, size_t* bytes)
{
    if (!bytes) return fail(QG_ERR_INVALID_ARG, "qgemm_tiles_workspace_size: bytes is null");
    qg_status st = check_qweight(w, "qgemm_tiles_workspace_size");
    if (st != QG_OK) return st;
    if (M < 0) return fail(QG_ERR_INVALID_ARG, "qgemm_tiles_workspace_size: M < 0");
    *bytes = M ? gemm_workspace_bytes(M, *w) : 0;
    return QG_OK;
}

qg_status qgemm_forward_tiles(const uint16_t* x, int32_t M, int32_t ldx, const qg_qweight* w, const void* tiles,
                              void* y, int32_t ldy, qg_ydtype yt, void* ws, size_t ws_bytes, void* stream)
{
    qg_status st = check_qweight(w, "qgemm_forward_tiles");
    if (st != QG_OK) return st;
    if (M < 0) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_tiles: M < 0");
    if (M == 0) return QG_OK;
    if (!x || !y || !tiles) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_tiles: x, y or tiles is null");
    if (ldx < w->K || ldy < w->N) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_tiles: ldx < K or ldy < N");
    if (yt != QG_Y_F32 && yt != QG_Y_BF16) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_tiles: bad y dtype");
    if (!aligned(x, 2) || !aligned(y, yt == QG_Y_F32 ? 4 : 2) || !aligned(tiles, 128))
        return fail(QG_ERR_ALIGNMENT, "qgemm_forward_tiles: x, y or tiles misaligned");
    const size_t need = gemm_workspace_bytes(M, *w);
    if (!ws || ws_bytes < need)
        return fail(QG_ERR_WORKSPACE, "qgemm_forward_tiles: workspace %zu bytes < %zu", ws ? ws_bytes : (size_t)0, need);
    if (!aligned(ws, 256)) return fail(QG_ERR_ALIGNMENT, "qgemm_forward_tiles: workspace must be 256-byte aligned");
    return launch_gemm_tiles(x, M, ldx, *w, tiles, y, ldy, yt, ws, static_cast<cudaStream_t>(stream));
}

qg_status qgemm_w8a8_workspace_size(int32_t M, const qg_qweight* w, size_t* bytes)
{
    if (!bytes) return fail(QG_ERR_INVALID_ARG, "qgemm_w8a8_workspace_size: bytes is null");
    qg_status st = check_qweight(w, "qgemm_w8a8_workspace_size");
    if (st != QG_OK) return st;
    if (M < 0 || M > kW8A8MaxM) return fail(QG_ERR_UNSUPPORTED, "qgemm_w8a8: M=%d not in 0..%d", M, kW8A8MaxM);
    *bytes = M ? w8a8_workspace_bytes(M, w->K) : 0;
    return QG_OK;
}

qg_status qgemm_forward_w8a8(const uint16_t* x, int32_t M, int32_t ldx, const qg_qweight* w, void* y, int32_t ldy,
                             qg_ydtype yt, void* ws, size_t ws_bytes, void* stream)
{
    qg_status st = check_qweight(w, "qgemm_forward_w8a8");
    if (st != QG_OK) return st;
    if (w->bits != 8) return fail(QG_ERR_UNSUPPORTED, "qgemm_forward_w8a8: weights must be 8-bit (bits=%d)", w->bits);
    if (M < 0 || M > kW8A8MaxM) return fail(QG_ERR_UNSUPPORTED, "qgemm_forward_w8a8: M=%d not in 0..%d", M, kW8A8MaxM);
    if (M == 0) return QG_OK;
    if (!x || !y) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_w8a8: x or y is null");
    if (ldx < w->K || ldy < w->N) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_w8a8: ldx < K or ldy < N");
    if (yt != QG_Y_F32 && yt != QG_Y_BF16) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_w8a8: bad y dtype");
    if (!aligned(x, 2) || !aligned(y, yt == QG_Y_F32 ? 4 : 2))
        return fail(QG_ERR_ALIGNMENT, "qgemm_forward_w8a8: x or y misaligned");
    const size_t need = w8a8_workspace_bytes(M, w->K);
    if (!ws || ws_bytes < need)
        return fail(QG_ERR_WORKSPACE, "qgemm_forward_w8a8: workspace %zu bytes < %zu", ws ? ws_bytes : (size_t)0, need);
    if (!aligned(ws, 256)) return fail(QG_ERR_ALIGNMENT, "qgemm_forward_w8a8: workspace must be 256-byte aligned");
    return launch_w8a8(x, M, ldx, *w, y, ldy, yt, ws, static_cast<cudaStream_t>(stream));
}

qg_status qdiag_workspace_size(int32_t N, int32_t K, int32_t group, size_t* bytes)
{
    if (!bytes) return fail(QG_ERR_INVALID_ARG, "qdiag_workspace_size: bytes is null");
    qg_status st = check_shape(N, K, 4, group);
    if (st != QG_OK) return st;
    *bytes = diag_workspace_bytes(N, K, group);
    return QG_OK;
}

qg_status qdiag_layer(const uint16_t* W, const qg_qweight* w, float threshold, float* group_ratio, qg_diag* out,
                      void* ws, size_t ws_bytes, void* stream)
{
    qg_status st = check_qweight(w, "qdiag_layer");
    if (st != QG_OK) return st;
    if (!W || !out) return fail(QG_ERR_INVALID_ARG, "qdiag_layer: W or out is null");
    if (!aligned(W, 16)) return fail(QG_ERR_ALIGNMENT, "qdiag_layer: W must be 16-byte aligned");
    if (!aligned(out, 8) || (group_ratio && !aligned(group_ratio, 4)))
        return fail(QG_ERR_ALIGNMENT, "qdiag_layer: out or group_ratio misaligned");
    if (!(threshold == threshold)) return fail(QG_ERR_INVALID_ARG, "qdiag_layer: threshold is NaN");
    const size_t need = diag_workspace_bytes(w->N, w->K, w->group);
    if (!ws || ws_bytes < need)
        return fail(QG_ERR_WORKSPACE, "qdiag_layer: workspace %zu bytes < %zu", ws ? ws_bytes : (size_t)0, need);
    if (!aligned(ws, 256)) return fail(QG_ERR_ALIGNMENT, "qdiag_layer: workspace must be 256-byte aligned");
    return launch_diag(W, *w, threshold, group_ratio, out, ws, static_cast<cudaStream_t>(stream));
}

qg_status qgemm_selftest_bounded_wait(int32_t poll_limit, void* stream)
{
    if (poll_limit < 1 || poll_limit > 64)
        return fail(QG_ERR_INVALID_ARG, "qgemm_selftest_bounded_wait: poll_limit=%d not in 1..64", poll_limit);
    return launch_wait_selftest((uint32_t)poll_limit, static_cast<cudaStream_t>(stream));
}

qg_status qpack_query_sizes(int32_t N, int32_t K, int32_t bits, int32_t group, float outlier_frac,
                            size_t* packed_bytes, size_t* scale_bytes, size_t* zp_bytes,
                            size_t* codebook_bytes, int32_t* nnz)
{
    qg_status st = check_shape(N, K, bits, group);
    if (st != QG_OK) return st;
    if (!(outlier_frac >= 0.0f && outlier_frac < 1.0f))
        return fail(QG_ERR_INVALID_ARG, "outlier_frac must be in [0, 1)");
    const int64_t ng = K / group;
    const int64_t n = nnz_of(N, K, outlier_frac);
    if (n > INT32_MAX) return fail(QG_ERR_INVALID_ARG, "too many outliers");
    if (packed_bytes) *packed_bytes = (size_t)N * K * bits / 8;
    if (scale_bytes) *scale_bytes = bits == 2 ? 0 : (size_t)N * ng * 2;
    if (zp_bytes) *zp_bytes = bits == 2 ? 0 : (size_t)N * ng;
    if (codebook_bytes) *codebook_bytes = bits == 2 ? (size_t)N * ng * 8 : 0;
    if (nnz) *nnz = (int32_t)n;
    return QG_OK;
}

qg_status qpack_workspace_size(int32_t N, int32_t K, size_t* bytes)
{
    if (!bytes) return fail(QG_ERR_INVALID_ARG, "bytes is null");
    if (N <= 0 || K <= 0) return fail(QG_ERR_INVALID_ARG, "N and K must be positive");
    *bytes = quantize_workspace_bytes(N, K);
    return QG_OK;
}

qg_status qpack_quantize_mode(const uint16_t* W, float outlier_frac, qg_quant_mode mode, const qg_qweight* out,
                              void* ws, size_t ws_bytes, void* stream)
{
    qg_status st = check_quantize_args(W, outlier_frac, out, "qpack_quantize_mode");
    if (st != QG_OK) return st;
    if (mode != QG_QUANT_ASYMMETRIC && mode != QG_QUANT_SYMMETRIC && mode != QG_QUANT_LINEAR2)
        return fail(QG_ERR_INVALID_ARG, "qpack_quantize_mode: unknown mode %d", (int)mode);
    if (mode == QG_QUANT_LINEAR2 && out->bits != 2)
        return fail(QG_ERR_UNSUPPORTED, "qpack_quantize_mode: QG_QUANT_LINEAR2 is a 2-bit format (bits=%d)", out->bits);
    const size_t need = quantize_workspace_bytes(out->N, out->K);
    if (!ws || ws_bytes < need)
        return fail(QG_ERR_WORKSPACE, "qpack_quantize_mode: workspace %zu bytes < %zu", ws ? ws_bytes : (size_t)0, need);
    if (!aligned(ws, 256)) return fail(QG_ERR_ALIGNMENT, "qpack_quantize_mode: workspace must be 256-byte aligned");
    return launch_quantize(W, outlier_frac, *out, ws, static_cast<cudaStream_t>(stream), (int)mode);
}

qg_status qpack_quantize(const uint16_t* W, float outlier_frac, const qg_qweight* out, void* ws,
                         size_t ws_bytes, void* stream)
{
    qg_status st = check_quantize_args(W, outlier_frac, out, "qpack_quantize");
    if (st != QG_OK) return st;
    const size_t need = quantize_workspace_bytes(out->N, out->K);
    if (!ws || ws_bytes < need)
        return fail(QG_ERR_WORKSPACE, "qpack_quantize: workspace %zu bytes < %zu", ws ? ws_bytes : (size_t)0, need);
    if (!aligned(ws, 256)) return fail(QG_ERR_ALIGNMENT, "qpack_quantize: workspace must be 256-byte aligned");
    return launch_quantize(W, outlier_frac, *out, ws, static_cast<cudaStream_t>(stream));
}

qg_status qgemm_forward_multi(const uint16_t* x, int32_t M, int32_t ldx, const qg_qweight* ws, int32_t n,
                              void* const* ys, const int32_t* ldys, qg_ydtype yt, void* work, size_t work_bytes,
                              void* stream)
{
    if (n < 1 || n > kMultiMax) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: n=%d not in 1..%d", n, kMultiMax);
    if (!ws || !ys || !ldys) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: null ws/ys/ldys");
    for (int q = 0; q < n; q++) {
        qg_status st = check_qweight(&ws[q], "qgemm_forward_multi");
        if (st != QG_OK) return st;
        if (ws[q].K != ws[0].K || ws[q].bits != ws[0].bits || ws[q].group != ws[0].group)
            return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: weights differ in K/bits/group");
    }
    if (M < 0) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: M < 0");
    if (M == 0) return QG_OK;
    if (!x) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: x is null");
    if (ldx < ws[0].K) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: ldx=%d < K=%d", ldx, ws[0].K);
    if (yt != QG_Y_F32 && yt != QG_Y_BF16) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: bad y dtype");
    if (!aligned(x, 2)) return fail(QG_ERR_ALIGNMENT, "qgemm_forward_multi: x misaligned");
    for (int q = 0; q < n; q++) {
        if (!ys[q]) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: ys[%d] is null", q);
        if (ldys[q] < ws[q].N) return fail(QG_ERR_INVALID_ARG, "qgemm_forward_multi: ldys[%d] < N", q);
        if (!aligned(ys[q], yt == QG_Y_F32 ? 4 : 2)) return fail(QG_ERR_ALIGNMENT, "qgemm_forward_multi: ys[%d] misaligned", q);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M <= kGemvMaxM) return launch_gemv_multi(x, M, ldx, ws, n, ys, ldys, yt, work, work_bytes, s);
    // above the decode range: one tensor-core product after the other in the
    // caller's workspace, x converted to fp16 by the first (same K and width:
    // the same operand order) and read by all
    for (int q = 0; q < n; q++) {
        const size_t need = gemm_workspace_bytes(M, ws[q]);
        if (need && (!work || work_bytes < need))
            return fail(QG_ERR_WORKSPACE, "qgemm_forward_multi: workspace %zu bytes < %zu", work ? work_bytes : (size_t)0, need);
        if (need && !aligned(work, 256)) return fail(QG_ERR_ALIGNMENT, "qgemm_forward_multi: workspace must be 256-byte aligned");
        qg_status st = launch_gemm(x, M, ldx, ws[q], ys[q], ldys[q], yt, work, work_bytes, q == 0, s);
        if (st != QG_OK) return st;
    }
    return QG_OK;
}

qg_status qgemm_workspace_size(int32_t M, const qg_qweight* w, size_t* bytes)
{
    if (!bytes) return fail(QG_ERR_INVALID_ARG, "bytes is null");
    qg_status st = check_qweight(w, "qgemm_workspace_size");
    if (st != QG_OK) return st;
    if (M < 0) return fail(QG_ERR_INVALID_ARG, "M < 0");
    *bytes = M <= kGemvMaxM ? gemv_workspace_bytes(M, w->K) : gemm_workspace_bytes(M, *w);
    return QG_OK;
}

qg_status qgemm_forward(const uint16_t* x, int32_t M, int32_t ldx, const qg_qweight* w, void* y,
                        int32_t ldy, qg_ydtype yt, void* ws, size_t ws_bytes, void* stream)
{
    qg_status st = check_qweight(w, "qgemm_forward");
    if (st != QG_OK) return st;
    if (M < 0) return fail(QG_ERR_INVALID_ARG, "qgemm_forward: M < 0");
    if (M == 0) return QG_OK;
    if (!x || !y) return fail(QG_ERR_INVALID_ARG, "qgemm_forward: x or y is null");
    if (ldx < w->K) return fail(QG_ERR_INVALID_ARG, "qgemm_forward: ldx=%d < K=%d", ldx, w->K);
    if (ldy < w->N) return fail(QG_ERR_INVALID_ARG, "qgemm_forward: ldy=%d < N=%d", ldy, w->N);
    if (yt != QG_Y_F32 && yt != QG_Y_BF16) return fail(QG_ERR_INVALID_ARG, "qgemm_forward: bad y dtype");
    if (!aligned(x, 2) || !aligned(y, yt == QG_Y_F32 ? 4 : 2))
        return fail(QG_ERR_ALIGNMENT, "qgemm_forward: x or y misaligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M <= kGemvMaxM) return launch_gemv(x, M, ldx, *w, y, ldy, yt, ws, ws_bytes, s);
    const size_t need = gemm_workspace_bytes(M, *w);
    if (need && (!ws || ws_bytes < need))
        return fail(QG_ERR_WORKSPACE, "qgemm_forward: workspace %zu bytes < %zu", ws ? ws_bytes : (size_t)0, need);
    if (need && !aligned(ws, 256)) return fail(QG_ERR_ALIGNMENT, "qgemm_forward: workspace must be 256-byte aligned");
    return launch_gemm(x, M, ldx, *w, y, ldy, yt, ws, ws_bytes, true, s);
}

qg_status qgemm_moe_workspace_size(int32_t T, int32_t k, int32_t E, const qg_qweight* experts,
                                   size_t* bytes)
{
    if (!bytes) return fail(QG_ERR_INVALID_ARG, "bytes is null");
    if (T < 0 || k <= 0 || E <= 0 || E > kMoeMaxExperts || !experts)
        return fail(QG_ERR_INVALID_ARG, "qgemm_moe_workspace_size: bad T/k/E");
    *bytes = moe_workspace_bytes(T, k, E, 1, experts);   // enough for any number of products per call
    return QG_OK;
}

static qg_status moe_checked(const char* fn, const uint16_t* x, int32_t T, const int32_t* topk_ids, int32_t k,
                             const qg_qweight* experts, int32_t E, int32_t n, void* const* ys, qg_ydtype yt,
                             void* ws, size_t ws_bytes, void* stream)
{
    if (T < 0 || k <= 0) return fail(QG_ERR_INVALID_ARG, "%s: T < 0 or k <= 0", fn);
    if (E <= 0 || E > kMoeMaxExperts) return fail(QG_ERR_INVALID_ARG, "%s: E must be in 1..%d", fn, kMoeMaxExperts);
    if (n < 1 || n > kMoeMaxProducts)
        return fail(QG_ERR_INVALID_ARG, "%s: n must be in 1..%d", fn, kMoeMaxProducts);
    if (!experts) return fail(QG_ERR_INVALID_ARG, "%s: experts is null", fn);
    for (int e = 0; e < E * n; e++) {
        qg_status st = check_qweight(&experts[e], fn);
        if (st != QG_OK) return st;
        if (experts[e].N != experts[0].N || experts[e].K != experts[0].K || experts[e].bits != experts[0].bits ||
            experts[e].group != experts[0].group)
            return fail(QG_ERR_INVALID_ARG, "%s: experts differ in N/K/bits/group", fn);
    }
    if (T == 0) return QG_OK;
    if (!x || !topk_ids || !ys) return fail(QG_ERR_INVALID_ARG, "%s: null x/topk_ids/y", fn);
    for (int q = 0; q < n; q++)
        if (!ys[q]) return fail(QG_ERR_INVALID_ARG, "%s: null y", fn);
    if (yt != QG_Y_F32 && yt != QG_Y_BF16) return fail(QG_ERR_INVALID_ARG, "%s: bad y dtype", fn);
    if (!aligned(x, 2) || !aligned(topk_ids, 4)) return fail(QG_ERR_ALIGNMENT, "%s: misaligned x/topk_ids/y", fn);
    for (int q = 0; q < n; q++)
        if (!aligned(ys[q], yt == QG_Y_F32 ? 4 : 2)) return fail(QG_ERR_ALIGNMENT, "%s: misaligned x/topk_ids/y", fn);
    const size_t need = moe_workspace_bytes(T, k, E, n, experts);
    if (need && (!ws || ws_bytes < need))
        return fail(QG_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu", fn, ws ? ws_bytes : (size_t)0, need);
    if (need && !aligned(ws, 256)) return fail(QG_ERR_ALIGNMENT, "%s: workspace must be 256-byte aligned", fn);
    return launch_moe(x, T, topk_ids, k, experts, E, n, ys, yt, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

qg_status qgemm_moe_grouped(const uint16_t* x, int32_t T, const int32_t* topk_ids, int32_t k,
                            const qg_qweight* experts, int32_t E, void* y, qg_ydtype yt, void* ws,
                            size_t ws_bytes, void* stream)
{
    void* ys[1] = {y};
    return moe_checked("qgemm_moe_grouped", x, T, topk_ids, k, experts, E, 1, y ? ys : nullptr, yt, ws, ws_bytes,
                       stream);
}

qg_status qgemm_moe_grouped_multi(const uint16_t* x, int32_t T, const int32_t* topk_ids, int32_t k,
                                  const qg_qweight* experts, int32_t E, int32_t n, void* const* ys, qg_ydtype yt,
                                  void* ws, size_t ws_bytes, void* stream)
{
    return moe_checked("qgemm_moe_grouped_multi", x, T, topk_ids, k, experts, E, n, ys, yt, ws, ws_bytes, stream);
}

}  // extern "C"
