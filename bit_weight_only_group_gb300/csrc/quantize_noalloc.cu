// qpack_quantize_noalloc: the quantize-and-pack entry point for callers that
// cannot hand the library a workspace.
//
// Who cannot allocate: code that runs inside a host application owning the
// device allocator (a plugin or an inference server that reserves its memory
// pool up front and forbids further cudaMalloc), code on a latency-critical
// path where cudaMalloc / cudaFree's implicit device-wide synchronization is
// not acceptable, and code that runs after a fixed memory budget has been
// frozen.  For them the scratch the quantizer needs (a 32768-bin histogram of
// |w| keys, the selection parameters and three per-row counters) lives in
// one file-scope device array of a fixed size.  Every GPU that loads this
// library holds that array until the process exits.
//
// The kernels are the same ones qpack_quantize launches; only the scratch
// pointer differs.  Every call shares the array, which keeps the last call's
// contents: the part that must start at zero (the histogram) is cleared on
// the stream by each call, and everything else is written before it is read.
// Calls whose work overlaps on the GPU (different streams, no ordering
// between them) race on the array.
#include <cmath>
#include <mutex>

#include "qg_internal.h"

namespace qg {
namespace {

// 1 MiB: the histogram takes 128 KiB; the per-row counters take 12 bytes per
// row, so matrices up to about 76,000 rows fit.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the name g_noalloc_scratch is only a host-side stand-in, so the address is
// looked up once per device, with that device current, and cached.
qg_status scratch_address(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "qpack_quantize_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(QG_ERR_UNSUPPORTED, "qpack_quantize_noalloc: device index %d above %d", dev, kMaxDevices - 1);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "qpack_quantize_noalloc: cudaGetSymbolAddress of the scratch array");
        if (!p) return fail(QG_ERR_CUDA, "qpack_quantize_noalloc: scratch array has no device address");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return QG_OK;
}

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" QG_API qg_status qpack_quantize_noalloc(const uint16_t* W, float outlier_frac, const qg_qweight* out,
                                                   void* stream)
{
    if (!W) return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: W is null");
    if (!is_aligned(W, 16)) return fail(QG_ERR_ALIGNMENT, "qpack_quantize_noalloc: W must be 16-byte aligned");
    if (!out) return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: null weight descriptor");
    const qg_qweight& w = *out;
    if (w.N <= 0 || w.K <= 0) return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: N and K must be positive");
    if (w.bits < 2 || w.bits > 6) return fail(QG_ERR_UNSUPPORTED, "qpack_quantize_noalloc: bits must be 2..6");
    if (w.group != 64 && w.group != 128) return fail(QG_ERR_UNSUPPORTED, "qpack_quantize_noalloc: group must be 64 or 128");
    if (w.K % w.group) return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: K is not a multiple of group");
    if (!(outlier_frac >= 0.0f && outlier_frac < 1.0f))
        return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: outlier_frac must be in [0, 1)");
    if (!w.packed || !is_aligned(w.packed, 16))
        return fail(w.packed ? QG_ERR_ALIGNMENT : QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: packed null or not 16-byte aligned");
    if (w.bits == 2 ? (!w.codebook || !is_aligned(w.codebook, 8)) : (!w.scale || !w.zp || !is_aligned(w.scale, 2)))
        return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: scale/zp or codebook missing or misaligned");
    const int64_t nnz = outlier_frac <= 0.0f ? 0 : (int64_t)std::floor((double)outlier_frac * (double)w.N * (double)w.K);
    if (nnz != w.nnz)
        return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: nnz=%d but floor(frac*N*K)=%lld", w.nnz, (long long)nnz);
    if (w.nnz > 0 && (!w.out_row_ptr || !w.out_col || !w.out_val))
        return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: outlier arrays null with nnz=%d", w.nnz);
    if (w.nnz > 0 && (int64_t)w.N * w.K > 0xFFFFFFFFll)
        return fail(QG_ERR_INVALID_ARG, "qpack_quantize_noalloc: N*K above 2^32 with outliers");
    const size_t need = quantize_workspace_bytes(w.N, w.K);
    if (need > kNoAllocScratchBytes)
        return fail(QG_ERR_WORKSPACE,
                    "qpack_quantize_noalloc: N=%d needs %zu bytes of scratch, above the fixed %zu-byte array "
                    "(use qpack_quantize with a workspace)", w.N, need, kNoAllocScratchBytes);
    void* scratch = nullptr;
    qg_status st = scratch_address(&scratch);
    if (st != QG_OK) return st;
    return launch_quantize(W, outlier_frac, w, scratch, static_cast<cudaStream_t>(stream));
}
