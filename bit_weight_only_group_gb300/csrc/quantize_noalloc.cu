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
#include <mutex>

#include "qg_internal.h"

namespace qg {
namespace {

// 1 MiB: the histogram takes 128 KiB; the per-row counters take 12 bytes per
// row, so matrices with outliers (or 8-bit scales) up to about 76,000 rows
// fit.  Without either the quantizer touches no scratch, and any size is
// accepted.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the current context.  In host code
// the name g_noalloc_scratch is only a host-side stand-in, so the address is
// looked up with the device current, once per device and context, and
// cached; a context created anew (after cudaDeviceReset) gets a new lookup.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

qg_status scratch_address(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "qpack_quantize_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(QG_ERR_UNSUPPORTED, "qpack_quantize_noalloc: device index %d above %d", dev, kMaxDevices - 1);
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_addr[dev] || !ctx || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "qpack_quantize_noalloc: cudaGetSymbolAddress of the scratch array");
        if (!p) return fail(QG_ERR_CUDA, "qpack_quantize_noalloc: scratch array has no device address");
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = current_context_id();   // the lookup made the context current
    }
    *out = g_scratch_addr[dev];
    return QG_OK;
}

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" QG_API qg_status qpack_quantize_noalloc(const uint16_t* W, float outlier_frac, const qg_qweight* out,
                                                   void* stream)
{
    // the same checks, in the same order, as qpack_quantize (same status codes)
    qg_status st = check_quantize_args(W, outlier_frac, out, "qpack_quantize_noalloc");
    if (st != QG_OK) return st;
    const qg_qweight& w = *out;
    void* scratch = nullptr;
    if (w.nnz > 0 || w.scale8) {   // only the outlier selection and the 8-bit scales use scratch
        const size_t need = quantize_workspace_bytes(w.N, w.K);
        if (need > kNoAllocScratchBytes)
            return fail(QG_ERR_WORKSPACE,
                        "qpack_quantize_noalloc: N=%d with outliers or 8-bit scales needs %zu bytes of scratch, "
                        "above the fixed %zu-byte array (use qpack_quantize with a workspace)", w.N, need,
                        kNoAllocScratchBytes);
        st = scratch_address(&scratch);
        if (st != QG_OK) return st;
    }
    return launch_quantize(W, outlier_frac, w, scratch, static_cast<cudaStream_t>(stream));
}
