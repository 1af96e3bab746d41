// Host dispatch of the decode kernels by bit width, and the grouped (MoE)
// entry: device-side routing (a stable counting sort of the (token, slot)
// pairs by expert) followed by the grouped decode kernel.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "gemv_impl.cuh"
#include "qg_internal.h"

namespace qg {
namespace gemv {
extern template qg_status launch_dense<2>(const Problem&, int, cudaStream_t);
extern template qg_status launch_multi<2>(const MultiTable&, int, cudaStream_t);
extern template qg_status launch_dense<3>(const Problem&, int, cudaStream_t);
extern template qg_status launch_multi<3>(const MultiTable&, int, cudaStream_t);
extern template qg_status launch_dense<4>(const Problem&, int, cudaStream_t);
extern template qg_status launch_multi<4>(const MultiTable&, int, cudaStream_t);
extern template qg_status launch_dense<5>(const Problem&, int, cudaStream_t);
extern template qg_status launch_multi<5>(const MultiTable&, int, cudaStream_t);
extern template qg_status launch_dense<6>(const Problem&, int, cudaStream_t);
extern template qg_status launch_multi<6>(const MultiTable&, int, cudaStream_t);
extern template qg_status launch_grouped<2>(const MoeTable&, int, int, int, int, cudaStream_t);
extern template qg_status launch_grouped<3>(const MoeTable&, int, int, int, int, cudaStream_t);
extern template qg_status launch_grouped<4>(const MoeTable&, int, int, int, int, cudaStream_t);
extern template qg_status launch_grouped<5>(const MoeTable&, int, int, int, int, cudaStream_t);
extern template qg_status launch_grouped<6>(const MoeTable&, int, int, int, int, cudaStream_t);
extern template qg_status launch_dense<8>(const Problem&, int, cudaStream_t);
extern template qg_status launch_multi<8>(const MultiTable&, int, cudaStream_t);
extern template qg_status launch_grouped<8>(const MoeTable&, int, int, int, int, cudaStream_t);
}  // namespace gemv

// Device status word of the library's kernels (QG_OK, or QG_ERR_TIMEOUT after
// a bounded wait gave up), one per device; kernels write it through a pointer
// argument, qgemm_device_status() reads and clears it.
__device__ int g_device_status;

namespace {
constexpr int kMaxStatusDevices = 64;
std::mutex g_status_mu;
int* g_status_addr[kMaxStatusDevices];
unsigned long long g_status_ctx[kMaxStatusDevices];
}  // namespace

// Address of g_device_status in the current context, looked up once per
// device and context (a context created anew gets a new lookup).
int* device_status_ptr()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxStatusDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_status_addr[dev] || !ctx || ctx != g_status_ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_addr[dev] = static_cast<int*>(p);
        g_status_ctx[dev] = current_context_id();
    }
    return g_status_addr[dev];
}

qg_status read_device_status(int* out, int reset)
{
    int* p = device_status_ptr();
    if (!p) return fail(QG_ERR_CUDA, "qgemm_device_status: no device status word on the current device");
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "qgemm_device_status: read");
    if (reset && v != 0) {
        const int zero = 0;
        e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "qgemm_device_status: reset");
    }
    *out = v;
    return QG_OK;
}

// Self-check of the bounded waits: one mbarrier that nothing ever arrives on,
// waited on with a poll limit; the wait gives up and the kernel reports
// QG_ERR_TIMEOUT through the status word, as a tensor-core kernel does when
// one of its waits runs out.  It issues no TMA and no MMA, and holds nothing
// when it exits.
__global__ void k_wait_selftest(int* status, uint32_t limit)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !ptx::mbar_wait_bounded(b, 0, limit) && status) atomicExch(status, (int)QG_ERR_TIMEOUT);
}

qg_status launch_wait_selftest(uint32_t limit, cudaStream_t s)
{
    int* st = device_status_ptr();
    if (!st) return fail(QG_ERR_CUDA, "qgemm_selftest_bounded_wait: no device status word on the current device");
    k_wait_selftest<<<1, 32, 0, s>>>(st, limit);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "qgemm_selftest_bounded_wait: launch");
    return QG_OK;
}

namespace {

gemv::Problem make_problem(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy,
                           qg_ydtype yt)
{
    gemv::Problem p;
    p.x = reinterpret_cast<const __nv_bfloat16*>(x);
    p.ldx = ldx; p.M = M; p.N = w.N; p.K = w.K;
    p.rowmap = nullptr; p.xdiv = 1;
    p.packed = w.packed;
    p.scale = w.scale;
    p.zp = w.zp;
    p.cb = reinterpret_cast<const uint2*>(w.codebook);
    p.row_ptr = w.out_row_ptr;
    p.col = w.out_col;
    p.val = w.out_val;
    p.nnz = w.nnz;
    p.y = y; p.ldy = ldy; p.y_bf16 = yt == QG_Y_BF16;
    p.magic = gemv::kF16Magic;
    p.scale8 = w.scale8;
    p.scale8_exp = w.scale8_exp;
    p.fb_row_ptr = w.fb_row_ptr;
    p.fb_col = w.fb_col;
    p.fb_val = w.fb_val;
    p.fb_cap = w.fb_cap;
    p.xfrag = nullptr;
    p.status = device_status_ptr();
    p.xg = p.xp_off = p.xslot_off = p.xbar_off = 0;
    return p;
}

qg_status dense_by_bits(const gemv::Problem& p, int bits, int group, cudaStream_t s)
{
    switch (bits) {
        case 2: return gemv::launch_dense<2>(p, group, s);
        case 3: return gemv::launch_dense<3>(p, group, s);
        case 4: return gemv::launch_dense<4>(p, group, s);
        case 5: return gemv::launch_dense<5>(p, group, s);
        case 6: return gemv::launch_dense<6>(p, group, s);
        default: return gemv::launch_dense<8>(p, group, s);
    }
}

// ---------------------------------------------------------------- routing
// One block.  counts -> exclusive offsets -> stable placement: pair i goes
// to offsets[e] + (number of earlier pairs with the same expert).
constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads) k_route(const int* __restrict__ topk, int P, int E, int chunk,
                                                         int* __restrict__ offsets, int* __restrict__ perm,
                                                         int2* __restrict__ items, int* __restrict__ n_items)
{
    __shared__ int cnt[kMoeMaxExperts];
    __shared__ int off[kMoeMaxExperts];
    __shared__ int carry[kMoeMaxExperts];
    __shared__ int wtab[kRouteThreads / 32][kMoeMaxExperts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kRouteThreads) cnt[e] = 0, carry[e] = 0;
    __syncthreads();
    for (int i = tid; i < P; i += kRouteThreads) {
        const int e = topk[i];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0, ni = 0;
        for (int e = 0; e < E; e++) {
            off[e] = acc;
            offsets[e] = acc;
            acc += cnt[e];
            for (int c = 0; c * chunk < cnt[e]; c++) items[ni++] = make_int2(e, c);
        }
        offsets[E] = acc;
        *n_items = ni;
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < P; base += kRouteThreads) {
        for (int q = tid; q < (kRouteThreads / 32) * E; q += kRouteThreads) wtab[q / E][q % E] = 0;
        __syncthreads();
        const int i = base + tid;
        const int e = i < P ? topk[i] : -1;
        const bool valid = e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        const int wrank = __popc(peers & lt);
        if (valid && wrank == 0) wtab[warp][e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int before = carry[e];
            for (int w = 0; w < warp; w++) before += wtab[w][e];
            perm[off[e] + before + wrank] = i;
        }
        __syncthreads();
        for (int q = tid; q < E; q += kRouteThreads) {
            int s = 0;
            for (int w = 0; w < kRouteThreads / 32; w++) s += wtab[w][q];
            carry[q] += s;
        }
        __syncthreads();
    }
}

struct MoeWs {
    int* offsets;
    int* perm;
    int2* items;
    int* n_items;
    void* x16;   // x in routed order, fp16 (tensor-core path only)
};

// Upper bound on work items: sum over experts of ceil(count / chunk) with the
// smallest chunk (1 pair).
inline int max_items_for(int P, int E, int chunk) { return (int)ceil_div(P, chunk) + E; }

size_t moe_ws_layout(int T, int k, int E, int n, const qg_qweight* experts, MoeWs* p, void* base)
{
    const size_t P = (size_t)T * k;
    const size_t o_off = 0;
    const size_t o_n = align_up(sizeof(int) * ((size_t)E + 1), 256);
    const size_t o_perm = o_n + 256;
    const size_t o_items = align_up(o_perm + sizeof(int) * P, 256);
    const size_t o_x16 = align_up(o_items + sizeof(int2) * (size_t)max_items_for((int)P, E, 1), 256);
    const size_t x16 = moe_tc_eligible(experts, E, n) ? moe_tc_x16_bytes((int)P, experts[0].K) : 0;
    const size_t total = o_x16 + x16;
    if (p && base) {
        char* b = static_cast<char*>(base);
        p->offsets = reinterpret_cast<int*>(b + o_off);
        p->n_items = reinterpret_cast<int*>(b + o_n);
        p->perm = reinterpret_cast<int*>(b + o_perm);
        p->items = reinterpret_cast<int2*>(b + o_items);
        p->x16 = x16 ? static_cast<void*>(b + o_x16) : nullptr;
    }
    return total;
}

}  // namespace

// The caller's workspace as the fragment-order copy of x, when M calls for it
// and it is large enough (else null: the CTAs convert x themselves).
static const unsigned char* xfrag_buffer(int M, int K, void* ws, size_t ws_bytes)
{
    const size_t need = gemv_workspace_bytes(M, K);
    return need && ws && ws_bytes >= need && aligned(ws, 256) ? static_cast<const unsigned char*>(ws) : nullptr;
}

qg_status launch_gemv(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy,
                      qg_ydtype yt, void* ws, size_t ws_bytes, cudaStream_t s)
{
    gemv::Problem p = make_problem(x, M, ldx, w, y, ldy, yt);
    p.xfrag = xfrag_buffer(M, w.K, ws, ws_bytes);
    return dense_by_bits(p, w.bits, w.group, s);
}

qg_status launch_gemv_multi(const uint16_t* x, int M, int ldx, const qg_qweight* ws, int n, void* const* ys,
                            const int32_t* ldys, qg_ydtype yt, void* work, size_t work_bytes, cudaStream_t s)
{
    static_assert(kMultiMax == gemv::kMultiMax, "one limit on products per launch");
    gemv::MultiTable t;
    memset(&t, 0, sizeof(t));
    t.n = n;
    t.tile_start[0] = 0;
    for (int q = 0; q < n; q++) {
        t.p[q] = make_problem(x, M, ldx, ws[q], ys[q], ldys[q], yt);
        t.p[q].xfrag = xfrag_buffer(M, ws[q].K, work, work_bytes);   // one copy of x for every product
        t.tile_start[q + 1] = t.tile_start[q] + (int)ceil_div(ws[q].N, gemv::kRowsPerCta);
    }
    for (int q = n; q < gemv::kMultiMax; q++) t.tile_start[q + 1] = t.tile_start[n];
    switch (ws[0].bits) {
        case 2: return gemv::launch_multi<2>(t, ws[0].group, s);
        case 3: return gemv::launch_multi<3>(t, ws[0].group, s);
        case 4: return gemv::launch_multi<4>(t, ws[0].group, s);
        case 5: return gemv::launch_multi<5>(t, ws[0].group, s);
        case 6: return gemv::launch_multi<6>(t, ws[0].group, s);
        default: return gemv::launch_multi<8>(t, ws[0].group, s);
    }
}

size_t moe_workspace_bytes(int T, int k, int E, int n, const qg_qweight* experts)
{
    return moe_ws_layout(T, k, E, n, experts, nullptr, nullptr);
}

qg_status launch_moe(const uint16_t* x, int T, const int32_t* topk, int k, const qg_qweight* experts, int E,
                     int n, void* const* ys, qg_ydtype yt, void* ws, size_t, cudaStream_t s)
{
    MoeWs p{};
    moe_ws_layout(T, k, E, n, experts, &p, ws);
    const int P = T * k;
    const qg_qweight& w0 = experts[0];
    if (p.x16) {
        // tensor cores: every expert's tokens in chunks of up to kMoeTcChunk, weights as the MMA's M side
        k_route<<<1, kRouteThreads, 0, s>>>(topk, P, E, kMoeTcChunk, p.offsets, p.perm, p.items, p.n_items);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "routing kernel launch");
        return launch_moe_tc(x, T, k, experts, E, n, ys, yt, p.offsets, p.perm, p.items, p.n_items,
                             max_items_for(P, E, kMoeTcChunk), p.x16, s);
    }
    // tokens per CTA chunk from the mean load per expert
    const int mean = (P + E - 1) / E;
    const int mp = gemv::mp_for(std::max(1, mean));
    k_route<<<1, kRouteThreads, 0, s>>>(topk, P, E, mp, p.offsets, p.perm, p.items, p.n_items);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "routing kernel launch");

    // one grouped decode launch per product over the shared routing
    for (int q = 0; q < n; q++) {
        const qg_qweight* ex = experts + (size_t)q * E;
        gemv::MoeTable t;
        memset(&t, 0, sizeof(t));
        t.x = reinterpret_cast<const __nv_bfloat16*>(x);
        t.ldx = w0.K; t.N = w0.N; t.K = w0.K; t.topk = k;
        t.chunk = mp;
        t.offsets = p.offsets;
        t.perm = p.perm;
        t.items = p.items;
        t.n_items = p.n_items;
        t.y = ys[q];
        t.y_bf16 = yt == QG_Y_BF16;
        t.magic = gemv::kF16Magic;
        for (int i = 0; i < E; i++) {
            t.packed[i] = ex[i].packed;
            t.scale[i] = ex[i].scale;
            t.zp[i] = ex[i].zp;
            t.cb[i] = reinterpret_cast<const uint2*>(ex[i].codebook);
            t.row_ptr[i] = ex[i].out_row_ptr;
            t.col[i] = ex[i].out_col;
            t.val[i] = ex[i].out_val;
            t.nnz[i] = ex[i].nnz;
            t.scale8[i] = ex[i].scale8;
            t.scale8_exp[i] = ex[i].scale8_exp;
            t.fb_row_ptr[i] = ex[i].fb_row_ptr;
            t.fb_col[i] = ex[i].fb_col;
            t.fb_val[i] = ex[i].fb_val;
            t.fb_cap[i] = ex[i].fb_cap;
        }
        const int maxi = max_items_for(P, E, t.chunk);
        const int expect = std::min(maxi, (int)ceil_div(P, t.chunk) + E / 2);
        qg_status st;
        switch (w0.bits) {
            case 2: st = gemv::launch_grouped<2>(t, maxi, expect, w0.group, mp, s); break;
            case 3: st = gemv::launch_grouped<3>(t, maxi, expect, w0.group, mp, s); break;
            case 4: st = gemv::launch_grouped<4>(t, maxi, expect, w0.group, mp, s); break;
            case 5: st = gemv::launch_grouped<5>(t, maxi, expect, w0.group, mp, s); break;
            case 6: st = gemv::launch_grouped<6>(t, maxi, expect, w0.group, mp, s); break;
            default: st = gemv::launch_grouped<8>(t, maxi, expect, w0.group, mp, s); break;
        }
        if (st != QG_OK) return st;
    }
    return QG_OK;
}

}  // namespace qg
