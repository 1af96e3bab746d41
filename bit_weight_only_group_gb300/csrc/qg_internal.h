// Internal declarations shared by the translation units of libqgemm.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "qgemm.h"

namespace qg {

// Thread-local message behind qgemm_last_error().
void set_error(const char* fmt, ...);
qg_status fail(qg_status st, const char* fmt, ...);
qg_status cuda_fail(cudaError_t e, const char* what);

// Number of SMs of the current device (cached per device).
int num_sms();
// Dynamic shared memory per CTA that lets at most `cap` CTAs share an SM of
// the current device (1 <= cap <= 8).
int smem_for_cap(int cap);

// Argument checks shared by the entry points (each sets the error message).
bool aligned(const void* p, size_t a);
int64_t nnz_of(int64_t N, int64_t K, float frac);
qg_status check_shape(int64_t N, int64_t K, int bits, int group);
qg_status check_qweight(const qg_qweight* w, const char* who);
qg_status check_quantize_args(const uint16_t* W, float outlier_frac, const qg_qweight* out, const char* who);
// Identity of the thread's current CUDA context (0 if none).
unsigned long long current_context_id();

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------- quantizer
size_t quantize_workspace_bytes(int N, int K);
// mode: 0 asymmetric (codebook at 2 bits), 1 symmetric, 2 linear 2-bit (qg_quant_mode)
qg_status launch_quantize(const uint16_t* W, float frac, const qg_qweight& w, void* ws,
                          cudaStream_t s, int mode = 0);

// ---------------------------------------------------------------- decode GEMV
// Largest M the register-dequant (decode) kernel takes; above it the
// tensor-core kernel runs (split over K up to 256 tokens).  Measured with
// the tensor-core kernel's split K: on two 70B-shaped INT4 layers (L2
// flushed) M = 16 decode 0.614 ms against 0.885 on the tensor cores, M = 24
// 1.125 against 1.043 (planar), M = 32 1.295 against 1.055; on the 7B-shaped
// mixed-width stack at M = 32, 354 GB/s on the decode kernel against 361.
constexpr int kGemvMaxM = 16;
// From this M on, a decode call converts x once into the fp16 fragment order
// the CTAs stage (in the caller's workspace) and the CTAs bulk-copy their x
// blocks, instead of every CTA converting them.
constexpr int kXFragMinM = 8;
inline int padded_tokens(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : 64; }
// Workspace of a decode call: the fragment-order copy of x (0 below kXFragMinM).
inline size_t gemv_workspace_bytes(int M, int K)
{
    return M >= kXFragMinM ? align_up((size_t)2 * K * padded_tokens(M), 256) : 0;
}
// ws: the decode workspace, or null (or too small): each CTA then converts its own x blocks.
qg_status launch_gemv(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy,
                      qg_ydtype yt, void* ws, size_t ws_bytes, cudaStream_t s);

// Device status word of the library's kernels with bounded waits (nullptr if
// it has no address on the current device) and its synchronous read
// (optionally cleared).
int* device_status_ptr();
// Programmatic dependent launch of the decode and tensor-core kernels
// (qgemm_set_dependent_launch).
bool dependent_launch_enabled();
qg_status read_device_status(int* out, int reset);
// A kernel whose one mbarrier wait (limit polls) must give up (QG_ERR_TIMEOUT).
qg_status launch_wait_selftest(uint32_t limit, cudaStream_t s);

// Up to kMultiMax products sharing x (same M, K, bits, group) in one decode launch.
constexpr int kMultiMax = 4;
qg_status launch_gemv_multi(const uint16_t* x, int M, int ldx, const qg_qweight* ws, int n, void* const* ys,
                            const int32_t* ldys, qg_ydtype yt, void* work, size_t work_bytes, cudaStream_t s);

// ---------------------------------------------------------------- tensor-core GEMM
size_t gemm_workspace_bytes(int M, const qg_qweight& w);
// convert_x = false: x is already in the workspace in fp16 (the later
// products of a fused call, after the first one converted it).
qg_status launch_gemm(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy,
                      qg_ydtype yt, void* ws, size_t ws_bytes, bool convert_x, cudaStream_t s);

// Tile-ordered copy of a quantized weight for the tensor-core kernel: for
// every 256-row tile and 64-wide K block, one contiguous block of the
// block's codes (word i of dequantization thread t = 2 * row + half at word
// i * 512 + t) followed by its group parameters (per row, for each group
// the block touches -- two at group 32, else one -- a 32-bit word fp16
// scale | zero-point << 16, or at 2 bits the 4 fp16 codebook entries),
// blocks in (row tile, K block) order.  Rows beyond N are zero.
constexpr int kTileRows = 256, kTileK = 64;
__host__ __device__ constexpr int tile_groups_per_block(int group) { return group == 32 ? 2 : 1; }
__host__ __device__ constexpr size_t tile_block_bytes(int bits, int group)
{
    return (size_t)2048 * bits + (size_t)256 * (bits == 2 ? 8 : 4) * tile_groups_per_block(group);
}
inline size_t tiles_bytes(const qg_qweight& w)
{
    return (size_t)ceil_div(w.N, kTileRows) * (size_t)(w.K / kTileK) * tile_block_bytes(w.bits, w.group);
}
qg_status launch_repack(const qg_qweight& w, void* tiles, cudaStream_t s);
// Tensor-core product over the tile-ordered copy (workspace: x in fp16, as
// gemm_workspace_bytes).
qg_status launch_gemm_tiles(const uint16_t* x, int M, int ldx, const qg_qweight& w, const void* tiles, void* y,
                            int ldy, qg_ydtype yt, void* ws, cudaStream_t s);

// ---------------------------------------------------------------- grouped MoE
constexpr int kMoeMaxExperts = 256;
constexpr int kMoeMaxProducts = 2;   // products sharing one routing per call (gate and up)
// n products over the same routing: experts[p * E + e] is expert e of
// product p, ys[p] its output.
size_t moe_workspace_bytes(int T, int k, int E, int n, const qg_qweight* experts);
qg_status launch_moe(const uint16_t* x, int T, const int32_t* topk, int k, const qg_qweight* experts,
                     int E, int n, void* const* ys, qg_ydtype yt, void* ws, size_t ws_bytes, cudaStream_t s);

// Grouped product on the tensor cores (4-bit, K a multiple of 64, at most 32
// experts over all n products): tokens of an expert in chunks of kMoeTcChunk; x16p is workspace
// for x gathered in routed order (moe_tc_x16_bytes).  Chunks of 64 tokens
// keep a token tile's K block at 8 KB, so the token ring holds ten of them;
// an expert with more tokens reads its weights once per chunk, mostly from
// L2 (the chunks' CTAs run together).
constexpr int kMoeTcChunk = 64;
bool moe_tc_eligible(const qg_qweight* experts, int E, int n);
size_t moe_tc_x16_bytes(int P, int K);
qg_status launch_moe_tc(const uint16_t* x, int T, int k, const qg_qweight* experts, int E, int n, void* const* ys,
                        qg_ydtype yt, const int* offsets, const int* perm, const int2* items, const int* n_items,
                        int max_items, void* x16p, cudaStream_t s);

// ---------------------------------------------------------------- W8A8 (int8 weights and activations)
constexpr int kW8A8MaxM = 16;
size_t w8a8_workspace_bytes(int M, int K);
qg_status launch_w8a8(const uint16_t* x, int M, int ldx, const qg_qweight& w, void* y, int ldy, qg_ydtype yt,
                      void* ws, cudaStream_t s);

// ---------------------------------------------------------------- diagnostics
size_t diag_workspace_bytes(int N, int K, int group);
qg_status launch_diag(const uint16_t* W, const qg_qweight& w, float threshold, float* ratio, qg_diag* out, void* ws,
                      cudaStream_t s);

}  // namespace qg
