/*
 * qgemm.h -- C ABI of the fused-dequantization linear layer for weight-only,
 * group-wise, asymmetric low-bit weights, built for NVIDIA GB300 (sm_103a).
 *
 *     y = x . dequant(W)^T  (+ FP16 outliers added back)
 *
 * The method (from the pages this library follows):
 *  - affine asymmetric quantizer: scale = (max - min) / (qmax - qmin),
 *    zero_point = qmin - round(min / scale), q = round(w / scale) +
 *    zero_point, w_hat = (q - zero_point) * scale  ("Inference acceleration guide" page,
 *    section 1.1 "quantization is a lossy mapping");
 *  - statistics per group of consecutive weights along K (32, 64 or 128;
 *    the "Mixed-width quantization" page, section 2.3, pairs the narrow
 *    widths with blocks of 32 and the wide ones with 64 or 128), after
 *    excluding the largest-magnitude 0.1 % of weights, which are kept in FP16
 *    and added back after the product  ("70B on one GPU" page, section 2,
 *    "group-wise outlier-aware quantization", steps 1-3);
 *  - widths 2, 3, 4, 5, 6 bits, and 8 bits (a weight-only int8 path, the
 *    width the pages' GPU unpack targets: "Mixed-width quantization" page,
 *    section 4.2); 2-bit groups use a 4-entry non-uniform
 *    codebook found by k-means  ("Mixed-width quantization" page, section 2.1 table and 4.1);
 *  - codes packed LSB-first in a little-endian bit stream: 3-bit 8 values
 *    in 3 bytes, 5-bit 8 values in 5 bytes, 6-bit 4 values in 3 bytes,
 *    2-bit 4 values per byte, 4-bit two per byte with the even index in the
 *    low half  ("Mixed-width quantization" page, sections 3.1-3.2 and the 2.1 table);
 *  - unpacking happens on the computing device, fused into the product,
 *    with fp32 accumulation  ("Mixed-width quantization" page, sections 1.2 and 4.1-4.2;
 *    "70B on one GPU" page, section 3 "kernel fusion").
 *
 * Conventions shared by every entry point:
 *  - Every pointer in a qg_qweight, every x / y / topk_ids / W argument and
 *    the workspace are DEVICE memory owned by the caller.  The library never
 *    allocates, frees or retains them past the call.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *    enqueued on it; the calls never synchronize the stream or the device.
 *  - Arguments are validated on the host before anything is launched; a
 *    rejected call launches nothing and returns a negative qg_status.  No
 *    call throws.  qgemm_last_error() returns a human-readable message for
 *    the calling thread's last failure.
 *  - Inputs must not alias outputs.
 */
#ifndef QGEMM_H_
#define QGEMM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = -1,   /* a null pointer, a bad size, an out-of-range value */
    QG_ERR_UNSUPPORTED = -2,   /* valid in principle, not built (e.g. bits = 7) */
    QG_ERR_ALIGNMENT = -3,     /* a pointer or leading dimension is misaligned */
    QG_ERR_WORKSPACE = -4,     /* workspace missing or smaller than the size query */
    QG_ERR_CUDA = -5,          /* a CUDA runtime call or launch failed */
    QG_ERR_TIMEOUT = -6,       /* reserved: a bounded device-side wait gave up */
    QG_ERR_DEVICE_STATUS = -7  /* reserved: a device-side check reported an error */
} qg_status;

typedef enum { QG_Y_F32 = 0, QG_Y_BF16 = 1 } qg_ydtype;

/*
 * A quantized weight matrix W [N, K] in the planar layout (codes in one
 * array, per-group parameters in others; "Mixed-width quantization" page, section 3.3).
 *
 *  N, K        output and input features.  K % group == 0.
 *  bits        2, 3, 4, 5, 6 or 8 (8: one byte per code).
 *  group       32, 64 or 128 consecutive weights along K share a scale/zp
 *              (or, at 2 bits, a codebook).  ng = K / group.
 *  packed      uint8 [N, K*bits/8], row-major; row n holds the K codes of
 *              row n as one LSB-first stream.  16-byte aligned.
 *  scale       fp16 [N, ng]  (bits != 2; NULL at 2 bits).  2-byte aligned.
 *  zp          uint8 [N, ng] (bits != 2; NULL at 2 bits).
 *  codebook    fp16 [N, ng, 4], ascending per group (bits == 2; NULL
 *              otherwise).  8-byte aligned.
 *  nnz         number of FP16 outliers = floor(outlier_frac * N * K).
 *  out_row_ptr int32 [N+1] CSR row pointer (may be NULL when nnz == 0).
 *  out_col     int32 [nnz] column of each outlier, ascending within a row.
 *  out_val     fp16 [nnz]  the value added back at (row, col): the weight
 *              itself (bits 3..8) or the residual w - codebook entry (2 bits).
 *
 * Optional 8-bit float group scales with an fp16 fallback ("Mixed-width
 * quantization" page, section 2.3: the scale stored as an 8-bit float,
 * groups whose scale the 8-bit format cannot hold kept at fp16).  When
 * scale8 is not NULL (bits 3..8) it replaces `scale`, which may be NULL:
 *  scale8      uint8 [N, ng]: the E4M3 code (1 sign, 4 exponent bits with
 *              bias 7, 3 fraction bits; only positive normal codes 0x08 ..
 *              0x7E occur) of the group's scale times 2^-E, or 0x7F: the
 *              group keeps an fp16 scale, found in the fallback list.  The
 *              group's scale is then code value * 2^E, an fp16 number.
 *  scale8_exp  int32 [1]: the matrix exponent E (written by the quantizer).
 *              4-byte aligned.
 *  fb_row_ptr  int32 [N+1] the fallback list's CSR row pointer.
 *  fb_col      int32 [fb_cap] group index j of each fallback group,
 *              ascending within a row.
 *  fb_val      fp16 [fb_cap] that group's fp16 scale.
 *  fb_cap      capacity of fb_col / fb_val (entries); the quantizer reports
 *              more fallback groups than that through the device status
 *              word (QG_ERR_WORKSPACE, see qgemm_device_status).
 */
typedef struct {
    int32_t N, K, bits, group;
    uint8_t* packed;
    uint16_t* scale;
    uint8_t* zp;
    uint16_t* codebook;
    int32_t nnz;
    int32_t* out_row_ptr;
    int32_t* out_col;
    uint16_t* out_val;
    uint8_t* scale8;
    int32_t* scale8_exp;
    int32_t* fb_row_ptr;
    int32_t* fb_col;
    uint16_t* fb_val;
    int32_t fb_cap;
} qg_qweight;

/*
 * Bytes of every buffer of a quantized [N, K] matrix.  Host-only, no GPU.
 * nnz = floor(outlier_frac * N * K) evaluated in double; the outlier arrays
 * take (N+1)*4 + nnz*4 + nnz*2 bytes.  Any output pointer may be NULL.
 * Effective bits per weight = bits + 24/group (fp16 scale + u8 zp) or
 * 2 + 64/group (2-bit codebook of 4 fp16 entries); "Mixed-width quantization" page, section 2.3
 * gives the same accounting for the scale overhead.
 * Errors: QG_ERR_INVALID_ARG for N, K <= 0, K % group, outlier_frac outside
 * [0, 1); QG_ERR_UNSUPPORTED for bits outside {2..6, 8} or group not 32/64/128.
 */
QG_API qg_status qpack_query_sizes(int32_t N, int32_t K, int32_t bits, int32_t group, float outlier_frac,
                            size_t* packed_bytes, size_t* scale_bytes, size_t* zp_bytes,
                            size_t* codebook_bytes, int32_t* nnz);

/* Workspace bytes qpack_quantize needs for an [N, K] matrix.  Host-only. */
QG_API qg_status qpack_workspace_size(int32_t N, int32_t K, size_t* bytes);

/*
 * Quantize and pack W [N, K] (fp16, row-major, DEVICE, 16-byte aligned, all
 * values finite) into the buffers of `out`, whose N, K, bits, group and nnz
 * the caller fills (nnz from qpack_query_sizes) and whose pointers the
 * caller allocates.  Steps ("70B on one GPU" page, section 2; "Inference acceleration guide"
 * page, section 1.1; "Mixed-width quantization" page, sections 3-4):
 *   1. outliers: the nnz largest |w| of the whole matrix (ties: lower
 *      linear index n*K + k), stored as CSR, columns ascending;
 *   2. per (row, group): min/max over the non-outliers with 0 included;
 *      bits 3..6: scale = fp16 rounded up of (max-min)/(2^bits - 1) (1.0 if
 *      max == min), zp = clamp(-rint(min/scale), 0, 2^bits-1),
 *      q = clamp(rint(w/scale) + zp, 0, 2^bits - 1), q = zp at outliers;
 *      bits 2: 16 Lloyd iterations from 4 evenly spaced levels, entries
 *      rounded to fp16 and sorted, q = nearest entry (ties: lower index),
 *      the entry nearest 0 at an outlier, whose stored value becomes the
 *      residual fp16(w - entry);
 *   3. codes packed LSB-first along K.
 * All rounding is IEEE round-to-nearest-even except the scale (toward +inf);
 * the results are bit-exact and deterministic.
 * With out->scale8 set (bits 3..8), step 2 stores 8-bit scales: the fp16
 * scale s16 of every group is found as above; E = the lower median of
 * floor(log2 s16) over all N * ng groups; a group's code is the least normal
 * E4M3 value >= s16 * 2^-E; the group falls back (code 0x7F, s16 in the
 * fallback list) when s16 * 2^-E < 2^-6, when that value would exceed 448,
 * or when value * 2^E is not a normal fp16 number; zp and q are then
 * computed with the group's stored scale.  When more groups fall back than
 * out->fb_cap, the first fb_cap are listed, fb_row_ptr still counts all of
 * them, and the device status word becomes QG_ERR_WORKSPACE: the weight must
 * not be used.
 * `ws` must hold qpack_workspace_size bytes (256-byte aligned).  Errors:
 * QG_ERR_INVALID_ARG (nulls, sizes, nnz mismatch), QG_ERR_ALIGNMENT,
 * QG_ERR_WORKSPACE, QG_ERR_CUDA.  Non-finite W gives unspecified output.
 */
QG_API qg_status qpack_quantize(const uint16_t* W, float outlier_frac, const qg_qweight* out, void* ws,
                         size_t ws_bytes, void* stream);

/* Quantizer variants ("Mixed-width quantization" page, sections 2.3 and
 * 4.1-4.2), all stored in the formats above, so every product entry point
 * takes them unchanged:
 *  QG_QUANT_ASYMMETRIC  qpack_quantize's quantizer (affine with a zero point
 *                       at 3..6 bits, a 4-entry k-means codebook at 2 bits).
 *  QG_QUANT_SYMMETRIC   no zero point (section 2.3 prefers it for the narrow
 *                       widths): with qs = 2^(bits-1) - 1 (the symmetric
 *                       integer range of the inference-acceleration guide
 *                       page's INT8 example, section 1.1, [-qs, qs]) and amax
 *                       the group's largest |w| over its non-outliers,
 *                       scale = fp16 rounded up of amax / qs (1.0 if amax is
 *                       0), q = clamp(round(w / scale), -qs, qs).  Widths
 *                       3..6: stored as codes q + 2^(bits-1) with the zero
 *                       point fixed at 2^(bits-1).  2 bits: levels -s, 0, s
 *                       stored as the constants (-s, 0, s, s), codes q + 1.
 *  QG_QUANT_LINEAR2     2 bits only: the affine grid (qpack_quantize's
 *                       formula at qmax = 3) stored as its four constants
 *                       fp16((i - zp) * scale), i = 0..3, which the code
 *                       selects (section 4.2: a linear 2-bit grid maps codes
 *                       to four constants, no k-means codebook).
 * In every mode the constant or grid point of the zero code is exactly 0,
 * outliers take that code, and their stored value is the weight itself. */
typedef enum { QG_QUANT_ASYMMETRIC = 0, QG_QUANT_SYMMETRIC = 1, QG_QUANT_LINEAR2 = 2 } qg_quant_mode;

/* qpack_quantize with a quantizer variant.  Arguments, workspace, results
 * and errors as qpack_quantize, plus QG_ERR_INVALID_ARG for an unknown mode
 * and QG_ERR_UNSUPPORTED for QG_QUANT_LINEAR2 at bits != 2. */
QG_API qg_status qpack_quantize_mode(const uint16_t* W, float outlier_frac, qg_quant_mode mode,
                                     const qg_qweight* out, void* ws, size_t ws_bytes, void* stream);

/*
 * qpack_quantize without a workspace argument, for callers that cannot
 * allocate device memory when they quantize: code inside a host application
 * that owns the device allocator (a plugin, a server that reserves its memory
 * pool up front), code where cudaMalloc's implicit device synchronization is
 * not acceptable, or code running after a fixed memory budget is frozen.
 * The pages have no counterpart to this entry point; it exists for such
 * callers only.  Same operation, arguments and results as qpack_quantize
 * (bit-identical output).
 *  - Scratch: a fixed 1 MiB array in the library's own device memory, held
 *    by every GPU that loads the library until the process exits.  Only the
 *    outlier selection uses it: without outliers (outlier_frac = 0) any size
 *    is accepted; with outliers, matrices whose scratch need
 *    (qpack_workspace_size) exceeds it -- more than about 76,000 rows -- are
 *    rejected with QG_ERR_WORKSPACE before anything runs.
 *  - Argument checks and their status codes are exactly qpack_quantize's.
 *  - The first call with outliers on each device looks up the array's
 *    device address (cudaGetSymbolAddress, with that device current) and
 *    caches it for that device's current context; make that first call
 *    before any stream capture.  A context created anew (after
 *    cudaDeviceReset) gets a new lookup on its first such call.
 *  - Every call shares the array and it keeps the last call's contents; each
 *    call clears what must start at zero.  Calls that overlap on the GPU
 *    (e.g. on two unordered streams) race on the array: order them.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
QG_API qg_status qpack_quantize_noalloc(const uint16_t* W, float outlier_frac, const qg_qweight* out,
                                        void* stream);

/* Workspace bytes qgemm_forward needs for M rows of x against w.  Host-only. */
QG_API qg_status qgemm_workspace_size(int32_t M, const qg_qweight* w, size_t* bytes);

/*
 * y[m, n] = sum_k x[m, k] * (w_hat[n, k] + S[n, k])   for m < M, n < N,
 * with w_hat the dequantized weight and S the FP16 outliers ("70B on one GPU"
 * page, sections 2-3).  Dequantization happens in registers / on-chip
 * memory inside the product; accumulation is fp32.
 *   x   bf16 [M, K] row-major with row stride ldx >= K elements (DEVICE).
 *   y   [M, N] row-major with row stride ldy >= N elements, fp32 or bf16
 *       per `yt` (DEVICE).
 * M = 0 is a no-op.  M <= 16 runs the decode kernel (register dequant, split
 * K across a thread-block cluster); larger M runs the tensor-core kernel
 * (tcgen05 with TMEM accumulators), which converts x to fp16 in the workspace;
 * up to M = 256 it also splits K over several CTAs per tile, whose partial
 * tiles (in the workspace) a second small kernel sums in a fixed order.
 * From M = 8 the decode call also uses the workspace: x is converted once
 * into the fp16 fragment order the kernel stages (2 * K * Mpad bytes, Mpad
 * 8 or 16), and every CTA copies its blocks of it; with no or a
 * smaller workspace each CTA converts its own blocks instead, with the same
 * result, more slowly.  `ws` may be NULL when qgemm_workspace_size reports 0.
 * |x| must stay below 65520: x is converted to fp16 on every path.
 * Ordering: the product's kernels are launched with programmatic dependent
 * launch, so a product may start, and read the weight buffers (packed,
 * scale, zp, codebook, outlier CSR, 8-bit scale arrays), before the kernel
 * launched just before it on the same stream has finished; it reads x and
 * writes y and the workspace only after that kernel has completed.
 * The kernel launched immediately before qgemm_forward on the stream must
 * therefore not write w's buffers (qpack_quantize ends with an empty kernel,
 * and copies are not kernels, so quantizing or uploading on the same stream
 * just before is safe).
 * Errors: QG_ERR_INVALID_ARG, QG_ERR_ALIGNMENT, QG_ERR_WORKSPACE, QG_ERR_CUDA.
 */
QG_API qg_status qgemm_forward(const uint16_t* x, int32_t M, int32_t ldx, const qg_qweight* w, void* y,
                        int32_t ldy, qg_ydtype yt, void* ws, size_t ws_bytes, void* stream);

/*
 * Several products that share one input in one call (a fused projection,
 * e.g. the q, k and v, or the gate and up, matrices of a transformer layer):
 *     ys[q][m, n] = sum_k x[m, k] * (w_hat_q[n, k] + S_q[n, k])   for q < n.
 * The pages define the single product ("70B on one GPU" page, sections
 * 2-3); this call computes exactly that product for each weight, so each
 * ys[q] equals what qgemm_forward would write for ws[q].  In the decode range
 * (M <= 16) all n products run as one kernel launch over their concatenated
 * row tiles; above it they run one after the other on the tensor cores in
 * the caller's workspace (size: the largest qgemm_workspace_size of the ws),
 * with x converted to fp16 once for all of them.
 *   x     bf16 [M, K], row stride ldx >= K (DEVICE), shared by all products.
 *   ws    host array of n descriptors, 1 <= n <= 4, same K, bits and group.
 *   ys    host array of n DEVICE pointers, ys[q] [M, ws[q].N] with row stride
 *         ldys[q] >= ws[q].N (host array), fp32 or bf16 per `yt`.
 * Ordering as for qgemm_forward.
 * Errors: QG_ERR_INVALID_ARG, QG_ERR_ALIGNMENT, QG_ERR_WORKSPACE, QG_ERR_CUDA.
 */
QG_API qg_status qgemm_forward_multi(const uint16_t* x, int32_t M, int32_t ldx, const qg_qweight* ws, int32_t n,
                                     void* const* ys, const int32_t* ldys, qg_ydtype yt, void* work,
                                     size_t work_bytes, void* stream);

/*
 * One-time device repack into the tile-ordered layout the tensor-core
 * (prefill) kernel streams ("Mixed-width quantization" page, sections 3.1
 * and 3.3: codes laid out for aligned vector access, the scales next to the
 * codes they scale -- misalignment costs 5-15 %, cache-line-aligned scales
 * gain about 8 %; "70B on one GPU" page, section 3: the weights are
 * repacked once, when the model is loaded, for the fused kernel).
 * Layout: for every 256-row tile (rows n0 .. n0+255) and 64-wide K block kb,
 * one contiguous block of tile_block_bytes = 2048*bits + 256*P*G bytes
 * (P = 8 at 2 bits, else 4; G = 2 at group 32, else 1), at byte
 * (tile * (K/64) + kb) * tile_block_bytes:
 *   words [0, 512*bits): word i of thread t = 2*r + h at word i*512 + t,
 *     where the thread's chunk is the 32 codes [64 kb + 32 h, 64 kb + 32 h +
 *     32) of row n0 + r as 4*bits bytes of the planar LSB-first stream;
 *   then per row r, for each of the G groups the block touches (in K
 *     order): one 32-bit word fp16 scale | zero-point << 16 (bits != 2), or
 *     the group's 4 fp16 codebook entries (8 bytes, bits == 2).
 * Rows beyond N are zero.  Every block starts on a 128-byte boundary, so
 * the kernel stages one block with one bulk copy and reads codes and
 * parameters from shared memory.  The outlier CSR stays in the descriptor.
 */
QG_API qg_status qrepack_tiles_size(const qg_qweight* w, size_t* bytes);
/* Writes the tile-ordered copy of w into `tiles` (DEVICE, 128-byte aligned,
 * at least qrepack_tiles_size bytes), stream-ordered.  w is unchanged.
 * Errors: QG_ERR_INVALID_ARG, QG_ERR_ALIGNMENT, QG_ERR_CUDA. */
QG_API qg_status qrepack_tiles(const qg_qweight* w, void* tiles, size_t tiles_bytes, void* stream);
/* Workspace bytes qgemm_forward_tiles needs for M rows of x.  Host-only. */
QG_API qg_status qgemm_tiles_workspace_size(int32_t M, const qg_qweight* w, size_t* bytes);
/* qgemm_forward on the tensor cores with the codes and group parameters
 * read from the tile-ordered copy `tiles` of w (made by qrepack_tiles from
 * the same w); w supplies the shape, the scales (for the per-row operand
 * exponent) and the outlier CSR.  Any M >= 1 (every M runs the tensor-core
 * kernel).  Same result as qgemm_forward's tensor-core path, bit for bit.
 * Ordering as for qgemm_forward (the kernel launched just before must not
 * write w's buffers or `tiles`; qrepack_tiles is safe).
 * Errors: QG_ERR_INVALID_ARG, QG_ERR_ALIGNMENT, QG_ERR_WORKSPACE, QG_ERR_CUDA. */
QG_API qg_status qgemm_forward_tiles(const uint16_t* x, int32_t M, int32_t ldx, const qg_qweight* w,
                                     const void* tiles, void* y, int32_t ldy, qg_ydtype yt, void* ws,
                                     size_t ws_bytes, void* stream);

/*
 * W8A8 product for decode (M <= 16): int8 weights (bits = 8, affine or
 * symmetric format, FP16 outliers as usual) and int8 activations quantized
 * dynamically per token inside the call ("Inference acceleration guide"
 * page, section 1.2: W8A8 quantizes weights and activations to INT8, the
 * activations per token; section 1.1: the symmetric range [-127, 127]):
 *   s_m = max_k |x[m,k]| / 127 (fp32; 1 if the maximum is 0),
 *   q[m,k] = clamp(round(x[m,k] / s_m), -127, 127)  (fp32 division, round half
 *   to even),
 *   y[m, n] = sum_k (q[m,k] s_m) * (w_hat[n,k] + S[n,k]).
 * Integer sums are exact (32-bit four-way int8 dot products on the CUDA
 * cores: GB300's int8 tensor-core rate is far below its fp16 rate), scales
 * and outliers are applied in fp32.  x, y, ldx, ldy, yt as qgemm_forward;
 * `ws` at least qgemm_w8a8_workspace_size bytes (q and s_m), 256-byte aligned.
 * Errors: QG_ERR_UNSUPPORTED (bits != 8, M > 16), QG_ERR_INVALID_ARG,
 * QG_ERR_ALIGNMENT, QG_ERR_WORKSPACE, QG_ERR_CUDA.
 */
QG_API qg_status qgemm_w8a8_workspace_size(int32_t M, const qg_qweight* w, size_t* bytes);
QG_API qg_status qgemm_forward_w8a8(const uint16_t* x, int32_t M, int32_t ldx, const qg_qweight* w, void* y,
                                    int32_t ldy, qg_ydtype yt, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes qgemm_moe_grouped (and qgemm_moe_grouped_multi with the
 * same T, k, E and experts[0 .. E-1]) needs.  Host-only. */
QG_API qg_status qgemm_moe_workspace_size(int32_t T, int32_t k, int32_t E, const qg_qweight* experts,
                                   size_t* bytes);

/*
 * Grouped product over top-k routed experts ("On-device MoE" page,
 * sections 1-2: each token activates its top-k of the experts):
 *   y[t, j, :] = x[t, :] . (w_hat + S)_{e}^T   with e = topk_ids[t, j],
 * for t < T, j < k.  No gate weights are applied.
 *   x         bf16 [T, K] row-major, contiguous (DEVICE).
 *   topk_ids  int32 [T, k] expert ids in [0, E) (DEVICE).
 *   experts   HOST array of E descriptors; all share N, K, bits and group.
 *   y         [T, k, N] contiguous, fp32 or bf16 per `yt` (DEVICE).
 * Routing (a counting sort of the T*k pairs by expert) runs on the device.
 * Ids outside [0, E) are skipped (their y rows are left untouched).
 * E <= 256.  Errors: QG_ERR_INVALID_ARG, QG_ERR_ALIGNMENT, QG_ERR_WORKSPACE,
 * QG_ERR_CUDA.
 */
QG_API qg_status qgemm_moe_grouped(const uint16_t* x, int32_t T, const int32_t* topk_ids, int32_t k,
                            const qg_qweight* experts, int32_t E, void* y, qg_ydtype yt, void* ws,
                            size_t ws_bytes, void* stream);

/*
 * n grouped products over one routing: products that read the same routed x
 * (an MoE layer's gate and up projections) share the routing, the gathered
 * x and one launch.  For each product p < n:
 *   y_p[t, j, :] = x[t, :] . (w_hat + S)_{p, e}^T   with e = topk_ids[t, j],
 * exactly as qgemm_moe_grouped computes it for experts[p * E .. p * E + E - 1].
 *   experts   HOST array of n * E descriptors (product p's experts at
 *             p * E .. p * E + E - 1); all share N, K, bits and group.
 *   n         1 <= n <= 2.
 *   ys        HOST array of n DEVICE pointers, each [T, k, N] contiguous, fp32
 *             or bf16 per `yt`.
 *   ws        at least qgemm_moe_workspace_size(T, k, E, experts) bytes.
 * Other arguments, ordering and errors as for qgemm_moe_grouped.
 */
QG_API qg_status qgemm_moe_grouped_multi(const uint16_t* x, int32_t T, const int32_t* topk_ids, int32_t k,
                                         const qg_qweight* experts, int32_t E, int32_t n, void* const* ys,
                                         qg_ydtype yt, void* ws, size_t ws_bytes, void* stream);

/* Status word of the library's kernels on the current device: QG_OK, or
 * QG_ERR_TIMEOUT once a bounded wait of the tensor-core product (M above the
 * decode range) on its shared-memory rings gave up (the kernel then finished
 * without hanging, and the outputs of that call are not valid).  The pages define no such call; it exists because
 * the kernels never trap or spin without a limit.
 *   status  host int32: receives the word.
 *   reset   non-zero: clear the word after reading it.
 * Synchronous: waits for the device (cudaMemcpy), so it is a check between
 * steps, not a call for the hot path.  Returns QG_ERR_INVALID_ARG if status
 * is NULL and QG_ERR_CUDA if the device cannot be read. */
QG_API qg_status qgemm_device_status(int32_t* status, int32_t reset);

/*
 * Programmatic dependent launch of the dense products (decode and
 * tensor-core kernels, with their x conversion and split-K sum), process-wide
 * (default on).  On, a product may start, and read its weight buffers,
 * before the kernel launched just before it on the stream has finished (see
 * qgemm_forward's ordering note).  enable = 0 turns this off for every later
 * call: each kernel then starts only after the previous kernel on its
 * stream has finished, so the product may follow a kernel that writes its
 * weights (a device-side copy or repack of them).  The results are the same
 * either way.  Host-only; never fails.
 */
QG_API qg_status qgemm_set_dependent_launch(int32_t enable);

/*
 * Diagnostics of one quantized layer against its original weights
 * ("Mixed-width quantization" page, section 6.1: unpack the quantized weights
 * and compare them element by element with the original fp16 weights --
 * maximum absolute error, root mean square error, cosine similarity --
 * section 6.2: a block whose largest value is far above its second largest
 * holds one extreme value that stretches its scale).  Over all N*K elements,
 * e = w - (w_hat + S) (the FP16 outliers are part of the layer's weight):
 */
typedef struct {
    double max_abs_err;      /* max |e| */
    double rmse;             /* sqrt(sum e^2 / (N*K)) */
    double cosine;           /* sum w*v / (|w| |v|), v = w_hat + S; 1 if both are 0, 0 if one is */
    double max_range_ratio;  /* largest group ratio (see group_ratio) */
    int64_t groups_over;     /* groups whose ratio exceeds the threshold */
} qg_diag;

/* Workspace bytes qdiag_layer needs (one partial per 128 groups).  Host-only.
 * Errors: QG_ERR_INVALID_ARG / QG_ERR_UNSUPPORTED as qpack_query_sizes. */
QG_API qg_status qdiag_workspace_size(int32_t N, int32_t K, int32_t group, size_t* bytes);

/*
 *   W            fp16 [N, K] the original weights (DEVICE, 16-byte aligned).
 *   w            the quantized layer (any width, group, outliers).
 *   threshold    groups with ratio > threshold are counted in groups_over.
 *   group_ratio  DEVICE fp32 [N, K/group] or NULL: per group, its largest
 *                |w| over its second largest |w| (magnitudes counted with
 *                multiplicity): 1 for an all-zero group, +inf when exactly
 *                one element is nonzero.
 *   out          DEVICE pointer to one qg_diag (8-byte aligned), written by
 *                the call's last kernel; read it after the stream reaches it.
 * Sums are fp32 within a group and fp64 across groups, reduced in a fixed
 * order (deterministic).  Errors: QG_ERR_INVALID_ARG, QG_ERR_ALIGNMENT,
 * QG_ERR_WORKSPACE, QG_ERR_CUDA.
 */
QG_API qg_status qdiag_layer(const uint16_t* W, const qg_qweight* w, float threshold, float* group_ratio,
                             qg_diag* out, void* ws, size_t ws_bytes, void* stream);

/* Self-check of the failure path of the bounded waits: launches one small
 * kernel on `stream` whose single mbarrier wait (at most poll_limit polls,
 * each suspending up to 0.1 ms) has nothing to wait for and gives up, so the
 * kernel sets the status word to QG_ERR_TIMEOUT and returns, exactly as a
 * tensor-core kernel does when one of its waits runs out.  It issues no TMA
 * and no MMA.  Read the result with qgemm_device_status (which also clears
 * it).  The pages define no such call; it exists so that this path can be
 * exercised without breaking a product kernel.
 *   poll_limit  1 .. 64.
 * Errors: QG_ERR_INVALID_ARG, QG_ERR_CUDA. */
QG_API qg_status qgemm_selftest_bounded_wait(int32_t poll_limit, void* stream);

/* Message describing the calling thread's most recent failure ("" if none). */
QG_API const char* qgemm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H_ */
