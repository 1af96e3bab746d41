// qgemv_cpu.cc -- the CPU baseline of the benchmark: a fused low-bit qGEMV
// (y = x . (w_hat + S)^T at M = 1) on all host cores.
//
// MEASUREMENT INFRASTRUCTURE: only the benchmark and its tests load this
// library.  It is neither the oracle (that is the plain fp64 definition) nor
// a fallback of the GPU library; it times the CPU method the pages describe
// so the GPU figures have a CPU figure beside them:
//  - unpack and multiply-accumulate in one loop, the unpacked value living
//    only in a register ("Mixed-width quantization" page, section 4.1), with
//    fp32 accumulation (section 4.2);
//  - the group scale factored out of the inner sum: per group
//    sum_k x_k (q_k - zp) = sum_k x_k q_k - zp * sum_k x_k is accumulated
//    first (sum_k x_k once per call, shared by every row) and multiplied by
//    the scale once (section 4.1); a group's codes are unpacked into a
//    128-float buffer that stays in L1, then dotted with x;
//  - rows split into contiguous blocks over std::thread workers, one per
//    hardware thread (std::thread::hardware_concurrency).
// Portable C++17 (no SIMD intrinsics; the compiler vectorizes what it can).
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// IEEE binary16 bit pattern -> float (from the format: 1 sign, 5 exponent
// bits with bias 15, 10 fraction bits).
float half_to_float(uint16_t h)
{
    const uint32_t s = (uint32_t)(h >> 15) << 31;
    const uint32_t e = (h >> 10) & 0x1F, m = h & 0x3FF;
    uint32_t bits;
    if (e == 0) {
        if (m == 0) {
            bits = s;
        } else {   // subnormal: m * 2^-24, renormalized
            int sh = 0;
            uint32_t mm = m;
            while (!(mm & 0x400)) { mm <<= 1; sh++; }
            bits = s | ((uint32_t)(127 - 15 - sh + 1) << 23) | ((mm & 0x3FF) << 13);
        }
    } else if (e == 31) {
        bits = s | 0x7F800000u | (m << 13);
    } else {
        bits = s | ((e + 112) << 23) | (m << 13);
    }
    float f;
    std::memcpy(&f, &bits, 4);
    return f;
}

struct Weight {
    int N, K, bits, group;
    const uint8_t* packed;
    const uint16_t* scale;
    const uint8_t* zp;
    const uint16_t* cb;
    const int32_t* row_ptr;
    const int32_t* col;
    const uint16_t* val;
    int nnz;
};

// Codes of one group -> float values q (exact small integers), written to a
// 128-entry buffer that stays in L1: a unit of 8 codes is `bits` bytes, code
// i at bit bits*i of the little-endian unit.
template <int BITS>
inline void unpack_group(const uint8_t* p, int g, float* q)
{
    if constexpr (BITS == 4) {
        for (int b = 0; b < g / 2; b++) {
            q[2 * b] = (float)(p[b] & 15u);
            q[2 * b + 1] = (float)(p[b] >> 4);
        }
    } else {
        for (int u = 0; u < g / 8; u++) {
            uint64_t v = 0;
            for (int i = 0; i < BITS; i++) v |= (uint64_t)p[u * BITS + i] << (8 * i);
            for (int i = 0; i < 8; i++) q[8 * u + i] = (float)((v >> (BITS * i)) & ((1u << BITS) - 1u));
        }
    }
}

inline float dot(const float* a, const float* b, int n)
{
    float s[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // eight partial sums: vectorizable
    for (int i = 0; i < n; i += 8)
        for (int j = 0; j < 8; j++) s[j] += a[i + j] * b[i + j];
    return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// One row, affine widths: per group sum x (q - zp) = sum x q - zp * sum x,
// with sum x of each group computed once per call (xsum), times the scale.
template <int BITS>
float row_affine(const Weight& w, const float* x, const float* xsum, int n)
{
    const int ng = w.K / w.group;
    const uint8_t* pr = w.packed + (size_t)n * w.K * BITS / 8;
    alignas(64) float q[128];
    float acc = 0.0f;
    for (int j = 0; j < ng; j++) {
        unpack_group<BITS>(pr + (size_t)j * w.group * BITS / 8, w.group, q);
        const float sq = dot(x + (size_t)j * w.group, q, w.group);
        const float zp = (float)w.zp[(size_t)n * ng + j];
        acc += half_to_float(w.scale[(size_t)n * ng + j]) * (sq - zp * xsum[j]);
    }
    return acc;
}

// One row, 2-bit codebook: the group's values are its fp16 entries.
float row_codebook(const Weight& w, const float* x, int n)
{
    const int ng = w.K / w.group;
    const uint8_t* pr = w.packed + (size_t)n * w.K / 4;
    alignas(64) float v[128];
    float acc = 0.0f;
    for (int j = 0; j < ng; j++) {
        const uint16_t* e = w.cb + ((size_t)n * ng + j) * 4;
        const float t[4] = {half_to_float(e[0]), half_to_float(e[1]), half_to_float(e[2]), half_to_float(e[3])};
        const uint8_t* pg = pr + (size_t)j * w.group / 4;
        for (int b = 0; b < w.group / 4; b++)
            for (int i = 0; i < 4; i++) v[4 * b + i] = t[(pg[b] >> (2 * i)) & 3u];
        acc += dot(x + (size_t)j * w.group, v, w.group);
    }
    return acc;
}

void rows(const Weight& w, const float* x, const float* xsum, float* y, int n0, int n1)
{
    for (int n = n0; n < n1; n++) {
        float v;
        switch (w.bits) {
            case 2: v = row_codebook(w, x, n); break;
            case 3: v = row_affine<3>(w, x, xsum, n); break;
            case 4: v = row_affine<4>(w, x, xsum, n); break;
            case 5: v = row_affine<5>(w, x, xsum, n); break;
            case 6: v = row_affine<6>(w, x, xsum, n); break;
            default: v = row_affine<8>(w, x, xsum, n); break;
        }
        if (w.nnz > 0)
            for (int p = w.row_ptr[n]; p < w.row_ptr[n + 1]; p++) v += x[w.col[p]] * half_to_float(w.val[p]);
        y[n] = v;
    }
}

}  // namespace

extern "C" {

int cpuq_hardware_concurrency(void)
{
    const unsigned c = std::thread::hardware_concurrency();
    return c ? (int)c : 1;
}

// y[n] = sum_k x[k] * (w_hat[n, k] + S[n, k]) for one token.  x is fp32 [K]
// (the bf16 input widened once by the caller); the weight arrays are the
// library's planar layout.  threads <= 0: one per hardware thread.  Returns
// the number of threads used, or -1 on bad arguments.
int cpuq_gemv(const float* x, int N, int K, int bits, int group, const uint8_t* packed, const uint16_t* scale,
              const uint8_t* zp, const uint16_t* cb, const int32_t* row_ptr, const int32_t* col,
              const uint16_t* val, int nnz, float* y, int threads)
{
    if (!x || !y || !packed || N <= 0 || K <= 0 || ((bits < 2 || bits > 6) && bits != 8) || (group != 64 && group != 128) ||
        K % group || (bits == 2 ? !cb : (!scale || !zp)) || (nnz > 0 && (!row_ptr || !col || !val)))
        return -1;
    const Weight w{N, K, bits, group, packed, scale, zp, cb, row_ptr, col, val, nnz};
    std::vector<float> xsum((size_t)(K / group));
    for (int j = 0; j < K / group; j++) {
        float s = 0.0f;
        for (int i = 0; i < group; i++) s += x[(size_t)j * group + i];
        xsum[j] = s;
    }
    const float* xs = xsum.data();
    int T = threads > 0 ? threads : cpuq_hardware_concurrency();
    if (T > N) T = N;
    std::vector<std::thread> pool;
    pool.reserve(T);
    for (int t = 0; t < T; t++) {
        const int n0 = (int)((long long)N * t / T), n1 = (int)((long long)N * (t + 1) / T);
        pool.emplace_back([&w, x, xs, y, n0, n1] { rows(w, x, xs, y, n0, n1); });
    }
    for (auto& th : pool) th.join();
    return T;
}

}  // extern "C"
