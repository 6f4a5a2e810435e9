// wquant.cu -- weight storage as int8 or int4 codes with one scale per
// channel, and its dequantization.
//
// "Precision" manual (docs.presk-lang.org/presk_manual/precision), section
// "Integer weights": a K x N weight contracted over K keeps one scale per
// column j,
//   s_j = max_k |W[k][j]| / (2^(b-1) - 1) rounded to f32 (b = 8 or 4),
// or, with the "pow2" scheme, that scale rounded up to a power of two (so
// that q * s is exact); an all-zero column gets s = 0 and stores zeros; the
// codes are q = w / s rounded to nearest, and a stored weight means f32(q*s).
// Readings where the page is open: "round to nearest" is IEEE's (the integer
// nearest the exact quotient, ties to even); a column whose scale rounds to
// zero is stored like an all-zero one; "up to a power of two" is the smallest
// power of two >= the scale; int4 codes are 4-bit two's complement packed two
// to a byte along each row (column 2i in bits 0-3 of byte i, 2i+1 in bits
// 4-7, the high nibble of a last odd column zero).
//
// One CTA per strip of 32 columns reads the strip twice: once for the column
// maxima, once (from L2) to quantize.  The quotient is taken in f64 and
// rounded to an integer with ties to even: its f64 rounding error (2^-53
// relative) is far below the distance (~2^-25 relative) at which an f32
// quotient that is not exactly k + 1/2 can lie from k + 1/2, so the integer
// is the one nearest the exact quotient.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsg_internal.h"

namespace bsg {
namespace {

constexpr int kWStrip = 32;

__device__ __forceinline__ uint32_t wq_absbits(float x) { return __float_as_uint(x) & 0x7fffffffu; }

// The smallest power of two >= s (s >= 0, finite); 0 stays 0.
__device__ __forceinline__ float wq_pow2_up(float s) {
    uint32_t b = __float_as_uint(s);
    if (b == 0) return 0.0f;
    if (b >= 0x00800000u) {                       // normal
        if (b & 0x007fffffu) b = (b & 0x7f800000u) + 0x00800000u;
        return __uint_as_float(b);
    }
    uint32_t p = 1;                               // subnormal: a power of two of its bits
    while (p < b) p <<= 1;
    return __uint_as_float(p);
}

template <int BITS, bool POW2>
__global__ void __launch_bounds__(256)
    wquant_cols_kernel(const float *__restrict__ W, int64_t K, int64_t N, int64_t ldw,
                       uint8_t *__restrict__ Q, int64_t ldq, float *__restrict__ scale,
                       int32_t *__restrict__ dstatus) {
    constexpr float kQmax = BITS == 8 ? 127.0f : 7.0f;
    __shared__ uint32_t red[32][33];
    __shared__ float s_col[kWStrip];
    __shared__ int s_bad;
    const int t = threadIdx.x;
    const int c4 = t & 7, rs = t >> 3;
    const int64_t col = (int64_t)blockIdx.x * kWStrip + 4 * c4;
    auto load = [&](int64_t r, int u) -> float {
        return col + u < N ? __ldg(W + r * ldw + col + u) : 0.0f;
    };
    if (t == 0) s_bad = 0;
    uint32_t m[4] = {0u, 0u, 0u, 0u};  // |x| bit patterns: NaN left out, Inf kept
    bool bad = false;
    for (int64_t r = rs; r < K; r += 32) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t a = wq_absbits(load(r, u));
            if (a <= 0x7f800000u) m[u] = max(m[u], a);
            bad = bad || a >= 0x7f800000u;
        }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) red[rs][4 * c4 + u] = m[u];
    __syncthreads();
    if (bad) s_bad = 1;
    if (t < kWStrip) {
        uint32_t mm = 0;
        for (int i = 0; i < 32; ++i) mm = max(mm, red[i][t]);
        const int64_t j = (int64_t)blockIdx.x * kWStrip + t;
        float s = __fdiv_rn(__uint_as_float(mm), kQmax);
        if (POW2 && isfinite(s)) s = wq_pow2_up(s);
        s_col[t] = s;
        if (j < N) scale[j] = s;
    }
    __syncthreads();
    if (t == 0 && s_bad && dstatus) atomicOr(dstatus, 1);  // Inf or NaN in this strip
    float sv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) sv[u] = s_col[4 * c4 + u];
    for (int64_t r = rs; r < K; r += 32) {
        int q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float w = load(r, u);
            int v = 0;
            if (sv[u] != 0.0f && isfinite(sv[u]) && isfinite(w))
                v = __double2int_rn(__ddiv_rn((double)w, (double)sv[u]));
            q[u] = v < -(int)kQmax ? -(int)kQmax : (v > (int)kQmax ? (int)kQmax : v);
        }
        uint8_t *row = Q + r * ldq;
        if (BITS == 8) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (col + u < N) row[col + u] = (uint8_t)(int8_t)q[u];
        } else {
            // columns col..col+3 (col even) -> bytes col/2 and col/2 + 1
            if (col < N)
                row[col / 2] = (uint8_t)((q[0] & 0xf) | ((col + 1 < N ? q[1] & 0xf : 0) << 4));
            if (col + 2 < N)
                row[col / 2 + 1] = (uint8_t)((q[2] & 0xf) | ((col + 3 < N ? q[3] & 0xf : 0) << 4));
        }
    }
}

template <int BITS>
__global__ void wdequant_cols_kernel(const uint8_t *__restrict__ Q, int64_t K, int64_t N,
                                     int64_t ldq, const float *__restrict__ scale,
                                     float *__restrict__ out, int64_t ldo) {
    const int64_t total = K * N;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k = e / N, j = e - k * N;
        int q;
        if (BITS == 8) {
            q = (int8_t)Q[k * ldq + j];
        } else {
            const uint8_t byte = Q[k * ldq + j / 2];
            const int nib = (j & 1) ? (byte >> 4) : (byte & 0xf);
            q = nib >= 8 ? nib - 16 : nib;
        }
        out[k * ldo + j] = __fmul_rn((float)q, scale[j]);
    }
}

}  // namespace

cudaError_t launch_wquant_cols(const float *W, int64_t K, int64_t N, int64_t ldw, int bits,
                               int pow2, void *Q, int64_t ldq, float *scale, int32_t *dstatus,
                               cudaStream_t st) {
    const unsigned grid = (unsigned)((N + kWStrip - 1) / kWStrip);
    uint8_t *q = static_cast<uint8_t *>(Q);
    if (bits == 8 && !pow2)
        wquant_cols_kernel<8, false><<<grid, 256, 0, st>>>(W, K, N, ldw, q, ldq, scale, dstatus);
    else if (bits == 8)
        wquant_cols_kernel<8, true><<<grid, 256, 0, st>>>(W, K, N, ldw, q, ldq, scale, dstatus);
    else if (!pow2)
        wquant_cols_kernel<4, false><<<grid, 256, 0, st>>>(W, K, N, ldw, q, ldq, scale, dstatus);
    else
        wquant_cols_kernel<4, true><<<grid, 256, 0, st>>>(W, K, N, ldw, q, ldq, scale, dstatus);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_wdequant_cols(const void *Q, int64_t K, int64_t N, int64_t ldq, int bits,
                                 const float *scale, float *out, int64_t ldo, cudaStream_t st) {
    const int64_t blocks = (K * N + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const unsigned grid = (unsigned)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
    const uint8_t *q = static_cast<const uint8_t *>(Q);
    if (bits == 8)
        wdequant_cols_kernel<8><<<grid, 256, 0, st>>>(q, K, N, ldq, scale, out, ldo);
    else
        wdequant_cols_kernel<4><<<grid, 256, 0, st>>>(q, K, N, ldq, scale, out, ldo);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace bsg
