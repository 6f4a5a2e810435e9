// quantize.cu -- per-row and per-column absmax quantization to int8.
//
// "Verification -- why you can trust the numbers", section "The verified
// INT8 units", step 1: scale = max|row| / 127 floored at 1e-8, values to
// int8.  The scale is an IEEE f64 quotient rounded to f32 (the page derives
// scales in f64, which is exactly rounded), inv = f32(1 / f64(scale)), and
// q = floor(RN(RN(x * inv) + 0.5)) with two f32 roundings (section "Hardware
// ground truth"; a fused multiply-add is not used because it changes q just
// below x*inv = -1/2 and +1/2).
//
// Memory plan: rows are read once with 128-bit loads (the row stays in
// registers when it is short), absmax by a warp-shuffle max of |x| bit
// patterns (non-negative floats order like their bits; Inf/NaN show up as
// >= 0x7f800000).  Columns take a partial-max pass over row slices and a
// quantize pass over 64 x 64 tiles that also transposes for the GEMM.
#include <cuda_fp16.h>
#include <stdint.h>

#include "bsg_internal.h"

namespace bsg {
namespace {

constexpr uint32_t kNonfiniteBits = 0x7f800000u;
constexpr int kRowWarps = 8;  // rows per 256-thread block
constexpr int kRowRegVec = 8; // float4 per lane kept in registers: rows up to 1024

// Scale and reciprocal of one row or column from its absmax bit pattern.
__device__ __forceinline__ void scale_from_max(uint32_t mbits, float &scale, float &inv) {
    const double m = static_cast<double>(__uint_as_float(mbits));
    double s = __ddiv_rn(m, 127.0);
    if (s < 1e-8) s = 1e-8;
    scale = __double2float_rn(s);
    inv = __double2float_rn(__ddiv_rn(1.0, static_cast<double>(scale)));
}

// floor(RN(RN(x*inv) + 0.5)), clamped so that non-finite input (whose
// output is unspecified) cannot leave int8.
__device__ __forceinline__ float quant(float x, float inv) {
    const float f = floorf(__fadd_rn(__fmul_rn(x, inv), 0.5f));
    return fminf(fmaxf(f, -127.0f), 127.0f);
}

__device__ __forceinline__ uint32_t absbits(float x) { return __float_as_uint(x) & 0x7fffffffu; }

template <int OUT>
__device__ __forceinline__ void store4(void *Q, int64_t idx, float q0, float q1, float q2,
                                       float q3) {
    if (OUT == kOutInt8) {
        char4 c = make_char4((signed char)(int)q0, (signed char)(int)q1, (signed char)(int)q2,
                             (signed char)(int)q3);
        *reinterpret_cast<char4 *>(static_cast<int8_t *>(Q) + idx) = c;
    } else {
        __half2 a = __floats2half2_rn(q0, q1);
        __half2 b = __floats2half2_rn(q2, q3);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(static_cast<__half *>(Q) + idx) = u;
    }
}

template <int OUT>
__device__ __forceinline__ void store1(void *Q, int64_t idx, float q) {
    if (OUT == kOutInt8)
        static_cast<int8_t *>(Q)[idx] = (int8_t)(int)q;
    else
        static_cast<__half *>(Q)[idx] = __float2half_rn(q);
}

// One warp per row.  VEC: X rows and Q rows allow 16-byte (X) and 4/8-byte
// (Q) vector accesses.
template <int OUT, bool VEC>
__global__ void __launch_bounds__(kRowWarps * 32)
    quantize_rows_kernel(const float *__restrict__ X, int64_t rows, int64_t cols, int64_t ldx,
                         void *__restrict__ Q, int64_t ldq, float *__restrict__ scale,
                         float *__restrict__ inv, int32_t *__restrict__ dstatus) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_global = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5);
    const int64_t warp_stride = (int64_t)gridDim.x * kRowWarps;
    const int64_t c4n = VEC ? cols / 4 : 0;
    const bool in_regs = VEC && c4n <= 32 * kRowRegVec;

    for (int64_t r = warp_global; r < rows; r += warp_stride) {
        const float *xr = X + r * ldx;
        float4 v[kRowRegVec];
        uint32_t m = 0;
        if (VEC) {
            if (in_regs) {
#pragma unroll
                for (int i = 0; i < kRowRegVec; ++i) {
                    const int64_t c4 = lane + 32 * i;
                    if (c4 < c4n) {
                        v[i] = __ldcs(reinterpret_cast<const float4 *>(xr) + c4);
                        m = max(m, max(max(absbits(v[i].x), absbits(v[i].y)),
                                       max(absbits(v[i].z), absbits(v[i].w))));
                    }
                }
            } else {
                for (int64_t c4 = lane; c4 < c4n; c4 += 32) {
                    const float4 t = __ldg(reinterpret_cast<const float4 *>(xr) + c4);
                    m = max(m, max(max(absbits(t.x), absbits(t.y)), max(absbits(t.z), absbits(t.w))));
                }
            }
        }
        for (int64_t c = 4 * c4n + lane; c < cols; c += 32) m = max(m, absbits(__ldg(xr + c)));
        m = __reduce_max_sync(0xffffffffu, m);

        float sc = 0.f, iv = 0.f;
        if (lane == 0) {
            scale_from_max(m, sc, iv);
            scale[r] = sc;
            if (inv) inv[r] = iv;
            if (m >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
        }
        iv = __shfl_sync(0xffffffffu, iv, 0);

        const int64_t qrow = r * ldq;
        if (VEC) {
            if (in_regs) {
#pragma unroll
                for (int i = 0; i < kRowRegVec; ++i) {
                    const int64_t c4 = lane + 32 * i;
                    if (c4 < c4n)
                        store4<OUT>(Q, qrow + 4 * c4, quant(v[i].x, iv), quant(v[i].y, iv),
                                    quant(v[i].z, iv), quant(v[i].w, iv));
                }
            } else {
                for (int64_t c4 = lane; c4 < c4n; c4 += 32) {
                    const float4 t = __ldcs(reinterpret_cast<const float4 *>(xr) + c4);
                    store4<OUT>(Q, qrow + 4 * c4, quant(t.x, iv), quant(t.y, iv),
                                quant(t.z, iv), quant(t.w, iv));
                }
            }
        }
        for (int64_t c = 4 * c4n + lane; c < cols; c += 32)
            store1<OUT>(Q, qrow + c, quant(__ldg(xr + c), iv));
    }
}

// Partial column max over a slice of rows: block = 64 columns x 4 row lanes.
__global__ void __launch_bounds__(256)
    colmax_partial_kernel(const float *__restrict__ X, int64_t rows, int64_t cols, int64_t ldx,
                          int64_t rows_per_split, uint32_t *__restrict__ partial) {
    __shared__ uint32_t red[4][64];
    const int cc = threadIdx.x & 63;
    const int rg = threadIdx.x >> 6;
    const int64_t col = (int64_t)blockIdx.x * 64 + cc;
    const int64_t r0 = (int64_t)blockIdx.y * rows_per_split;
    const int64_t r1 = min(rows, r0 + rows_per_split);
    uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
    if (col < cols) {
        int64_t r = r0 + rg;
        for (; r + 12 < r1; r += 16) {
            m0 = max(m0, absbits(__ldg(X + r * ldx + col)));
            m1 = max(m1, absbits(__ldg(X + (r + 4) * ldx + col)));
            m2 = max(m2, absbits(__ldg(X + (r + 8) * ldx + col)));
            m3 = max(m3, absbits(__ldg(X + (r + 12) * ldx + col)));
        }
        for (; r < r1; r += 4) m0 = max(m0, absbits(__ldg(X + r * ldx + col)));
    }
    red[rg][cc] = max(max(m0, m1), max(m2, m3));
    __syncthreads();
    if (rg == 0 && col < cols)
        partial[(int64_t)blockIdx.y * cols + col] =
            max(max(red[0][cc], red[1][cc]), max(red[2][cc], red[3][cc]));
}

// Quantize a 64 x 64 tile of X with per-column scales (from the partial
// maxima).  kOutInt8 writes Q in X's layout; kOutHalfKMajor writes the
// transposed tile, Q[col][row], as f16.
template <int OUT>
__global__ void __launch_bounds__(256)
    quantize_cols_kernel(const float *__restrict__ X, int64_t rows, int64_t cols, int64_t ldx,
                         const uint32_t *__restrict__ partial, int nsplit, void *__restrict__ Q,
                         int64_t ldq, float *__restrict__ scale, float *__restrict__ inv,
                         int32_t *__restrict__ dstatus) {
    __shared__ float s_inv[64];
    __shared__ __align__(16) __half tile[64][64 + 8];
    const int t = threadIdx.x;
    const int64_t c0 = (int64_t)blockIdx.x * 64;
    const int64_t r0 = (int64_t)blockIdx.y * 64;
    if (t < 64) {
        const int64_t col = c0 + t;
        float iv = 0.f;
        if (col < cols) {
            uint32_t m = 0;
            for (int s = 0; s < nsplit; ++s) m = max(m, partial[(int64_t)s * cols + col]);
            float sc;
            scale_from_max(m, sc, iv);
            if (blockIdx.y == 0) {
                scale[col] = sc;
                if (inv) inv[col] = iv;
                if (m >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
            }
        }
        s_inv[t] = iv;
    }
    __syncthreads();
    const int cc = t & 63;
    const int rg = t >> 6;
    const int64_t col = c0 + cc;
    const float iv = s_inv[cc];
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
        const int rr = rg + 4 * i;
        const int64_t row = r0 + rr;
        const bool ok = row < rows && col < cols;
        const float q = ok ? quant(__ldg(X + row * ldx + col), iv) : 0.0f;
        if (OUT == kOutInt8) {
            if (ok) static_cast<int8_t *>(Q)[row * ldq + col] = (int8_t)(int)q;
        } else {
            tile[cc][rr] = __float2half_rn(q);
        }
    }
    if (OUT == kOutHalfKMajor) {
        __syncthreads();
        // 64 output rows (columns of X) x 64 halves (128 bytes) each.
        const int j = t >> 2;      // output row within the tile
        const int part = t & 3;    // 16 halves each
        const int64_t orow = c0 + j;
        if (orow < cols) {
            const uint4 *src = reinterpret_cast<const uint4 *>(&tile[j][part * 16]);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__half *>(Q) + orow * ldq + r0 +
                                                   part * 16);
            dst[0] = src[0];
            dst[1] = src[1];
        }
    }
}

__global__ void i8_rows_to_half_kernel(const int8_t *__restrict__ Q, int64_t rows, int64_t cols,
                                       int64_t ldq, __half *__restrict__ out, int64_t ldo) {
    const int64_t total = rows * cols;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / cols, c = e % cols;
        out[r * ldo + c] = __int2half_rn((int)Q[r * ldq + c]);
    }
}

// Q: rows x cols int8 -> out[c][r] f16 (64 x 64 tiles through shared memory).
__global__ void __launch_bounds__(256)
    i8_cols_to_half_kernel(const int8_t *__restrict__ Q, int64_t rows, int64_t cols, int64_t ldq,
                           __half *__restrict__ out, int64_t ldo) {
    __shared__ __half tile[64][64 + 2];
    const int t = threadIdx.x;
    const int64_t c0 = (int64_t)blockIdx.x * 64, r0 = (int64_t)blockIdx.y * 64;
    const int cc = t & 63, rg = t >> 6;
    for (int i = 0; i < 16; ++i) {
        const int rr = rg + 4 * i;
        const int64_t r = r0 + rr, c = c0 + cc;
        tile[cc][rr] = __int2half_rn((r < rows && c < cols) ? (int)Q[r * ldq + c] : 0);
    }
    __syncthreads();
    for (int i = 0; i < 16; ++i) {
        const int j = rg + 4 * i;       // output row (a column of Q)
        const int64_t orow = c0 + j, ocol = r0 + cc;
        if (orow < cols) out[orow * ldo + ocol] = tile[j][cc];
    }
}

}  // namespace

int colmax_nsplit(int64_t rows) {
    const int64_t s = (rows + 127) / 128;
    return (int)(s < 1 ? 1 : (s > 256 ? 256 : s));
}

size_t colmax_partial_bytes(int64_t rows, int64_t cols) {
    return (size_t)colmax_nsplit(rows) * (size_t)cols * sizeof(uint32_t);
}

static int grid_for(int64_t work, int per_block) {
    const int64_t b = (work + per_block - 1) / per_block;
    const int64_t cap = (int64_t)device_sm_count() * 32;
    return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

cudaError_t launch_quantize_rows(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                 int out_kind, void *Q, int64_t ldq, float *scale, float *inv,
                                 int32_t *dstatus, cudaStream_t st) {
    const int grid = grid_for(rows, kRowWarps);
    const size_t qalign = out_kind == kOutInt8 ? 4 : 8;
    const size_t qesz = out_kind == kOutInt8 ? 1 : 2;
    const bool vec = (ldx % 4 == 0) && (reinterpret_cast<uintptr_t>(X) % 16 == 0) &&
                     ((ldq * qesz) % qalign == 0) && (reinterpret_cast<uintptr_t>(Q) % qalign == 0);
    if (out_kind == kOutInt8) {
        if (vec)
            quantize_rows_kernel<kOutInt8, true><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
        else
            quantize_rows_kernel<kOutInt8, false><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
    } else {
        if (vec)
            quantize_rows_kernel<kOutHalfKMajor, true><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
        else
            quantize_rows_kernel<kOutHalfKMajor, false><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
    }
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_quantize_cols(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                 int out_kind, void *Q, int64_t ldq, float *scale, float *inv,
                                 uint32_t *partial, int32_t *dstatus, cudaStream_t st) {
    const int nsplit = colmax_nsplit(rows);
    const int64_t rps = (rows + nsplit - 1) / nsplit;
    dim3 g1((unsigned)((cols + 63) / 64), (unsigned)nsplit);
    colmax_partial_kernel<<<g1, 256, 0, st>>>(X, rows, cols, ldx, rps, partial);
    dim3 g2((unsigned)((cols + 63) / 64), (unsigned)((rows + 63) / 64));
    if (out_kind == kOutInt8)
        quantize_cols_kernel<kOutInt8><<<g2, 256, 0, st>>>(X, rows, cols, ldx, partial, nsplit, Q,
                                                           ldq, scale, inv, dstatus);
    else
        quantize_cols_kernel<kOutHalfKMajor><<<g2, 256, 0, st>>>(
            X, rows, cols, ldx, partial, nsplit, Q, ldq, scale, inv, dstatus);
    count_launches(2);
    return cudaGetLastError();
}

cudaError_t launch_i8_rows_to_half(const int8_t *Q, int64_t rows, int64_t cols, int64_t ldq,
                                   __half *out, int64_t ldo, cudaStream_t st) {
    i8_rows_to_half_kernel<<<grid_for(rows * cols, 256), 256, 0, st>>>(Q, rows, cols, ldq, out,
                                                                      ldo);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_i8_cols_to_half(const int8_t *Q, int64_t rows, int64_t cols, int64_t ldq,
                                   __half *out, int64_t ldo, cudaStream_t st) {
    dim3 g((unsigned)((cols + 63) / 64), (unsigned)((rows + 63) / 64));
    i8_cols_to_half_kernel<<<g, 256, 0, st>>>(Q, rows, cols, ldq, out, ldo);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace bsg
