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
// >= 0x7f800000).  Columns of up to 4096 rows are read once too: a strip of
// 32 columns sits in the registers of a cluster of CTAs, which exchange
// their partial maxima through distributed shared memory (fused with the
// row quantize of A in one launch when K <= 2048).  Longer columns are read
// once from HBM into the GEMM's K-major operand by a list of max and
// quantize items whose second read of each tile comes from L2; the int8
// codes in X's layout take a partial-max pass over row slices, then a
// quantize pass.
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "bsg_internal.h"
#include "bsg_ptx.cuh"
#include "lag_list.cuh"

namespace cg = cooperative_groups;

namespace bsg {
namespace {

constexpr uint32_t kNonfiniteBits = 0x7f800000u;
constexpr int kRowWarps = 8;  // rows per 256-thread block
constexpr int kRowRegVec = 8; // float4 per lane kept in registers: rows up to 1024

// Scale and reciprocal of one row or column from its absmax bit pattern.
//
// The definition is f64: scale = RN32(max(RN64(m / 127), RN64(1e-8))) and
// inv = RN32(RN64(1 / scale)).  GB300's FP64 pipe is far too slow for a
// divide per row, and two IEEE f32 divides give the same bits:
//   * RN32(RN64(x)) differs from RN32(x) only if RN64(x) lands exactly on a
//     midpoint of the f32 grid.  For x = m/127 with m = M 2^E (M a 24-bit
//     integer) x is either exact (127 | M) or at least 1/(127 2^u) from any
//     25-bit dyadic p/2^u -- a relative gap near 2^-32, far wider than the
//     2^-53 an f64 rounding can close.  For y = 1/scale with scale = S 2^F,
//     |1/S - k 2^-48| >= 1/(S 2^48): a relative gap >= 2^-48, again wider
//     than 2^-53 (y is exact when S is a power of two).  So the f64 step is
//     invisible and each value is one correctly rounded f32 divide.
//   * The floor: max commutes with the monotone RN32, and f64(1e-8) sits
//     0.07 ulp from its f32 rounding, so max(RN32(m/127), f32(f64(1e-8)))
//     equals the f64 definition, ties at the boundary included.
// The derivation is checked exhaustively against the f64 definition by
// bsg_selftest_scales and against the CPU oracle by the tests.
constexpr uint32_t kScaleFloorBits = 0x322bcc77u;  // RN32(RN64(1e-8))

__device__ __forceinline__ void scale_from_max(uint32_t mbits, float &scale, float &inv) {
    scale = fmaxf(__fdiv_rn(__uint_as_float(mbits), 127.0f), __uint_as_float(kScaleFloorBits));
    inv = __fdiv_rn(1.0f, scale);
}

// The f64 definition itself, for the self-test only.
__device__ __forceinline__ void scale_from_max_f64(uint32_t mbits, float &scale, float &inv) {
    double s = __ddiv_rn(static_cast<double>(__uint_as_float(mbits)), 127.0);
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
        int64_t c0 = 4 * c4n + lane;
        if (!VEC) {
            // unaligned rows: scalar loads, eight in flight per lane
            uint32_t m1 = 0;
            for (; c0 + 224 < cols; c0 += 256) {
                float a[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) a[u] = __ldg(xr + c0 + 32 * u);
#pragma unroll
                for (int u = 0; u < 8; u += 2) {
                    m = max(m, absbits(a[u]));
                    m1 = max(m1, absbits(a[u + 1]));
                }
            }
            m = max(m, m1);
        }
        for (int64_t c = c0; c < cols; c += 32) m = max(m, absbits(__ldg(xr + c)));
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
        int64_t cq = 4 * c4n + lane;
        if (!VEC) {
            for (; cq + 224 < cols; cq += 256) {
                float a[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) a[u] = __ldg(xr + cq + 32 * u);
#pragma unroll
                for (int u = 0; u < 8; ++u) store1<OUT>(Q, qrow + cq + 32 * u, quant(a[u], iv));
            }
        }
        for (int64_t c = cq; c < cols; c += 32)
            store1<OUT>(Q, qrow + c, quant(__ldg(xr + c), iv));
    }
}

// Rows that are not 16-byte aligned (ldx % 4 != 0, e.g. K = 8191): one warp
// per row.  The maximum: the few elements before the row's first 16-byte
// boundary and after its last read one by one, the body with 128-bit loads,
// eight in flight per lane.  The codes: the row read again (mostly from
// L1/L2) with lanes on consecutive elements, so that every store instruction
// writes one contiguous span (the codes are as unaligned as the row).
template <int OUT>
__global__ void __launch_bounds__(kRowWarps * 32)
    quantize_rows_peel_kernel(const float *__restrict__ X, int64_t rows, int64_t cols,
                              int64_t ldx, void *__restrict__ Q, int64_t ldq,
                              float *__restrict__ scale, float *__restrict__ inv,
                              int32_t *__restrict__ dstatus) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_global = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5);
    const int64_t warp_stride = (int64_t)gridDim.x * kRowWarps;
    for (int64_t r = warp_global; r < rows; r += warp_stride) {
        const float *xr = X + r * ldx;
        // elements before the first 16-byte boundary (X is 4-byte aligned)
        int64_t h = (int64_t)((16u - (uint32_t)(reinterpret_cast<uintptr_t>(xr) & 15u)) & 15u) / 4;
        if (h > cols) h = cols;
        const int64_t nb4 = (cols - h) / 4;  // float4 of the body
        const int64_t t0 = h + 4 * nb4;      // first element of the tail
        const float4 *body = reinterpret_cast<const float4 *>(xr + h);
        uint32_t m = 0, m1 = 0;
        if (lane < h) m = absbits(__ldg(xr + lane));
        if (t0 + lane < cols) m = max(m, absbits(__ldg(xr + t0 + lane)));
        int64_t c4 = lane;
        for (; c4 + 224 < nb4; c4 += 256) {
            float4 a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = __ldg(body + c4 + 32 * u);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                m = max(m, max(absbits(a[u].x), absbits(a[u].y)));
                m1 = max(m1, max(absbits(a[u].z), absbits(a[u].w)));
            }
        }
        for (; c4 < nb4; c4 += 32) {
            const float4 a = __ldg(body + c4);
            m = max(m, max(absbits(a.x), absbits(a.y)));
            m1 = max(m1, max(absbits(a.z), absbits(a.w)));
        }
        m = __reduce_max_sync(0xffffffffu, max(m, m1));
        float sc = 0.f, iv = 0.f;
        if (lane == 0) {
            scale_from_max(m, sc, iv);
            scale[r] = sc;
            if (inv) inv[r] = iv;
            if (m >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
        }
        iv = __shfl_sync(0xffffffffu, iv, 0);
        // the codes: the row again (mostly from L1/L2), lanes on consecutive
        // elements so that each store covers one contiguous span
        const int64_t qrow = r * ldq;
        int64_t c = lane;
        for (; c + 224 < cols; c += 256) {
            float a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = __ldcs(xr + c + 32 * u);
#pragma unroll
            for (int u = 0; u < 8; ++u) store1<OUT>(Q, qrow + c + 32 * u, quant(a[u], iv));
        }
        for (; c < cols; c += 32) store1<OUT>(Q, qrow + c, quant(__ldcs(xr + c), iv));
    }
}

// Column quantize, pass 1: partial |x| maxima of 128-column groups over
// slices of rows.  Block = 32 column lanes (VW columns each) x 8 row lanes;
// each thread keeps 4 row loads in flight.
constexpr int kColLanes = 32;
constexpr int kColRows = 8;

template <int VW>
__global__ void __launch_bounds__(256)
    colmax_partial_kernel(const float *__restrict__ X, int64_t rows, int64_t cols, int64_t ldx,
                          int64_t rows_per_split, uint32_t *__restrict__ partial) {
    __shared__ uint32_t red[kColRows][kColLanes * VW];
    const int cl = threadIdx.x % kColLanes;
    const int rg = threadIdx.x / kColLanes;
    const int64_t col = (int64_t)blockIdx.x * (kColLanes * VW) + cl * VW;
    const int64_t r0 = (int64_t)blockIdx.y * rows_per_split;
    const int64_t r1 = min(rows, r0 + rows_per_split);
    uint32_t m[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) m[v] = 0;
    if (col < cols) {
        int64_t r = r0 + rg;
        if (VW == 4) {
            for (; r + 3 * kColRows < r1; r += 4 * kColRows) {
                float4 t[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    t[u] = __ldg(reinterpret_cast<const float4 *>(X + (r + u * kColRows) * ldx + col));
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    m[0] = max(m[0], absbits(t[u].x));
                    m[VW > 1 ? 1 : 0] = max(m[VW > 1 ? 1 : 0], absbits(t[u].y));
                    m[VW > 2 ? 2 : 0] = max(m[VW > 2 ? 2 : 0], absbits(t[u].z));
                    m[VW > 3 ? 3 : 0] = max(m[VW > 3 ? 3 : 0], absbits(t[u].w));
                }
            }
            for (; r < r1; r += kColRows) {
                const float4 t = __ldg(reinterpret_cast<const float4 *>(X + r * ldx + col));
                m[0] = max(m[0], absbits(t.x));
                m[VW > 1 ? 1 : 0] = max(m[VW > 1 ? 1 : 0], absbits(t.y));
                m[VW > 2 ? 2 : 0] = max(m[VW > 2 ? 2 : 0], absbits(t.z));
                m[VW > 3 ? 3 : 0] = max(m[VW > 3 ? 3 : 0], absbits(t.w));
            }
        } else {
            // scalar columns: sixteen row loads in flight per thread
            for (; r + 15 * kColRows < r1; r += 16 * kColRows) {
                float t[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) t[u] = __ldg(X + (r + u * kColRows) * ldx + col);
#pragma unroll
                for (int u = 0; u < 16; ++u) m[0] = max(m[0], absbits(t[u]));
            }
            for (; r < r1; r += kColRows) m[0] = max(m[0], absbits(__ldg(X + r * ldx + col)));
        }
    }
#pragma unroll
    for (int v = 0; v < VW; ++v) red[rg][cl * VW + v] = m[v];
    __syncthreads();
    for (int c = threadIdx.x; c < kColLanes * VW; c += blockDim.x) {
        const int64_t gc = (int64_t)blockIdx.x * (kColLanes * VW) + c;
        if (gc < cols) {
            uint32_t mm = red[0][c];
#pragma unroll
            for (int g = 1; g < kColRows; ++g) mm = max(mm, red[g][c]);
            partial[(int64_t)blockIdx.y * cols + gc] = mm;
        }
    }
}

// Column quantize, pass 2: a 64-row x (32 * VW)-column tile with per-column
// scales from the partial maxima (at most kMaxSplit of them), int8 codes in
// X's layout.  (The GEMM's transposed f16 operand takes quantize_cols_t16_kernel
// as its second pass.)
constexpr int kMaxSplit = 32;

template <int VW>
__global__ void __launch_bounds__(256)
    quantize_cols_kernel(const float *__restrict__ X, int64_t rows, int64_t cols, int64_t ldx,
                         const uint32_t *__restrict__ partial, int nsplit, int8_t *__restrict__ Q,
                         int64_t ldq, float *__restrict__ scale, float *__restrict__ inv,
                         int32_t *__restrict__ dstatus) {
    constexpr int TC = kColLanes * VW;  // tile columns
    __shared__ float s_inv[TC];
    const int t = threadIdx.x;
    const int64_t c0 = (int64_t)blockIdx.x * TC;
    const int64_t r0 = (int64_t)blockIdx.y * 64;
    for (int c = t; c < TC; c += blockDim.x) {
        const int64_t col = c0 + c;
        float iv = 0.f;
        if (col < cols) {
            uint32_t mm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mm[u] = 0;
            for (int s = 0; s < nsplit; s += 8) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (s + u < nsplit) mm[u] = max(mm[u], partial[(int64_t)(s + u) * cols + col]);
            }
            uint32_t m = max(max(max(mm[0], mm[1]), max(mm[2], mm[3])),
                             max(max(mm[4], mm[5]), max(mm[6], mm[7])));
            float sc;
            scale_from_max(m, sc, iv);
            if (blockIdx.y == 0) {
                scale[col] = sc;
                if (inv) inv[col] = iv;
                if (m >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
            }
        }
        s_inv[c] = iv;
    }
    __syncthreads();
    const int cl = t % kColLanes;
    const int rg = t / kColLanes;
    const int64_t col = c0 + cl * VW;
    float ivv[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) ivv[v] = s_inv[cl * VW + v];
    float x[8][VW];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = r0 + rg + kColRows * i;
        const bool ok = row < rows && col < cols;
        if (VW == 4) {
            float4 v4 = ok ? __ldg(reinterpret_cast<const float4 *>(X + row * ldx + col))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            x[i][0] = v4.x;
            x[i][VW > 1 ? 1 : 0] = v4.y;
            x[i][VW > 2 ? 2 : 0] = v4.z;
            x[i][VW > 3 ? 3 : 0] = v4.w;
        } else {
            x[i][0] = ok ? __ldg(X + row * ldx + col) : 0.f;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = r0 + rg + kColRows * i;
        if (row < rows && col < cols) {
            if (VW == 4) {
                const char4 q = make_char4((signed char)(int)quant(x[i][0], ivv[0]),
                                           (signed char)(int)quant(x[i][VW > 1 ? 1 : 0], ivv[VW > 1 ? 1 : 0]),
                                           (signed char)(int)quant(x[i][VW > 2 ? 2 : 0], ivv[VW > 2 ? 2 : 0]),
                                           (signed char)(int)quant(x[i][VW > 3 ? 3 : 0], ivv[VW > 3 ? 3 : 0]));
                *reinterpret_cast<char4 *>(Q + row * ldq + col) = q;
            } else {
                Q[row * ldq + col] = (int8_t)(int)quant(x[i][0], ivv[0]);
            }
        }
    }
}

// Rows, single pass: WPR warps share a row and each lane keeps RV float4 of
// it in registers (rows up to 128 * RV * WPR elements), so the row is read
// once, reduced (shuffles, then shared memory across the row's warps) and
// quantized from registers.  8 warps per block: 8 / WPR rows per block.
template <int OUT, int WPR, int RV>
__device__ __forceinline__ void rows_wide_block(int64_t blk, const float *__restrict__ X,
                                                int64_t rows, int64_t cols, int64_t ldx,
                                                void *__restrict__ Q, int64_t ldq,
                                                float *__restrict__ scale,
                                                float *__restrict__ inv,
                                                int32_t *__restrict__ dstatus,
                                                unsigned int *__restrict__ zrows) {
    constexpr int RPB = 8 / WPR;
    __shared__ uint32_t red[8];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rloc = warp / WPR;
    const int wr = warp % WPR;
    const int64_t r = blk * RPB + rloc;
    const bool live = r < rows;
    // one word per row set to zero (may be NULL): the row maxima a GEMM
    // epilogue gathers for this matrix's rows
    if (zrows && live && wr == 0 && lane == 0) zrows[r] = 0u;
    const int64_t c4n = cols / 4;
    const float4 *xr = reinterpret_cast<const float4 *>(X + (live ? r : 0) * ldx);
    float4 v[RV];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < RV; ++i) {
        const int64_t c4 = lane + 32 * (i + RV * wr);
        if (live && c4 < c4n) {
            v[i] = __ldcs(xr + c4);
            m = max(m, max(max(absbits(v[i].x), absbits(v[i].y)), max(absbits(v[i].z), absbits(v[i].w))));
        } else {
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if (WPR > 1) {
        if (lane == 0) red[warp] = m;
        __syncthreads();
        m = 0;
#pragma unroll
        for (int w = 0; w < WPR; ++w) m = max(m, red[rloc * WPR + w]);
    }
    float sc, iv;
    scale_from_max(m, sc, iv);
    if (!live) return;
    if (wr == 0 && lane == 0) {
        scale[r] = sc;
        if (inv) inv[r] = iv;
        if (m >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
    }
#pragma unroll
    for (int i = 0; i < RV; ++i) {
        const int64_t c4 = lane + 32 * (i + RV * wr);
        if (c4 < c4n)
            store4<OUT>(Q, r * ldq + 4 * c4, quant(v[i].x, iv), quant(v[i].y, iv), quant(v[i].z, iv),
                        quant(v[i].w, iv));
    }
}

// Rows whose start is not 16-byte aligned (a row pitch that is not a
// multiple of 4 floats), of up to 4096 RV + 3 columns, one row per block:
// the row is held in registers as 128-bit loads from its first 16-byte
// boundary (consecutive threads on consecutive chunks), the 0-3 elements
// before that boundary and the 0-3 after the last whole chunk are loaded one
// by one; the codes are then staged in shared memory at their column
// positions and copied out in 16-byte pieces (the output rows are 16-byte
// aligned).  One read of X from HBM, like the aligned rows.  Measured on a
// GB300 (rows alone, L2 flushed): 4097 x 8191 79.5 -> 49.1 us against the
// peeling kernel, 1024 x 16383 57.2 -> 34.8 us; at 2049 columns it was
// slower (8192 rows 39.0 -> 42.9 us), so it takes rows above 4096 columns.
template <int OUT, int RV>
__global__ void __launch_bounds__(256, RV == 8 ? 4 : 2)
    quantize_rows_shift_kernel(const float *__restrict__ X, int64_t rows, int64_t cols,
                               int64_t ldx, void *__restrict__ Q, int64_t ldq,
                               float *__restrict__ scale, float *__restrict__ inv,
                               int32_t *__restrict__ dstatus) {
    constexpr int kQ = OUT == kOutInt8 ? 1 : 2;  // bytes per code
    __shared__ __align__(16) uint8_t stage[(1024 * RV + 16) * kQ];
    __shared__ uint32_t red[8];
    griddep_wait();  // programmatic launch: the previous kernel is done from here on
    griddep_launch_dependents();
    const int64_t r = blockIdx.x;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const float *xr = X + r * ldx;
    int hd = (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(xr) & 15u)) & 15u) >> 2);
    if (hd > cols) hd = (int)cols;
    const int64_t nb = (cols - hd) / 4;             // whole 16-byte chunks
    const int tl = (int)(cols - hd - 4 * nb);       // elements after them (0-3)
    const float4 *xb = reinterpret_cast<const float4 *>(xr + hd);
    float4 v[RV];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < RV; ++i) {
        const int64_t c4 = t + 256 * i;
        if (c4 < nb) {
            v[i] = __ldcs(xb + c4);
            m = max(m, max(max(absbits(v[i].x), absbits(v[i].y)), max(absbits(v[i].z), absbits(v[i].w))));
        } else {
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    float ends[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // thread 0: the head, then the tail
    if (t == 0) {
        for (int j = 0; j < hd; ++j) ends[j] = xr[j];
        for (int j = 0; j < tl; ++j) ends[3 + j] = xr[hd + 4 * nb + j];
#pragma unroll
        for (int j = 0; j < 6; ++j) m = max(m, absbits(ends[j]));
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = max(m, red[w]);
    float sc, iv;
    scale_from_max(m, sc, iv);
    if (t == 0) {
        scale[r] = sc;
        if (inv) inv[r] = iv;
        if (m >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
    }
    // the codes at their column positions
#pragma unroll
    for (int i = 0; i < RV; ++i) {
        const int64_t c4 = t + 256 * i;
        if (c4 < nb) {
            const int c = hd + 4 * (int)c4;
            const float q[4] = {quant(v[i].x, iv), quant(v[i].y, iv), quant(v[i].z, iv),
                                quant(v[i].w, iv)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (OUT == kOutInt8)
                    stage[c + j] = (uint8_t)(int8_t)(int)q[j];
                else
                    reinterpret_cast<__half *>(stage)[c + j] = __float2half_rn(q[j]);
            }
        }
    }
    if (t == 0) {
        for (int j = 0; j < hd + tl; ++j) {
            const int c = j < hd ? j : hd + 4 * (int)nb + (j - hd);
            const float q = quant(ends[j < hd ? j : 3 + (j - hd)], iv);
            if (OUT == kOutInt8)
                stage[c] = (uint8_t)(int8_t)(int)q;
            else
                reinterpret_cast<__half *>(stage)[c] = __float2half_rn(q);
        }
    }
    __syncthreads();
    const int64_t nbytes = cols * kQ;
    uint8_t *qr = static_cast<uint8_t *>(Q) + r * ldq * kQ;
    for (int64_t b = 16 * (int64_t)t; b < nbytes; b += 16 * 256) {
        if (b + 16 <= nbytes) {
            *reinterpret_cast<uint4 *>(qr + b) = *reinterpret_cast<const uint4 *>(stage + b);
        } else {
            for (int64_t j = b; j < nbytes; ++j) qr[j] = stage[j];
        }
    }
}

// zero2 (may be NULL): two words set to zero by one thread -- the tile
// counter of the GEMM that reads this launch's output.  The explicit minimum
// of one block per SM changes how ptxas schedules the loads: measured on a
// GB300 (A alone, L2 flushed), 16384 x 16384 330 -> 301 us and 8192 x 8192
// 86 -> 70 us, the same register count at 8192 columns; giving every kernel
// of this file that bound made others slower (4096^3's quantize 55 -> 61 us).
template <int OUT, int WPR, int RV>
__global__ void __launch_bounds__(256, 1)
    quantize_rows_wide_kernel(const float *__restrict__ X, int64_t rows, int64_t cols,
                              int64_t ldx, void *__restrict__ Q, int64_t ldq,
                              float *__restrict__ scale, float *__restrict__ inv,
                              int32_t *__restrict__ dstatus, unsigned int *__restrict__ zero2,
                              unsigned int *__restrict__ zrows) {
    griddep_wait();  // programmatic launch: the previous kernel is done from here on
    // the next kernel may be placed on SMs as this one drains; it waits for
    // this grid's completion before it touches memory
    griddep_launch_dependents();
    if (zero2 && blockIdx.x == 0 && threadIdx.x == 0) zero2[0] = zero2[1] = 0u;
    rows_wide_block<OUT, WPR, RV>((int64_t)blockIdx.x, X, rows, cols, ldx, Q, ldq, scale, inv,
                                  dstatus, zrows);
}

// Columns, single pass: a cluster of CS CTAs shares a strip of 32 columns;
// CTA `rank` stages rows [rank * R, rank * R + R) of the strip in shared
// memory (one HBM read), the CTAs exchange their partial |x| maxima through
// distributed shared memory, and each quantizes its rows from shared memory
// into int8 codes in X's layout.  (The GEMM's transposed f16 operand takes
// the strip, one-read or two-pass kernels below.)
constexpr int kStripCols = 32;

// The second cluster barrier of the strip kernels, split in two: a CTA
// arrives as soon as it has read its peers' partial maxima -- before any
// global store, so the release has nothing of its own to wait for -- and
// waits only before it exits, so that no CTA leaves while a peer may still
// read its shared memory.  (A full barrier after the stores made each CTA's
// release wait for them.)  Measured on a GB300: the standalone strip kernel
// dropped from 54 to 48 registers and 4096^3's quantize went 50.5 -> 48.2 us;
// the fused launch at 768 rows did not change.  Every thread of every CTA
// executes both, once (the forms without .aligned: a warp need not be
// converged there).
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__global__ void __launch_bounds__(256)
    quantize_cols_cluster_kernel(const float *__restrict__ X, int64_t rows, int64_t cols,
                                 int64_t ldx, int R, int vec, int8_t *__restrict__ Q, int64_t ldq,
                                 float *__restrict__ scale, float *__restrict__ inv,
                                 int32_t *__restrict__ dstatus) {
    extern __shared__ __align__(16) uint8_t dsm[];
    float *xs = reinterpret_cast<float *>(dsm);  // [R][32]
    __shared__ uint32_t red[8][kStripCols];
    __shared__ uint32_t part[kStripCols];
    __shared__ float s_inv[kStripCols];
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int cs = (int)cluster.num_blocks();
    const int t = threadIdx.x;
    const int64_t c0 = (int64_t)blockIdx.x * kStripCols;
    const int64_t r0 = (int64_t)rank * R;
    const int64_t left = rows - r0;
    const int nr = left <= 0 ? 0 : (left < R ? (int)left : R);

    // stage the block: 8 chunks of 16 bytes per row
    for (int q = t; q < nr * 8; q += blockDim.x) {
        const int row = q >> 3, c4 = q & 7;
        const int64_t col = c0 + 4 * c4;
        float *dst = xs + row * kStripCols + 4 * c4;
        const float *src = X + (r0 + row) * ldx + col;
        if (vec && col + 3 < cols) {
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                             static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                         "l"(src)
                         : "memory");
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) dst[u] = (col + u < cols) ? __ldg(src + u) : 0.0f;
        }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    // partial column max over this CTA's rows
    const int c = t & 31, g = t >> 5;
    uint32_t m = 0;
    for (int row = g; row < nr; row += 8) m = max(m, absbits(xs[row * kStripCols + c]));
    red[g][c] = m;
    __syncthreads();
    if (t < kStripCols) {
        uint32_t mm = red[0][t];
#pragma unroll
        for (int gg = 1; gg < 8; ++gg) mm = max(mm, red[gg][t]);
        part[t] = mm;
    }
    cluster.sync();  // every CTA's partial maxima are visible cluster-wide
    uint32_t mm = 0;
    float sc = 0.f, iv0 = 0.f;
    if (t < kStripCols) {
        for (int rk = 0; rk < cs; ++rk) mm = max(mm, *cluster.map_shared_rank(&part[t], rk));
        scale_from_max(mm, sc, iv0);
        s_inv[t] = iv0;
    }
    cluster_arrive_release();  // done with the peers' maxima
    if (t < kStripCols && rank == 0 && c0 + t < cols) {
        scale[c0 + t] = sc;
        if (inv) inv[c0 + t] = iv0;
        if (mm >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
    }
    __syncthreads();
    const float iv = s_inv[c];
    if (c0 + c < cols)
        for (int row = g; row < nr; row += 8)
            Q[(r0 + row) * ldq + c0 + c] = (int8_t)(int)quant(xs[row * kStripCols + c], iv);
    cluster_wait_acquire();  // no CTA leaves while another may still read its maxima
}

// Both operands of the unit in one launch, for the common layout (A stored
// M x K, quantized per row; B stored K x N, quantized per column, written
// transposed).  The column work is latency-bound (a small matrix, a max
// before any output) and the row work bandwidth-bound, so they share the
// launch: clusters of CS CTAs each take one 32-column strip of B and come
// first in launch order, and the row blocks of A fill the rest of the grid
// (grid (strips + row clusters, CS), cluster (1, CS, 1); row clusters do
// not interact).  A strip CTA holds its (at most 256) rows of the strip in
// registers -- one read, all loads in flight at once -- reduces its partial
// column maxima, combines them across the cluster through distributed
// shared memory, quantizes from registers and writes the strip transposed
// (Q[col][row], f16) through shared memory, each store a whole 128-byte row
// segment.
constexpr int kStripRows = 256;  // rows of a strip per CTA: 8 per thread

__device__ __forceinline__ void cols_strip_block(const float *__restrict__ X, int64_t rows,
                                                 int64_t cols, int64_t ldx, int R, int64_t strip,
                                                 __half *__restrict__ Q, int64_t ldq,
                                                 float *__restrict__ scale,
                                                 int32_t *__restrict__ dstatus) {
    __shared__ uint32_t red[32][33];  // [row phase][column] partial maxima
    __shared__ uint32_t part[kStripCols];
    __shared__ float s_inv[kStripCols];
    __shared__ __align__(16) __half ts[kStripCols][kStripRows + 2];  // [column][row]
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int cs = (int)cluster.num_blocks();
    const int t = threadIdx.x;
    const int c4 = t & 7;   // float4 column group of the strip
    const int rs = t >> 3;  // row phase, 0..31
    const int64_t c0 = strip * kStripCols;
    const int64_t r0 = (int64_t)rank * R;
    const int64_t left = rows - r0;
    const int nr = left <= 0 ? 0 : (left < R ? (int)left : R);  // R <= kStripRows
    const int64_t col = c0 + 4 * c4;
    const bool full4 = col + 3 < cols;

    float4 v[kStripRows / 32];
#pragma unroll
    for (int i = 0; i < kStripRows / 32; ++i) {
        const int r = rs + 32 * i;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < nr) {
            const float *src = X + (r0 + r) * ldx + col;
            if (full4) {
                // read once: streaming, so B's f32 leaves L2 before the f16
                // operands the GEMM reads next (qkv's quantize 9.8 -> 9.5 us)
                v[i] = __ldcs(reinterpret_cast<const float4 *>(src));
            } else {
                if (col < cols) v[i].x = __ldg(src);
                if (col + 1 < cols) v[i].y = __ldg(src + 1);
                if (col + 2 < cols) v[i].z = __ldg(src + 2);
            }
        }
    }
    uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
#pragma unroll
    for (int i = 0; i < kStripRows / 32; ++i) {
        m0 = max(m0, absbits(v[i].x));
        m1 = max(m1, absbits(v[i].y));
        m2 = max(m2, absbits(v[i].z));
        m3 = max(m3, absbits(v[i].w));
    }
    red[rs][4 * c4 + 0] = m0;
    red[rs][4 * c4 + 1] = m1;
    red[rs][4 * c4 + 2] = m2;
    red[rs][4 * c4 + 3] = m3;
    __syncthreads();
    if (t < kStripCols) {
        uint32_t mm = 0;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) mm = max(mm, red[i][t]);
        part[t] = mm;
    }
    cluster.sync();  // every CTA's partial maxima are visible cluster-wide
    uint32_t mm = 0;
    float sc = 0.f;
    if (t < kStripCols) {
        for (int k = 0; k < cs; ++k) mm = max(mm, *cluster.map_shared_rank(&part[t], k));
        float iv;
        scale_from_max(mm, sc, iv);
        s_inv[t] = iv;
    }
    cluster_arrive_release();  // done with the peers' maxima
    if (t < kStripCols && rank == 0 && c0 + t < cols) {
        scale[c0 + t] = sc;
        if (mm >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
    }
    __syncthreads();
    const float i0 = s_inv[4 * c4], i1 = s_inv[4 * c4 + 1], i2 = s_inv[4 * c4 + 2],
                i3 = s_inv[4 * c4 + 3];
#pragma unroll
    for (int i = 0; i < kStripRows / 32; ++i) {
        const int r = rs + 32 * i;
        ts[4 * c4 + 0][r] = __float2half_rn(quant(v[i].x, i0));
        ts[4 * c4 + 1][r] = __float2half_rn(quant(v[i].y, i1));
        ts[4 * c4 + 2][r] = __float2half_rn(quant(v[i].z, i2));
        ts[4 * c4 + 3][r] = __float2half_rn(quant(v[i].w, i3));
    }
    __syncthreads();
    // 32 output rows (columns of X), nr halves each from row r0: one warp
    // per output row at a time, 4-byte pairs, 128 bytes per store
    const int w = t >> 5, lane = t & 31;
    for (int n = w; n < kStripCols; n += 8) {
        if (c0 + n >= cols) continue;
        __half *dst = Q + (c0 + n) * ldq + r0;
#pragma unroll
        for (int k2 = 2 * lane; k2 < kStripRows; k2 += 64) {
            if (k2 + 1 < nr)
                *reinterpret_cast<__half2 *>(dst + k2) = *reinterpret_cast<const __half2 *>(&ts[n][k2]);
            else if (k2 < nr)
                dst[k2] = ts[n][k2];
        }
    }
    cluster_wait_acquire();  // no CTA leaves while another may still read its maxima
}

// One-warp rows of at most 768 columns (the GPT-2 linears, the LM head) are
// held to 48 registers, five CTAs per SM instead of four, without spills.
// Measured on a GB300: fc's quantize 10.5 -> 10.1 us, the LM head unit 520.9
// -> 516.7 us, qkv's quantize 9.6 -> 10.0 us (the GPT-2 step 164.5 -> 163.9
// us).  Wider rows (up to K = 2048, the fused launch's limit) keep the
// unbounded register count (they spill at 48).
template <int WPR, int RV>
__global__ void __launch_bounds__(256, WPR == 1 && RV <= 6 ? 5 : 0)
    quantize_ab_kernel(const float *__restrict__ A, int64_t M, int64_t K, int64_t lda,
                       __half *__restrict__ Aop, float *__restrict__ sa,
                       const float *__restrict__ B, int64_t N, int64_t ldb,
                       __half *__restrict__ Bop, float *__restrict__ sb, int64_t ldk, int R,
                       int strips, int32_t *__restrict__ dstatus, unsigned int *__restrict__ zero2,
                       unsigned int *__restrict__ zrows) {
    griddep_wait();  // programmatic launch: the previous kernel is done from here on
    griddep_launch_dependents();  // see quantize_rows_wide_kernel
    if (zero2 && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        zero2[0] = zero2[1] = 0u;  // the GEMM's tile counter
    if ((int)blockIdx.x < strips) {
        cols_strip_block(B, K, N, ldb, R, (int64_t)blockIdx.x, Bop, ldk, sb, dstatus);
    } else {
        const int64_t blk = (int64_t)(blockIdx.x - strips) * gridDim.y + blockIdx.y;
        rows_wide_block<kOutHalfKMajor, WPR, RV>(blk, A, M, K, lda, Aop, ldk, sa, nullptr,
                                                 dstatus, zrows);
    }
}

// The strip CTAs alone, for a column quantize that is not fused with a row
// quantize: grid (strips, CS), cluster (1, CS, 1).
__global__ void __launch_bounds__(256)
    quantize_cols_strip_kernel(const float *__restrict__ X, int64_t rows, int64_t cols,
                               int64_t ldx, int R, __half *__restrict__ Q, int64_t ldq,
                               float *__restrict__ scale, int32_t *__restrict__ dstatus) {
    griddep_wait();  // programmatic launch: the previous kernel is done from here on
    griddep_launch_dependents();  // see quantize_rows_wide_kernel
    cols_strip_block(X, rows, cols, ldx, R, (int64_t)blockIdx.x, Q, ldq, scale, dstatus);
}

// Column quantize, pass 2, into the GEMM's K-major f16 operand (Q[col][row]):
// a tile of 64 rows x 128 columns.  Each thread quantizes 32 consecutive rows
// of one column -- the lanes of a warp take consecutive columns, so each row
// load is one 128-byte line -- and stores them as f16 pairs into a [128][66]
// tile whose 33-word row stride puts the 32 lanes' stores in 32 distinct
// banks.  Each warp then copies whole output rows (one column of X, 64
// halves) from the tile to Q, 128 bytes per store.  Loads are scalar, so X
// may have any alignment and stride.
constexpr int kT16Cols = 128;
constexpr int kT16Rows = 64;

__global__ void __launch_bounds__(256)
    quantize_cols_t16_kernel(const float *__restrict__ X, int64_t rows, int64_t cols, int64_t ldx,
                             const uint32_t *__restrict__ partial, int nsplit,
                             __half *__restrict__ Q, int64_t ldq, float *__restrict__ scale,
                             float *__restrict__ inv, int32_t *__restrict__ dstatus) {
    __shared__ float s_inv[kT16Cols];
    __shared__ __align__(16) __half tile[kT16Cols][kT16Rows + 2];
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int64_t c0 = (int64_t)blockIdx.x * kT16Cols;
    const int64_t r0 = (int64_t)blockIdx.y * kT16Rows;
    if (t < kT16Cols) {
        const int64_t col = c0 + t;
        float iv = 0.f;
        if (col < cols) {
            uint32_t mm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mm[u] = 0;
            for (int s = 0; s < nsplit; s += 8) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (s + u < nsplit) mm[u] = max(mm[u], partial[(int64_t)(s + u) * cols + col]);
            }
            const uint32_t m = max(max(max(mm[0], mm[1]), max(mm[2], mm[3])),
                                   max(max(mm[4], mm[5]), max(mm[6], mm[7])));
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
    const int cj = 32 * (w & 3) + lane;  // tile column = output row of the tile
    const int rh = 32 * (w >> 2);        // this thread's first row in the tile
    const int64_t col = c0 + cj;
    const float iv = s_inv[cj];
    float x[32];
    if (col < cols && r0 + rh + 32 <= rows) {
        // the common case: 32 rows in range, the address stepped by ldx
        const float *xp = X + (r0 + rh) * ldx + col;
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = __ldg(xp + k * ldx);
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int64_t row = r0 + rh + k;
            x[k] = (row < rows && col < cols) ? __ldg(X + row * ldx + col) : 0.f;
        }
    }
#pragma unroll
    for (int k2 = 0; k2 < 16; ++k2)
        *reinterpret_cast<__half2 *>(&tile[cj][rh + 2 * k2]) =
            __floats2half2_rn(quant(x[2 * k2], iv), quant(x[2 * k2 + 1], iv));
    __syncthreads();
    const int64_t nr = rows - r0 < kT16Rows ? rows - r0 : kT16Rows;  // valid halves per row
    const int jmax = cols - c0 < kT16Cols ? (int)(cols - c0) : kT16Cols;
    const int e = 2 * lane;
    __half *dst = Q + (c0 + w) * ldq + r0 + e;
    if (e + 1 < nr) {
        for (int j = w; j < jmax; j += 8, dst += 8 * ldq)
            *reinterpret_cast<__half2 *>(dst) = *reinterpret_cast<const __half2 *>(&tile[j][e]);
    } else if (e < nr) {
        for (int j = w; j < jmax; j += 8, dst += 8 * ldq) dst[0] = tile[j][e];
    }
}

// Column quantize into the GEMM's K-major f16 operand with one read of X
// from HBM, for columns too long for the strip kernel, through the item list
// of lag_list.cuh: a max item takes its rows' |x| maxima (atomicMax into the
// panel's column maxima, then one count on the panel's counter); a quantize
// item waits (bounded) until its panel's count is complete and writes the
// transposed codes.
//
// Each thread reads one column of 32 rows straight into registers (the
// lanes of a warp take consecutive columns, so each load instruction reads
// one 128-byte line); a slice is 32 RQ rows (RQ warps per 32-column group)
// and an item covers kLagChunk consecutive slices of its panel, so the
// atomics, the fence and the wait are paid once per item.  Measured on a
// GB300 (16384 x 16384 B): RQ = 2 with 2 slices per item 344 us, RQ = 4 or
// one slice per item 380-410 us, 4 or 8 slices 400-570 us; the two-pass
// kernels 442 us.  A version that staged the tiles in a 3-stage
// shared-memory ring by cp.async, one CTA per SM, ran at half this speed:
// the chain of barriers, atomics and waits of each item then stalls the SM.
constexpr int kLagRq = 2;

// Load one thread's 32 rows of its column (zero past X's edge).  LAST: the
// last read of these lines (evict first).
template <bool LAST>
__device__ __forceinline__ void lag_load(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                         int64_t col, int64_t r0, float (&x)[32]) {
    const float *xp = X + r0 * ldx + col;
    if (col < cols && r0 + 32 <= rows) {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = LAST ? __ldcs(xp + i * ldx) : __ldg(xp + i * ldx);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            x[i] = (col < cols && r0 + i < rows) ? __ldg(xp + i * ldx) : 0.0f;
    }
}

// ws: [0] the item counter, [1, 1 + P) the panels' counts, then the column
// maxima (bit patterns); all zero at launch.  An item covers C consecutive
// slices (32 RQ rows each) of its panel; S is the number of items per panel.
template <int RQ>
__global__ void __launch_bounds__(128 * RQ, 8 / RQ)
    quantize_cols_lag_kernel(const float *__restrict__ X, int64_t rows, int64_t cols,
                             int64_t ldx, int64_t P, int64_t S, int64_t L, int C,
                             uint32_t *__restrict__ ws, __half *__restrict__ Q, int64_t ldq,
                             float *__restrict__ scale, float *__restrict__ inv,
                             int32_t *__restrict__ dstatus) {
    constexpr int kThreads = 128 * RQ, kRows = 32 * RQ;
    __shared__ __align__(16) __half tile[kLagCols][kRows + 2];  // [column][row]
    __shared__ uint32_t red[RQ][kLagCols];
    __shared__ float s_inv[kLagCols];
    __shared__ unsigned int s_item[2];
    unsigned int *claim = ws;
    uint32_t *count = ws + 1;
    uint32_t *colmax = ws + 1 + P;
    griddep_wait();  // programmatic launch: the previous kernel is done from here on
    griddep_launch_dependents();
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int cj = 32 * (w & 3) + lane;  // this thread's column of the tile
    const int rq = w >> 2;               // and its 32 rows of each slice: 32 rq .. 32 rq + 31
    const int64_t total = 2 * P * S;
    const int64_t nslices = (rows + kRows - 1) / kRows;
    if (t == 0) s_item[0] = atomicAdd(claim, 1u);
    __syncthreads();
    for (int k = 0;; k ^= 1) {
        const int64_t it = s_item[k];
        if (it >= total) break;
        if (t == 0) s_item[k ^ 1] = atomicAdd(claim, 1u);  // the next item, claimed early
        bool quantize;
        int64_t panel, chunk;
        lag_item(it, P, S, L, quantize, panel, chunk);
        const int64_t col = panel * kLagCols + cj;
        const int64_t sl0 = chunk * C;
        const int64_t sl1 = sl0 + C < nslices ? sl0 + C : nslices;
        float x[32];
        if (!quantize) {
            uint32_t m = 0;
            for (int64_t sl = sl0; sl < sl1; ++sl) {
                lag_load<false>(X, rows, cols, ldx, col, sl * kRows + 32 * rq, x);
#pragma unroll
                for (int i = 0; i < 32; ++i) m = max(m, absbits(x[i]));
            }
            red[rq][cj] = m;
            __syncthreads();
            if (t < kLagCols) {
                const int64_t c = panel * kLagCols + t;
                uint32_t mm = red[0][t];
#pragma unroll
                for (int q = 1; q < RQ; ++q) mm = max(mm, red[q][t]);
                if (c < cols && mm != 0) atomicMax(colmax + c, mm);
            }
            __syncthreads();
            if (t == 0) {
                // the barrier orders the CTA's maxima before this release
                __threadfence();
                atomicAdd(count + panel, 1u);
            }
        } else {
            lag_load<true>(X, rows, cols, ldx, col, sl0 * kRows + 32 * rq, x);
            if (t == 0) {
                // every max item of the panel has counted (bounded wait)
                bool ok = ld_acquire_gpu(count + panel) >= (uint32_t)S;
                const long long t0 = clock64();
                while (!ok) {
                    __nanosleep(64);
                    ok = ld_acquire_gpu(count + panel) >= (uint32_t)S;
                    if (!ok && clock64() - t0 > kWaitLimitCycles) break;
                }
                if (!ok && dstatus) atomicOr(dstatus, BSG_DSTATUS_TIMEOUT);
            }
            __syncthreads();
            if (t < kLagCols) {
                const int64_t c = panel * kLagCols + t;
                float iv = 0.0f;
                if (c < cols) {
                    const uint32_t m = ld_relaxed_gpu(colmax + c);
                    float sc;
                    scale_from_max(m, sc, iv);
                    if (chunk == 0) {
                        scale[c] = sc;
                        if (inv) inv[c] = iv;
                        if (m >= kNonfiniteBits && dstatus) atomicOr(dstatus, BSG_DSTATUS_NONFINITE);
                    }
                }
                s_inv[t] = iv;
            }
            __syncthreads();
            const float iv = s_inv[cj];
            const int64_t cc = cols - panel * kLagCols;
            const int jmax = cc < kLagCols ? (int)cc : kLagCols;
            for (int64_t sl = sl0; sl < sl1; ++sl) {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    *reinterpret_cast<__half2 *>(&tile[cj][32 * rq + 2 * i]) =
                        __floats2half2_rn(quant(x[2 * i], iv), quant(x[2 * i + 1], iv));
                __syncthreads();
                // the next slice's loads are in flight while the tile is copied out
                if (sl + 1 < sl1) lag_load<true>(X, rows, cols, ldx, col, (sl + 1) * kRows + 32 * rq, x);
                // each warp copies whole output rows (columns of X) to Q
                const int64_t rr = rows - sl * kRows;
                const int nr = rr < kRows ? (int)rr : kRows;  // valid halves per row
                for (int j = w; j < jmax; j += kThreads / 32) {
                    __half *dst = Q + (panel * kLagCols + j) * ldq + sl * kRows;
#pragma unroll
                    for (int e = 2 * lane; e < kRows; e += 64) {
                        if (e + 1 < nr)
                            *reinterpret_cast<__half2 *>(dst + e) =
                                *reinterpret_cast<const __half2 *>(&tile[j][e]);
                        else if (e < nr)
                            dst[e] = tile[j][e];
                    }
                }
                __syncthreads();  // the tile is free again
            }
        }
        __syncthreads();  // s_item[k ^ 1] is visible; red and s_inv are free again
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

// Compare the f32 derivation with the f64 definition for every absmax bit
// pattern in [first, last]; count the mismatches.
__global__ void selftest_scales_kernel(uint32_t first, uint32_t last,
                                       unsigned long long *__restrict__ bad) {
    unsigned long long local = 0;
    const uint64_t n = (uint64_t)last - first + 1;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t m = first + (uint32_t)i;
        float s1, i1, s2, i2;
        scale_from_max(m, s1, i1);
        scale_from_max_f64(m, s2, i2);
        if (__float_as_uint(s1) != __float_as_uint(s2) || __float_as_uint(i1) != __float_as_uint(i2))
            ++local;
    }
    if (local) atomicAdd(bad, local);
}

}  // namespace

cudaError_t launch_selftest_scales(uint32_t first, uint32_t last, unsigned long long *bad,
                                   cudaStream_t st) {
    selftest_scales_kernel<<<device_sm_count() * 8, 256, 0, st>>>(first, last, bad);
    count_launches(1);
    return cudaGetLastError();
}

// Row slices of the column absmax: enough blocks to fill the GPU, at most
// kMaxSplit (the quantize pass reads them all), at least 8 rows each.
int colmax_nsplit(int64_t rows, int64_t cols) {
    const int64_t groups = (cols + 127) / 128;
    int64_t s = (1216 + groups - 1) / groups;
    const int64_t cap_rows = (rows + 7) / 8;
    if (s > cap_rows) s = cap_rows;
    if (s > kMaxSplit) s = kMaxSplit;
    return (int)(s < 1 ? 1 : s);
}

size_t colmax_partial_bytes(int64_t rows, int64_t cols) {
    // the two-pass kernels' partial maxima, or the one-read kernel's item
    // counter, panel counts and column maxima, whichever is larger
    const size_t split = (size_t)colmax_nsplit(rows, cols) * (size_t)cols;
    const size_t lag = 1 + (size_t)((cols + kLagCols - 1) / kLagCols) + (size_t)cols;
    return (split > lag ? split : lag) * sizeof(uint32_t);
}

namespace {

// Rows longer than the register-resident kernel takes (> 16384 columns):
// each 256-thread block reduces one 8192-column segment of a row to its max
// |x| bit pattern and folds it into rowmax[r] (zeroed before) by atomicMax;
// the requantize kernel then quantizes the rows in one streaming pass.  X
// must be 16-byte aligned with ldx % 4 == 0 (the launcher's condition);
// cols % 4 may be anything: the tail is read element by element.
constexpr int kRmSeg = 256 * 4 * 8;  // columns per block

__global__ void __launch_bounds__(256)
    rowmax_seg_kernel(const float *__restrict__ X, int64_t rows, int64_t cols, int64_t ldx,
                      uint32_t *__restrict__ rowmax) {
    __shared__ uint32_t wmax[8];
    const int64_t c0 = (int64_t)blockIdx.x * kRmSeg;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const float *xr = X + r * ldx;
        uint32_t m = 0;
        const int64_t c4n = cols / 4;
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t c4 = c0 / 4 + threadIdx.x + 256 * i;
            v[i] = c4 < c4n ? __ldcs(reinterpret_cast<const float4 *>(xr) + c4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            m = max(m, max(max(absbits(v[i].x), absbits(v[i].y)),
                           max(absbits(v[i].z), absbits(v[i].w))));
        // the tail past the last whole float4, in the last segment
        for (int64_t c = 4 * c4n + threadIdx.x; c < cols && c >= c0 && c < c0 + kRmSeg; c += 256)
            m = max(m, absbits(__ldg(xr + c)));
        m = __reduce_max_sync(0xffffffffu, m);
        if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t mm = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) mm = max(mm, wmax[w]);
            atomicMax(rowmax + r, mm);
        }
        __syncthreads();
    }
}

// scale[r] and inv[r] from the max bit pattern left in scale[r] (in place).
__global__ void scales_from_bits_kernel(int64_t rows, float *__restrict__ scale,
                                        float *__restrict__ inv) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
         r += (int64_t)gridDim.x * blockDim.x) {
        float sc, iv;
        scale_from_max(__float_as_uint(scale[r]), sc, iv);
        scale[r] = sc;
        if (inv) inv[r] = iv;
    }
}

}  // namespace

static int grid_for(int64_t work, int per_block) {
    const int64_t b = (work + per_block - 1) / per_block;
    const int64_t cap = (int64_t)device_sm_count() * 32;
    return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

template <int OUT, int WPR, int RV>
static void launch_rows_wide(const float *X, int64_t rows, int64_t cols, int64_t ldx, void *Q,
                             int64_t ldq, float *scale, float *inv, int32_t *dstatus,
                             unsigned int *zero2, unsigned int *zrows, cudaStream_t st) {
    constexpr int RPB = 8 / WPR;
    const int64_t blocks = (rows + RPB - 1) / RPB;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, quantize_rows_wide_kernel<OUT, WPR, RV>, X, rows, cols, ldx, Q, ldq,
                       scale, inv, dstatus, zero2, zrows);
}

// Smallest single-pass layout (warps per row, float4 per lane) that holds a
// row of `cols` elements; -1 when the row is too long.
static int row_layout(int64_t cols) {
    static const int cap[9] = {256, 512, 768, 1024, 2048, 3072, 4096, 8192, 16384};
    for (int i = 0; i < 9; ++i)
        if (cols <= cap[i]) return i;
    return -1;
}

template <int OUT>
static bool dispatch_rows_wide(int layout, const float *X, int64_t rows, int64_t cols,
                               int64_t ldx, void *Q, int64_t ldq, float *scale, float *inv,
                               int32_t *dstatus, unsigned int *zero2, unsigned int *zrows,
                               cudaStream_t st) {
    switch (layout) {
        case 0: launch_rows_wide<OUT, 1, 2>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
        case 1: launch_rows_wide<OUT, 1, 4>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
        case 2: launch_rows_wide<OUT, 1, 6>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
        case 3: launch_rows_wide<OUT, 1, 8>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
        case 4: launch_rows_wide<OUT, 2, 8>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
        case 5: launch_rows_wide<OUT, 4, 6>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
        case 6: launch_rows_wide<OUT, 4, 8>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
        case 7: launch_rows_wide<OUT, 8, 8>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
        case 8: launch_rows_wide<OUT, 8, 16>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus, zero2, zrows, st); return true;
    }
    return false;
}

cudaError_t launch_quantize_rows(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                 int out_kind, void *Q, int64_t ldq, float *scale, float *inv,
                                 int32_t *dstatus, cudaStream_t st, unsigned int *zero2,
                                 unsigned int *zrows) {
    const size_t qalign = out_kind == kOutInt8 ? 4 : 8;
    const size_t qesz = out_kind == kOutInt8 ? 1 : 2;
    const bool vec = (cols % 4 == 0) && (ldx % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(X) % 16 == 0) && ((ldq * qesz) % qalign == 0) &&
                     (reinterpret_cast<uintptr_t>(Q) % qalign == 0);
    const int layout = vec ? row_layout(cols) : -1;
    if (layout >= 0) {
        if (out_kind == kOutInt8)
            dispatch_rows_wide<kOutInt8>(layout, X, rows, cols, ldx, Q, ldq, scale, inv, dstatus,
                                         zero2, zrows, st);
        else
            dispatch_rows_wide<kOutHalfKMajor>(layout, X, rows, cols, ldx, Q, ldq, scale, inv, dstatus,
                                              zero2, zrows, st);
        count_launches(1);
        return cudaGetLastError();
    }
    if (zero2 && cudaMemsetAsync(zero2, 0, 2 * sizeof(unsigned int), st) != cudaSuccess)
        return cudaErrorInvalidValue;
    if (zrows && cudaMemsetAsync(zrows, 0, (size_t)rows * sizeof(unsigned int), st) != cudaSuccess)
        return cudaErrorInvalidValue;
    // rows beyond the register-resident kernel: row maxima by segments (kept
    // in scale[] as bit patterns), the streaming requantize, then the scales
    if (cols > 16384 && ldx % 4 == 0 && reinterpret_cast<uintptr_t>(X) % 16 == 0) {
        uint32_t *mx = reinterpret_cast<uint32_t *>(scale);
        if (cudaMemsetAsync(mx, 0, (size_t)rows * sizeof(uint32_t), st) != cudaSuccess)
            return cudaErrorInvalidValue;
        const int64_t nseg = (cols + kRmSeg - 1) / kRmSeg;
        const dim3 g1((unsigned)nseg, (unsigned)(rows < 65535 ? rows : 65535), 1);
        rowmax_seg_kernel<<<g1, 256, 0, st>>>(X, rows, cols, ldx, mx);
        count_launches(1);
        cudaError_t e = launch_requant_rows(X, rows, cols, ldx, mx, out_kind, Q, ldq, nullptr,
                                            nullptr, dstatus, st, nullptr);
        if (e != cudaSuccess) return e;
        scales_from_bits_kernel<<<grid_for(rows, 256), 256, 0, st>>>(rows, scale, inv);
        count_launches(1);
        return cudaGetLastError();
    }
    const int grid = grid_for(rows, kRowWarps);
    const bool vec2 = (ldx % 4 == 0) && (reinterpret_cast<uintptr_t>(X) % 16 == 0) &&
                      ((ldq * qesz) % qalign == 0) && (reinterpret_cast<uintptr_t>(Q) % qalign == 0);
    // long rows that are not 16-byte aligned, into 16-byte aligned output
    // rows: held in registers from their first 16-byte boundary
    const char *se = getenv("BSG_ROWS_SHIFT");
    if (!vec2 && cols > 4096 && cols <= 16384 && rows <= 0x7fffffff &&
        reinterpret_cast<uintptr_t>(X) % 4 == 0 && (ldq * qesz) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(Q) % 16 == 0 && !(se && se[0] == '0')) {
        const bool r8 = cols <= 8192;
        if (out_kind == kOutInt8) {
            if (r8)
                quantize_rows_shift_kernel<kOutInt8, 8><<<(unsigned)rows, 256, 0, st>>>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
            else
                quantize_rows_shift_kernel<kOutInt8, 16><<<(unsigned)rows, 256, 0, st>>>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
        } else {
            if (r8)
                quantize_rows_shift_kernel<kOutHalfKMajor, 8><<<(unsigned)rows, 256, 0, st>>>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
            else
                quantize_rows_shift_kernel<kOutHalfKMajor, 16><<<(unsigned)rows, 256, 0, st>>>(X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
        }
        count_launches(1);
        return cudaGetLastError();
    }
    // rows long enough to gain from 128-bit loads take the peeling kernel
    // when they are not 16-byte aligned (BSG_ROWS_PEEL=0 keeps the scalar one)
    const char *pe = getenv("BSG_ROWS_PEEL");
    const bool peel = !vec2 && cols >= 64 && !(pe && pe[0] == '0');
    if (out_kind == kOutInt8) {
        if (vec2)
            quantize_rows_kernel<kOutInt8, true><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
        else if (peel)
            quantize_rows_peel_kernel<kOutInt8><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
        else
            quantize_rows_kernel<kOutInt8, false><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
    } else {
        if (vec2)
            quantize_rows_kernel<kOutHalfKMajor, true><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
        else if (peel)
            quantize_rows_peel_kernel<kOutHalfKMajor><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
        else
            quantize_rows_kernel<kOutHalfKMajor, false><<<grid, kRowWarps * 32, 0, st>>>(
                X, rows, cols, ldx, Q, ldq, scale, inv, dstatus);
    }
    count_launches(1);
    return cudaGetLastError();
}

// Cluster shape of the single-pass column quantize: CS CTAs of R rows each
// (R a multiple of 8, at most 1024), enough CTAs to cover the SMs twice.
// Returns false when the columns are too long for one pass.
static bool cols_cluster_shape(int64_t rows, int64_t cols, int &cs, int &R) {
    const int64_t strips = (cols + kStripCols - 1) / kStripCols;
    int64_t c = (2 * (int64_t)device_sm_count() + strips - 1) / strips;
    const int64_t by_rows = (rows + 255) / 256;  // keep a CTA at or under 256 rows when possible
    if (c < by_rows) c = by_rows;
    if (c > 8) c = 8;
    if (c < 1) c = 1;
    int64_t r = (rows + c - 1) / c;
    r = (r + 7) / 8 * 8;
    if (r > 1024) return false;
    cs = (int)c;
    R = (int)r;
    return true;
}

static size_t cols_cluster_smem(int R) { return (size_t)R * kStripCols * 4 + 16; }

static cudaError_t launch_cols_cluster(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                       int cs, int R, int8_t *Q, int64_t ldq, float *scale,
                                       float *inv, int32_t *dstatus, cudaStream_t st) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(quantize_cols_cluster_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)cols_cluster_smem(1024));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int vec = (ldx % 4 == 0) && (reinterpret_cast<uintptr_t>(X) % 16 == 0);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)((cols + kStripCols - 1) / kStripCols), (unsigned)cs, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = cols_cluster_smem(R);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)cs;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_cols_cluster_kernel, X, rows, cols, ldx, R, vec,
                              Q, ldq, scale, inv, dstatus);
}

// Cluster size and rows per CTA of the register-resident strip kernels:
// CTAs of at most 256 rows, clusters of at most `max_cs` CTAs.
static bool strip_shape(int64_t rows, int max_cs, int &cs, int &R) {
    if (rows < 1 || rows > (int64_t)max_cs * kStripRows) return false;
    cs = (int)((rows + kStripRows - 1) / kStripRows);
    R = (int)round_up((rows + cs - 1) / cs, 8);
    return true;
}

static cudaError_t allow_big_clusters(const void *kernel, bool *ready) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev]) {  // clusters of up to 16 CTAs
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        ready[dev] = true;
    }
    return cudaSuccess;
}

template <int WPR, int RV>
static cudaError_t launch_ab(const float *A, int64_t M, int64_t K, int64_t lda, __half *Aop,
                             float *sa, const float *B, int64_t N, int64_t ldb, __half *Bop,
                             float *sb, int64_t ldk, int cs, int R, int32_t *dstatus,
                             unsigned int *zero2, unsigned int *zrows, cudaStream_t st) {
    constexpr int RPB = 8 / WPR;
    const int64_t strips = (N + kStripCols - 1) / kStripCols;
    const int64_t row_blocks = (M + RPB - 1) / RPB;
    const int64_t row_clusters = (row_blocks + cs - 1) / cs;
    if (strips + row_clusters > 0x7fffffff) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(strips + row_clusters), (unsigned)cs, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)cs;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, quantize_ab_kernel<WPR, RV>, A, M, K, lda, Aop, sa, B, N, ldb,
                              Bop, sb, ldk, R, (int)strips, dstatus, zero2, zrows);
}

cudaError_t launch_quantize_ab(const float *A, int64_t M, int64_t K, int64_t lda,
                               const float *B, int64_t N, int64_t ldb, __half *Aop,
                               __half *Bop, int64_t ldk, float *sa, float *sb,
                               int32_t *dstatus, unsigned int *zero2, cudaStream_t st,
                               unsigned int *zrows) {
    const bool vecA = (K % 4 == 0) && (lda % 4 == 0) &&
                      (reinterpret_cast<uintptr_t>(A) % 16 == 0) && ((ldk * 2) % 8 == 0) &&
                      (reinterpret_cast<uintptr_t>(Aop) % 8 == 0);
    const int layout = vecA ? row_layout(K) : -1;
    const bool vecB = (ldb % 4 == 0) && (reinterpret_cast<uintptr_t>(B) % 16 == 0) &&
                      (ldk % 2 == 0) && (reinterpret_cast<uintptr_t>(Bop) % 4 == 0);
    // Strip CTAs of at most 256 rows, at most 8 to a cluster (K <= 2048):
    // every row block of the grid is launched in a cluster of the same size,
    // and larger clusters (with the strip CTAs' registers) slowed the row
    // blocks down more than the fusion saved.
    int cs = 0, R = 0;
    if (layout < 0 || !vecB || !strip_shape(K, 8, cs, R)) return cudaErrorNotSupported;
    cudaError_t e = cudaErrorNotSupported;
    switch (layout) {
        case 0: e = launch_ab<1, 2>(A, M, K, lda, Aop, sa, B, N, ldb, Bop, sb, ldk, cs, R, dstatus, zero2, zrows, st); break;
        case 1: e = launch_ab<1, 4>(A, M, K, lda, Aop, sa, B, N, ldb, Bop, sb, ldk, cs, R, dstatus, zero2, zrows, st); break;
        case 2: e = launch_ab<1, 6>(A, M, K, lda, Aop, sa, B, N, ldb, Bop, sb, ldk, cs, R, dstatus, zero2, zrows, st); break;
        case 3: e = launch_ab<1, 8>(A, M, K, lda, Aop, sa, B, N, ldb, Bop, sb, ldk, cs, R, dstatus, zero2, zrows, st); break;
        case 4: e = launch_ab<2, 8>(A, M, K, lda, Aop, sa, B, N, ldb, Bop, sb, ldk, cs, R, dstatus, zero2, zrows, st); break;
        default: return cudaErrorNotSupported;  // not reached: strip_shape caps K at 2048
    }
    count_launches(1);
    return e;
}

// Column quantize path: BSG_COLS_PATH=strip|lag|twopass forces one (strips
// only where their layout conditions hold; results are the same), for the
// tests; read on every call.  0 = no preference.
static int forced_cols_path() {
    const char *e = getenv("BSG_COLS_PATH");
    if (!e) return 0;
    if (!strcmp(e, "strip")) return 1;
    if (!strcmp(e, "lag")) return 2;
    if (!strcmp(e, "twopass")) return 3;
    return 0;
}

static cudaError_t launch_cols_lag(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                   __half *Q, int64_t ldq, float *scale, float *inv,
                                   uint32_t *ws, int32_t *dstatus, cudaStream_t st) {
    constexpr int kThreads = 128 * kLagRq, kRows = 32 * kLagRq;
    static int per_sm[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (per_sm[dev] == 0) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_cols_lag_kernel<kLagRq>,
                                                          kThreads, 0);
        if (e != cudaSuccess) return e;
        per_sm[dev] = n > 0 ? n : 1;
    }
    const int64_t P = (cols + kLagCols - 1) / kLagCols;
    const int64_t S = ((rows + kRows - 1) / kRows + kLagChunk - 1) / kLagChunk;  // items per panel
    if (2 * P * S >= 0xffff0000LL) return cudaErrorInvalidValue;  // the 32-bit item counter
    int64_t grid = (int64_t)per_sm[dev] * device_sm_count();
    if (grid > 2 * P * S) grid = 2 * P * S;
    const int64_t L = colq_lag(rows);
    e = cudaMemsetAsync(ws, 0, (size_t)(1 + P + cols) * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    quantize_cols_lag_kernel<kLagRq><<<(unsigned)grid, kThreads, 0, st>>>(
        X, rows, cols, ldx, P, S, L, kLagChunk, ws, Q, ldq, scale, inv, dstatus);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_quantize_cols(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                 int out_kind, void *Q, int64_t ldq, float *scale, float *inv,
                                 uint32_t *partial, int32_t *dstatus, cudaStream_t st) {
    int cs = 0, R = 0;
    const int forced = forced_cols_path();
    // the GEMM's transposed f16 operand, no inv wanted, 16-byte rows: strip CTAs
    if (forced != 3 && forced != 2 && out_kind == kOutHalfKMajor && !inv && ldx % 4 == 0 &&
        reinterpret_cast<uintptr_t>(X) % 16 == 0 && ldq % 2 == 0 &&
        reinterpret_cast<uintptr_t>(Q) % 4 == 0 && strip_shape(rows, 16, cs, R)) {
        static bool ready[64] = {false};
        cudaError_t e = allow_big_clusters((const void *)quantize_cols_strip_kernel, ready);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3((unsigned)((cols + kStripCols - 1) / kStripCols), (unsigned)cs, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)cs;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, quantize_cols_strip_kernel, X, rows, cols, ldx, R,
                               static_cast<__half *>(Q), ldq, scale, dstatus);
        count_launches(1);
        return e;
    }
    // Single pass in clusters only for columns of at most 3072 rows (int8 in
    // X's layout): beyond, two passes measured faster (8192 rows 108 against
    // 191 us, 4096 rows 30 against 35 us), the cluster kernel's CTAs holding
    // up to ~200 KB of shared memory, one per SM.  The GEMM's f16 operand past
    // the strip kernel's rows takes the one-read list of items (two passes
    // only when BSG_COLS_PATH=twopass asks for them).
    if (forced != 3 && out_kind == kOutInt8 && rows <= 3072 &&
        cols_cluster_shape(rows, cols, cs, R)) {
        const cudaError_t e = launch_cols_cluster(X, rows, cols, ldx, cs, R,
                                                  static_cast<int8_t *>(Q), ldq, scale, inv,
                                                  dstatus, st);
        count_launches(1);
        return e;
    }
    const int nsplit = colmax_nsplit(rows, cols);
    const int64_t rps = (rows + nsplit - 1) / nsplit;
    const bool vec = (cols % 4 == 0) && (ldx % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(X) % 16 == 0) &&
                     (out_kind != kOutInt8 || ((ldq % 4 == 0) && reinterpret_cast<uintptr_t>(Q) % 4 == 0));
    const int vw = vec ? 4 : 1;
    const unsigned gx = (unsigned)((cols + 32 * vw - 1) / (32 * vw));
    dim3 g1(gx, (unsigned)nsplit), g2(gx, (unsigned)((rows + 63) / 64));
    if (out_kind == kOutHalfKMajor) {
        if (reinterpret_cast<uintptr_t>(Q) % 4 != 0 || ldq % 2 != 0) return cudaErrorInvalidValue;
        if (forced != 3)
            return launch_cols_lag(X, rows, cols, ldx, static_cast<__half *>(Q), ldq, scale, inv,
                                   partial, dstatus, st);
        if (vec)
            colmax_partial_kernel<4><<<g1, 256, 0, st>>>(X, rows, cols, ldx, rps, partial);
        else
            colmax_partial_kernel<1><<<g1, 256, 0, st>>>(X, rows, cols, ldx, rps, partial);
        const dim3 g3((unsigned)((cols + kT16Cols - 1) / kT16Cols),
                      (unsigned)((rows + kT16Rows - 1) / kT16Rows));
        quantize_cols_t16_kernel<<<g3, 256, 0, st>>>(X, rows, cols, ldx, partial, nsplit,
                                                     static_cast<__half *>(Q), ldq, scale, inv,
                                                     dstatus);
        count_launches(2);
        return cudaGetLastError();
    }
    // int8 codes in X's layout
    int8_t *q8 = static_cast<int8_t *>(Q);
    if (vec) {
        colmax_partial_kernel<4><<<g1, 256, 0, st>>>(X, rows, cols, ldx, rps, partial);
        quantize_cols_kernel<4><<<g2, 256, 0, st>>>(X, rows, cols, ldx, partial, nsplit, q8, ldq,
                                                    scale, inv, dstatus);
    } else {
        colmax_partial_kernel<1><<<g1, 256, 0, st>>>(X, rows, cols, ldx, rps, partial);
        quantize_cols_kernel<1><<<g2, 256, 0, st>>>(X, rows, cols, ldx, partial, nsplit, q8, ldq,
                                                    scale, inv, dstatus);
    }
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

namespace {

// Rows whose absmax is already known (the per-row maxima of |C| that the
// GEMM's epilogue gathered): no reduction is left, so each 256-thread block
// quantizes one 4096-column segment of one row in a single streaming pass,
// 4 bytes read and 1 (int8) or 2 (f16 operand) written per element, for any
// row length.  VEC: 16-byte loads of X (all four issued before any store)
// and 4/8-byte stores of Q.
constexpr int kRqThreads = 256;
constexpr int kRqVec = 4;                         // float4 per thread
constexpr int kRqSeg = kRqThreads * 4 * kRqVec;   // columns per block

template <int OUT, bool VEC>
__global__ void __launch_bounds__(kRqThreads)
    requant_rows_kernel(const float *__restrict__ X, int64_t rows, int64_t cols, int64_t ldx,
                        const uint32_t *__restrict__ rowmax, void *__restrict__ Q, int64_t ldq,
                        float *__restrict__ scale, float *__restrict__ inv,
                        int32_t *__restrict__ dstatus, unsigned int *__restrict__ zero2) {
    griddep_wait();  // programmatic launch: the GEMM that gathered rowmax is done
    griddep_launch_dependents();
    if (zero2 && blockIdx.x == 0 && threadIdx.x == 0) zero2[0] = zero2[1] = 0u;
    const int64_t nseg = (cols + kRqSeg - 1) / kRqSeg;
    for (int64_t b = blockIdx.x; b < rows * nseg; b += gridDim.x) {
        const int64_t r = b / nseg;
        const int64_t seg = b - r * nseg;
        const uint32_t m = __ldg(rowmax + r);
        float s, iv;
        scale_from_max(m, s, iv);
        if (seg == 0 && threadIdx.x == 0) {
            if (scale) scale[r] = s;
            if (inv) inv[r] = iv;
            if (m >= kNonfiniteBits && dstatus) atomicOr(dstatus, 1);
        }
        const float *xr = X + r * ldx;
        const int64_t qrow = r * ldq;
        if (VEC) {
            float4 x[kRqVec];
#pragma unroll
            for (int h = 0; h < kRqVec; ++h) {
                const int64_t c = seg * kRqSeg + 4 * (threadIdx.x + h * kRqThreads);
                if (c < cols)  // cols % 4 == 0 here
                    x[h] = __ldcs(reinterpret_cast<const float4 *>(xr + c));
            }
#pragma unroll
            for (int h = 0; h < kRqVec; ++h) {
                const int64_t c = seg * kRqSeg + 4 * (threadIdx.x + h * kRqThreads);
                if (c < cols)
                    store4<OUT>(Q, qrow + c, quant(x[h].x, iv), quant(x[h].y, iv),
                                quant(x[h].z, iv), quant(x[h].w, iv));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4 * kRqVec; ++i) {
                const int64_t c = seg * kRqSeg + threadIdx.x + i * kRqThreads;
                if (c < cols) store1<OUT>(Q, qrow + c, quant(__ldg(xr + c), iv));
            }
        }
    }
}

}  // namespace

cudaError_t launch_requant_rows(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                const uint32_t *rowmax, int out_kind, void *Q, int64_t ldq,
                                float *scale, float *inv, int32_t *dstatus, cudaStream_t st,
                                unsigned int *zero2) {
    const size_t qsz = out_kind == kOutInt8 ? 1 : 2;
    const bool vec = cols % 4 == 0 && ldx % 4 == 0 && ldq % 4 == 0 &&
                     reinterpret_cast<uintptr_t>(X) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(Q) % (4 * qsz) == 0;
    const int64_t blocks = rows * ((cols + kRqSeg - 1) / kRqSeg);
    const int64_t cap = (int64_t)device_sm_count() * 16;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(blocks < cap ? blocks : cap), 1, 1);
    cfg.blockDim = dim3(kRqThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (out_kind == kOutInt8)
        e = vec ? cudaLaunchKernelEx(&cfg, requant_rows_kernel<kOutInt8, true>, X, rows, cols, ldx,
                                     rowmax, Q, ldq, scale, inv, dstatus, zero2)
                : cudaLaunchKernelEx(&cfg, requant_rows_kernel<kOutInt8, false>, X, rows, cols, ldx,
                                     rowmax, Q, ldq, scale, inv, dstatus, zero2);
    else
        e = vec ? cudaLaunchKernelEx(&cfg, requant_rows_kernel<kOutHalfKMajor, true>, X, rows, cols,
                                     ldx, rowmax, Q, ldq, scale, inv, dstatus, zero2)
                : cudaLaunchKernelEx(&cfg, requant_rows_kernel<kOutHalfKMajor, false>, X, rows, cols,
                                     ldx, rowmax, Q, ldq, scale, inv, dstatus, zero2);
    count_launches(1);
    return e;
}

}  // namespace bsg
