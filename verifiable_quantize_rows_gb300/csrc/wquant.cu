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
// A strip of 32 columns is quantized by a cluster of CTAs, each owning a slice
// of its rows: each reads its slice for the column maxima, the cluster
// combines them through distributed shared memory, and each reads its slice
// again (from L2) to quantize it; long columns take the one-read item list
// of lag_list.cuh instead.  The code is the integer
// nearest the exact quotient w / s, ties to even: almost always rint of
// RN(w * RN(1/s)), which lies within 2^-16 of the exact quotient, when that
// product is more than 2^-14 from a half-integer; otherwise found with
// integer arithmetic on the two floats' significands (2|w|/s = mw * 2^sh /
// ms exactly; its integer part and remainder decide the rounding).  The f64
// divide the first version used per element ran on GB300's FP64 pipe, and
// an f32 divide per element still made the kernel compute-bound.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "bsg_internal.h"
#include "bsg_ptx.cuh"
#include "lag_list.cuh"

namespace cg = cooperative_groups;

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

// The integer nearest w / s, ties to even, clamped to [-qmax, qmax]; w and s
// finite, s > 0.  With w = mw 2^(ew-150) and s = ms 2^(es-150) (significands
// with the implicit bit; subnormals take exponent field 1 and no implicit
// bit), 2|w|/s = mw 2^sh / ms with sh = ew - es + 1, a ratio of integers.
__device__ __forceinline__ int wq_round_quotient_exact(float w, float s, int qmax) {
    const uint32_t wb = __float_as_uint(w);
    const uint32_t aw = wb & 0x7fffffffu;
    const int neg = (int)(wb >> 31);
    if (aw == 0) return 0;
    const uint32_t sb = __float_as_uint(s);
    const int ew = (int)(aw >> 23), es = (int)(sb >> 23);
    const uint64_t mw = (aw & 0x7fffffu) | (ew ? 0x800000u : 0u);
    const uint64_t ms = (sb & 0x7fffffu) | (es ? 0x800000u : 0u);
    const int sh = (ew ? ew : 1) - (es ? es : 1) + 1;
    // sh <= -25: 2|w|/s < 2^24 2^-25 = 1/2, so |w|/s < 1/4 and the code is 0;
    // sh >= 33: 2|w|/s > 2^33 / 2^24 = 512, beyond any qmax
    if (sh <= -25) return 0;
    if (sh >= 33) return neg ? -qmax : qmax;
    const uint64_t num = sh >= 0 ? mw << sh : mw;          // < 2^56
    const uint64_t den = sh >= 0 ? ms : ms << (-sh);        // < 2^48
    if (num >= (uint64_t)(2 * qmax + 2) * den) return neg ? -qmax : qmax;  // |w|/s >= qmax + 1
    // q2 = floor(2|w|/s) <= 2 qmax + 1: a float estimate, corrected exactly
    uint32_t q2 = (uint32_t)__fdividef((float)num, (float)den);
    if ((uint64_t)q2 * den > num) --q2;
    if ((uint64_t)(q2 + 1) * den <= num) ++q2;
    const uint64_t rem = num - (uint64_t)q2 * den;
    uint32_t q = q2 >> 1;                                   // |w|/s = q + (q2 odd) / 2 + rem / (2 den)
    if (q2 & 1) q += (rem != 0 || (q & 1)) ? 1u : 0u;       // above a half: up; on it: to even
    if ((int)q > qmax) q = (uint32_t)qmax;
    return neg ? -(int)q : (int)q;
}

// The same integer, first from x = RN(w * r) with r = RN(1 / s) (one
// reciprocal per column instead of a divide per element): x is within
// |w/s| 2^-23 of the exact quotient (two roundings of 2^-24; r is a normal
// float, since s <= FLT_MAX / 7 < 2^126), below 2^-16 while |x| < 128, so
// when x lies more than 2^-14 from the nearest half-integer h, the exact
// quotient lies on the same side of h and rounds to rint(x).  (x - h is
// exact there: for |x| >= 1, x and h are within a factor of two; below,
// h = +-1/2 and |x - h| >= 1/4 unless |x| >= 1/4.)  Quotients near a
// half-integer, and any x that is not finite (r overflowing for a tiny s),
// take the exact path.
__device__ __forceinline__ bool wq_fast_code(float w, float r, int qmax, int &q) {
    const float x = __fmul_rn(w, r);
    if (!(fabsf(x) < 128.0f)) return false;
    const float h = __fadd_rn(floorf(x), 0.5f);
    if (!(fabsf(__fsub_rn(x, h)) > 0x1p-14f)) return false;
    q = (int)rintf(x);
    q = q < -qmax ? -qmax : (q > qmax ? qmax : q);
    return true;
}

__device__ __forceinline__ int wq_round_quotient(float w, float s, float r, int qmax) {
    int q;
    return wq_fast_code(w, r, qmax, q) ? q : wq_round_quotient_exact(w, s, qmax);
}

// grid (strips, CS), cluster (1, CS, 1): CTA `rank` owns rows [rank R, rank R + R).
// VEC: W 16-byte aligned with ldw % 4 == 0 (float4 loads of each 4-column group).
template <int BITS, bool POW2, bool VEC>
__global__ void __launch_bounds__(256)
    wquant_cols_kernel(const float *__restrict__ W, int64_t K, int64_t N, int64_t ldw, int R,
                       uint8_t *__restrict__ Q, int64_t ldq, int qvec,
                       float *__restrict__ scale, int32_t *__restrict__ dstatus) {
    constexpr int kQmax = BITS == 8 ? 127 : 7;
    __shared__ uint32_t red[32][33];
    __shared__ uint32_t part[kWStrip];
    __shared__ float s_col[kWStrip];
    __shared__ int s_bad;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int cs = (int)cluster.num_blocks();
    const int t = threadIdx.x;
    const int c4 = t & 7, rs = t >> 3;
    const int64_t col = (int64_t)blockIdx.x * kWStrip + 4 * c4;
    const int64_t r0 = (int64_t)rank * R;
    const int64_t left = K - r0;
    const int nr = left <= 0 ? 0 : (left < R ? (int)left : R);
    const bool full4 = col + 3 < N;
    auto load4 = [&](int r) {
        const float *p = W + (r0 + r) * ldw + col;
        if (VEC && full4) return __ldg(reinterpret_cast<const float4 *>(p));
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < N) v.x = __ldg(p);
        if (col + 1 < N) v.y = __ldg(p + 1);
        if (col + 2 < N) v.z = __ldg(p + 2);
        if (col + 3 < N) v.w = __ldg(p + 3);
        return v;
    };
    if (t == 0) s_bad = 0;
    uint32_t m[4] = {0u, 0u, 0u, 0u};  // |x| bit patterns: NaN left out, Inf kept
    bool bad = false;
#pragma unroll 4
    for (int r = rs; r < nr; r += 32) {
        const float4 v = load4(r);
        const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t a = wq_absbits(x[u]);
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
#pragma unroll 8
        for (int i = 0; i < 32; ++i) mm = max(mm, red[i][t]);
        part[t] = mm;
    }
    cluster.sync();  // every CTA's partial maxima are visible cluster-wide
    if (t < kWStrip) {
        uint32_t mm = 0;
        for (int k = 0; k < cs; ++k) mm = max(mm, *cluster.map_shared_rank(&part[t], k));
        const int64_t j = (int64_t)blockIdx.x * kWStrip + t;
        float sc = __fdiv_rn(__uint_as_float(mm), (float)kQmax);
        if (POW2 && isfinite(sc)) sc = wq_pow2_up(sc);
        s_col[t] = sc;
        if (rank == 0 && j < N) scale[j] = sc;
    }
    if (t == 0 && s_bad && dstatus) atomicOr(dstatus, 1);  // Inf or NaN in this slice
    cluster.sync();  // s_col is complete; no CTA leaves while another reads its maxima
    float sv[4], rv[4];
    bool use[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        sv[u] = s_col[4 * c4 + u];
        use[u] = sv[u] != 0.0f && isfinite(sv[u]);
        rv[u] = use[u] ? __frcp_rn(sv[u]) : 0.0f;
    }
#pragma unroll 4
    for (int r = rs; r < nr; r += 32) {
        const float4 v = load4(r);
        const float x[4] = {v.x, v.y, v.z, v.w};
        int q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            q[u] = (use[u] && isfinite(x[u])) ? wq_round_quotient(x[u], sv[u], rv[u], kQmax) : 0;
        uint8_t *row = Q + (r0 + r) * ldq;
        if (BITS == 8) {
            if (qvec && full4) {
                *reinterpret_cast<char4 *>(row + col) =
                    make_char4((signed char)q[0], (signed char)q[1], (signed char)q[2],
                               (signed char)q[3]);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (col + u < N) row[col + u] = (uint8_t)(int8_t)q[u];
            }
        } else {
            // columns col..col+3 (col % 4 == 0) -> bytes col/2 and col/2 + 1
            const uint8_t b0 = (uint8_t)((q[0] & 0xf) | ((col + 1 < N ? q[1] & 0xf : 0) << 4));
            const uint8_t b1 = (uint8_t)((q[2] & 0xf) | ((col + 3 < N ? q[3] & 0xf : 0) << 4));
            if (qvec && col + 2 < N) {
                *reinterpret_cast<uint16_t *>(row + col / 2) = (uint16_t)(b0 | (b1 << 8));
            } else {
                if (col < N) row[col / 2] = b0;
                if (col + 2 < N) row[col / 2 + 1] = b1;
            }
        }
    }
}

// Long weight columns: the one-read item list of lag_list.cuh, with this
// scheme's maxima (NaN left out, Inf kept and reported), scales and codes;
// the codes go to Q in W's layout.  Each thread takes one column of 32 rows
// of each 64-row slice (lanes on consecutive columns, so each load reads one
// 128-byte line); a slice's codes are staged in shared memory and leave in
// 16-byte (int8) or 4-byte (packed int4) pieces where Q's rows allow, else
// one code (or code pair) at a time.
constexpr int kWqRows = 64;  // rows per slice

template <bool LAST>
__device__ __forceinline__ void wq_load32(const float *W, int64_t K, int64_t N, int64_t ldw,
                                          int64_t col, int64_t r0, float (&x)[32]) {
    const float *p = W + r0 * ldw + col;
    if (col < N && r0 + 32 <= K) {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = LAST ? __ldcs(p + i * ldw) : __ldg(p + i * ldw);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = (col < N && r0 + i < K) ? __ldg(p + i * ldw) : 0.0f;
    }
}

// ws: [0] the item counter, [1, 1 + P) the panels' counts, then the column
// maxima (bit patterns); all zero at launch.
template <int BITS, bool POW2>
__global__ void __launch_bounds__(256, 4)
    wquant_cols_lag_kernel(const float *__restrict__ W, int64_t K, int64_t N, int64_t ldw,
                           int64_t P, int64_t S, int64_t L, uint32_t *__restrict__ ws,
                           uint8_t *__restrict__ Q, int64_t ldq, int qvec,
                           float *__restrict__ scale, int32_t *__restrict__ dstatus) {
    constexpr int kQmax = BITS == 8 ? 127 : 7;
    __shared__ uint32_t red[2][kLagCols];
    __shared__ float s_sc[kLagCols];
    __shared__ unsigned int s_item[2];
    __shared__ int s_bad;
    __shared__ __align__(16) int8_t qt[kWqRows][kLagCols];  // a slice's codes, then copied out
    unsigned int *claim = ws;
    uint32_t *count = ws + 1;
    uint32_t *colmax = ws + 1 + P;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int cj = 32 * (w & 3) + lane;  // this thread's column of the panel
    const int rq = w >> 2;               // and its 32 rows of each slice
    const int64_t total = 2 * P * S;
    const int64_t nslices = (K + kWqRows - 1) / kWqRows;
    if (t == 0) {
        s_item[0] = atomicAdd(claim, 1u);
        s_bad = 0;
    }
    __syncthreads();
    for (int k = 0;; k ^= 1) {
        const int64_t it = s_item[k];
        if (it >= total) break;
        if (t == 0) s_item[k ^ 1] = atomicAdd(claim, 1u);  // the next item, claimed early
        bool quantize;
        int64_t panel, chunk;
        lag_item(it, P, S, L, quantize, panel, chunk);
        const int64_t col = panel * kLagCols + cj;
        const int64_t sl0 = chunk * kLagChunk;
        const int64_t sl1 = sl0 + kLagChunk < nslices ? sl0 + kLagChunk : nslices;
        float x[32];
        if (!quantize) {
            uint32_t m = 0;
            bool bad = false;
            for (int64_t sl = sl0; sl < sl1; ++sl) {
                wq_load32<false>(W, K, N, ldw, col, sl * kWqRows + 32 * rq, x);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint32_t a = wq_absbits(x[i]);
                    if (a <= 0x7f800000u) m = max(m, a);
                    bad = bad || a >= 0x7f800000u;
                }
            }
            if (bad) s_bad = 1;
            red[rq][cj] = m;
            __syncthreads();
            if (t < kLagCols) {
                const int64_t c = panel * kLagCols + t;
                const uint32_t mm = max(red[0][t], red[1][t]);
                if (c < N && mm != 0) atomicMax(colmax + c, mm);
            }
            __syncthreads();
            if (t == 0) {
                // the barrier orders the CTA's maxima before this release
                __threadfence();
                atomicAdd(count + panel, 1u);
            }
        } else {
            wq_load32<true>(W, K, N, ldw, col, sl0 * kWqRows + 32 * rq, x);
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
                float sc = 0.0f;
                if (c < N) {
                    sc = __fdiv_rn(__uint_as_float(ld_relaxed_gpu(colmax + c)), (float)kQmax);
                    if (POW2 && isfinite(sc)) sc = wq_pow2_up(sc);
                    if (chunk == 0) scale[c] = sc;
                }
                s_sc[t] = sc;
            }
            __syncthreads();
            const float sv = s_sc[cj];
            const bool use = sv != 0.0f && isfinite(sv);
            const float rv = use ? __frcp_rn(sv) : 0.0f;
            for (int64_t sl = sl0; sl < sl1; ++sl) {
                if (sl > sl0) wq_load32<true>(W, K, N, ldw, col, sl * kWqRows + 32 * rq, x);
                const int64_t r0 = sl * kWqRows + 32 * rq;
                // the 32 codes as bytes: the fast test of wq_fast_code decides
                // almost every one; the few it leaves are redone exactly, from
                // W read again
                uint32_t pk[8];
                uint32_t slow = 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    int q = 0;
                    if (use && isfinite(x[i]) && !wq_fast_code(x[i], rv, kQmax, q)) {
                        q = 0;
                        slow |= 1u << i;
                    }
                    if ((i & 3) == 0) pk[i >> 2] = 0u;
                    pk[i >> 2] |= (uint32_t)(q & 0xff) << (8 * (i & 3));
                }
                // Zero padding past K or N (never stored) reaches this loop when
                // rv = +Inf (a column of subnormal maxima: 0 * rv is NaN); it
                // is not read again, and its exact code is 0.
                const bool in_cols = col < N;
                while (slow) {
                    const int i = __ffs(slow) - 1;
                    slow &= slow - 1;
                    const float wv = (in_cols && r0 + i < K) ? __ldg(W + (r0 + i) * ldw + col) : 0.0f;
                    const int q = wq_round_quotient_exact(wv, sv, kQmax);
                    const uint32_t sh = 8u * (uint32_t)(i & 3);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j == (i >> 2)) pk[j] = (pk[j] & ~(0xffu << sh)) | ((uint32_t)(q & 0xff) << sh);
                }
                if (qvec) {
                    // through the tile: each row of codes leaves in 16-byte
                    // (int8) or 4-byte (int4, two codes a byte) pieces
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        qt[32 * rq + i][cj] = (int8_t)(uint8_t)(pk[i >> 2] >> (8 * (i & 3)));
                    __syncthreads();
                    const int64_t cc = N - panel * kLagCols;
                    const int ncol = cc < kLagCols ? (int)cc : kLagCols;  // valid columns
                    const int64_t rbase = sl * kWqRows;
                    if (BITS == 8) {
                        for (int e = t; e < kWqRows * (kLagCols / 16); e += 256) {
                            const int r = e >> 3, c16 = (e & 7) * 16;
                            if (rbase + r >= K || c16 >= ncol) continue;
                            uint8_t *dst = Q + (rbase + r) * ldq + panel * kLagCols + c16;
                            if (c16 + 16 <= ncol)
                                *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(&qt[r][c16]);
                            else
                                for (int j = 0; j < ncol - c16; ++j) dst[j] = (uint8_t)qt[r][c16 + j];
                        }
                    } else {
                        const int nbyte = (ncol + 1) / 2;  // a last odd column's high nibble is 0
                        for (int e = t; e < kWqRows * (kLagCols / 8); e += 256) {
                            const int r = e >> 4, c8 = (e & 15) * 8;
                            if (rbase + r >= K || c8 >= ncol) continue;
                            const uint2 v = *reinterpret_cast<const uint2 *>(&qt[r][c8]);
                            uint32_t packed = 0;
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t word = j < 2 ? v.x : v.y;
                                const uint32_t lo = (word >> (16 * (j & 1))) & 0xfu;
                                const uint32_t hi = (word >> (16 * (j & 1) + 8)) & 0xfu;
                                packed |= (lo | (hi << 4)) << (8 * j);
                            }
                            uint8_t *dst = Q + (rbase + r) * ldq + panel * (kLagCols / 2) + c8 / 2;
                            if (c8 / 2 + 4 <= nbyte)
                                *reinterpret_cast<uint32_t *>(dst) = packed;
                            else
                                for (int j = 0; j < nbyte - c8 / 2; ++j) dst[j] = (uint8_t)(packed >> (8 * j));
                        }
                    }
                    __syncthreads();  // the tile is free for the next slice
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int q = (int)(int8_t)(uint8_t)(pk[i >> 2] >> (8 * (i & 3)));
                        const int64_t row = r0 + i;
                        if (BITS == 8) {
                            if (row < K && col < N) Q[row * ldq + col] = (uint8_t)(int8_t)q;
                        } else {
                            // lanes 2i and 2i + 1 hold columns 2c and 2c + 1: one byte
                            const int qn = __shfl_down_sync(0xffffffffu, q, 1);
                            if (!(lane & 1) && row < K && col < N)
                                Q[row * ldq + col / 2] =
                                    (uint8_t)((q & 0xf) | ((col + 1 < N ? qn & 0xf : 0) << 4));
                        }
                    }
                }
            }
        }
        __syncthreads();  // s_item[k ^ 1] is visible; red and s_sc are free again
    }
    if (t == 0 && s_bad && dstatus) atomicOr(dstatus, BSG_DSTATUS_NONFINITE);
}

// out[k][j] = f32(q * s_j).  grid (column blocks of 1024, row groups); each
// thread takes 4 consecutive columns of one row at a time.  VEC: 4-byte (int8)
// or 2-byte (int4) code loads and 16-byte stores.
template <int BITS, bool VEC>
__global__ void __launch_bounds__(256)
    wdequant_cols_kernel(const uint8_t *__restrict__ Q, int64_t K, int64_t N, int64_t ldq,
                         const float *__restrict__ scale, float *__restrict__ out,
                         int64_t ldo) {
    const int64_t c = ((int64_t)blockIdx.x * 256 + threadIdx.x) * 4;
    if (c >= N) return;
    const bool full4 = c + 3 < N;
    float sv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) sv[u] = c + u < N ? __ldg(scale + c + u) : 0.0f;
    for (int64_t r = blockIdx.y; r < K; r += gridDim.y) {
        const uint8_t *qr = Q + r * ldq;
        int q[4] = {0, 0, 0, 0};
        if (BITS == 8) {
            if (VEC && full4) {
                const char4 v = *reinterpret_cast<const char4 *>(qr + c);
                q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (c + u < N) q[u] = (int8_t)qr[c + u];
            }
        } else {
            uint32_t bytes;
            if (VEC && c + 2 < N)
                bytes = *reinterpret_cast<const uint16_t *>(qr + c / 2);
            else
                bytes = qr[c / 2] | (c + 2 < N ? (uint32_t)qr[c / 2 + 1] << 8 : 0u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int nib = (int)((bytes >> (4 * u)) & 0xfu);
                q[u] = nib >= 8 ? nib - 16 : nib;
            }
        }
        float o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) o[u] = __fmul_rn((float)q[u], sv[u]);
        float *orow = out + r * ldo;
        if (VEC && full4) {
            *reinterpret_cast<float4 *>(orow + c) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c + u < N) orow[c + u] = o[u];
        }
    }
}


template <int BITS, bool POW2, bool VEC>
static cudaError_t launch_wq(const float *W, int64_t K, int64_t N, int64_t ldw, uint8_t *Q,
                            int64_t ldq, int qvec, float *scale, int32_t *dstatus,
                            cudaStream_t st) {
    static bool ready[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev]) {  // clusters of up to 16 CTAs
        const cudaError_t e = cudaFuncSetAttribute(wquant_cols_kernel<BITS, POW2, VEC>,
                                                   cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        ready[dev] = true;
    }
    // a CTA per 256 rows of the strip, at most 16 (longer slices beyond 4096 rows)
    int cs = (int)((K + 255) / 256);
    cs = cs < 1 ? 1 : (cs > 16 ? 16 : cs);
    const int R = (int)((K + cs - 1) / cs);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)((N + kWStrip - 1) / kWStrip), (unsigned)cs, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)cs;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, wquant_cols_kernel<BITS, POW2, VEC>, W, K, N,
                                             ldw, R, Q, ldq, qvec, scale, dstatus);
    count_launches(1);
    return e;
}

template <int BITS, bool POW2>
static cudaError_t launch_wq_vec(const float *W, int64_t K, int64_t N, int64_t ldw, uint8_t *Q,
                                int64_t ldq, int qvec, float *scale, int32_t *dstatus,
                                cudaStream_t st) {
    const bool vec = ldw % 4 == 0 && reinterpret_cast<uintptr_t>(W) % 16 == 0;
    return vec ? launch_wq<BITS, POW2, true>(W, K, N, ldw, Q, ldq, qvec, scale, dstatus, st)
               : launch_wq<BITS, POW2, false>(W, K, N, ldw, Q, ldq, qvec, scale, dstatus, st);
}

template <int BITS, bool POW2>
static cudaError_t launch_wq_lag(const float *W, int64_t K, int64_t N, int64_t ldw, uint8_t *Q,
                                 int64_t ldq, float *scale, uint32_t *ws, int32_t *dstatus,
                                 cudaStream_t st) {
    static int per_sm[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (per_sm[dev] == 0) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, wquant_cols_lag_kernel<BITS, POW2>,
                                                          256, 0);
        if (e != cudaSuccess) return e;
        per_sm[dev] = n > 0 ? n : 1;
    }
    const int64_t P = (N + kLagCols - 1) / kLagCols;
    const int64_t S = ((K + kWqRows - 1) / kWqRows + kLagChunk - 1) / kLagChunk;
    if (2 * P * S >= 0xffff0000LL) return cudaErrorInvalidValue;  // the 32-bit item counter
    int64_t grid = (int64_t)per_sm[dev] * device_sm_count();
    if (grid > 2 * P * S) grid = 2 * P * S;
    e = cudaMemsetAsync(ws, 0, (size_t)(1 + P + N) * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    // whole-piece stores of the code rows: 16 bytes (int8) or 4 (int4)
    const uintptr_t qa = reinterpret_cast<uintptr_t>(Q);
    const int qvec = BITS == 8 ? (ldq % 16 == 0 && qa % 16 == 0) : (ldq % 4 == 0 && qa % 4 == 0);
    wquant_cols_lag_kernel<BITS, POW2><<<(unsigned)grid, 256, 0, st>>>(
        W, K, N, ldw, P, S, colq_lag(K), ws, Q, ldq, qvec, scale, dstatus);
    count_launches(1);
    return cudaGetLastError();
}

// Long columns take the one-read item list (the cluster kernel reads its
// rows twice and waits on two cluster barriers per strip), and so do
// columns of 2048 rows or more in weights of 2^23 elements or more.
// Measured (int8 / int4): 4096 x 4096 61 / 72 us in clusters against
// 52 / 53 us on the list, 2048 x 8192 51 / 59 against 52 / 52-56 us, but
// 3072 x 768 18 / 19 against 21 / 22 us.  BSG_WQ_PATH=cluster|lag forces
// one (same results), for the tests.
static bool wq_use_lag(int64_t K, int64_t N) {
    const char *e = getenv("BSG_WQ_PATH");
    if (e && !strcmp(e, "cluster")) return false;
    if (e && !strcmp(e, "lag")) return true;
    return K > 4096 || (K >= 2048 && K * N >= ((int64_t)1 << 23));
}

}  // namespace

size_t wquant_workspace_bytes(int64_t K, int64_t N) {
    (void)K;
    const size_t words = 1 + (size_t)((N + kLagCols - 1) / kLagCols) + (size_t)N;
    return (words * sizeof(uint32_t) + 255) / 256 * 256;
}

cudaError_t launch_wquant_cols(const float *W, int64_t K, int64_t N, int64_t ldw, int bits,
                               int pow2, void *Q, int64_t ldq, float *scale, void *ws,
                               int32_t *dstatus, cudaStream_t st) {
    if (wq_use_lag(K, N)) {
        uint8_t *q8 = static_cast<uint8_t *>(Q);
        uint32_t *w32 = static_cast<uint32_t *>(ws);
        if (bits == 8)
            return pow2 ? launch_wq_lag<8, true>(W, K, N, ldw, q8, ldq, scale, w32, dstatus, st)
                        : launch_wq_lag<8, false>(W, K, N, ldw, q8, ldq, scale, w32, dstatus, st);
        return pow2 ? launch_wq_lag<4, true>(W, K, N, ldw, q8, ldq, scale, w32, dstatus, st)
                    : launch_wq_lag<4, false>(W, K, N, ldw, q8, ldq, scale, w32, dstatus, st);
    }
    uint8_t *q = static_cast<uint8_t *>(Q);
    const uintptr_t qa = reinterpret_cast<uintptr_t>(Q);
    const int qvec = bits == 8 ? (ldq % 4 == 0 && qa % 4 == 0) : (ldq % 2 == 0 && qa % 2 == 0);
    if (bits == 8)
        return pow2 ? launch_wq_vec<8, true>(W, K, N, ldw, q, ldq, qvec, scale, dstatus, st)
                    : launch_wq_vec<8, false>(W, K, N, ldw, q, ldq, qvec, scale, dstatus, st);
    return pow2 ? launch_wq_vec<4, true>(W, K, N, ldw, q, ldq, qvec, scale, dstatus, st)
                : launch_wq_vec<4, false>(W, K, N, ldw, q, ldq, qvec, scale, dstatus, st);
}

cudaError_t launch_wdequant_cols(const void *Q, int64_t K, int64_t N, int64_t ldq, int bits,
                                 const float *scale, float *out, int64_t ldo, cudaStream_t st) {
    const uint8_t *q = static_cast<const uint8_t *>(Q);
    const uintptr_t qa = reinterpret_cast<uintptr_t>(Q);
    const bool vec = ldo % 4 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0 &&
                     (bits == 8 ? (ldq % 4 == 0 && qa % 4 == 0) : (ldq % 2 == 0 && qa % 2 == 0));
    const int64_t xblocks = (N + 1023) / 1024;
    int64_t yblocks = ((int64_t)device_sm_count() * 16 + xblocks - 1) / xblocks;
    if (yblocks > K) yblocks = K;
    if (yblocks > 65535) yblocks = 65535;
    if (yblocks < 1) yblocks = 1;
    const dim3 grid((unsigned)xblocks, (unsigned)yblocks, 1);
    if (bits == 8) {
        if (vec)
            wdequant_cols_kernel<8, true><<<grid, 256, 0, st>>>(q, K, N, ldq, scale, out, ldo);
        else
            wdequant_cols_kernel<8, false><<<grid, 256, 0, st>>>(q, K, N, ldq, scale, out, ldo);
    } else {
        if (vec)
            wdequant_cols_kernel<4, true><<<grid, 256, 0, st>>>(q, K, N, ldq, scale, out, ldo);
        else
            wdequant_cols_kernel<4, false><<<grid, 256, 0, st>>>(q, K, N, ldq, scale, out, ldo);
    }
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace bsg
