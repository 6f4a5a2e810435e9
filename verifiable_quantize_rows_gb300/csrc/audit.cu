// audit.cu -- the live audit: sampled output cells recomputed by a path that
// shares nothing with the quantize and tensor-core kernels.
//
// "Verification -- why you can trust the numbers", section "Layer 2: the live
// audit": cells of a live GEMM, chosen at random, are recomputed
// independently and compared bit for bit; section "Layer 1: exact init gates"
// uses the same comparison on fixed inputs before the kernels are trusted
// (bsg_selftest).
//
// The independent path runs on the CUDA cores, one warp per sampled cell:
//   * it reads the cell's row of A and column of B straight from the f32
//     inputs (no quantized operand, no scale array of the main path);
//   * it derives both scales from the f64 definition -- scale =
//     f32(max(f64(m) / 127, 1e-8)), inv = f32(1 / f64(scale)) -- where the main
//     path uses f32 divides proven equal to it;
//   * it quantizes every element with two f32 roundings and a floor, without
//     the main path's clamp, and sums the products in int64 on the integer
//     units, where the main path accumulates in fp32 on the tensor cores;
//   * it applies f32(f32(f32(S) * a) * b) and the ReLU and compares the bits
//     with C.
// Cells whose row or column holds a non-finite value are skipped (their
// output is unspecified).  The cells come from SplitMix64 (Steele, Lea, Flood,
// OOPSLA 2014) seeded by the caller: output 2s picks sample s's row (mod M),
// output 2s + 1 its column (mod N).
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsg_internal.h"

namespace bsg {
namespace {

__device__ __forceinline__ uint64_t audit_splitmix(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1ull) * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// The f64 definition of the scale and its reciprocal from an absmax.
__device__ __forceinline__ void audit_scale(float m, float &scale, float &inv) {
    double s = __ddiv_rn((double)m, 127.0);
    if (s < 1e-8) s = 1e-8;
    scale = __double2float_rn(s);
    inv = __double2float_rn(__ddiv_rn(1.0, (double)scale));
}

__device__ __forceinline__ int audit_q(float x, float inv) {
    return (int)floorf(__fadd_rn(__fmul_rn(x, inv), 0.5f));
}

constexpr int kAuditWarps = 8;

__global__ void __launch_bounds__(kAuditWarps * 32)
    audit_kernel(const float *__restrict__ A, int64_t lda, const float *__restrict__ B,
                 int64_t ldb, const float *__restrict__ C, int64_t ldc, int64_t M, int64_t N,
                 int64_t K, int relu, uint64_t seed, int nsamples,
                 uint32_t *__restrict__ mismatches, int64_t *__restrict__ cells) {
    const int s = blockIdx.x * kAuditWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= nsamples) return;
    const int64_t i = (int64_t)(audit_splitmix(seed, 2ull * (uint64_t)s) % (uint64_t)M);
    const int64_t j = (int64_t)(audit_splitmix(seed, 2ull * (uint64_t)s + 1ull) % (uint64_t)N);
    const float *arow = A + i * lda;
    const float *bcol = B + j;
    float ma = 0.0f, mb = 0.0f;
    bool finite = true;
    for (int64_t k = lane; k < K; k += 32) {
        const float a = arow[k], b = bcol[k * ldb];
        finite = finite && isfinite(a) && isfinite(b);
        ma = fmaxf(ma, fabsf(a));
        mb = fmaxf(mb, fabsf(b));
    }
    for (int o = 16; o > 0; o >>= 1) {
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, o));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    }
    finite = __all_sync(0xffffffffu, finite);
    float sa, ia, sb, ib;
    audit_scale(ma, sa, ia);
    audit_scale(mb, sb, ib);
    long long acc = 0;
    for (int64_t k = lane; k < K; k += 32)
        acc += (long long)audit_q(arow[k], ia) * (long long)audit_q(bcol[k * ldb], ib);
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        if (cells) {
            cells[2 * (int64_t)s] = i;
            cells[2 * (int64_t)s + 1] = j;
        }
        if (finite) {
            float c = __fmul_rn(__fmul_rn(__ll2float_rn(acc), sa), sb);
            if (relu) c = c > 0.0f ? c : 0.0f;
            if (__float_as_uint(c) != __float_as_uint(C[i * ldc + j])) atomicAdd(mismatches, 1u);
        }
    }
}

}  // namespace

cudaError_t launch_audit(const float *A, int64_t lda, const float *B, int64_t ldb, const float *C,
                         int64_t ldc, int64_t M, int64_t N, int64_t K, int relu, uint64_t seed,
                         int nsamples, uint32_t *mismatches, int64_t *cells, cudaStream_t st) {
    const int blocks = (nsamples + kAuditWarps - 1) / kAuditWarps;
    audit_kernel<<<blocks, kAuditWarps * 32, 0, st>>>(A, lda, B, ldb, C, ldc, M, N, K, relu, seed,
                                                      nsamples, mismatches, cells);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace bsg
