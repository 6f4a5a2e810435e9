// epilogue.cu -- the standalone epilogue over stored int32 accumulators.
//
// "Verification -- why you can trust the numbers", section "The verified
// INT8 units", step 3: epi(s,a,b) = f32(f32(f32(s)*a)*b), rounding to f32
// after the int->float conversion and after each multiply; section "Layer
// 5": a fused-ReLU output is never negative (-0 and NaN become +0).
// Only __int2float_rn and __fmul_rn are used: no contraction, no flush to
// zero, so signed zeros and subnormals come out as IEEE-754 defines them.
#include <stdint.h>

#include "bsg_internal.h"

namespace bsg {
namespace {

__global__ void __launch_bounds__(256)
    epilogue_kernel(const int32_t *__restrict__ S, int64_t lds, const float *__restrict__ sa,
                    const float *__restrict__ sb, int64_t M, int64_t N, int relu,
                    float *__restrict__ C, int64_t ldc) {
    const int64_t total = M * N;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / N, j = e - i * N;
        const float c = __fmul_rn(__fmul_rn(__int2float_rn(S[i * lds + j]), sa[i]), sb[j]);
        C[i * ldc + j] = relu ? (c > 0.0f ? c : 0.0f) : c;
    }
}

}  // namespace

cudaError_t launch_epilogue(const int32_t *S, int64_t lds, const float *sa, const float *sb,
                            int64_t M, int64_t N, int relu, float *C, int64_t ldc,
                            cudaStream_t st) {
    const int64_t blocks = (M * N + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    const int grid = (int)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
    epilogue_kernel<<<grid, 256, 0, st>>>(S, lds, sa, sb, M, N, relu, C, ldc);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace bsg
