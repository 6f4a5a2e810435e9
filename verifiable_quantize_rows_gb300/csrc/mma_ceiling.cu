// mma_ceiling.cu -- the rate of the contraction's own tensor-core
// instruction with nothing else in the way: the pair MMA (tcgen05
// cta_group::2, kind::f16, 256 x 256 x 16, fp32 accumulators in tensor
// memory) issued back to back from operand tiles that stay in shared
// memory, on every SM pair the GEMM kernel can use.  No operand copies, no
// epilogue, no output.  A measurement aid for the roofline: the ceiling the
// exact GEMM can approach on this GPU at the clock it runs at.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "bsg_internal.h"
#include "bsg_ptx.cuh"

namespace bsg {
namespace {

constexpr int kCeilThreads = 128;
constexpr uint32_t kCeilTile = 128 * 64 * 2;  // A: 128 rows, B: 128 rows (half of 256), 64 f16 deep
constexpr uint32_t kCeilCols = 512;           // two 256-column accumulators
// Shared memory asked for: enough that one CTA fills an SM, so that the
// pairs never share an SM's tensor memory.
constexpr uint32_t kCeilSmem = 200 * 1024;
constexpr uint32_t kCeilIdesc = idesc_f16_f32(256, 256);

__global__ void __launch_bounds__(kCeilThreads, 1) mma_ceiling_kernel(int iters, int32_t *dstatus) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t *tile_a = smem;
    uint8_t *tile_b = smem + kCeilTile;
    uint64_t *done = reinterpret_cast<uint64_t *>(smem + 2 * kCeilTile);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *never = reinterpret_cast<volatile int *>(tmem_ptr + 1);
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_ctarank();

    // zero operands (f16 zeros): the products are exact zeros
    for (uint32_t i = threadIdx.x; i < 2 * kCeilTile / 16; i += kCeilThreads)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        *never = 0;
        fence_mbar_init();
    }
    fence_async_shared();  // the zeros are visible to the tensor core's reads
    if (warp == 1) {
        tmem_alloc_pair(tmem_ptr, kCeilCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_ptr;

    if (rank == 0 && threadIdx.x == 0) {
        const uint64_t adesc = sdesc_k128(smem_u32(tile_a));
        const uint64_t bdesc = sdesc_k128(smem_u32(tile_b));
        for (int it = 0; it < iters; ++it) {
            const uint32_t d = tmem + (uint32_t)(it & 1) * 256u;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_f16_ss_pair(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k),
                                kCeilIdesc, (it >= 2 || k > 0) ? 1u : 0u);
        }
        mma_commit_pair_mc(done, 0x3);
    }
    // both CTAs wait (bounded) until every MMA has finished
    if (threadIdx.x == 0 && !mbar_wait_cl(done, 0, never) && dstatus) atomicOr(dstatus, 2);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kCeilCols);
    }
}

}  // namespace
}  // namespace bsg

using namespace bsg;

extern "C" bsg_status bsg_mma_ceiling(int iters, int32_t *dstatus, double *flops_host,
                                      void *stream) {
    if (iters < 1 || iters > (1 << 18)) return BSG_ERR_ARG;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return BSG_ERR_CUDA;
    if (major != 10 || minor != 3) return BSG_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(mma_ceiling_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kCeilSmem) != cudaSuccess)
        return BSG_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kCeilThreads, 1, 1);
    cfg.dynamicSmemBytes = kCeilSmem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    // as many pairs as can be resident at once (a pair needs two SMs of one GPC)
    int pairs = device_sm_count() / 2;
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mma_ceiling_kernel, &cfg) == cudaSuccess && n > 0 &&
        n < pairs)
        pairs = n;
    cudaGetLastError();
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    if (flops_host) *flops_host = (double)pairs * iters * 4.0 * (2.0 * 256 * 256 * 16);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mma_ceiling_kernel, iters, dstatus);
    count_launches(1);
    return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}
