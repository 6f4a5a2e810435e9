// noalloc.cu -- bsgemm_i8 for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: a host framework that
// owns every device allocation through its own pool and exposes none to
// extensions, code that runs while a stream is being captured into a CUDA
// graph (where it must not call cudaMalloc), or an embedding in which the
// library may not touch the allocator at all.  For them this file keeps the
// unit's scratch in a device array compiled into the library and runs the
// ordinary bsgemm_i8 on it.  Nothing here allocates: the array exists from
// the moment the library's module is loaded on a device until the process
// exits (every GPU that loads it holds BSG_NOALLOC_SCRATCH_BYTES).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "bsg_internal.h"
#include "bsgemm.h"

namespace {

// The scratch itself.  In host code this name only stands in for the
// device array; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BSG_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
bsg_status scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSG_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return BSG_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return BSG_OK;
}

}  // namespace

extern "C" bsg_status bsgemm_i8_noalloc(const float *A, const float *B, int64_t M, int64_t N,
                                        int64_t K, int relu, float *C, int32_t *dstatus,
                                        void *stream) {
    if (!A || !B || !C || M < 1 || N < 1 || K < 1) return BSG_ERR_ARG;
    if (K > BSG_MAX_K) return BSG_ERR_K_TOO_LARGE;
    const size_t need = bsgemm_i8_workspace_size(M, N, K);
    if (need == 0) return BSG_ERR_ARG;
    if (need > (size_t)BSG_NOALLOC_SCRATCH_BYTES) return BSG_ERR_WORKSPACE;
    void *scratch = nullptr;
    const bsg_status s = scratch_address(&scratch);
    if (s != BSG_OK) return s;
    // Every byte of the scratch that the unit reads is written earlier in
    // the same call (operands, scales, partial maxima), so nothing needs
    // clearing between calls.
    // overlap = false: the second quantize stream would be a created object
    return bsg::run_unit(A, K, 0, B, N, 0, M, N, K, relu, C, N, scratch,
                         (size_t)BSG_NOALLOC_SCRATCH_BYTES, dstatus,
                         static_cast<cudaStream_t>(stream), false);
}
