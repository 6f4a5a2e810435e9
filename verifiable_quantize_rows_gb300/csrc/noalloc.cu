// noalloc.cu -- bsgemm_i8 for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: a host framework that
// owns every device allocation through its own pool and lends none to
// extensions, or an embedding in which the library may not touch the
// allocator at all (a plug-in loaded into someone else's process, a
// real-time loop that forbids allocation after start-up).  For them this
// file keeps the unit's scratch in a device array compiled into the library
// and runs the ordinary unit on it.  Nothing here allocates: the array exists
// from the moment the library's module is loaded on a device until the
// process exits (every GPU that loads it holds BSG_NOALLOC_SCRATCH_BYTES).
#include <cuda.h>
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
struct Cached {
    void *addr;
    unsigned long long ctx_id;  // the context the address belongs to
};
Cached g_cached[kMaxDevices] = {};

// Identity of the current context (0 if it cannot be read).  A context that
// is destroyed and created again (cudaDeviceReset) gets a new id, and its
// module -- with the array -- may be loaded at another address.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch on the current device.  Looked up with that
// device current on the first call there (cudaGetSymbolAddress, which also
// makes the runtime set up its context), then cached; looked up again only
// if the device's context has been replaced since.
bsg_status scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSG_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    Cached &c = g_cached[dev];
    const unsigned long long id = c.addr ? current_ctx_id() : 0;
    if (!c.addr || id != c.ctx_id) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            c.addr = nullptr;
            return BSG_ERR_CUDA;
        }
        c.addr = p;
        c.ctx_id = current_ctx_id();
    }
    *addr = c.addr;
    return BSG_OK;
}

}  // namespace

extern "C" bsg_status bsgemm_i8_noalloc(const float *A, const float *B, int64_t M, int64_t N,
                                        int64_t K, int relu, float *C, int32_t *dstatus,
                                        void *stream) {
    if (!A || !B || !C || M < 1 || N < 1 || K < 1) return BSG_ERR_ARG;
    if (K > BSG_MAX_K) return BSG_ERR_K_TOO_LARGE;
    // the layout this entry point runs: A and B as stored, not transposed
    const size_t need = bsg::unit_workspace_bytes(M, N, K, 0, 0);
    if (need == 0) return BSG_ERR_ARG;
    if (need > (size_t)BSG_NOALLOC_SCRATCH_BYTES) return BSG_ERR_WORKSPACE;
    void *scratch = nullptr;
    const bsg_status s = scratch_address(&scratch);
    if (s != BSG_OK) return s;
    // What the unit reads from the scratch is written earlier in the same
    // call (operands, scales, partial maxima, the zeroed tile counter), except
    // the column scales past N, which the epilogue loads for whole tiles but
    // applies to no stored column; so nothing needs clearing between calls.
    // overlap = false: the second quantize stream would be a created object
    return bsg::run_unit(A, K, 0, B, N, 0, M, N, K, relu, C, N, scratch,
                         (size_t)BSG_NOALLOC_SCRATCH_BYTES, dstatus,
                         static_cast<cudaStream_t>(stream), false);
}
