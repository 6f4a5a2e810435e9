// bsgemm_api.cu -- the C ABI: argument checks, workspace layout, launches.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "bsg_internal.h"
#include "bsgemm.h"

namespace bsg {

static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

int device_sm_count() {
    static int count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (count[dev] == 0) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
            c = 148;
        count[dev] = c;
    }
    return count[dev];
}

namespace {

// The kernels are built for sm_103a only.
bsg_status check_device() {
    static int ok[64] = {0};  // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BSG_ERR_CUDA;
    if (ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return BSG_ERR_CUDA;
        ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return ok[dev] == 1 ? BSG_OK : BSG_ERR_UNSUPPORTED;
}

bsg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA; }

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the whole unit:
//   Aop  f16 [M][ldk]        (ldk = K rounded up to 64)
//   Bop  f16 [N][ldk]
//   sa   f32 [round_up(M, 128)]
//   sb   f32 [round_up(N, 256) + 256] (a tile of any width may read its
//        whole last tile of scales; entries past N are never used)
//   the GEMM's tile counter (one uint32 in 256 bytes)
//   column-quantize scratch (uint32: partial or whole column maxima and
//   the one-read path's counters) of op(A), then of op(B), for columns
//   longer than the strip kernel holds (separate, since the two operands
//   may be quantized at the same time)
struct UnitLayout {
    size_t aop, bop, sa, sb, ticket, part, part_b, total;
};

UnitLayout unit_layout(int64_t M, int64_t N, int64_t K, int transA, int transB) {
    UnitLayout L;
    const int64_t ldk = operand_ld(K);
    size_t off = 0;
    L.aop = off;
    off = align256(off + (size_t)M * ldk * 2);
    L.bop = off;
    off = align256(off + (size_t)N * ldk * 2);
    L.sa = off;
    off = align256(off + (size_t)round_up(M, kBM) * 4);
    L.sb = off;
    off = align256(off + (size_t)(round_up(N, kBN) + kBN) * 4);
    L.ticket = off;  // the GEMM's tile counter
    off += 256;
    L.part = off;
    if (transA) off = align256(off + colmax_partial_bytes(K, M));
    L.part_b = off;
    if (!transB) off = align256(off + colmax_partial_bytes(K, N));
    L.total = off;
    return L;
}

bool ws_ok(const void *ws, size_t have, size_t need) {
    return ws != nullptr && (reinterpret_cast<uintptr_t>(ws) % 256) == 0 && have >= need;
}

// Sizes the kernels index: M, N below 2^31, and C at most 2^40 elements (4 TiB
// of f32, beyond any GPU's memory), which keeps every tile count and element
// offset inside the kernels' integer types.
bool dims_ok(int64_t M, int64_t N, int64_t K) {
    return M >= 1 && N >= 1 && K >= 1 && M <= INT32_MAX && N <= INT32_MAX &&
           M <= (int64_t(1) << 40) / N;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

bsg_status check_unit_args(const float *A, int64_t lda, int transA, const float *B, int64_t ldb,
                           int transB, int64_t M, int64_t N, int64_t K) {
    if (!A || !B) return BSG_ERR_ARG;
    if (!dims_ok(M, N, K)) return BSG_ERR_ARG;
    if (K > BSG_MAX_K) return BSG_ERR_K_TOO_LARGE;
    if (transA ? lda < M : lda < K) return BSG_ERR_ARG;
    if (transB ? ldb < K : ldb < N) return BSG_ERR_ARG;
    return BSG_OK;
}

// A second stream per device on which op(B) is quantized while op(A) is
// quantized on the caller's stream: the two kernels are independent, and
// the smaller one (usually the weight) is latency-bound, so running it beside
// the larger one hides it.  It is forked from and joined back into the
// caller's stream with two events, which also works while the caller's
// stream is being captured into a CUDA graph (the side stream joins the
// capture).  Created on the first call on each device and kept until the
// process exits; one host thread at a time uses it.
struct SideStream {
    cudaStream_t st = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool tried = false;
};
std::mutex g_side_lock;
SideStream g_side[64];

// The side stream of the current device, or nullptr if it could not be
// created (the operands are then quantized one after the other).  Called
// with g_side_lock held.
SideStream *side_stream() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    SideStream &s = g_side[dev];
    if (!s.tried) {
        s.tried = true;
        int least = 0, greatest = 0;
        cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (cudaStreamCreateWithPriority(&s.st, cudaStreamNonBlocking, greatest) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            s.st = nullptr;
        }
    }
    return s.st ? &s : nullptr;
}

// Step 1 into the workspace: op(A) per row, op(B) per column, as f16
// K-major operands plus scales.  With `overlap`, op(B) is quantized on the
// side stream at the same time as op(A).
bsg_status unit_quantize(const float *A, int64_t lda, int transA, const float *B, int64_t ldb,
                         int transB, int64_t M, int64_t N, int64_t K, void *ws, size_t ws_bytes,
                         int32_t *dstatus, cudaStream_t st, bool overlap = true,
                         unsigned int *zrows = nullptr) {
    bsg_status s = check_unit_args(A, lda, transA, B, ldb, transB, M, N, K);
    if (s != BSG_OK) return s;
    const UnitLayout L = unit_layout(M, N, K, transA, transB);
    if (!ws_ok(ws, ws_bytes, L.total)) return BSG_ERR_WORKSPACE;
    s = check_device();
    if (s != BSG_OK) return s;
    const int64_t ldk = operand_ld(K);
    __half *aop = at<__half>(ws, L.aop);
    __half *bop = at<__half>(ws, L.bop);
    float *sa = at<float>(ws, L.sa);
    float *sb = at<float>(ws, L.sb);
    uint32_t *part_a = at<uint32_t>(ws, L.part);
    uint32_t *part_b = at<uint32_t>(ws, L.part_b);
    // The GEMM claims tiles from a counter in the workspace that must start
    // at zero: the quantize launch of op(A) zeroes it (the GEMM sets it back
    // to zero whenever it completes).
    unsigned int *ticket = at<unsigned int>(ws, L.ticket);
    if (transA && cudaMemsetAsync(ticket, 0, 2 * sizeof(unsigned int), st) != cudaSuccess)
        return BSG_ERR_CUDA;
    // zrows (the chained units' row maxima of C, one word per row of op(A))
    // is zeroed by op(A)'s row quantize; a column quantize of a stored A^T
    // cannot, so it is cleared here
    if (zrows && transA && cudaMemsetAsync(zrows, 0, (size_t)M * 4, st) != cudaSuccess)
        return BSG_ERR_CUDA;
    // op(A) per row: a row quantize of A, or a column quantize of the stored K x M.
    auto quant_a = [&](cudaStream_t s) {
        return !transA ? launch_quantize_rows(A, M, K, lda, kOutHalfKMajor, aop, ldk, sa, nullptr,
                                              dstatus, s, ticket, zrows)
                       : launch_quantize_cols(A, K, M, lda, kOutHalfKMajor, aop, ldk, sa, nullptr,
                                              part_a, dstatus, s);
    };
    // op(B) per column: a column quantize of B, or a row quantize of the stored N x K.
    auto quant_b = [&](cudaStream_t s) {
        return !transB ? launch_quantize_cols(B, K, N, ldb, kOutHalfKMajor, bop, ldk, sb, nullptr,
                                              part_b, dstatus, s)
                       : launch_quantize_rows(B, N, K, ldb, kOutHalfKMajor, bop, ldk, sb, nullptr,
                                              dstatus, s);
    };
    if (!transA && !transB) {
        // the common layout: one launch for both operands
        const cudaError_t ef = launch_quantize_ab(A, M, K, lda, B, N, ldb, aop, bop, ldk, sa, sb,
                                                  dstatus, ticket, st, zrows);
        if (ef == cudaSuccess) return BSG_OK;
        if (ef != cudaErrorNotSupported) return BSG_ERR_CUDA;
    }
    if (overlap) {
        std::lock_guard<std::mutex> guard(g_side_lock);
        SideStream *side = side_stream();
        if (side) {
            if (cudaEventRecord(side->fork, st) != cudaSuccess ||
                cudaStreamWaitEvent(side->st, side->fork, 0) != cudaSuccess)
                return BSG_ERR_CUDA;
            const cudaError_t eb = quant_b(side->st);
            const cudaError_t ea = quant_a(st);
            // join even after a failed launch, so that no captured fork is left open
            const cudaError_t ej = cudaEventRecord(side->join, side->st);
            const cudaError_t ew = ej == cudaSuccess ? cudaStreamWaitEvent(st, side->join, 0) : ej;
            return (ea == cudaSuccess && eb == cudaSuccess && ew == cudaSuccess) ? BSG_OK
                                                                                 : BSG_ERR_CUDA;
        }
    }
    if (quant_a(st) != cudaSuccess) return BSG_ERR_CUDA;
    return quant_b(st) == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}

// Steps 2-3 from the workspace: the tensor-core contraction with the fused
// epilogue.
bsg_status unit_contract(int64_t M, int64_t N, int64_t K, int relu, float *C, int64_t ldc,
                         void *ws, size_t ws_bytes, int32_t *dstatus, cudaStream_t st,
                         int tile_width = 0) {
    if (!C || !dims_ok(M, N, K) || ldc < N) return BSG_ERR_ARG;
    if (K > BSG_MAX_K) return BSG_ERR_K_TOO_LARGE;
    const UnitLayout L = unit_layout(M, N, K, 0, 0);
    if (!ws_ok(ws, ws_bytes, L.part)) return BSG_ERR_WORKSPACE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    return from_cuda(launch_gemm_tc(at<__half>(ws, L.aop), at<__half>(ws, L.bop), M, N, K,
                                    at<float>(ws, L.sa), at<float>(ws, L.sb), relu, 0, C, ldc,
                                    dstatus, at<unsigned int>(ws, L.ticket), st, tile_width));
}

}  // namespace

size_t unit_workspace_bytes(int64_t M, int64_t N, int64_t K, int transA, int transB) {
    if (!dims_ok(M, N, K)) return 0;
    return unit_layout(M, N, K, transA, transB).total;
}

bsg_status run_unit(const float *A, int64_t lda, int transA, const float *B, int64_t ldb,
                    int transB, int64_t M, int64_t N, int64_t K, int relu, float *C, int64_t ldc,
                    void *ws, size_t ws_bytes, int32_t *dstatus, cudaStream_t st, bool overlap) {
    if (!C || ldc < N) return BSG_ERR_ARG;
    bsg_status s = unit_quantize(A, lda, transA, B, ldb, transB, M, N, K, ws, ws_bytes, dstatus,
                                 st, overlap);
    if (s != BSG_OK) return s;
    return unit_contract(M, N, K, relu, C, ldc, ws, ws_bytes, dstatus, st);
}

namespace {
bsg_status unit(const float *A, int64_t lda, int transA, const float *B, int64_t ldb,
                int transB, int64_t M, int64_t N, int64_t K, int relu, float *C, int64_t ldc,
                void *ws, size_t ws_bytes, int32_t *dstatus, cudaStream_t st) {
    return run_unit(A, lda, transA, B, ldb, transB, M, N, K, relu, C, ldc, ws, ws_bytes, dstatus,
                    st, true);
}
}  // namespace
}  // namespace bsg

using namespace bsg;

extern "C" {

const char *bsg_status_str(bsg_status s) {
    switch (s) {
        case BSG_OK: return "BSG_OK";
        case BSG_ERR_ARG: return "BSG_ERR_ARG: invalid argument";
        case BSG_ERR_K_TOO_LARGE: return "BSG_ERR_K_TOO_LARGE: K > 133144 can overflow int32";
        case BSG_ERR_WORKSPACE: return "BSG_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case BSG_ERR_CUDA: return "BSG_ERR_CUDA: a CUDA call failed";
        case BSG_ERR_NONFINITE: return "BSG_ERR_NONFINITE: non-finite input";
        case BSG_ERR_TIMEOUT: return "BSG_ERR_TIMEOUT: a bounded device wait expired";
        case BSG_ERR_UNSUPPORTED: return "BSG_ERR_UNSUPPORTED: device is not sm_103";
        case BSG_ERR_SELFTEST: return "BSG_ERR_SELFTEST: the self-test found a wrong result";
    }
    return "unknown bsg_status";
}

int bsg_version(void) { return 100; }

bsg_status bsg_quantize_rows(const float *X, int64_t rows, int64_t cols, int64_t ldx, int8_t *Q,
                             int64_t ldq, float *scale, float *inv, int32_t *dstatus,
                             void *stream) {
    if (!X || !Q || !scale || rows < 1 || cols < 1 || ldx < cols || ldq < cols) return BSG_ERR_ARG;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    return from_cuda(launch_quantize_rows(X, rows, cols, ldx, kOutInt8, Q, ldq, scale, inv,
                                          dstatus, static_cast<cudaStream_t>(stream)));
}

size_t bsg_quantize_cols_workspace_size(int64_t rows, int64_t cols) {
    if (rows < 1 || cols < 1) return 0;
    return align256(colmax_partial_bytes(rows, cols));
}

bsg_status bsg_quantize_cols(const float *X, int64_t rows, int64_t cols, int64_t ldx, int8_t *Q,
                             int64_t ldq, float *scale, float *inv, void *workspace,
                             size_t ws_bytes, int32_t *dstatus, void *stream) {
    if (!X || !Q || !scale || rows < 1 || cols < 1 || ldx < cols || ldq < cols) return BSG_ERR_ARG;
    if (!ws_ok(workspace, ws_bytes, bsg_quantize_cols_workspace_size(rows, cols)))
        return BSG_ERR_WORKSPACE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    return from_cuda(launch_quantize_cols(X, rows, cols, ldx, kOutInt8, Q, ldq, scale, inv,
                                          static_cast<uint32_t *>(workspace), dstatus,
                                          static_cast<cudaStream_t>(stream)));
}

size_t bsg_gemm_s32_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (!dims_ok(M, N, K)) return 0;
    const int64_t ldk = operand_ld(K);
    return align256((size_t)M * ldk * 2) + align256((size_t)N * ldk * 2) + 256;  // + tile counter
}

bsg_status bsg_gemm_s32(const int8_t *Aq, int64_t lda, const int8_t *Bq, int64_t ldb, int64_t M,
                        int64_t N, int64_t K, int32_t *S, int64_t lds, void *workspace,
                        size_t ws_bytes, int32_t *dstatus, void *stream) {
    if (!Aq || !Bq || !S || !dims_ok(M, N, K) || lda < K || ldb < N || lds < N) return BSG_ERR_ARG;
    if (K > BSG_MAX_K) return BSG_ERR_K_TOO_LARGE;
    if (!ws_ok(workspace, ws_bytes, bsg_gemm_s32_workspace_size(M, N, K))) return BSG_ERR_WORKSPACE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t ldk = operand_ld(K);
    __half *aop = static_cast<__half *>(workspace);
    __half *bop = at<__half>(workspace, align256((size_t)M * ldk * 2));
    if (launch_i8_rows_to_half(Aq, M, K, lda, aop, ldk, st) != cudaSuccess) return BSG_ERR_CUDA;
    if (launch_i8_cols_to_half(Bq, K, N, ldb, bop, ldk, st) != cudaSuccess) return BSG_ERR_CUDA;
    unsigned int *ticket =
        at<unsigned int>(workspace, align256((size_t)M * ldk * 2) + align256((size_t)N * ldk * 2));
    if (cudaMemsetAsync(ticket, 0, 2 * sizeof(unsigned int), st) != cudaSuccess) return BSG_ERR_CUDA;
    return from_cuda(
        launch_gemm_tc(aop, bop, M, N, K, nullptr, nullptr, 0, 1, S, lds, dstatus, ticket, st));
}

bsg_status bsg_epilogue(const int32_t *S, int64_t lds, const float *sa, const float *sb,
                        int64_t M, int64_t N, int relu, float *C, int64_t ldc, void *stream) {
    if (!S || !sa || !sb || !C || M < 1 || N < 1 || lds < N || ldc < N) return BSG_ERR_ARG;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    return from_cuda(
        launch_epilogue(S, lds, sa, sb, M, N, relu, C, ldc, static_cast<cudaStream_t>(stream)));
}

size_t bsgemm_i8_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (!dims_ok(M, N, K)) return 0;
    // large enough for every transpose combination
    const size_t a = unit_layout(M, N, K, 0, 0).total;
    const size_t b = unit_layout(M, N, K, 1, 0).total;
    return a > b ? a : b;
}

bsg_status bsgemm_i8(const float *A, const float *B, int64_t M, int64_t N, int64_t K, int relu,
                     float *C, void *workspace, size_t ws_bytes, int32_t *dstatus,
                     void *stream) {
    return unit(A, K, 0, B, N, 0, M, N, K, relu, C, N, workspace, ws_bytes, dstatus,
                static_cast<cudaStream_t>(stream));
}

bsg_status bsgemm_i8_ex(const float *A, int64_t lda, int transA, const float *B, int64_t ldb,
                        int transB, int64_t M, int64_t N, int64_t K, int relu, float *C,
                        int64_t ldc, void *workspace, size_t ws_bytes, int32_t *dstatus,
                        void *stream) {
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return BSG_ERR_ARG;
    return unit(A, lda, transA, B, ldb, transB, M, N, K, relu, C, ldc, workspace, ws_bytes,
                dstatus, static_cast<cudaStream_t>(stream));
}

bsg_status bsgemm_i8_group(const bsg_gemm_item *items, int count, int32_t *dstatus,
                           void *stream) {
    if (!items || count < 1 || count > BSG_MAX_GROUP) return BSG_ERR_ARG;
    for (int i = 0; i < count; ++i) {
        const bsg_gemm_item &it = items[i];
        if ((it.transA != 0 && it.transA != 1) || (it.transB != 0 && it.transB != 1))
            return BSG_ERR_ARG;
        bsg_status s = check_unit_args(it.A, it.lda, it.transA, it.B, it.ldb, it.transB, it.M,
                                       it.N, it.K);
        if (s != BSG_OK) return s;
        if (!it.C || it.ldc < it.N || (it.relu != 0 && it.relu != 1)) return BSG_ERR_ARG;
        if (!ws_ok(it.workspace, it.ws_bytes, bsgemm_i8_workspace_size(it.M, it.N, it.K)))
            return BSG_ERR_WORKSPACE;
    }
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    GemmJob jobs[BSG_MAX_GROUP];
    for (int i = 0; i < count; ++i) {
        const bsg_gemm_item &it = items[i];
        s = unit_quantize(it.A, it.lda, it.transA, it.B, it.ldb, it.transB, it.M, it.N, it.K,
                          it.workspace, it.ws_bytes, dstatus, st);
        if (s != BSG_OK) return s;
        const UnitLayout L = unit_layout(it.M, it.N, it.K, 0, 0);
        jobs[i].Aop = at<__half>(it.workspace, L.aop);
        jobs[i].Bop = at<__half>(it.workspace, L.bop);
        jobs[i].M = it.M;
        jobs[i].N = it.N;
        jobs[i].K = it.K;
        jobs[i].sa = at<float>(it.workspace, L.sa);
        jobs[i].sb = at<float>(it.workspace, L.sb);
        jobs[i].relu = it.relu;
        jobs[i].out = it.C;
        jobs[i].ldo = it.ldc;
    }
    // the tile counter of the first item's workspace (its quantize zeroed it)
    const UnitLayout L0 = unit_layout(items[0].M, items[0].N, items[0].K, 0, 0);
    return from_cuda(launch_gemm_tc_group(jobs, count, 0, dstatus,
                                          at<unsigned int>(items[0].workspace, L0.ticket), st));
}

bsg_status bsgemm_i8_quantize(const float *A, int64_t lda, int transA, const float *B,
                              int64_t ldb, int transB, int64_t M, int64_t N, int64_t K,
                              void *workspace, size_t ws_bytes, int32_t *dstatus, void *stream) {
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return BSG_ERR_ARG;
    return unit_quantize(A, lda, transA, B, ldb, transB, M, N, K, workspace, ws_bytes, dstatus,
                         static_cast<cudaStream_t>(stream));
}

bsg_status bsgemm_i8_contract(int64_t M, int64_t N, int64_t K, int relu, float *C, int64_t ldc,
                              void *workspace, size_t ws_bytes, int32_t *dstatus, void *stream) {
    return unit_contract(M, N, K, relu, C, ldc, workspace, ws_bytes, dstatus,
                         static_cast<cudaStream_t>(stream));
}

bsg_status bsg_selftest_scales(uint32_t first_bits, uint32_t last_bits,
                               uint64_t *mismatches_host) {
    if (!mismatches_host || first_bits > last_bits) return BSG_ERR_ARG;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    unsigned long long *d = nullptr;
    if (cudaMalloc(&d, sizeof(*d)) != cudaSuccess) return BSG_ERR_CUDA;
    unsigned long long h = 0;
    cudaError_t e = cudaMemset(d, 0, sizeof(*d));
    if (e == cudaSuccess) e = launch_selftest_scales(first_bits, last_bits, d, 0);
    if (e == cudaSuccess) e = cudaMemcpy(&h, d, sizeof(h), cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return BSG_ERR_CUDA;
    *mismatches_host = h;
    return BSG_OK;
}

int bsg_gemm_tile_width(int64_t M, int64_t N, int sms) {
    if (M < 1 || N < 1 || sms < 1) return -1;
    return gemm_tile_width(M, N, sms);
}

uint64_t bsg_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

// Host-buffer form: device copies of A, B, C and a status word sit in front
// of the unit's own workspace.
static size_t host_prefix(int64_t M, int64_t N, int64_t K) {
    return align256((size_t)M * K * 4) + align256((size_t)K * N * 4) +
           align256((size_t)M * N * 4) + 256;
}

size_t bsgemm_i8_host_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (!dims_ok(M, N, K)) return 0;
    return host_prefix(M, N, K) + bsgemm_i8_workspace_size(M, N, K);
}

}  // extern "C"

namespace bsg {
namespace {

// Copy streams of the host-buffer entry point, one pair per device: uploads
// on one, downloads on the other, so that both directions of the link and the
// kernels on the caller's stream run at once.  Created on the first call on
// each device and kept until the process exits; one host thread at a time
// uses them (the entry point is synchronous).
// A in 4 row chunks per unit: 2, 3, 4, 6, 8 and 16 were measured, and 4 gave the
// shortest batch of the three GPT-2 linears (1.39 against 1.43 ms at 8) with
// no single unit slower; two copy streams per direction were slower still.
constexpr int kHostChunks = 4;
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, b_in = nullptr, done = nullptr;
    cudaEvent_t a_in[kHostChunks] = {}, c_ready[kHostChunks] = {};
    bool tried = false;
};
std::mutex g_host_lock;
HostPipe g_host[64];

HostPipe *host_pipe() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    HostPipe &h = g_host[dev];
    if (!h.tried) {
        h.tried = true;
        bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.b_in, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&h.done, cudaEventDisableTiming) == cudaSuccess;
        for (int c = 0; ok && c < kHostChunks; ++c)
            ok = cudaEventCreateWithFlags(&h.a_in[c], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&h.c_ready[c], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            h.in = nullptr;
        }
    }
    return h.in ? &h : nullptr;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return na && nb && pa < pb + nb && pb < pa + na;
}

// Byte offset of the status word inside a host-entry workspace.
size_t host_status_offset(int64_t M, int64_t N, int64_t K) {
    return align256((size_t)M * K * 4) + align256((size_t)K * N * 4) + align256((size_t)M * N * 4);
}

// One unit on host buffers, enqueued: B and then A in row chunks upload on
// h->in; on `st`, B is quantized per column once, then per chunk the rows of
// A and the GEMM of those rows; each chunk of C downloads on h->out as soon
// as its GEMM is done.  A chunk is a multiple of 256 rows (the GEMM's pair
// tile).  Per-row quantize and the GEMM's tiling do not depend on the
// chunking, so neither does any bit of C.  The events of `h` are re-recorded
// per item; every wait is enqueued right after the record it pairs with.
cudaError_t host_enqueue(const bsg_host_item &it, int32_t *dstat, cudaStream_t st, HostPipe *h) {
    const int64_t M = it.M, N = it.N, K = it.K;
    size_t off = 0;
    float *dA = at<float>(it.workspace, off);
    off += align256((size_t)M * K * 4);
    float *dB = at<float>(it.workspace, off);
    off += align256((size_t)K * N * 4);
    float *dC = at<float>(it.workspace, off);
    off += align256((size_t)M * N * 4);
    off += 256;  // the status word
    void *uws = at<void>(it.workspace, off);
    const UnitLayout L = unit_layout(M, N, K, 0, 0);
    const int64_t ldk = operand_ld(K);
    __half *aop = at<__half>(uws, L.aop);
    __half *bop = at<__half>(uws, L.bop);
    float *sa = at<float>(uws, L.sa);
    float *sb = at<float>(uws, L.sb);
    unsigned int *ticket = at<unsigned int>(uws, L.ticket);
    uint32_t *part_b = at<uint32_t>(uws, L.part_b);
    int64_t rows = (M + kHostChunks - 1) / kHostChunks;
    rows = (rows + 255) / 256 * 256;
    const int nchunks = (int)((M + rows - 1) / rows);
    cudaError_t e;
#define BSG_TRY(x)                         \
    if ((e = (x)) != cudaSuccess) return e;
    BSG_TRY(cudaMemcpyAsync(dB, it.B_host, (size_t)K * N * 4, cudaMemcpyHostToDevice, h->in));
    BSG_TRY(cudaEventRecord(h->b_in, h->in));
    for (int c = 0; c < nchunks; ++c) {
        const int64_t r0 = c * rows, mc = M - r0 < rows ? M - r0 : rows;
        BSG_TRY(cudaMemcpyAsync(dA + r0 * K, it.A_host + r0 * K, (size_t)(mc * K) * 4,
                                cudaMemcpyHostToDevice, h->in));
        BSG_TRY(cudaEventRecord(h->a_in[c], h->in));
    }
    BSG_TRY(cudaStreamWaitEvent(st, h->b_in, 0));
    BSG_TRY(launch_quantize_cols(dB, K, N, N, kOutHalfKMajor, bop, ldk, sb, nullptr, part_b, dstat,
                                 st));
    for (int c = 0; c < nchunks; ++c) {
        const int64_t r0 = c * rows, mc = M - r0 < rows ? M - r0 : rows;
        BSG_TRY(cudaStreamWaitEvent(st, h->a_in[c], 0));
        BSG_TRY(launch_quantize_rows(dA + r0 * K, mc, K, K, kOutHalfKMajor, aop + r0 * ldk, ldk,
                                     sa + r0, nullptr, dstat, st, ticket));
        BSG_TRY(launch_gemm_tc(aop + r0 * ldk, bop, mc, N, K, sa + r0, sb, it.relu, 0, dC + r0 * N,
                               N, dstat, ticket, st));
        BSG_TRY(cudaEventRecord(h->c_ready[c], st));
        BSG_TRY(cudaStreamWaitEvent(h->out, h->c_ready[c], 0));
        BSG_TRY(cudaMemcpyAsync(it.C_host + r0 * N, dC + r0 * N, (size_t)(mc * N) * 4,
                                cudaMemcpyDeviceToHost, h->out));
    }
#undef BSG_TRY
    return cudaSuccess;
}

}  // namespace
}  // namespace bsg

extern "C" {

bsg_status bsgemm_i8_host(const float *A_host, const float *B_host, int64_t M, int64_t N,
                          int64_t K, int relu, float *C_host, void *workspace, size_t ws_bytes,
                          int32_t *dstatus_host, void *stream) {
    const bsg_host_item item = {A_host, B_host, M, N, K, relu, C_host, workspace, ws_bytes};
    return bsgemm_i8_host_batch(&item, 1, dstatus_host, stream);
}

bsg_status bsgemm_i8_host_batch(const bsg_host_item *items, int n, int32_t *dstatus_host,
                                void *stream) {
    if (!items || n < 1 || n > BSG_MAX_HOST_BATCH) return BSG_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        const bsg_host_item &it = items[i];
        if (!it.A_host || !it.B_host || !it.C_host || !dims_ok(it.M, it.N, it.K))
            return BSG_ERR_ARG;
        if (it.K > BSG_MAX_K) return BSG_ERR_K_TOO_LARGE;
    }
    // no two items may share device workspace or C (their copies and kernels
    // are in flight together)
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < i; ++j) {
            const bsg_host_item &a = items[i], &b = items[j];
            if (ranges_overlap(a.workspace, a.ws_bytes, b.workspace, b.ws_bytes) ||
                ranges_overlap(a.C_host, (size_t)(a.M * a.N) * 4, b.C_host,
                               (size_t)(b.M * b.N) * 4))
                return BSG_ERR_ARG;
        }
    for (int i = 0; i < n; ++i)
        if (!ws_ok(items[i].workspace, items[i].ws_bytes,
                   bsgemm_i8_host_workspace_size(items[i].M, items[i].N, items[i].K)))
            return BSG_ERR_WORKSPACE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // every item's kernels report into the first item's status word
    int32_t *dstat = at<int32_t>(items[0].workspace, host_status_offset(items[0].M, items[0].N,
                                                                         items[0].K));

    std::lock_guard<std::mutex> guard(g_host_lock);
    HostPipe *h = host_pipe();
    if (!h) return BSG_ERR_CUDA;
    // One fork for the whole batch: the copy streams start after the work
    // already on `stream`, then run ahead of it -- item i+1 uploads while
    // item i computes and downloads.
    if (!ok(cudaEventRecord(h->start, st)) || !ok(cudaStreamWaitEvent(h->in, h->start, 0)) ||
        !ok(cudaStreamWaitEvent(h->out, h->start, 0)) ||
        !ok(cudaMemsetAsync(dstat, 0, sizeof(int32_t), st)))
        return BSG_ERR_CUDA;
    // Items are independent, so they may run in any order: Johnson's rule for
    // a two-stage flow (upload, then download) minimises the makespan.
    // Items that download more than they upload go first, by increasing
    // upload; the others follow, by decreasing download.
    int order[BSG_MAX_HOST_BATCH];
    for (int i = 0; i < n; ++i) order[i] = i;
    auto up = [&](int i) { return (items[i].M + items[i].N) * items[i].K; };
    auto down = [&](int i) { return items[i].M * items[i].N; };
    std::stable_sort(order, order + n, [&](int a, int b) {
        const bool fa = up(a) < down(a), fb = up(b) < down(b);
        if (fa != fb) return fa;
        return fa ? up(a) < up(b) : down(a) > down(b);
    });
    for (int k = 0; k < n; ++k)
        if (!ok(host_enqueue(items[order[k]], dstat, st, h))) return BSG_ERR_CUDA;
    int32_t hstat = 0;
    if (!ok(cudaMemcpyAsync(&hstat, dstat, sizeof(int32_t), cudaMemcpyDeviceToHost, h->out)) ||
        !ok(cudaEventRecord(h->done, h->out)) || !ok(cudaStreamWaitEvent(st, h->done, 0)) ||
        !ok(cudaStreamSynchronize(st)))
        return BSG_ERR_CUDA;
    if (dstatus_host) *dstatus_host = hstat;
    return BSG_OK;
}

size_t bsg_hash_f32_workspace_size(int64_t M, int64_t N) {
    if (M < 0 || N < 0) return 0;
    return hash_workspace_bytes(M, N);
}

bsg_status bsg_hash_f32(const float *C, int64_t M, int64_t N, int64_t ldc, uint8_t *out32,
                        void *workspace, size_t ws_bytes, void *stream) {
    if (!out32 || M < 0 || N < 0 || ldc < N || (M * N > 0 && !C)) return BSG_ERR_ARG;
    if (!ws_ok(workspace, ws_bytes, bsg_hash_f32_workspace_size(M, N))) return BSG_ERR_WORKSPACE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    return from_cuda(launch_hash_f32(C, M, N, ldc, out32, workspace,
                                     static_cast<cudaStream_t>(stream)));
}

// Probe workspace: A (M x K), B (K x N), C (M x N) floats, the unit's
// workspace, the hash workspace, and a status word.
static size_t probe_parts(int64_t M, int64_t N, int64_t K, size_t *offs) {
    size_t off = 0;
    offs[0] = off;  // A
    off += align256((size_t)M * K * 4);
    offs[1] = off;  // B
    off += align256((size_t)K * N * 4);
    offs[2] = off;  // C
    off += align256((size_t)M * N * 4);
    offs[3] = off;  // unit workspace
    off += align256(bsgemm_i8_workspace_size(M, N, K));
    offs[4] = off;  // hash workspace
    off += align256(hash_workspace_bytes(M, N));
    offs[5] = off;  // status word + device digest
    off += 256;
    return off;
}

size_t bsg_probe_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (!dims_ok(M, N, K)) return 0;
    size_t offs[6];
    return probe_parts(M, N, K, offs);
}

bsg_status bsg_probe_hash_async(uint64_t seed, int64_t M, int64_t N, int64_t K, uint8_t *out32,
                                void *workspace, size_t ws_bytes, int32_t *dstatus,
                                void *stream) {
    if (!out32 || !dims_ok(M, N, K)) return BSG_ERR_ARG;
    if (K > BSG_MAX_K) return BSG_ERR_K_TOO_LARGE;
    size_t offs[6];
    const size_t need = probe_parts(M, N, K, offs);
    if (!ws_ok(workspace, ws_bytes, need)) return BSG_ERR_WORKSPACE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *A = at<float>(workspace, offs[0]);
    float *B = at<float>(workspace, offs[1]);
    float *C = at<float>(workspace, offs[2]);
    if (launch_probe_fill(seed, M, N, K, A, B, st) != cudaSuccess) return BSG_ERR_CUDA;
    // The probe runs beside other work: the widest tiles keep its GEMM on
    // the fewest SMs (1024^3: 16 pair tiles on 32 SMs), the same results.
    void *uws = at<void>(workspace, offs[3]);
    s = unit_quantize(A, K, 0, B, N, 0, M, N, K, uws, offs[4] - offs[3], dstatus, st);
    if (s != BSG_OK) return s;
    s = unit_contract(M, N, K, 0, C, N, uws, offs[4] - offs[3], dstatus, st, 256);
    if (s != BSG_OK) return s;
    return from_cuda(launch_hash_f32(C, M, N, N, out32, at<void>(workspace, offs[4]), st));
}

bsg_status bsg_probe_hash(uint64_t seed, int64_t M, int64_t N, int64_t K, uint8_t *out32_host,
                          void *workspace, size_t ws_bytes, void *stream) {
    if (!out32_host || !dims_ok(M, N, K)) return BSG_ERR_ARG;
    size_t offs[6];
    const size_t need = probe_parts(M, N, K, offs);
    if (!ws_ok(workspace, ws_bytes, need)) return BSG_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *dstat = at<int32_t>(workspace, offs[5]);
    uint8_t *ddig = at<uint8_t>(workspace, offs[5] + 64);
    if (cudaMemsetAsync(dstat, 0, sizeof(int32_t), st) != cudaSuccess) return BSG_ERR_CUDA;
    bsg_status s = bsg_probe_hash_async(seed, M, N, K, ddig, workspace, ws_bytes, dstat, stream);
    if (s != BSG_OK) return s;
    int32_t hstat = 0;
    if (cudaMemcpyAsync(out32_host, ddig, 32, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(&hstat, dstat, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return BSG_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return BSG_ERR_CUDA;
    if (hstat & BSG_DSTATUS_TIMEOUT) return BSG_ERR_TIMEOUT;
    if (hstat & BSG_DSTATUS_NONFINITE) return BSG_ERR_NONFINITE;
    return BSG_OK;
}

bsg_status bsg_audit(const float *A, int64_t lda, const float *B, int64_t ldb, const float *C,
                     int64_t ldc, int64_t M, int64_t N, int64_t K, int relu, uint64_t seed,
                     int nsamples, uint32_t *mismatches, int64_t *cells, void *stream) {
    if (!A || !B || !C || !mismatches || !dims_ok(M, N, K)) return BSG_ERR_ARG;
    if (lda < K || ldb < N || ldc < N || nsamples < 1 || nsamples > (1 << 24)) return BSG_ERR_ARG;
    if (K > BSG_MAX_K) return BSG_ERR_K_TOO_LARGE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    return from_cuda(launch_audit(A, lda, B, ldb, C, ldc, M, N, K, relu, seed, nsamples,
                                  mismatches, cells, static_cast<cudaStream_t>(stream)));
}

// The probe hash of seed 0 at M = N = K = 1024, as the CPU oracle computes it
// (its SplitMix64 inputs, its quantize, exact contraction and epilogue, its
// BLAKE2s tree): the self-test's known answer.
static const uint8_t kProbeKnownAnswer[32] = {
    0xdd, 0x11, 0x9c, 0x18, 0x51, 0xaf, 0x87, 0x41, 0xe7, 0x50, 0xdd, 0x2a, 0x3f, 0x14, 0xa0, 0x42,
    0x72, 0x4f, 0x6c, 0xce, 0xd2, 0x6e, 0xd2, 0x08, 0xf6, 0xfc, 0x07, 0xd8, 0xdd, 0xc9, 0x41, 0xe8};
static const int64_t kSelftestN = 1024;
static const int kSelftestSamples = 4096;

size_t bsg_selftest_workspace_size(void) {
    return bsg_probe_workspace_size(kSelftestN, kSelftestN, kSelftestN) + 256;
}

bsg_status bsg_selftest(void *workspace, size_t ws_bytes, uint32_t *audit_mismatches_host,
                        int *hash_ok_host) {
    const size_t pws = bsg_probe_workspace_size(kSelftestN, kSelftestN, kSelftestN);
    if (!ws_ok(workspace, ws_bytes, pws + 256)) return BSG_ERR_WORKSPACE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    uint8_t digest[32];
    s = bsg_probe_hash(0, kSelftestN, kSelftestN, kSelftestN, digest, workspace, pws, nullptr);
    if (s != BSG_OK) return s;
    int hash_ok = memcmp(digest, kProbeKnownAnswer, 32) == 0;
    // audit the probe's GEMM, whose A, B and C are still in the probe workspace
    size_t offs[6];
    probe_parts(kSelftestN, kSelftestN, kSelftestN, offs);
    uint32_t *dmis = at<uint32_t>(workspace, pws);
    if (cudaMemsetAsync(dmis, 0, sizeof(uint32_t), nullptr) != cudaSuccess) return BSG_ERR_CUDA;
    if (launch_audit(at<float>(workspace, offs[0]), kSelftestN, at<float>(workspace, offs[1]),
                     kSelftestN, at<float>(workspace, offs[2]), kSelftestN, kSelftestN,
                     kSelftestN, kSelftestN, 0, 0x5eed, kSelftestSamples, dmis, nullptr,
                     nullptr) != cudaSuccess)
        return BSG_ERR_CUDA;
    uint32_t mis = 0;
    if (cudaMemcpy(&mis, dmis, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return BSG_ERR_CUDA;
    if (audit_mismatches_host) *audit_mismatches_host = mis;
    if (hash_ok_host) *hash_ok_host = hash_ok;
    return (hash_ok && mis == 0) ? BSG_OK : BSG_ERR_SELFTEST;
}

size_t bsg_wquant_cols_workspace_size(int64_t K, int64_t N) {
    if (K < 1 || N < 1) return 0;
    return wquant_workspace_bytes(K, N);
}

bsg_status bsg_wquant_cols(const float *W, int64_t K, int64_t N, int64_t ldw, int bits, int pow2,
                           void *Q, int64_t ldq, float *scale, void *workspace, size_t ws_bytes,
                           int32_t *dstatus, void *stream) {
    if (!W || !Q || !scale || K < 1 || N < 1 || ldw < N || (bits != 8 && bits != 4) ||
        (pow2 != 0 && pow2 != 1))
        return BSG_ERR_ARG;
    if (ldq < (bits == 8 ? N : (N + 1) / 2)) return BSG_ERR_ARG;
    if (!ws_ok(workspace, ws_bytes, wquant_workspace_bytes(K, N))) return BSG_ERR_WORKSPACE;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    return from_cuda(launch_wquant_cols(W, K, N, ldw, bits, pow2, Q, ldq, scale, workspace,
                                        dstatus, static_cast<cudaStream_t>(stream)));
}

bsg_status bsg_wdequant_cols(const void *Q, int64_t K, int64_t N, int64_t ldq, int bits,
                             const float *scale, float *W_hat, int64_t ldo, void *stream) {
    if (!Q || !scale || !W_hat || K < 1 || N < 1 || ldo < N || (bits != 8 && bits != 4))
        return BSG_ERR_ARG;
    if (ldq < (bits == 8 ? N : (N + 1) / 2)) return BSG_ERR_ARG;
    bsg_status s = check_device();
    if (s != BSG_OK) return s;
    return from_cuda(launch_wdequant_cols(Q, K, N, ldq, bits, scale, W_hat, ldo,
                                          static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ------------------------------------------------------------ chained units
// The epilogue of one unit also gathers, per row of C, the maximum of |C|
// (bit patterns, combined by atomicMax: exact in any order), so that C's
// per-row quantize for the next unit needs no reduction pass of its own.
namespace bsg {
namespace {

// rowmax (uint32 [M]) after the unit workspace of (M, N, K).
size_t requant_layout(int64_t M, int64_t N, int64_t K, size_t *rowmax_off) {
    const size_t unit_bytes = unit_layout(M, N, K, 0, 0).total;
    *rowmax_off = unit_bytes;
    return unit_bytes + align256((size_t)M * 4);
}

// Unit (M, N, K) from its quantized workspace into C, with the row maxima of
// |C| gathered into rowmax (zeroed by the unit's row quantize).
bsg_status contract_with_rowmax(int64_t M, int64_t N, int64_t K, int relu, float *C,
                                void *ws, uint32_t *rowmax, int32_t *dstatus, cudaStream_t st) {
    const UnitLayout L = unit_layout(M, N, K, 0, 0);
    GemmJob j;
    j.Aop = at<__half>(ws, L.aop);
    j.Bop = at<__half>(ws, L.bop);
    j.M = M;
    j.N = N;
    j.K = K;
    j.sa = at<float>(ws, L.sa);
    j.sb = at<float>(ws, L.sb);
    j.relu = relu;
    j.out = C;
    j.ldo = N;
    j.rowmax = rowmax;
    return from_cuda(launch_gemm_tc_group(&j, 1, 0, dstatus, at<unsigned int>(ws, L.ticket), st));
}

}  // namespace
}  // namespace bsg

extern "C" {

size_t bsgemm_i8_requant_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (!dims_ok(M, N, K)) return 0;
    size_t off = 0;
    return requant_layout(M, N, K, &off);
}

bsg_status bsgemm_i8_requant(const float *A, const float *B, int64_t M, int64_t N, int64_t K,
                             int relu, float *C, int8_t *Cq, float *scale, float *inv,
                             void *workspace, size_t ws_bytes, int32_t *dstatus, void *stream) {
    if (!C || !Cq || !scale) return BSG_ERR_ARG;
    bsg_status s = check_unit_args(A, K, 0, B, N, 0, M, N, K);
    if (s != BSG_OK) return s;
    size_t rm_off = 0;
    if (!ws_ok(workspace, ws_bytes, requant_layout(M, N, K, &rm_off))) return BSG_ERR_WORKSPACE;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t *rowmax = at<uint32_t>(workspace, rm_off);
    s = unit_quantize(A, K, 0, B, N, 0, M, N, K, workspace, ws_bytes, dstatus, st, true, rowmax);
    if (s != BSG_OK) return s;
    s = contract_with_rowmax(M, N, K, relu, C, workspace, rowmax, dstatus, st);
    if (s != BSG_OK) return s;
    return from_cuda(
        launch_requant_rows(C, M, N, N, rowmax, kOutInt8, Cq, N, scale, inv, dstatus, st));
}

// Layer 1 (M, N1, K) in front, layer 2 (M, N2, N1) after it, then the row
// maxima of C1.
static size_t chain_layout(int64_t M, int64_t K, int64_t N1, int64_t N2, size_t *ws2_off,
                           size_t *rowmax_off) {
    const size_t u1 = align256(unit_layout(M, N1, K, 0, 0).total);
    *ws2_off = u1;
    const size_t u2 = align256(unit_layout(M, N2, N1, 0, 0).total);
    *rowmax_off = u1 + u2;
    return u1 + u2 + align256((size_t)M * 4);
}

size_t bsgemm_i8_chain_workspace_size(int64_t M, int64_t K, int64_t N1, int64_t N2) {
    if (!dims_ok(M, N1, K) || !dims_ok(M, N2, N1)) return 0;
    size_t a = 0, b = 0;
    return chain_layout(M, K, N1, N2, &a, &b);
}

bsg_status bsgemm_i8_chain(const float *A, const float *B1, const float *B2, int64_t M,
                           int64_t K, int64_t N1, int64_t N2, int relu1, int relu2, float *C1,
                           float *C2, void *workspace, size_t ws_bytes, int32_t *dstatus,
                           void *stream) {
    if (!C1 || !C2 || !B2) return BSG_ERR_ARG;
    bsg_status s = check_unit_args(A, K, 0, B1, N1, 0, M, N1, K);
    if (s != BSG_OK) return s;
    s = check_unit_args(C1, N1, 0, B2, N2, 0, M, N2, N1);
    if (s != BSG_OK) return s;
    size_t ws2_off = 0, rm_off = 0;
    if (!ws_ok(workspace, ws_bytes, chain_layout(M, K, N1, N2, &ws2_off, &rm_off)))
        return BSG_ERR_WORKSPACE;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *ws1 = workspace;
    void *ws2 = static_cast<uint8_t *>(workspace) + ws2_off;
    uint32_t *rowmax = at<uint32_t>(workspace, rm_off);
    const UnitLayout L2 = unit_layout(M, N2, N1, 0, 0);
    // layer 1's operands (A's row quantize also zeroes C1's row maxima)
    s = unit_quantize(A, K, 0, B1, N1, 0, M, N1, K, ws1, ws2_off, dstatus, st, true, rowmax);
    if (s != BSG_OK) return s;
    // layer 2's weights per column, on the library's second stream beside
    // layer 1 (it depends on nothing of it), joined before layer 2's GEMM
    std::lock_guard<std::mutex> guard(g_side_lock);
    SideStream *side = side_stream();
    cudaStream_t qs = side ? side->st : st;
    if (side && (cudaEventRecord(side->fork, st) != cudaSuccess ||
                 cudaStreamWaitEvent(side->st, side->fork, 0) != cudaSuccess))
        return BSG_ERR_CUDA;
    const cudaError_t eq = launch_quantize_cols(B2, N1, N2, N2, kOutHalfKMajor,
                                                at<__half>(ws2, L2.bop), operand_ld(N1),
                                                at<float>(ws2, L2.sb), nullptr,
                                                at<uint32_t>(ws2, L2.part_b), dstatus, qs);
    // record the join even after a failed launch, so that no fork is left open
    if (side && cudaEventRecord(side->join, side->st) != cudaSuccess) return BSG_ERR_CUDA;
    if (eq != cudaSuccess) return BSG_ERR_CUDA;
    // layer 1, gathering C1's row maxima
    s = contract_with_rowmax(M, N1, K, relu1, C1, ws1, rowmax, dstatus, st);
    if (s != BSG_OK) return s;
    // C1 per row, straight into layer 2's f16 operand and row scales; the same
    // launch zeroes layer 2's tile counter
    if (launch_requant_rows(C1, M, N1, N1, rowmax, kOutHalfKMajor, at<__half>(ws2, L2.aop),
                            operand_ld(N1), at<float>(ws2, L2.sa), nullptr, dstatus, st,
                            at<unsigned int>(ws2, L2.ticket)) != cudaSuccess)
        return BSG_ERR_CUDA;
    if (side && cudaStreamWaitEvent(st, side->join, 0) != cudaSuccess) return BSG_ERR_CUDA;
    return unit_contract(M, N2, N1, relu2, C2, N2, ws2, L2.total, dstatus, st);
}

}  // extern "C"
