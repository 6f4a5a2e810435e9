// bsg_internal.h -- launchers shared by the library's translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "bsgemm.h"

namespace bsg {

// Output encodings of the quantize kernels.
enum QuantOut : int {
    kOutInt8 = 0,        // int8, same layout as the input
    kOutHalfKMajor = 1,  // f16-encoded int8 in the GEMM's K-major operand layout
};

// GEMM tile: 128 x (64, 128, 192 or 256) output per CTA, K in blocks of 64.
// kBN is the widest tile; per-column arrays hold round_up(N, kBN) + kBN
// entries so that any tile width's last tile stays inside them.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
// fp32 accumulation of int8 x int8 products stays exact while every partial
// sum stays below 2^24: 1024 * 127 * 127 = 16,516,096 < 16,777,216.
constexpr int kChunkK = 1024;

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Padded row length (elements) of the f16 operand arrays: a whole number of
// K-blocks, so the quantize kernels can write full 64-wide blocks.
inline int64_t operand_ld(int64_t K) { return round_up(K, kBK); }

// Column absmax is reduced in `nsplit` slices of rows.
int colmax_nsplit(int64_t rows, int64_t cols);
size_t colmax_partial_bytes(int64_t rows, int64_t cols);

int device_sm_count();

// Host-side count of kernel launches made by this library.
void count_launches(int n);

// zero2 (may be NULL): two words zeroed by the launch (a GEMM tile counter);
// zrows (may be NULL): one word per row zeroed (row maxima a GEMM gathers).
cudaError_t launch_quantize_rows(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                 int out_kind, void *Q, int64_t ldq, float *scale, float *inv,
                                 int32_t *dstatus, cudaStream_t st,
                                 unsigned int *zero2 = nullptr, unsigned int *zrows = nullptr);

// Bytes of the unit workspace for one operand layout (transA / transB as in
// bsgemm_i8_ex); bsgemm_i8_workspace_size is the largest over the layouts.
size_t unit_workspace_bytes(int64_t M, int64_t N, int64_t K, int transA, int transB);

// Columns.  kOutInt8 keeps X's layout (Q is rows x cols): clusters, or a
// partial-max pass over row slices then a quantize pass.  kOutHalfKMajor
// writes the transpose (Q is cols x ldq, each row a column of X): register
// strips in clusters, or one HBM read through a list of max and quantize
// items.  `partial` is colmax_partial_bytes(rows, cols) of scratch.
cudaError_t launch_quantize_cols(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                 int out_kind, void *Q, int64_t ldq, float *scale, float *inv,
                                 uint32_t *partial, int32_t *dstatus, cudaStream_t st);

// Rows of X quantized with absmax bit patterns given per row (rowmax[r]):
// scale / inv as in launch_quantize_rows (either may be NULL), codes as int8
// (Q rows x cols, ldq) or f16 (the GEMM's K-major operand layout); zero2 as
// in launch_quantize_rows.  Launched programmatically after the GEMM.
cudaError_t launch_requant_rows(const float *X, int64_t rows, int64_t cols, int64_t ldx,
                                const uint32_t *rowmax, int out_kind, void *Q, int64_t ldq,
                                float *scale, float *inv, int32_t *dstatus, cudaStream_t st,
                                unsigned int *zero2 = nullptr);

// Both operands of the unit in one launch: A (M x K, lda) per row into Aop
// (M x ldk f16) and sa, B (K x N, ldb) per column into Bop (N x ldk f16,
// transposed) and sb.  cudaErrorNotSupported (nothing launched) when the
// layout or size is outside the fused kernel's range.
cudaError_t launch_quantize_ab(const float *A, int64_t M, int64_t K, int64_t lda,
                               const float *B, int64_t N, int64_t ldb, __half *Aop,
                               __half *Bop, int64_t ldk, float *sa, float *sb,
                               int32_t *dstatus, unsigned int *zero2, cudaStream_t st,
                               unsigned int *zrows = nullptr);

// The live audit: `nsamples` seeded cells of C recomputed on the CUDA cores
// from the f32 inputs; mismatching cells are counted into *mismatches.
cudaError_t launch_audit(const float *A, int64_t lda, const float *B, int64_t ldb, const float *C,
                         int64_t ldc, int64_t M, int64_t N, int64_t K, int relu, uint64_t seed,
                         int nsamples, uint32_t *mismatches, int64_t *cells, cudaStream_t st);

// Weight storage as int8 / int4 codes with per-column scales, and back.
// ws: wquant_workspace_bytes(K, N) of scratch (the one-read path's
// counters and column maxima; columns of up to 4096 rows use none of it).
size_t wquant_workspace_bytes(int64_t K, int64_t N);
cudaError_t launch_wquant_cols(const float *W, int64_t K, int64_t N, int64_t ldw, int bits,
                               int pow2, void *Q, int64_t ldq, float *scale, void *ws,
                               int32_t *dstatus, cudaStream_t st);
cudaError_t launch_wdequant_cols(const void *Q, int64_t K, int64_t N, int64_t ldq, int bits,
                                 const float *scale, float *out, int64_t ldo, cudaStream_t st);

// Device check of the scale derivation over absmax bit patterns [first, last].
cudaError_t launch_selftest_scales(uint32_t first, uint32_t last, unsigned long long *bad,
                                   cudaStream_t st);

// int8 -> f16 operand conversions for the integer-only entry point.
cudaError_t launch_i8_rows_to_half(const int8_t *Q, int64_t rows, int64_t cols, int64_t ldq,
                                   __half *out, int64_t ldo, cudaStream_t st);
cudaError_t launch_i8_cols_to_half(const int8_t *Q, int64_t rows, int64_t cols, int64_t ldq,
                                   __half *out, int64_t ldo, cudaStream_t st);

// The tile width (64, 128, 192 or 256) the GEMM uses for an M x N problem (or
// a launch of n of them), and whether it runs 256-row tiles on CTA pairs
// when M > 128.
int gemm_tile_width(int64_t M, int64_t N, int sms);
int gemm_group_tile_width(const int64_t *M, const int64_t *N, int n, int sms);
bool gemm_pairs_enabled();
int gemm_group_m();
int gemm_snake();
// The tensor-core GEMM.  Aop: M x ldk f16, Bop: N x ldk f16 (both K-major,
// ldk = operand_ld(K)).  mode 0: C = epi(S, sa, sb) (+ReLU) as float;
// mode 1: S stored as int32.  sa / sb must hold round_up(M, kBM) /
// round_up(N, kBN) + kBN floats (mode 0).  `tile_width` 64/128/192/256
// fixes the tile width, 0 leaves it to gemm_tile_width.  `ticket`: two unsigned ints of
// device memory, the tile counter: zero before the first launch on it (the
// quantize step that fills a unit workspace zeroes it), and zero again after
// every launch that completes.
// One GEMM of a grouped launch (the arguments of launch_gemm_tc).
struct GemmJob {
    const __half *Aop, *Bop;
    int64_t M, N, K;
    const float *sa, *sb;
    int relu;
    void *out;
    int64_t ldo;
    // f32 mode only, may be NULL: per row of C, the running maximum of |C|
    // bit patterns (stored columns only), combined by atomicMax; must hold
    // M uint32 set to zero before the launch.
    uint32_t *rowmax = nullptr;
};
// Up to 3 GEMMs in one launch: their tiles form one list that the launch's
// CTAs share (one tail instead of three).  Same mode, status word and tile
// counter for all.
cudaError_t launch_gemm_tc_group(const GemmJob *jobs, int n, int mode, int32_t *dstatus,
                                 unsigned int *ticket, cudaStream_t st, int tile_width = 0);
cudaError_t launch_gemm_tc(const __half *Aop, const __half *Bop, int64_t M, int64_t N,
                           int64_t K, const float *sa, const float *sb, int relu, int mode,
                           void *out, int64_t ldo, int32_t *dstatus, unsigned int *ticket,
                           cudaStream_t st, int tile_width = 0);

cudaError_t launch_epilogue(const int32_t *S, int64_t lds, const float *sa, const float *sb,
                            int64_t M, int64_t N, int relu, float *C, int64_t ldc,
                            cudaStream_t st);

cudaError_t launch_probe_fill(uint64_t seed, int64_t M, int64_t N, int64_t K, float *A,
                              float *B, cudaStream_t st);

size_t hash_workspace_bytes(int64_t M, int64_t N);

// The whole unit (quantize both operands, contract, epilogue) from a
// workspace of bsgemm_i8_workspace_size(M, N, K) bytes.  `overlap`: quantize op(B)
// on a second stream of this library beside op(A); false keeps every launch
// on `st` and creates nothing.
bsg_status run_unit(const float *A, int64_t lda, int transA, const float *B, int64_t ldb,
                    int transB, int64_t M, int64_t N, int64_t K, int relu, float *C, int64_t ldc,
                    void *ws, size_t ws_bytes, int32_t *dstatus, cudaStream_t st, bool overlap);
cudaError_t launch_hash_f32(const float *C, int64_t M, int64_t N, int64_t ldc, uint8_t *out32,
                            void *ws, cudaStream_t st);

}  // namespace bsg
