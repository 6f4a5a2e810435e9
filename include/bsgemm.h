/*
 * bsgemm.h -- C ABI of the bit-exact block-scaled int8 GEMM for GB300.
 *
 * The operation ("Verification -- why you can trust the numbers",
 * DaisyChain-Train web/docs/VERIFICATION.md, section "The verified INT8
 * units", steps 1-3):
 *
 *   1. A (M x K) is quantized per row and B (K x N) per column:
 *        m      = max |x| over the row (column)
 *        scale  = f32( max( f64(m) / 127, 1e-8 ) )      -- an IEEE f64 divide
 *        inv    = f32( 1 / f64(scale) )                 -- an IEEE f64 divide
 *        q      = floor( RN32( RN32(x * inv) + 0.5 ) )  -- int8 in [-127, 127]
 *   2. S = Aq . Bq, exact int32 accumulation;
 *   3. C = f32( f32( f32(S) * sa[i] ) * sb[j] ), each step rounded to
 *      nearest-even binary32; with relu != 0, C = (C > 0) ? C : +0.
 *
 * and the kernel probe (same page, section "Layer 3: the kernel probe"): a
 * seeded GEMM whose output bytes are hashed to 32 bytes.
 *
 * Readings of points the page leaves open (the floor is applied to the f64
 * quotient; inv is the reciprocal of the stored f32 scale; the quantize uses
 * two f32 roundings; ReLU maps -0 and NaN to +0; the probe's inputs come
 * from SplitMix64 and its hash is a BLAKE2s tree over 256-byte leaves)
 * are stated per entry point below.
 *
 * Conventions for every entry point:
 *   - Matrices are row-major float32 / int8 / int32 with a leading dimension
 *     in elements.  Unless an argument says "host", every pointer is a
 *     DEVICE pointer owned by the caller; the library keeps no pointer after
 *     it returns and frees nothing.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream) unless stated otherwise.
 *   - Argument errors are returned synchronously before anything is
 *     launched.  A failed launch returns BSG_ERR_CUDA.
 *   - Data-dependent conditions are OR-ed into `*dstatus` (a device int32,
 *     may be NULL) as BSG_DSTATUS_* bits; read it after the stream
 *     synchronizes.  With a non-finite input the outputs are unspecified.
 *   - Every wait inside a kernel is bounded; on expiry the kernel sets
 *     BSG_DSTATUS_TIMEOUT, drains its own copies, frees its tensor memory and
 *     returns.  Nothing traps or aborts.
 *   - K <= BSG_MAX_K (133144): above it 127*127*K can leave int32.
 */
#ifndef BSGEMM_H
#define BSGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BSG_OK = 0,
    BSG_ERR_ARG = 1,         /* a size, pointer, leading dimension or flag is invalid */
    BSG_ERR_K_TOO_LARGE = 2, /* K > BSG_MAX_K */
    BSG_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned (256 B) or too small */
    BSG_ERR_CUDA = 4,        /* a CUDA call or launch failed */
    BSG_ERR_NONFINITE = 5,   /* only as a host-side summary; see BSG_DSTATUS_NONFINITE */
    BSG_ERR_TIMEOUT = 6,     /* only as a host-side summary; see BSG_DSTATUS_TIMEOUT */
    BSG_ERR_UNSUPPORTED = 7, /* the current device is not sm_103 */
    BSG_ERR_SELFTEST = 8     /* bsg_selftest found a wrong result */
} bsg_status;

#define BSG_MAX_K 133144
#define BSG_DSTATUS_NONFINITE 0x1 /* an input row or column held Inf or NaN */
#define BSG_DSTATUS_TIMEOUT 0x2   /* a bounded wait inside a kernel expired */

/* Human-readable name of a status code (static storage). */
const char *bsg_status_str(bsg_status s);

/* Library version, major*10000 + minor*100 + patch. */
int bsg_version(void);

/* ---- step 1: quantize ---------------------------------------------------- */

/* Rows of X (rows x cols, leading dimension ldx >= cols) to int8.
 * Q: rows x cols int8 with leading dimension ldq >= cols.
 * scale, inv: `rows` floats each (inv may be NULL).
 * Page: "The verified INT8 units", step 1; "Hardware ground truth" for the
 * floor(x*inv + 0.5) rule.  rows, cols >= 1. */
bsg_status bsg_quantize_rows(const float *X, int64_t rows, int64_t cols, int64_t ldx, int8_t *Q,
                             int64_t ldq, float *scale, float *inv, int32_t *dstatus,
                             void *stream);

/* Columns of X (rows x cols, leading dimension ldx >= cols) to int8: one
 * scale per column j, reduced over the rows.  Q has X's layout: rows x cols
 * int8 with leading dimension ldq >= cols.  scale, inv: `cols` floats (inv
 * may be NULL).  `workspace` must hold bsg_quantize_cols_workspace_size()
 * bytes (256-byte aligned).  Same passage as bsg_quantize_rows. */
size_t bsg_quantize_cols_workspace_size(int64_t rows, int64_t cols);
bsg_status bsg_quantize_cols(const float *X, int64_t rows, int64_t cols, int64_t ldx, int8_t *Q,
                             int64_t ldq, float *scale, float *inv, void *workspace,
                             size_t ws_bytes, int32_t *dstatus, void *stream);

/* ---- step 2: the exact integer contraction -------------------------------- */

/* S = Aq . Bq exactly, int32.  Aq: M x K int8 (lda >= K); Bq: K x N int8
 * (ldb >= N); S: M x N int32 (lds >= N).  Runs the same tensor-core kernel
 * as bsgemm_i8 with its int32 result stored instead of the epilogue.
 * Page: "The verified INT8 units", step 2. */
size_t bsg_gemm_s32_workspace_size(int64_t M, int64_t N, int64_t K);
bsg_status bsg_gemm_s32(const int8_t *Aq, int64_t lda, const int8_t *Bq, int64_t ldb, int64_t M,
                        int64_t N, int64_t K, int32_t *S, int64_t lds, void *workspace,
                        size_t ws_bytes, int32_t *dstatus, void *stream);

/* ---- step 3: the epilogue --------------------------------------------------- */

/* C[i][j] = epi(S[i][j], sa[i], sb[j]) (then ReLU if relu != 0), for any
 * int32 S and any float scales (subnormals and signed zeros are kept; a NaN
 * result's payload is unspecified).  S: M x N int32 (lds >= N); C: M x N
 * float (ldc >= N).  Page: "The verified INT8 units", step 3, and "Layer 5"
 * for the ReLU. */
bsg_status bsg_epilogue(const int32_t *S, int64_t lds, const float *sa, const float *sb,
                        int64_t M, int64_t N, int relu, float *C, int64_t ldc, void *stream);

/* ---- the whole unit ------------------------------------------------------------ */

/* C = epi(q(A) . q(B)) with A (M x K) quantized per row and B (K x N) per
 * column; all operands packed row-major.  `workspace`: at least
 * bsgemm_i8_workspace_size(M, N, K) bytes, 256-byte aligned, device memory;
 * its contents on return are unspecified.  Steps 1-3 of "The verified INT8
 * units".
 * The two operands are quantized at the same time: op(B) on a second stream
 * that the library creates on its first such call on each device (one
 * stream and two events, kept until the process exits), forked from
 * `stream` and joined back into it with events, so the call is ordered on
 * `stream` like any other and can be captured into a CUDA graph (make the
 * first call on each device outside a capture).  If that stream cannot be
 * created, the operands are quantized one after the other on `stream`.
 * This applies to bsgemm_i8, bsgemm_i8_ex, bsgemm_i8_quantize and
 * bsgemm_i8_host. */
size_t bsgemm_i8_workspace_size(int64_t M, int64_t N, int64_t K);
bsg_status bsgemm_i8(const float *A, const float *B, int64_t M, int64_t N, int64_t K, int relu,
                     float *C, void *workspace, size_t ws_bytes, int32_t *dstatus,
                     void *stream);

/* The general form: op(A) = A (M x K, lda >= K) or, with transA, the
 * transpose of a stored K x M matrix (lda >= M); op(B) = B (K x N, ldb >= N)
 * or, with transB, the transpose of a stored N x K matrix (ldb >= K).  op(A)
 * is quantized per row and op(B) per column, as if the transposes were
 * materialised (transposing floats is exact).  C: M x N, ldc >= N.  Same
 * workspace size as bsgemm_i8. */
bsg_status bsgemm_i8_ex(const float *A, int64_t lda, int transA, const float *B, int64_t ldb,
                        int transB, int64_t M, int64_t N, int64_t K, int relu, float *C,
                        int64_t ldc, void *workspace, size_t ws_bytes, int32_t *dstatus,
                        void *stream);

/* Several units in one GEMM launch (at most BSG_MAX_GROUP): each item is the
 * argument list of bsgemm_i8_ex, with its own workspace of
 * bsgemm_i8_workspace_size(M, N, K) bytes.  Every item's operands are
 * quantized as in bsgemm_i8_ex; then ONE tensor-core launch computes all the
 * products, its CTAs sharing the tiles of all items (one tail wave instead of
 * one per item) -- for instance the three GEMMs of a training step's linear
 * layer (forward X.W, grad-input dY.W^T, grad-weight X^T.dY).  The C of each
 * item is bit for bit what bsgemm_i8_ex gives it.  Items must not overlap in
 * C or workspace.  The pages have no grouped call; their units run one
 * product at a time. */
#define BSG_MAX_GROUP 3
typedef struct {
    const float *A;
    int64_t lda;
    int transA;
    const float *B;
    int64_t ldb;
    int transB;
    int64_t M, N, K;
    int relu;
    float *C;
    int64_t ldc;
    void *workspace;
    size_t ws_bytes;
} bsg_gemm_item;
bsg_status bsgemm_i8_group(const bsg_gemm_item *items, int count, int32_t *dstatus, void *stream);

/* The unit in two stages over one workspace (bsgemm_i8 is the pair):
 * bsgemm_i8_quantize runs step 1 -- op(A) per row and op(B) per column into
 * the workspace's f16 operands and scales (arguments as bsgemm_i8_ex) -- and
 * bsgemm_i8_contract runs steps 2-3 from that workspace into C (M x N,
 * ldc >= N).  Both on `stream`; the workspace must not be reused in between. */
bsg_status bsgemm_i8_quantize(const float *A, int64_t lda, int transA, const float *B,
                              int64_t ldb, int transB, int64_t M, int64_t N, int64_t K,
                              void *workspace, size_t ws_bytes, int32_t *dstatus, void *stream);
bsg_status bsgemm_i8_contract(int64_t M, int64_t N, int64_t K, int relu, float *C, int64_t ldc,
                              void *workspace, size_t ws_bytes, int32_t *dstatus, void *stream);

/* ---- chained units: the output quantized for the next unit ------------------ */

/* The unit, plus C quantized per row as the next unit's A operand: the
 * W8A8 chain of the presk "Precision" manual's closing list ("quantisation
 * beyond weights": int8 activations, i32 accumulation, requantisation) and
 * the B2B chain gate of "Layer 1: exact init gates", where one unit's output
 * feeds the next.  C = bsgemm_i8(A, B, relu) (M x N f32, packed), and
 *   Cq (M x N int8, packed), scale (M floats), inv (M floats, may be NULL)
 * are exactly what bsg_quantize_rows(C) gives.  The GEMM's epilogue gathers
 * each row's max |C| while C is still in registers (exact: a max of bit
 * patterns, in any order), so C is quantized in one streaming pass with no
 * reduction of its own.  A row of C that overflowed to +-Inf sets
 * BSG_DSTATUS_NONFINITE; that row's codes and scale are then unspecified, as
 * for any non-finite input of bsg_quantize_rows.  `workspace`:
 * bsgemm_i8_requant_workspace_size(M, N, K) bytes, 256-byte aligned; the
 * same second stream as bsgemm_i8 quantizes B. */
size_t bsgemm_i8_requant_workspace_size(int64_t M, int64_t N, int64_t K);
bsg_status bsgemm_i8_requant(const float *A, const float *B, int64_t M, int64_t N, int64_t K,
                             int relu, float *C, int8_t *Cq, float *scale, float *inv,
                             void *workspace, size_t ws_bytes, int32_t *dstatus, void *stream);

/* Two units in a chain, the second fed by the first:
 *   C1 = bsgemm_i8(A, B1, relu1)    A: M x K, B1: K x N1, C1: M x N1
 *   C2 = bsgemm_i8(C1, B2, relu2)   B2: N1 x N2, C2: M x N2
 * all packed row-major f32 in device memory; both C1 and C2 are written and
 * each is bit for bit what the two bsgemm_i8 calls give.  C1 is quantized
 * for the second unit straight from the row maxima its epilogue gathered
 * (see bsgemm_i8_requant), into the second GEMM's operand, with no separate
 * absmax pass over C1.  Pages: as bsgemm_i8_requant.  `workspace`:
 * bsgemm_i8_chain_workspace_size(M, K, N1, N2) bytes, 256-byte aligned.
 * B2 is quantized on the same second stream as bsgemm_i8 uses, beside the
 * first unit, and joined back into `stream` before the second GEMM. */
size_t bsgemm_i8_chain_workspace_size(int64_t M, int64_t K, int64_t N1, int64_t N2);
bsg_status bsgemm_i8_chain(const float *A, const float *B1, const float *B2, int64_t M,
                           int64_t K, int64_t N1, int64_t N2, int relu1, int relu2, float *C1,
                           float *C2, void *workspace, size_t ws_bytes, int32_t *dstatus,
                           void *stream);

/* Self-test of the scale derivation on the current device.  The kernels
 * derive scale and inv with IEEE f32 divides, which equal the f64 definition
 * for every input (the double rounding can never meet an f32 midpoint);
 * this call checks that claim for every absmax bit pattern in
 * [first_bits, last_bits] against the device's own f64 divide and stores
 * the number of mismatches in *mismatches_host.  Synchronous (default
 * stream); allocates 8 bytes of device memory.  In the spirit of the init
 * gates of "Layer 1: exact init gates". */
bsg_status bsg_selftest_scales(uint32_t first_bits, uint32_t last_bits,
                               uint64_t *mismatches_host);

/* The output tile width (64, 128, 192 or 256 columns) the GEMM kernel uses
 * for an M x N problem on `sms` SMs: the width with the fewest idle SMs in
 * the last wave, weighted by the narrower tiles' lower MMA efficiency.
 * Tiles are 256 rows on pairs of SMs (sms / 2 of them) when M > 128, else
 * 128 rows on single SMs.  Host-only; -1 on bad arguments.  No counterpart in the
 * pages: it documents this library's schedule. */
int bsg_gemm_tile_width(int64_t M, int64_t N, int sms);

/* Measurement aid for the roofline: one launch that issues `iters` x 4 pair
 * MMAs (tcgen05 cta_group::2, kind::f16, 256 x 256 x 16, fp32 accumulators)
 * back to back on every SM pair that can be resident, from operand tiles
 * that stay in shared memory -- the contraction's own instruction with no
 * operand copies and no epilogue.  Its duration (timed by the caller with
 * events on `stream`) gives the tensor pipe's ceiling for the GEMM at the
 * clock it runs at.  *flops_host receives the floating-point operations of
 * the launch (2 * 256 * 256 * 16 per MMA).  1 <= iters <= 2^18.  Asynchronous;
 * BSG_DSTATUS_TIMEOUT if its bounded final wait expires.  No counterpart in
 * the pages. */
bsg_status bsg_mma_ceiling(int iters, int32_t *dstatus, double *flops_host, void *stream);

/* Number of kernels this library has launched in this process (host-side
 * counter; every launch of every entry point counts). */
uint64_t bsg_launch_count(void);

/* bsgemm_i8 for callers that cannot allocate device memory -- a framework
 * that owns every device allocation and lends none to extensions, or an
 * embedding where the library may not touch the allocator (a plug-in in
 * someone else's process, a loop that forbids allocation after start-up).
 * It takes no workspace: its scratch is a device array compiled into the
 * library, BSG_NOALLOC_SCRATCH_BYTES (64 MiB) long, which every GPU that
 * loads the library holds until the process exits.  Arguments and results
 * are those of bsgemm_i8 (A and B as stored, never transposed).
 *   - Problems whose unit workspace for that layout exceeds the array are
 *     rejected with BSG_ERR_WORKSPACE before anything is launched (the GPT-2
 *     linears fit; an 8192 x 50304 x 768 LM head does not).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  The address is looked up
 *     again if the device's context has been replaced (cudaDeviceReset).
 *   - All calls share the one array and each leaves its contents behind:
 *     calls that may overlap on the GPU (other streams, other host threads)
 *     race on it and must be serialized by the caller.  Nothing in the array
 *     has to start at zero: what a call reads is written earlier in the same
 *     call, except column scales past N, which the epilogue loads for whole
 *     tiles but applies to no stored column.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine, and
 *     creates no stream or event: every launch goes to `stream`.
 * The pages have no counterpart: this is a deployment variant. */
#define BSG_NOALLOC_SCRATCH_BYTES (64u << 20)
bsg_status bsgemm_i8_noalloc(const float *A, const float *B, int64_t M, int64_t N, int64_t K,
                             int relu, float *C, int32_t *dstatus, void *stream);

/* ---- weight storage as int8 / int4 codes ------------------------------------ */

/* The weight storage of the presk "Precision" manual, section "Integer
 * weights": a K x N weight W contracted over K is stored as codes with one
 * scale per column j,
 *   s_j = max_k |W[k][j]| / (2^(bits-1) - 1) rounded to f32 (bits = 8 or 4),
 * or, with pow2 != 0, that scale rounded up to the smallest power of two >=
 * it (q * s is then exact); an all-zero column, or one whose scale rounds to
 * zero, gets s = 0 and stores zeros; the codes are q = W / s rounded to the
 * nearest integer, ties to even.  W: DEVICE f32, row-major, ldw >= N.
 * bits = 8: Q is K x N int8 (ldq >= N).  bits = 4: Q is K rows of ceil(N/2)
 * bytes (ldq >= ceil(N/2)), 4-bit two's complement codes, column 2i in bits
 * 0-3 of byte i and column 2i+1 in bits 4-7 (zero past the last column).
 * scale: DEVICE f32[N].  `workspace`: bsg_wquant_cols_workspace_size(K, N)
 * bytes of DEVICE memory (256-byte aligned; counters and column maxima of
 * the one-read path that long columns take: more than 4096 rows, or 2048 or
 * more in a weight of 2^23 elements or more), owned by the
 * caller and not used after the call's work completes on `stream`.  Inf or
 * NaN in W sets BSG_DSTATUS_NONFINITE in *dstatus (may be NULL); the codes
 * and scales of such columns are then unspecified.  Asynchronous.  These are
 * the pages' stored-weight semantics for a presk realization, a different
 * scheme from the block-scaled unit's floor(x * inv + 0.5) codes. */
size_t bsg_wquant_cols_workspace_size(int64_t K, int64_t N);
bsg_status bsg_wquant_cols(const float *W, int64_t K, int64_t N, int64_t ldw, int bits, int pow2,
                           void *Q, int64_t ldq, float *scale, void *workspace, size_t ws_bytes,
                           int32_t *dstatus, void *stream);

/* The stored weights: W_hat[k][j] = f32(q[k][j] * s_j), one rounding (exact
 * with pow2 scales).  Q and bits as written by bsg_wquant_cols; W_hat: DEVICE
 * f32 K x N, ldo >= N.  Asynchronous. */
bsg_status bsg_wdequant_cols(const void *Q, int64_t K, int64_t N, int64_t ldq, int bits,
                             const float *scale, float *W_hat, int64_t ldo, void *stream);

/* ---- verification of live results ----------------------------------------- */

/* The live audit ("Verification -- why you can trust the numbers", section
 * "Layer 2: the live audit"): `nsamples` cells of C, chosen by SplitMix64
 * seeded with `seed` (output 2s gives sample s's row mod M, output 2s+1 its
 * column mod N), are recomputed on the CUDA cores by a path that shares no
 * kernel with bsgemm_i8 -- the cell's row of A and column of B read from the
 * f32 inputs, scales from the f64 definition, int64 dot product, f32
 * epilogue -- and every cell whose bits differ from C adds 1 to *mismatches
 * (DEVICE uint32, not cleared by the call).  Cells whose row or column holds
 * Inf or NaN are skipped.  A (M x K, lda >= K), B (K x N, ldb >= N), C (M x N,
 * ldc >= N): the inputs and output of one bsgemm_i8(A, B, relu) call,
 * row-major device memory.  `cells` (DEVICE int64[2 * nsamples], may be NULL)
 * receives the sampled (row, column) pairs.  1 <= nsamples <= 1 << 24.
 * Asynchronous on `stream`. */
bsg_status bsg_audit(const float *A, int64_t lda, const float *B, int64_t ldb, const float *C,
                     int64_t ldc, int64_t M, int64_t N, int64_t K, int relu, uint64_t seed,
                     int nsamples, uint32_t *mismatches, int64_t *cells, void *stream);

/* The init gate ("Layer 1: exact init gates"): runs the probe (seed 0,
 * 1024^3) through the live kernels, compares its hash with the known answer
 * the CPU oracle computes for it, and audits 4096 cells of that GEMM with
 * bsg_audit.  Returns BSG_OK when both agree, BSG_ERR_SELFTEST when either
 * does not (other codes for argument or CUDA errors).  `workspace`: DEVICE
 * memory of bsg_selftest_workspace_size() bytes, 256-byte aligned.
 * *audit_mismatches_host and *hash_ok_host (each may be NULL) receive the
 * audit's mismatch count and 1 if the hash matched.  Synchronous (default
 * stream). */
size_t bsg_selftest_workspace_size(void);
bsg_status bsg_selftest(void *workspace, size_t ws_bytes, uint32_t *audit_mismatches_host,
                        int *hash_ok_host);

/* bsgemm_i8 on HOST buffers (packed row-major; pinned memory gives
 * asynchronous copies): copies A and B to the device, runs the unit, copies
 * C back, and synchronizes `stream` before returning.  A moves in row chunks
 * on a copy stream of the library's own and C comes back chunk by chunk on
 * another, so that uploads, the kernels (on `stream`) and downloads overlap
 * (the two copy streams are created on the first call on each device and
 * kept until the process exits); the result does not depend on the
 * chunking.  `workspace`: device
 * memory of at least bsgemm_i8_host_workspace_size(M, N, K) bytes.
 * *dstatus_host (may be NULL) receives the device status bits. */
size_t bsgemm_i8_host_workspace_size(int64_t M, int64_t N, int64_t K);
bsg_status bsgemm_i8_host(const float *A_host, const float *B_host, int64_t M, int64_t N,
                          int64_t K, int relu, float *C_host, void *workspace, size_t ws_bytes,
                          int32_t *dstatus_host, void *stream);

/* Several independent units on host buffers in one call (at most
 * BSG_MAX_HOST_BATCH): each item is the argument list of bsgemm_i8_host.
 * The items' copies and kernels are pipelined across items: one item uploads
 * while the previous one computes and downloads, so both directions of the
 * host link stay busy for the whole batch, where back-to-back bsgemm_i8_host
 * calls drain the pipeline at every call.  The library picks the order of
 * the items (Johnson's rule for the two stages, upload then download:
 * download-heavy items first by increasing upload, then the rest by
 * decreasing download).  Each C is bit for bit what
 * bsgemm_i8_host gives it.  Items may share A or B, but no two items may
 * overlap in workspace or in C (BSG_ERR_ARG); an item's A and B must not
 * overlap another item's C.  Synchronizes `stream` before returning;
 * *dstatus_host (may be NULL) receives the OR of every item's device status
 * bits.  The pages run one unit at a time; this call has no counterpart
 * there. */
#define BSG_MAX_HOST_BATCH 16
typedef struct {
    const float *A_host;
    const float *B_host;
    int64_t M, N, K;
    int relu;
    float *C_host;
    void *workspace;
    size_t ws_bytes;
} bsg_host_item;
bsg_status bsgemm_i8_host_batch(const bsg_host_item *items, int n, int32_t *dstatus_host,
                                void *stream);

/* ---- the probe --------------------------------------------------------------------- */

/* 32-byte hash of an M x N float matrix (leading dimension ldc >= N): the
 * matrix's little-endian bytes, row after row with no padding, hashed as a
 * BLAKE2s-256 tree (RFC 7693; BLAKE2 tree mode with fanout 4, unlimited
 * depth, leaf length 256, inner length 32): leaf i (256 bytes, the last may
 * be shorter) at node offset i, depth 0; then, level by level, groups of
 * four digests concatenated and hashed at node offset = group index, node
 * depth = level; the last node of each level carries the last-node flag;
 * the hash is the single digest of the first level that has one.
 * out32: 32 bytes of DEVICE memory.  `workspace`: bsg_hash_f32_workspace_size
 * (M, N) bytes.  Page: "Layer 3: the kernel probe" (the page names no hash
 * function; this tree is our reading). */
size_t bsg_hash_f32_workspace_size(int64_t M, int64_t N);
bsg_status bsg_hash_f32(const float *C, int64_t M, int64_t N, int64_t ldc, uint8_t *out32,
                        void *workspace, size_t ws_bytes, void *stream);

/* The probe: A (M x K) and B (K x N) filled from SplitMix64 (Steele, Lea,
 * Flood 2014) seeded with `seed` -- A takes outputs 0 .. M*K-1 row-major, B
 * the next K*N -- each output z mapped exactly to ((z >> 40) - 2^23) * 2^-23
 * in [-1, 1); then bsgemm_i8 without ReLU; then bsg_hash_f32 of C.
 * out32: 32 bytes of DEVICE memory (asynchronous).  `workspace`:
 * bsg_probe_workspace_size(M, N, K) bytes.  Page: "Layer 3: the kernel
 * probe". */
size_t bsg_probe_workspace_size(int64_t M, int64_t N, int64_t K);
bsg_status bsg_probe_hash_async(uint64_t seed, int64_t M, int64_t N, int64_t K, uint8_t *out32,
                                void *workspace, size_t ws_bytes, int32_t *dstatus,
                                void *stream);

/* As bsg_probe_hash_async, but out32_host is HOST memory and the call
 * synchronizes `stream` before returning.  Returns BSG_ERR_TIMEOUT or
 * BSG_ERR_NONFINITE if the device status says so. */
bsg_status bsg_probe_hash(uint64_t seed, int64_t M, int64_t N, int64_t K, uint8_t *out32_host,
                          void *workspace, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* BSGEMM_H */
