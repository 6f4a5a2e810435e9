// gemm_tc.cu -- the exact int8 contraction on the tcgen05 tensor cores, with
// the f32 epilogue (and ReLU) fused.
//
// "Verification -- why you can trust the numbers", section "The verified
// INT8 units", steps 2-3: exact int8 products accumulated in int32, then
// epi(s,a,b) = f32(f32(f32(s)*a)*b).
//
// sm_103a has no integer tensor-core MMA (ptxas rejects tcgen05.mma
// .kind::i8 for this target), so the contraction runs as kind::f16: every
// int8 in [-127, 127] is exact in f16, every product (|p| <= 16129) is exact,
// and an fp32 accumulation of integers stays exact while every partial sum
// is below 2^24 -- which holds for any 1024 consecutive products (1024 *
// 16129 < 2^24), whatever the order of the adds and whatever truncation the
// tensor core's adder applies below the integer bit (the tensor-core adder
// model of "The step oracle", section 3.4: products exact, aligned to the
// largest exponent, 25 fraction bits kept on Blackwell).  K is therefore cut
// into chunks of 1024; each chunk's fp32 tile is converted to int32 and the
// chunks are summed in int32, which is exact.
//
// Two kernels, one template:
//   * PAIR (M > 128): a cluster of two CTAs on two SMs computes a 256 x BN
//     tile with the pair MMA (tcgen05 cta_group::2, M = 256).  Each CTA
//     loads 128 rows of A and BN/2 rows of B per k-block, so each SM takes
//     in and its tensor core reads two thirds of what a 128 x BN tile per SM
//     needs for the same multiply-adds.  With one CTA per SM the 128 x 256
//     tile was bound by shared-memory traffic (TMA writes plus MMA reads),
//     not by the tensor pipe; the pair also frees shared memory for a deeper
//     operand ring (6 stages at the widest tiles) beside the output staging.
//   * single (M <= 128): one CTA computes a 128 x BN tile (cta_group::1).
// BN in {64, 128, 192, 256} is chosen per problem so that the last wave of tiles
// leaves few SMs idle; CTAs (pairs) are persistent, and after the first wave
// they claim tiles dynamically, so that a CTA that starts late, its SM busy
// with other work, takes fewer tiles (only its first, static tile waits for
// it).
//
// Roles (one CTA per SM):
//   warp 0      TMA producer: A and B k-blocks (64 wide, 128-byte swizzle)
//               into a shared-memory ring; in a pair both CTAs load and both
//               count their bytes on the even CTA's barrier;
//   warp 1      MMA issuer (one thread; in a pair, of the even CTA only):
//               4 x tcgen05.mma (K = 16) per k-block into a tensor-memory
//               accumulator, double-buffered (2 x BN columns) so the epilogue
//               of one chunk or tile overlaps the next one's MMAs;
//   warp 2      allocates / frees the tensor-memory columns;
//   warp 3      tile scheduler (one thread; in a pair, of the even CTA only):
//               the first tile of each CTA (pair) is its index, later tiles
//               are claimed from a counter, and each index is handed to every
//               role of both CTAs through a small shared-memory queue;
//   warps 4-11  epilogue: tcgen05.ld of each chunk into registers (the tensor
//               memory is released at once), then the f32 epilogue, ReLU,
//               staging in shared memory and TMA stores (or plain stores
//               where C's rows are not 16-byte aligned).
// Every mbarrier wait is bounded; on expiry the CTA records
// BSG_DSTATUS_TIMEOUT, drains its copies and MMAs, frees tensor memory and
// returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "bsg_internal.h"
#include "bsg_ptx.cuh"

namespace bsg {
namespace {

constexpr int kChunkBlocks = kChunkK / kBK;  // 16 k-blocks per exact chunk
constexpr int kEpiWarps = 8;
constexpr int kThreads = 128 + kEpiWarps * 32;
constexpr uint32_t kABytes = kBM * kBK * 2;     // 16 KiB
constexpr uint32_t kEpiBufBytes = 32 * 32 * 4;  // one 32 x 32 fp32 box
// Default tile raster: groups of 8 m-units, so that a wave of tiles (76 pairs)
// covers about 8 m-units x 9.5 n-tiles and the operand rows and columns in
// use at once stay in L2.  Measured on 16384^3 against 16 per group: DRAM
// reads per launch 8.6 against 11.2 GB, 2120 against 2092 TFLOP/s; 8192^3 and
// the ragged 4097 x 12289 x 8191 also fastest at 8, 4096^3 the same at any.
constexpr int kGroupM = 8;
constexpr int kTileQ = 2;                       // depth of the tile-index queue
constexpr uint32_t kMaxSmem = 232448;           // 227 KiB per CTA

// Compile-time layout of one tile width and kernel kind.
template <int BN, bool PAIR>
struct Cfg {
    static_assert(BN == 64 || BN == 128 || BN == 192 || BN == 256, "tile width");
    static constexpr int kBRows = PAIR ? BN / 2 : BN;  // B rows this CTA loads
    static constexpr uint32_t kBBytes = kBRows * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    // 6 stages with one staging box per epilogue warp measured better than 5
    // with two at the wide tiles (8192^3: 2000 vs 1896 TFLOP/s)
    static constexpr int kStages = PAIR ? (BN >= 192 ? 6 : BN == 128 ? 6 : 8)
                                        : (BN >= 192 ? 4 : BN == 128 ? 5 : 6);
    static constexpr int kBoxes = (BN >= 192) ? 1 : 2;  // staging boxes per warp
    // one accumulator buffer (192 wide tiles keep 256-column buffers, so
    // both start at a multiple of 256 and the allocation is a power of 2)
    static constexpr uint32_t kAccCols = BN == 192 ? 256 : BN;
    static constexpr uint32_t kTmemCols = 2 * kAccCols;
    static constexpr int kWarpCols = BN / 2;  // columns per epilogue warp
    static constexpr int kPieces = kWarpCols / 32;
    static constexpr uint32_t kOffEpi = kStages * kStageBytes;
    static constexpr uint32_t kOffBar = kOffEpi + kEpiWarps * kBoxes * kEpiBufBytes;
    // barriers: full[kStages], empty[kStages], tfull[2], tempty[2], drain,
    // qfull[kTileQ], qempty[kTileQ]; then the tile-index queue
    static constexpr uint32_t kNumBars = 2 * kStages + 5 + 2 * kTileQ;
    static constexpr uint32_t kOffTileQ = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffTmemPtr = kOffTileQ + kTileQ * 4;
    static constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
    static constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + 1024-byte alignment slack
    static constexpr uint32_t kIdesc = idesc_f16_f32(PAIR ? 2 * kBM : kBM, BN);
    static_assert(kSmemBytes <= kMaxSmem, "shared memory");
    static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle atoms stay aligned");
};

constexpr int kMaxGroup = 3;  // GEMMs per launch

// One GEMM of a launch.
struct Prob {
    int M, N, K;
    int num_kb;        // k-blocks per tile
    int num_m, num_n;  // 128-row m-blocks, BN-wide n-tiles
    int num_mu;        // m-units: m-blocks, or pairs of them (PAIR)
    int unit0;         // index of this GEMM's first tile in the launch
    const float *sa;
    const float *sb;
    void *out;
    int64_t ldo;
    int relu;
    int tma_store;  // 1: C's rows are 16-byte aligned; store through its tensor map
    uint32_t *rowmax;  // NULL, or per row the max of |C| bit patterns (atomicMax)
};

template <int NP>  // GEMMs the launch was compiled for (1, or kMaxGroup)
struct Params {
    Prob prob[NP];
    int nprob;
    int num_units;  // tiles of the launch, all GEMMs
    int mode;       // 0: f32 epilogue, 1: int32 accumulators
    int group_m;    // tile raster: m-units per group
    int snake;      // 1: odd raster groups take their n-tiles in reverse
    int32_t *dstatus;
    // ticket[0]: tiles claimed beyond the first wave; ticket[1]: CTAs (pairs)
    // done claiming.  Zero at launch; the last CTA to finish claiming sets
    // both back to zero for the next launch.
    unsigned int *ticket;
};

// The tensor maps of every GEMM: operands A and B (f16, K-major) and C.
template <int NP>
struct Maps {
    CUtensorMap a[NP], b[NP], c[NP];
};

// Tile u of the launch -> its GEMM (returned) and (m-unit, n-tile) there,
// rastered in groups of p.group_m m-units so that concurrent tiles share
// operand rows and columns in L2.  With NP = 1 the GEMM is a constant, so
// that a single GEMM's parameters are read at fixed offsets.
template <int NP>
__device__ __forceinline__ int tile_coords(const Params<NP> &p, int u, int &mu, int &nb) {
    int pi = 0;
    if (NP > 1)
        while (pi + 1 < p.nprob && u >= p.prob[pi + 1].unit0) ++pi;
    const Prob &q = p.prob[pi];
    u -= q.unit0;
    const int group_m = p.group_m;
    const int per_group = group_m * q.num_n;
    const int g = u / per_group;
    const int first_m = g * group_m;
    const int gm = (q.num_mu - first_m) < group_m ? (q.num_mu - first_m) : group_m;
    const int r = u - g * per_group;
    mu = first_m + r % gm;
    nb = r / gm;
    // serpentine: odd groups walk the n-tiles backwards, so that a group's
    // first waves use the B columns the previous group's last waves left in L2
    if (p.snake && (g & 1)) nb = q.num_n - 1 - nb;
    return pi;
}

__device__ __forceinline__ void record_abort(volatile int *abort_flag, int32_t *dstatus) {
    *abort_flag = 1;
    if (dstatus) atomicOr(dstatus, 2);
}

// Bounded wait on one of this CTA's barriers; PAIR barriers may be arrived
// on from the other CTA, so they are acquired at cluster scope.
template <bool PAIR>
__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity, const volatile int *abort) {
    return PAIR ? mbar_wait_cl(bar, parity, abort) : mbar_wait(bar, parity, abort);
}
template <bool PAIR>
__device__ __forceinline__ bool bar_try_wait(uint64_t *bar, uint32_t parity) {
    return PAIR ? mbar_try_wait_cl(bar, parity) : mbar_try_wait(bar, parity);
}

// Epilogue value of one accumulator: f32(S) * a * b, each step RN; ReLU maps
// everything that is not > 0 (including -0) to +0.
__device__ __forceinline__ float epi_value_f(float s, float a, float b, int relu) {
    const float c = __fmul_rn(__fmul_rn(s, a), b);
    return relu ? (c > 0.0f ? c : 0.0f) : c;
}

// The epilogue of 32 consecutive sums of one row, in place.  F32: v holds
// f32(S) bit patterns (+0 added to map -0 to +0); otherwise int32 S.  Lane j
// holds the column scale of column j of the piece in `bl`; the scales reach
// every lane by shuffles (they were loaded before the tile's sums were ready,
// so no global-memory latency sits between the sums and the stores).
template <bool F32>
__device__ __forceinline__ void epi_piece(uint32_t (&v)[32], float bl, float a, int relu) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float bj = __shfl_sync(0xffffffffu, bl, j);
        const uint32_t x = v[j];
        const float sv = F32 ? __fadd_rn(__uint_as_float(x), 0.0f) : __int2float_rn((int32_t)x);
        v[j] = __float_as_uint(epi_value_f(sv, a, bj, relu));
    }
}

// Write one thread's 32 values (row `lane` of a 32 x 32 box) into the next
// of the warp's NBOX swizzled staging boxes and store it with the TMA, or
// store directly to global memory.  `nstored` counts the warp's TMA stores;
// a box is rewritten only after the store that last used it has read it.
template <int NBOX>
__device__ __forceinline__ void emit_box(const Prob &p, const CUtensorMap *tmap_c,
                                         uint8_t *boxes, const uint32_t (&v)[32], int row0,
                                         int col0, int lane, int &nstored) {
    if (p.tma_store) {
        if (nstored >= NBOX) {
            if (lane == 0) {
                if (NBOX == 1)
                    bulk_wait_read0();
                else
                    bulk_wait_read1();
            }
            __syncwarp();
        }
        uint8_t *box = boxes + (nstored % NBOX) * kEpiBufBytes;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t off = lane * 128 + ((j ^ (lane & 7)) << 4);
            *reinterpret_cast<uint4 *>(box + off) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmap_c, box, col0, row0);
            bulk_commit();
        }
        ++nstored;
    } else {
        // C's rows are not 16-byte aligned (no TMA store): transpose the box
        // through the first staging box, so that each store instruction
        // writes 32 consecutive columns of one row (one 128-byte span)
        // instead of one column of 32 rows.
        if (nstored > 0) {  // a TMA store of an earlier GEMM of the launch may still read it
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            nstored = 0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t off = lane * 128 + ((j ^ (lane & 7)) << 4);
            *reinterpret_cast<uint4 *>(boxes + off) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        __syncwarp();
        const int col = col0 + lane;
        if (col < p.N) {
            uint32_t *dst = static_cast<uint32_t *>(p.out) + (int64_t)row0 * p.ldo + col;
            const uint32_t cw = (uint32_t)((lane >> 2) << 4) + (uint32_t)(lane & 3) * 4;
#pragma unroll 8
            for (int r = 0; r < 32; ++r) {
                if (row0 + r >= p.M) break;
                const uint32_t off = r * 128 + (cw ^ ((uint32_t)(r & 7) << 4));
                __stcs(dst + (int64_t)r * p.ldo, *reinterpret_cast<const uint32_t *>(boxes + off));
            }
        }
        __syncwarp();  // the box is read before the next piece overwrites it
    }
}

template <int BN, bool PAIR, int NP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ Maps<NP> maps, const __grid_constant__ Params<NP> p) {
    using K = Cfg<BN, PAIR>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + K::kOffBar);
    uint64_t *full = bars;
    uint64_t *empty = bars + K::kStages;
    uint64_t *tfull = bars + 2 * K::kStages;
    uint64_t *tempty = bars + 2 * K::kStages + 2;
    uint64_t *drain = bars + 2 * K::kStages + 4;
    uint64_t *qfull = bars + 2 * K::kStages + 5;
    uint64_t *qempty = qfull + kTileQ;
    volatile int *tileq = reinterpret_cast<volatile int *>(smem + K::kOffTileQ);
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(smem + K::kOffTmemPtr);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + K::kOffAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = PAIR ? (int)cluster_ctarank() : 0;  // 0: the pair's MMA-issuing CTA
    const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // first tile
    const int nunits = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    constexpr uint16_t kPairMask = 0x3;  // cluster ranks 0 and 1

    if (threadIdx.x == 0) {
        for (int s = 0; s < K::kStages; ++s) {
            mbar_init(&full[s], PAIR ? 2 : 1);  // PAIR: both CTAs' producers
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], PAIR ? 2 * kEpiWarps : kEpiWarps);  // PAIR: both epilogues
        }
        mbar_init(drain, 1);
        for (int q = 0; q < kTileQ; ++q) {
            mbar_init(&qfull[q], 1);
            // readers of a queue slot: the producer, the MMA thread and the
            // epilogue warps of this CTA, and in a pair the odd CTA's producer
            // and epilogue warps
            mbar_init(&qempty[q], PAIR ? 2 * (1 + kEpiWarps) + 1 : 2 + kEpiWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_async_shared();
    }
    if (warp == 2) {
        if (PAIR) {
            tmem_alloc_pair(tmem_ptr, K::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_ptr, K::kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_ptr;
    // everything above overlaps the end of the previous kernel in the stream
    // (programmatic launch); the operands, scales and tile counter it wrote
    // are read only from here on
    griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int i = 0; i < p.nprob; ++i) {
                prefetch_tmap(&maps.a[i]);
                prefetch_tmap(&maps.b[i]);
            }
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_parity[K::kStages];
            bool issued[K::kStages];
            for (int s = 0; s < K::kStages; ++s) issued[s] = false, issued_parity[s] = 0;
            bool ok = true;
            for (uint32_t t = 0; ok; ++t) {
                const int slot = (int)(t % kTileQ);
                const uint32_t qph = (t / kTileQ) & 1;
                if (!bar_wait<PAIR>(&qfull[slot], qph, abort_flag)) {
                    record_abort(abort_flag, p.dstatus);
                    ok = false;
                    break;
                }
                const int tile = tileq[slot];
                if (PAIR)
                    mbar_arrive_cl(cluster_addr(&qempty[slot], 0));
                else
                    mbar_arrive(&qempty[slot]);
                if (tile < 0) {
                    // no tiles left for this CTA: the next kernel may be placed
                    // on SMs as the grid drains (it waits for this grid's
                    // completion before it touches memory)
                    griddep_launch_dependents();
                    break;
                }
                int mu, nb;
                const int pi = tile_coords(p, tile, mu, nb);
                const CUtensorMap *tma = &maps.a[pi];
                const CUtensorMap *tmb = &maps.b[pi];
                const int mb = PAIR ? 2 * mu + rank : mu;
                const int num_kb = p.prob[pi].num_kb;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!bar_wait<PAIR>(&empty[stage], phase ^ 1, abort_flag)) {
                        record_abort(abort_flag, p.dstatus);
                        ok = false;
                        break;
                    }
                    uint8_t *sa_tile = smem + stage * K::kStageBytes;
                    uint8_t *sb_tile = sa_tile + kABytes;
                    if (PAIR) {
                        // the even CTA's full barrier, where both CTAs count their bytes
                        const uint32_t fb = cluster_addr(&full[stage], 0);
                        mbar_arrive_expect_tx_cl(fb, K::kStageBytes);
                        tma_load_2d_pair(tma, fb, sa_tile, kb * kBK, mb * kBM);
                        tma_load_2d_pair(tmb, fb, sb_tile, kb * kBK, nb * BN + rank * K::kBRows);
                    } else {
                        mbar_arrive_expect_tx(&full[stage], K::kStageBytes);
                        tma_load_2d(tma, &full[stage], sa_tile, kb * kBK, mb * kBM);
                        tma_load_2d(tmb, &full[stage], sb_tile, kb * kBK, nb * BN);
                    }
                    issued[stage] = true;
                    issued_parity[stage] = phase;
                    if (++stage == K::kStages) stage = 0, phase ^= 1;
                }
            }
            // Never leave with a copy still landing in shared memory (the
            // even CTA's full barriers count both CTAs' copies), nor, in a
            // pair, with an MMA commit still due to arrive here.
            if (!PAIR || rank == 0)
                for (int s = 0; s < K::kStages; ++s)
                    if (issued[s] && !bar_wait<PAIR>(&full[s], issued_parity[s], abort_flag)) {
                        const long long t0 = clock64();
                        while (!bar_try_wait<PAIR>(&full[s], issued_parity[s]) &&
                               clock64() - t0 < kWaitLimitCycles) {
                        }
                    }
            if (PAIR)
                for (int s = 0; s < K::kStages; ++s)
                    if (issued[s]) {
                        const long long t0 = clock64();
                        while (!bar_try_wait<PAIR>(&empty[s], issued_parity[s]) &&
                               clock64() - t0 < kWaitLimitCycles) {
                        }
                    }
        }
    } else if (warp == 3) {
        // ------------------------------------------------ tile scheduler
        // (one thread of the even CTA) The first wave is static (tile = unit
        // index); later tiles are claimed from the launch's counter, so that
        // a CTA that starts late (its SM busy with other work) takes fewer of
        // them.  Each tile index goes into a 2-deep queue read by every role
        // of both CTAs; claiming and publishing here keeps the latency of the
        // atomic and of the cluster-scope release off the operand path.
        if (lane == 0 && rank == 0) {
            for (uint32_t t = 0;; ++t) {
                const int slot = (int)(t % kTileQ);
                const uint32_t qph = (t / kTileQ) & 1;
                if (!bar_wait<PAIR>(&qempty[slot], qph ^ 1, abort_flag)) {
                    record_abort(abort_flag, p.dstatus);
                    break;
                }
                const unsigned int u = t == 0 ? (unsigned int)unit0
                                              : (unsigned int)nunits + atomicAdd(&p.ticket[0], 1u);
                const int tile = u < (unsigned int)p.num_units ? (int)u : -1;
                tileq[slot] = tile;
                if (PAIR) {
                    st_cluster_u32(cluster_addr(const_cast<int *>(&tileq[slot]), 1),
                                   (uint32_t)tile);
                    mbar_arrive_release_cl(cluster_addr(&qfull[slot], 1));
                }
                mbar_arrive(&qfull[slot]);
                if (tile < 0) break;
            }
            // The last CTA (pair) to stop claiming resets the counter for the
            // next launch; every CTA counts itself once, also after an abort.
            __threadfence();  // this CTA's last claim lands before its "done"
            if (atomicAdd(&p.ticket[1], 1u) == (unsigned int)nunits - 1u) {
                __threadfence();  // every claim of this launch is in before the reset
                atomicExch(&p.ticket[0], 0u);
                atomicExch(&p.ticket[1], 0u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_iter = 0;
            bool ok = true;
            bool any_mma = false;
            for (uint32_t t = 0; ok; ++t) {
                const int slot = (int)(t % kTileQ);
                const uint32_t qph = (t / kTileQ) & 1;
                if (!bar_wait<PAIR>(&qfull[slot], qph, abort_flag)) {
                    record_abort(abort_flag, p.dstatus);
                    ok = false;
                    break;
                }
                const int tile = tileq[slot];
                mbar_arrive(&qempty[slot]);
                if (tile < 0) break;
                int mu, nb;
                const int num_kb = p.prob[tile_coords(p, tile, mu, nb)].num_kb;
                const int num_chunks = (num_kb + kChunkBlocks - 1) / kChunkBlocks;
                for (int c = 0; ok && c < num_chunks; ++c) {
                    const int kb0 = c * kChunkBlocks;
                    const int kb1 = min(num_kb, kb0 + kChunkBlocks);
                    const uint32_t b = acc_iter & 1;
                    const uint32_t acc_phase = (acc_iter >> 1) & 1;
                    if (!bar_wait<PAIR>(&tempty[b], acc_phase ^ 1, abort_flag)) {
                        record_abort(abort_flag, p.dstatus);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + b * K::kAccCols;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!bar_wait<PAIR>(&full[stage], phase, abort_flag)) {
                            record_abort(abort_flag, p.dstatus);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + stage * K::kStageBytes);
                        const uint32_t b_addr = a_addr + kABytes;
                        const uint64_t adesc = sdesc_k128(a_addr);
                        const uint64_t bdesc = sdesc_k128(b_addr);
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            // advance 16 f16 = 32 bytes along K inside the swizzle atom
                            const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
                            if (PAIR)
                                mma_f16_ss_pair(d_tmem, adesc + (uint64_t)(2 * k),
                                                bdesc + (uint64_t)(2 * k), K::kIdesc, accum);
                            else
                                mma_f16_ss(d_tmem, adesc + (uint64_t)(2 * k),
                                           bdesc + (uint64_t)(2 * k), K::kIdesc, accum);
                        }
                        any_mma = true;
                        if (PAIR)
                            mma_commit_pair_mc(&empty[stage], kPairMask);
                        else
                            mma_commit(&empty[stage]);
                        if (++stage == K::kStages) stage = 0, phase ^= 1;
                    }
                    if (!ok) break;
                    if (PAIR)
                        mma_commit_pair_mc(&tfull[b], kPairMask);
                    else
                        mma_commit(&tfull[b]);
                    ++acc_iter;
                }
            }
            if (!ok && any_mma) {
                // drain: wait until every MMA issued so far has finished
                if (PAIR)
                    mma_commit_pair_mc(drain, 0x1);
                else
                    mma_commit(drain);
                const long long t0 = clock64();
                while (!mbar_try_wait(drain, 0) && clock64() - t0 < kWaitLimitCycles) {
                }
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;         // tensor-memory lane quadrant
        const int h = (warp - 4) >> 2;  // column half of the tile
        const int ew = warp - 4;        // epilogue warp index
        uint8_t *boxes = smem + K::kOffEpi + ew * K::kBoxes * kEpiBufBytes;
        int nstored = 0;
        uint32_t acc_iter = 0;
        bool ok = true;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        for (uint32_t t = 0; ok; ++t) {
            const int slot = (int)(t % kTileQ);
            const uint32_t qph = (t / kTileQ) & 1;
            if (!__all_sync(0xffffffffu, bar_wait<PAIR>(&qfull[slot], qph, abort_flag))) {
                if (lane == 0) record_abort(abort_flag, p.dstatus);
                ok = false;
                break;
            }
            const int tile = tileq[slot];
            __syncwarp();
            if (lane == 0) {
                if (PAIR)
                    mbar_arrive_cl(cluster_addr(&qempty[slot], 0));
                else
                    mbar_arrive(&qempty[slot]);
            }
            if (tile < 0) break;
            int mu, nb;
            const int pi = tile_coords(p, tile, mu, nb);
            const Prob &pr = p.prob[pi];
            const int num_chunks = (pr.num_kb + kChunkBlocks - 1) / kChunkBlocks;
            const int mb = PAIR ? 2 * mu + rank : mu;
            const bool rows_here = mb < pr.num_m;  // false: the odd CTA of a pair past the last m-block
            const int row0 = mb * kBM + q * 32;
            const int colh = nb * BN + h * K::kWarpCols;
            // The scales of this warp's rows and columns, loaded now so that
            // their latency overlaps the wait for the tile's sums (the scale
            // arrays are padded past M and N, like the tiles).
            float a = 0.0f;
            float bl[K::kPieces];
#pragma unroll
            for (int piece = 0; piece < K::kPieces; ++piece) bl[piece] = 0.0f;
            if (p.mode == 0 && rows_here) {
                a = __ldg(pr.sa + row0 + lane);
#pragma unroll
                for (int piece = 0; piece < K::kPieces; ++piece)
                    bl[piece] = __ldg(pr.sb + colh + piece * 32 + lane);
            }
            // With a single chunk (K <= 1024) the fp32 accumulator already is
            // f32(S): S is an integer below 2^24 in magnitude, held exactly.
            // The f32 epilogue then needs no conversion (float->int and back
            // run at a fraction of the ALU rate); adding +0 turns a -0 sum
            // (all products -0) into f32(0) = +0.
            const bool f32_sums = num_chunks == 1 && p.mode == 0;
            // ---- drain every chunk into int32 sums (or, f32_sums, f32(S))
            uint32_t acc[K::kWarpCols];  // int32 or f32 bit patterns
            for (int c = 0; c < num_chunks; ++c) {
                const uint32_t b = acc_iter & 1;
                const uint32_t acc_phase = (acc_iter >> 1) & 1;
                // warp-uniform: every lane must agree before the .sync.aligned loads
                if (!__all_sync(0xffffffffu, bar_wait<PAIR>(&tfull[b], acc_phase, abort_flag))) {
                    if (lane == 0) record_abort(abort_flag, p.dstatus);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase = tmem_base + b * K::kAccCols + h * K::kWarpCols + lane_addr;
                if (c == 0) {
#pragma unroll
                    for (int piece = 0; piece < K::kWarpCols / 16; ++piece)
                        tmem_ld16(tbase + piece * 16,
                                  *reinterpret_cast<uint32_t(*)[16]>(&acc[piece * 16]));
                    tmem_ld_wait();
                    if (!f32_sums) {
#pragma unroll
                        for (int j = 0; j < K::kWarpCols; ++j)
                            acc[j] = (uint32_t)__float2int_rn(__uint_as_float(acc[j]));
                    }
                } else {
#pragma unroll
                    for (int piece = 0; piece < K::kWarpCols / 16; ++piece) {
                        uint32_t r[16];
                        tmem_ld16(tbase + piece * 16, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            acc[piece * 16 + j] = (uint32_t)((int32_t)acc[piece * 16 + j] +
                                                             __float2int_rn(__uint_as_float(r[j])));
                    }
                }
                // the accumulator buffer is free again
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR)  // the even CTA's barrier: both epilogues release
                        mbar_arrive_cl(cluster_addr(&tempty[b], 0));
                    else
                        mbar_arrive(&tempty[b]);
                }
                ++acc_iter;
            }
            if (!ok) break;

            // ---- final epilogue of the tile from the sums
            if (!rows_here) continue;
            uint32_t rmax = 0;  // this thread's row: max |C| bits over its stored columns
#pragma unroll
            for (int piece = 0; piece < K::kPieces; ++piece) {
                uint32_t(&v)[32] = *reinterpret_cast<uint32_t(*)[32]>(&acc[piece * 32]);
                const int col0 = colh + piece * 32;
                if (p.mode == 0) {
                    // in place: the sums become the output bits
                    if (f32_sums)
                        epi_piece<true>(v, bl[piece], a, pr.relu);
                    else
                        epi_piece<false>(v, bl[piece], a, pr.relu);
                    if (pr.rowmax) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < pr.N) rmax = max(rmax, v[j] & 0x7fffffffu);
                    }
                }
                emit_box<K::kBoxes>(pr, &maps.c[pi], boxes, v, row0, col0, lane, nstored);
            }
            // exact in any order: the max of non-negative bit patterns
            if (pr.rowmax && row0 + lane < pr.M) atomicMax(pr.rowmax + row0 + lane, rmax);
        }
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }

    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();  // neither CTA leaves while the other may still signal it
    if (warp == 2) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, K::kTmemCols);
        else
            tmem_dealloc(tmem_base, K::kTmemCols);
    }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool make_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, size_t esz, const void *base,
                  uint64_t inner, uint64_t outer, uint64_t row_stride_elems, uint32_t box_inner,
                  uint32_t box_outer) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_elems * esz};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, bool PAIR, int NP>
cudaError_t launch_bn(Maps<NP> &maps, Params<NP> &p, const GemmJob *jobs, cudaStream_t st) {
    using C = Cfg<BN, PAIR>;
    // per device: the shared-memory attribute, and how many CTAs (pairs)
    // can be resident at once -- a pair needs two free SMs of one GPC, so
    // fewer than half the SMs may host pairs
    static bool ready[64] = {false};
    static int max_units[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const int sms = device_sm_count();
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 2 : 1;
    if (!ready[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN, PAIR, NP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmemBytes);
        if (e != cudaSuccess) return e;
        int units = PAIR ? sms / 2 : sms;
        if (PAIR) {
            cfg.gridDim = dim3((unsigned)(2 * units), 1, 1);
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, PAIR, NP>, &cfg) == cudaSuccess &&
                n > 0 && n < units)
                units = n;
            cudaGetLastError();
        }
        max_units[dev] = units;
        ready[dev] = true;
    }
    // per GEMM: B's tensor map (its box depends on the tile width) and the
    // GEMM's tiles, numbered after the previous GEMMs' tiles
    int units_total = 0;
    for (int i = 0; i < p.nprob; ++i) {
        const GemmJob &j = jobs[i];
        if (!make_tmap_2d(&maps.b[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, j.Bop, (uint64_t)j.K,
                          (uint64_t)j.N, (uint64_t)operand_ld(j.K), kBK, C::kBRows))
            return cudaErrorInvalidValue;
        Prob &q = p.prob[i];
        q.num_n = (int)((j.N + BN - 1) / BN);
        q.num_mu = PAIR ? (q.num_m + 1) / 2 : q.num_m;
        q.unit0 = units_total;
        units_total += q.num_mu * q.num_n;
    }
    p.num_units = units_total;
    const int units = p.num_units < max_units[dev] ? p.num_units : max_units[dev];
    cfg.gridDim = dim3((unsigned)(units * (PAIR ? 2 : 1)), 1, 1);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, PAIR, NP>, maps, p);
    count_launches(1);
    return e;
}

template <int BN, int NP>
cudaError_t launch_width(Maps<NP> &maps, Params<NP> &p, const GemmJob *jobs, bool pair,
                         cudaStream_t st) {
    if (pair) return launch_bn<BN, true, NP>(maps, p, jobs, st);
    return launch_bn<BN, false, NP>(maps, p, jobs, st);
}

}  // namespace

// CTA pairs are used whenever M spans two or more 128-row blocks, unless
// BSG_GEMM_PAIR=0 is set in the environment (the single-CTA kernel then runs
// every shape; same results).  Read on every call, like BSG_GEMM_BN below,
// so that tests can run each kernel on the same inputs.
bool gemm_pairs_enabled() {
    const char *e = getenv("BSG_GEMM_PAIR");
    return !(e && e[0] == '0' && e[1] == 0);
}

// m-units per group of the tile raster; BSG_GEMM_GROUP=1..64 overrides the
// default (same results, another order of the tiles).
int gemm_group_m() {
    const char *e = getenv("BSG_GEMM_GROUP");
    const int v = e ? atoi(e) : 0;
    return (v >= 1 && v <= 64) ? v : kGroupM;
}

// Serpentine raster (default on); BSG_GEMM_SNAKE=0 turns it off (same
// results, another order of the tiles).
int gemm_snake() {
    const char *e = getenv("BSG_GEMM_SNAKE");
    return (e && e[0] == '0' && e[1] == 0) ? 0 : 1;
}

// BSG_GEMM_BN=64|128|192|256 forces the tile width (same results); anything
// else, or nothing, leaves the choice to gemm_tile_width.
static int forced_tile_width() {
    const char *e = getenv("BSG_GEMM_BN");
    if (!e) return 0;
    const int v = atoi(e);
    return (v == 64 || v == 128 || v == 192 || v == 256) ? v : 0;
}

// Tile width for a launch of n GEMMs (M[i] x N[i]) on `sms` SMs: the one
// with the least estimated time, rounds of tiles (all GEMMs together) times
// the cost of one tile.  Tiles are 256 rows on CTA pairs (sms / 2 of them)
// when some M > 128, else 128 rows on single CTAs.  A tile of width BN costs
// BN/256 of a 256-wide one, times a penalty for the narrower MMAs (which
// read more shared memory per multiply-add) and for the fixed per-tile
// epilogue work.
int gemm_group_tile_width(const int64_t *M, const int64_t *N, int n, int sms) {
    const int widths[4] = {256, 192, 128, 64};
    const double penalty[4] = {1.0, 1.27, 1.65, 3.24};  // measured: 8192^3 at each width (pairs)
    int64_t max_m = 0;
    for (int i = 0; i < n; ++i) max_m = M[i] > max_m ? M[i] : max_m;
    const bool pair = (max_m + kBM - 1) / kBM >= 2 && gemm_pairs_enabled();
    const int64_t units = pair ? (sms / 2 > 0 ? sms / 2 : 1) : sms;
    int best = 256;
    double best_cost = 1e300;
    for (int w = 0; w < 4; ++w) {
        int64_t tiles = 0;
        for (int i = 0; i < n; ++i) {
            const int64_t num_m = (M[i] + kBM - 1) / kBM;
            const int64_t num_mu = pair ? (num_m + 1) / 2 : num_m;
            tiles += num_mu * ((N[i] + widths[w] - 1) / widths[w]);
        }
        const int64_t rounds = (tiles + units - 1) / units;
        const double cost = (double)rounds * widths[w] / 256.0 * penalty[w];
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best = widths[w];
        }
    }
    return best;
}

int gemm_tile_width(int64_t M, int64_t N, int sms) { return gemm_group_tile_width(&M, &N, 1, sms); }

template <int NP>
cudaError_t launch_group_np(const GemmJob *jobs, int n, int mode, int32_t *dstatus,
                            unsigned int *ticket, cudaStream_t st, int tile_width) {
    Maps<NP> maps;
    memset(&maps, 0, sizeof(maps));
    Params<NP> p;
    memset(&p, 0, sizeof(p));
    p.nprob = n;
    p.mode = mode;
    p.group_m = gemm_group_m();
    p.snake = gemm_snake();
    p.dstatus = dstatus;
    p.ticket = ticket;
    int64_t Ms[kMaxGroup], Ns[kMaxGroup];
    int max_m = 0;
    for (int i = 0; i < n; ++i) {
        const GemmJob &j = jobs[i];
        if (!make_tmap_2d(&maps.a[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, j.Aop, (uint64_t)j.K,
                          (uint64_t)j.M, (uint64_t)operand_ld(j.K), kBK, kBM))
            return cudaErrorInvalidValue;
        // TMA stores need 16-byte aligned rows, and a row length that is a
        // whole number of 16-byte chunks: at the right edge the store writes
        // whole chunks, so with N % 4 != 0 it would write up to 3 elements
        // past column N - 1 into the caller's row padding (ldc > N)
        const bool aligned = ((j.ldo * 4) % 16 == 0) && ((j.N * 4) % 16 == 0) &&
                             (reinterpret_cast<uintptr_t>(j.out) % 16 == 0);
        Prob &q = p.prob[i];
        q.tma_store = aligned && make_tmap_2d(&maps.c[i],
                                              mode == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                        : CU_TENSOR_MAP_DATA_TYPE_INT32,
                                              4, j.out, (uint64_t)j.N, (uint64_t)j.M,
                                              (uint64_t)j.ldo, 32, 32)
                          ? 1
                          : 0;
        q.M = (int)j.M;
        q.N = (int)j.N;
        q.K = (int)j.K;
        q.num_kb = (int)((j.K + kBK - 1) / kBK);
        q.num_m = (int)((j.M + kBM - 1) / kBM);
        q.sa = j.sa;
        q.sb = j.sb;
        q.out = j.out;
        q.ldo = j.ldo;
        q.relu = j.relu;
        q.rowmax = mode == 0 ? j.rowmax : nullptr;
        Ms[i] = j.M;
        Ns[i] = j.N;
        max_m = q.num_m > max_m ? q.num_m : max_m;
    }
    const bool pair = max_m >= 2 && gemm_pairs_enabled();
    const int forced = forced_tile_width();
    switch (forced ? forced
                   : tile_width ? tile_width : gemm_group_tile_width(Ms, Ns, n, device_sm_count())) {
        case 64: return launch_width<64, NP>(maps, p, jobs, pair, st);
        case 128: return launch_width<128, NP>(maps, p, jobs, pair, st);
        case 192: return launch_width<192, NP>(maps, p, jobs, pair, st);
        default: return launch_width<256, NP>(maps, p, jobs, pair, st);
    }
}

cudaError_t launch_gemm_tc_group(const GemmJob *jobs, int n, int mode, int32_t *dstatus,
                                 unsigned int *ticket, cudaStream_t st, int tile_width) {
    if (n < 1 || n > kMaxGroup) return cudaErrorInvalidValue;
    // a single GEMM gets the kernel compiled for one
    if (n == 1) return launch_group_np<1>(jobs, n, mode, dstatus, ticket, st, tile_width);
    return launch_group_np<kMaxGroup>(jobs, n, mode, dstatus, ticket, st, tile_width);
}

cudaError_t launch_gemm_tc(const __half *Aop, const __half *Bop, int64_t M, int64_t N,
                           int64_t K, const float *sa, const float *sb, int relu, int mode,
                           void *out, int64_t ldo, int32_t *dstatus, unsigned int *ticket,
                           cudaStream_t st, int tile_width) {
    GemmJob j;
    j.Aop = Aop;
    j.Bop = Bop;
    j.M = M;
    j.N = N;
    j.K = K;
    j.sa = sa;
    j.sb = sb;
    j.relu = relu;
    j.out = out;
    j.ldo = ldo;
    return launch_gemm_tc_group(&j, 1, mode, dstatus, ticket, st, tile_width);
}

}  // namespace bsg
