// probe.cu -- the kernel probe's inputs and its hash.
//
// "Verification -- why you can trust the numbers", section "Layer 3: the
// kernel probe": every device publishes the hash of the same seeded int8
// GEMM run through its live kernel.  The page fixes neither the generator
// nor the hash, so this library uses
//   * SplitMix64 (Steele, Lea, Flood, OOPSLA 2014): output i of the
//     generator seeded with s is mix(s + (i+1) * 0x9e3779b97f4a7c15), and an
//     output z becomes the float ((z >> 40) - 2^23) * 2^-23, exact, in
//     [-1, 1); A takes outputs 0 .. M*K-1, B the next K*N;
//   * a BLAKE2s-256 tree (RFC 7693, BLAKE2 tree mode: fanout 4, unlimited
//     depth, 256-byte leaves, inner length 32) over C's little-endian bytes,
//     rows packed: leaf i hashed with node offset i at depth 0; groups of
//     four digests hashed level by level (node offset = group index, node
//     depth = level); the last node of each level flagged; the hash is the
//     single node of the first level that has one.  Every leaf hashes in
//     parallel; the serial depth is 4 + 2 * levels compressions.
#include <stdint.h>

#include "bsg_internal.h"

namespace bsg {
namespace {

// ---------------------------------------------------------------- SplitMix64
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1ull) * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ float probe_float(uint64_t z) {
    const int32_t v = (int32_t)(uint32_t)(z >> 40) - (1 << 23);
    return __fmul_rn((float)v, 1.0f / 8388608.0f);  // exact: |v| < 2^24, times 2^-23
}

__global__ void probe_fill_kernel(uint64_t seed, int64_t nA, int64_t nB, float *__restrict__ A,
                                  float *__restrict__ B) {
    const int64_t total = nA + nB;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const float v = probe_float(splitmix64_at(seed, (uint64_t)e));
        if (e < nA)
            A[e] = v;
        else
            B[e - nA] = v;
    }
}

// ---------------------------------------------------------------- BLAKE2s
// BLAKE2s-256 (RFC 7693) in the BLAKE2 tree mode.  Messages here are always
// a whole number of 32-bit little-endian words: a leaf is C's float bits, an
// inner node its children's digests.
constexpr uint32_t kFanout = 4;
constexpr uint32_t kTreeDepth = 255;  // unlimited
constexpr uint32_t kLeafBytes = 256;

__device__ __forceinline__ uint32_t b2s_iv(int i) {
    constexpr uint32_t iv[8] = {0x6A09E667u, 0xBB67AE85u, 0x3C6EF372u, 0xA54FF53Au,
                                0x510E527Fu, 0x9B05688Cu, 0x1F83D9ABu, 0x5BE0CD19u};
    return iv[i];
}

__device__ __forceinline__ uint32_t ror(uint32_t x, int n) { return __funnelshift_r(x, x, n); }

#define B2S_G(a, b, c, d, x, y)          \
    do {                                 \
        v[a] = v[a] + v[b] + (x);        \
        v[d] = ror(v[d] ^ v[a], 16);     \
        v[c] = v[c] + v[d];              \
        v[b] = ror(v[b] ^ v[c], 12);     \
        v[a] = v[a] + v[b] + (y);        \
        v[d] = ror(v[d] ^ v[a], 8);      \
        v[c] = v[c] + v[d];              \
        v[b] = ror(v[b] ^ v[c], 7);      \
    } while (0)

// The compression function F (RFC 7693 section 3.2): t is the byte count so
// far, last_block / last_node the finalization flags.  Kept out of line: its
// ten unrolled rounds are about 18 KB of code, and one copy per call site
// (a leaf's four blocks, the tree levels) overflowed the instruction cache,
// so that warps stalled on instruction fetch rather than on arithmetic.
__device__ __noinline__ void b2s_compress(uint32_t (&h)[8], const uint32_t (&m)[16], uint32_t t,
                                          bool last_block, bool last_node) {
    constexpr uint8_t S[10][16] = {
        {0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15},
        {14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3},
        {11, 8, 12, 0, 5, 2, 15, 13, 10, 14, 3, 6, 7, 1, 9, 4},
        {7, 9, 3, 1, 13, 12, 11, 14, 2, 6, 5, 10, 4, 0, 15, 8},
        {9, 0, 5, 7, 2, 4, 10, 15, 14, 1, 11, 12, 6, 8, 3, 13},
        {2, 12, 6, 10, 0, 11, 8, 3, 4, 13, 7, 5, 15, 14, 1, 9},
        {12, 5, 1, 15, 14, 13, 4, 10, 0, 7, 6, 3, 9, 2, 8, 11},
        {13, 11, 7, 14, 12, 1, 3, 9, 5, 0, 15, 4, 8, 6, 2, 10},
        {6, 15, 14, 9, 11, 3, 0, 8, 12, 2, 13, 7, 1, 4, 10, 5},
        {10, 2, 8, 4, 7, 6, 1, 5, 15, 11, 9, 14, 3, 12, 13, 0}};
    uint32_t v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = h[i];
        v[i + 8] = b2s_iv(i);
    }
    v[12] ^= t;  // messages here stay far below 2^32 bytes
    if (last_block) v[14] = ~v[14];
    if (last_block && last_node) v[15] = ~v[15];
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        B2S_G(0, 4, 8, 12, m[S[r][0]], m[S[r][1]]);
        B2S_G(1, 5, 9, 13, m[S[r][2]], m[S[r][3]]);
        B2S_G(2, 6, 10, 14, m[S[r][4]], m[S[r][5]]);
        B2S_G(3, 7, 11, 15, m[S[r][6]], m[S[r][7]]);
        B2S_G(0, 5, 10, 15, m[S[r][8]], m[S[r][9]]);
        B2S_G(1, 6, 11, 12, m[S[r][10]], m[S[r][11]]);
        B2S_G(2, 7, 8, 13, m[S[r][12]], m[S[r][13]]);
        B2S_G(3, 4, 9, 14, m[S[r][14]], m[S[r][15]]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] ^= v[i] ^ v[i + 8];
}

// Initial state of a tree node: the IV xor the parameter block (digest 32,
// no key, fanout 4, unlimited depth, leaf 256 bytes, inner length 32).
__device__ __forceinline__ void b2s_node_init(uint32_t (&h)[8], uint64_t node_offset,
                                              uint32_t node_depth) {
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = b2s_iv(i);
    h[0] ^= 32u | (kFanout << 16) | (kTreeDepth << 24);
    h[1] ^= kLeafBytes;
    h[2] ^= (uint32_t)node_offset;
    h[3] ^= (uint32_t)((node_offset >> 32) & 0xFFFFu) | (node_depth << 16) | (32u << 24);
}

// Hash of W little-endian words supplied by word(i) as one tree node.
template <typename WordFn>
__device__ void b2s_node(int W, WordFn word, uint64_t node_offset, uint32_t node_depth,
                         bool last_node, uint32_t (&h)[8]) {
    b2s_node_init(h, node_offset, node_depth);
    const int nblocks = W == 0 ? 1 : (W + 15) / 16;
    for (int blk = 0; blk < nblocks; ++blk) {
        uint32_t m[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int wi = blk * 16 + j;
            m[j] = wi < W ? word(wi) : 0u;
        }
        const int words_done = min(W, (blk + 1) * 16);
        b2s_compress(h, m, 4u * (uint32_t)words_done, blk == nblocks - 1, last_node);
    }
}

// A full 64-word leaf at a 16-byte aligned address (the common case): 4
// blocks, each block's words loaded while the previous one is compressed.
__device__ __forceinline__ void b2s_leaf64(const uint4 *src, uint64_t node_offset,
                                           bool last_node, uint32_t (&h)[8]) {
    b2s_node_init(h, node_offset, 0);
    uint4 next[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) next[j] = __ldg(src + j);
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t m[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m[4 * j] = next[j].x; m[4 * j + 1] = next[j].y;
            m[4 * j + 2] = next[j].z; m[4 * j + 3] = next[j].w;
        }
        if (blk < 3) {
#pragma unroll
            for (int j = 0; j < 4; ++j) next[j] = __ldg(src + 4 * (blk + 1) + j);
        }
        b2s_compress(h, m, 64u * (blk + 1), blk == 3, last_node);
    }
}

// Leaves are hashed 1024 to a block (5 tree levels inside the block; a
// 1024 x 1024 output is 16 blocks), higher levels 256 to a block (4
// levels).  The hash is latency-bound (a chain of compressions), so few,
// full blocks are as fast as many small ones and leave most SMs to other
// work running beside the probe.
constexpr int kLeafThreads = 1024;
constexpr int kLeafLevels = 5;
constexpr int kNodeThreads = 256;
constexpr int kNodeLevels = 4;
constexpr int kLeafFloats = 64;  // 256-byte leaves

struct LeafWords {
    const float *C;
    int64_t first;  // flat float index of the leaf's first word
    int64_t N, ldc;
    bool packed;
    __device__ uint32_t operator()(int i) const {
        const int64_t e = first + i;
        const float *p = packed ? C + e : C + (e / N) * ldc + (e % N);
        return __float_as_uint(__ldg(p));
    }
};

struct SmemWords {
    const uint32_t *base;  // consecutive digests, 8 words each
    __device__ uint32_t operator()(int i) const { return base[i]; }
};

// LEAF: this block's level-0 inputs are leaves of C; otherwise they are the
// digests in `in` at tree depth `depth0`.  The block reduces its THREADS
// inputs through up to LEVELS levels (stopping once the whole tree has one
// node) and writes its last node; the block that produces the root also
// writes the digest's 32 bytes (its state words, little-endian) to out32.
template <bool LEAF, int THREADS, int LEVELS>
__global__ void __launch_bounds__(THREADS)
    hash_level_kernel(const float *__restrict__ C, int64_t M, int64_t N, int64_t ldc,
                      const uint32_t *__restrict__ in, int64_t count, uint32_t depth0,
                      uint32_t *__restrict__ out, uint8_t *__restrict__ out32) {
    static_assert((1 << (2 * LEVELS)) == THREADS, "THREADS must be 4^LEVELS");
    // two digest buffers of THREADS x 8 words, dynamic shared memory
    extern __shared__ uint32_t dig_raw[];
    uint32_t(*dig)[THREADS][8] = reinterpret_cast<uint32_t(*)[THREADS][8]>(dig_raw);
    const int t = threadIdx.x;
    const int64_t base = (int64_t)blockIdx.x * THREADS;
    const int64_t idx = base + t;
    uint32_t h[8];
    if (idx < count) {
        if (LEAF) {
            const int64_t nfloat = M * N;
            const int64_t first = idx * kLeafFloats;
            const int64_t left = nfloat - first;
            const bool last = idx == count - 1;
            if (left >= kLeafFloats && ldc == N &&
                (reinterpret_cast<uintptr_t>(C + first) & 15) == 0) {
                b2s_leaf64(reinterpret_cast<const uint4 *>(C + first), (uint64_t)idx, last, h);
            } else {
                const int W = (int)(left < kLeafFloats ? (left > 0 ? left : 0) : kLeafFloats);
                LeafWords lw{C, first, N, ldc, ldc == N};
                b2s_node(W, lw, (uint64_t)idx, 0u, last, h);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) h[j] = in[idx * 8 + j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) dig[0][t][j] = h[j];
    }
    __syncthreads();
    int64_t n = count;       // nodes at the current level, whole tree
    int64_t lbase = base;    // index of this block's first node at this level
    uint32_t depth = depth0;
    int cur = 0;
    int64_t width = THREADS;
    for (int level = 0; level < LEVELS && n > 1; ++level) {
        const int64_t nn = (n + 3) / 4;
        const int64_t nbase = lbase / 4;
        width /= 4;
        ++depth;
        if (t < width) {
            const int64_t node = nbase + t;
            if (node < nn) {
                const int64_t first = node * 4;
                const int g = (int)(n - first < 4 ? n - first : 4);
                SmemWords sw{&dig[cur][first - lbase][0]};
                b2s_node(8 * g, sw, (uint64_t)node, depth, node == nn - 1, h);
#pragma unroll
                for (int j = 0; j < 8; ++j) dig[cur ^ 1][t][j] = h[j];
            }
        }
        __syncthreads();
        cur ^= 1;
        n = nn;
        lbase = nbase;
    }
    // This block's surviving node (index lbase at the final level).
    if (t < 8 && lbase < n) out[lbase * 8 + t] = dig[cur][0][t];
    if (n == 1 && t < 32) out32[t] = (uint8_t)(dig[cur][0][t >> 2] >> (8 * (t & 3)));
}


}  // namespace

cudaError_t launch_probe_fill(uint64_t seed, int64_t M, int64_t N, int64_t K, float *A,
                              float *B, cudaStream_t st) {
    const int64_t total = M * K + K * N;
    const int64_t blocks = (total + 255) / 256;
    // half the SMs, one block each: the fill is ALU work that runs beside
    // other kernels in the probe's use, and a block on every SM would hold
    // each of them back
    const int64_t cap = (int64_t)device_sm_count() / 2 > 0 ? (int64_t)device_sm_count() / 2 : 1;
    probe_fill_kernel<<<(int)(blocks < cap ? blocks : cap), 256, 0, st>>>(seed, M * K, K * N, A, B);
    count_launches(1);
    return cudaGetLastError();
}

static int64_t num_leaves(int64_t M, int64_t N) {
    const int64_t nf = M * N;
    return nf <= 0 ? 1 : (nf + kLeafFloats - 1) / kLeafFloats;
}

size_t hash_workspace_bytes(int64_t M, int64_t N) {
    const int64_t n1 = (num_leaves(M, N) + kLeafThreads - 1) / kLeafThreads;
    return (size_t)round_up(2 * n1 * 32 + 64, 256);
}

cudaError_t launch_hash_f32(const float *C, int64_t M, int64_t N, int64_t ldc, uint8_t *out32,
                            void *ws, cudaStream_t st) {
    int64_t count = num_leaves(M, N);
    const int64_t n1cap = (count + kLeafThreads - 1) / kLeafThreads;
    uint32_t *bufs[2] = {static_cast<uint32_t *>(ws), static_cast<uint32_t *>(ws) + n1cap * 8};
    int which = 0;
    int nlaunch = 1;
    constexpr size_t kLeafSmem = 2 * kLeafThreads * 8 * sizeof(uint32_t);  // 64 KiB
    constexpr size_t kNodeSmem = 2 * kNodeThreads * 8 * sizeof(uint32_t);
    static bool ready[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(
            hash_level_kernel<true, kLeafThreads, kLeafLevels>,
            cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLeafSmem);
        if (e != cudaSuccess) return e;
        ready[dev] = true;
    }
    int64_t blocks = (count + kLeafThreads - 1) / kLeafThreads;
    hash_level_kernel<true, kLeafThreads, kLeafLevels><<<(int)blocks, kLeafThreads, kLeafSmem, st>>>(
        C, M, N, ldc, nullptr, count, 0u, bufs[which], out32);
    // tree depth reached inside the leaf blocks
    uint32_t depth = 0;
    for (int l = 0; l < kLeafLevels && count > 1; ++l) count = (count + 3) / 4, ++depth;
    while (count > 1) {
        blocks = (count + kNodeThreads - 1) / kNodeThreads;
        hash_level_kernel<false, kNodeThreads, kNodeLevels>
            <<<(int)blocks, kNodeThreads, kNodeSmem, st>>>(nullptr, 0, 0, 0, bufs[which], count,
                                                          depth, bufs[which ^ 1], out32);
        which ^= 1;
        for (int l = 0; l < kNodeLevels && count > 1; ++l) count = (count + 3) / 4, ++depth;
        ++nlaunch;
    }
    count_launches(nlaunch);
    return cudaGetLastError();
}

}  // namespace bsg
