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
//   * a 4-ary SHA-256 tree (FIPS 180-4) over C's little-endian bytes, rows
//     packed: leaves of 256 bytes hashed as SHA-256(0x00 || leaf), then
//     groups of four digests hashed as SHA-256(0x01 || d1 || ...), level by
//     level, until one digest is left.  The tree lets every leaf hash in
//     parallel; the serial depth is 5 + 3 * levels compressions.
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

// ---------------------------------------------------------------- SHA-256
// Round constants: FIPS 180-4 section 4.2.2 (first 32 bits of the
// fractional parts of the cube roots of the first 64 primes).
__constant__ uint32_t kRound[64] = {
    0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4,
    0xab1c5ed5, 0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe,
    0x9bdc06a7, 0xc19bf174, 0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f,
    0x4a7484aa, 0x5cb0a9dc, 0x76f988da, 0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7,
    0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967, 0x27b70a85, 0x2e1b2138, 0x4d2c6dfc,
    0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85, 0xa2bfe8a1, 0xa81a664b,
    0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070, 0x19a4c116,
    0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
    0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7,
    0xc67178f2};

__device__ __forceinline__ uint32_t ror(uint32_t x, int n) { return __funnelshift_r(x, x, n); }

// One compression of a 16-word big-endian block into state h (FIPS 180-4
// section 6.2.2), message schedule kept as a rolling 16-word window.
__device__ __forceinline__ void compress(uint32_t (&h)[8], uint32_t (&w)[16]) {
    uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
#pragma unroll
    for (int t = 0; t < 64; ++t) {
        uint32_t wt;
        if (t < 16) {
            wt = w[t];
        } else {
            const uint32_t w15 = w[(t - 15) & 15], w2 = w[(t - 2) & 15];
            const uint32_t s0 = ror(w15, 7) ^ ror(w15, 18) ^ (w15 >> 3);
            const uint32_t s1 = ror(w2, 17) ^ ror(w2, 19) ^ (w2 >> 10);
            wt = w[t & 15] + s0 + w[(t - 7) & 15] + s1;
            w[t & 15] = wt;
        }
        const uint32_t S1 = ror(e, 6) ^ ror(e, 11) ^ ror(e, 25);
        const uint32_t ch = (e & f) ^ (~e & g);
        const uint32_t t1 = hh + S1 + ch + kRound[t] + wt;
        const uint32_t S0 = ror(a, 2) ^ ror(a, 13) ^ ror(a, 22);
        const uint32_t mj = (a & b) ^ (a & c) ^ (b & c);
        const uint32_t t2 = S0 + mj;
        hh = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + t2;
    }
    h[0] += a; h[1] += b; h[2] += c; h[3] += d;
    h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
}

// SHA-256 of the byte string  prefix || D_0 || ... || D_{W-1}  where each
// D_i is a big-endian 32-bit word supplied by `word(i)`.  Words of the
// padded message are the stream shifted by the one prefix byte.
template <typename WordFn>
__device__ void sha256_prefixed(uint32_t prefix, int W, WordFn word, uint32_t (&h)[8]) {
    h[0] = 0x6a09e667; h[1] = 0xbb67ae85; h[2] = 0x3c6ef372; h[3] = 0xa54ff53a;
    h[4] = 0x510e527f; h[5] = 0x9b05688c; h[6] = 0x1f83d9ab; h[7] = 0x5be0cd19;
    const uint32_t nbytes = 1u + 4u * (uint32_t)W;
    const int nblocks = (int)((nbytes + 9u + 63u) / 64u);
    uint32_t prev = prefix;  // D_{-1}
    for (int blk = 0; blk < nblocks; ++blk) {
        uint32_t m[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int wi = blk * 16 + j;
            uint32_t v;
            if (wi < W) {
                const uint32_t cur = word(wi);
                v = (prev << 24) | (cur >> 8);
                prev = cur;
            } else if (wi == W) {
                v = (prev << 24) | 0x00800000u;
            } else {
                v = 0u;
            }
            m[j] = v;
        }
        if (blk == nblocks - 1) m[15] = nbytes * 8u;  // bit length < 2^32
        compress(h, m);
    }
}

constexpr int kHashThreads = 256;   // inputs per block = 4^4
constexpr int kLeafFloats = 64;     // 256-byte leaves

__device__ __forceinline__ uint32_t bswap32(uint32_t u) { return __byte_perm(u, 0, 0x0123); }

struct LeafWords {
    const float *C;
    int64_t first;  // flat float index of the leaf's first word
    int64_t N, ldc;
    bool packed;
    __device__ uint32_t operator()(int i) const {
        const int64_t e = first + i;
        const float *p = packed ? C + e : C + (e / N) * ldc + (e % N);
        return bswap32(__float_as_uint(__ldg(p)));
    }
};

struct SmemWords {
    const uint32_t *base;  // consecutive digests, 8 words each
    __device__ uint32_t operator()(int i) const { return base[i]; }
};

// LEAF: this block's level-0 inputs are leaves of C; otherwise they are
// digests in `in`.  The block reduces its 256 inputs through up to 4 levels
// (stopping once the whole tree has one node) and writes its last node.
template <bool LEAF>
__global__ void __launch_bounds__(kHashThreads)
    hash_level_kernel(const float *__restrict__ C, int64_t M, int64_t N, int64_t ldc,
                      const uint32_t *__restrict__ in, int64_t count, uint32_t *__restrict__ out) {
    __shared__ uint32_t dig[2][kHashThreads][8];
    const int t = threadIdx.x;
    const int64_t base = (int64_t)blockIdx.x * kHashThreads;
    const int64_t idx = base + t;
    uint32_t h[8];
    if (idx < count) {
        if (LEAF) {
            const int64_t nfloat = M * N;
            const int64_t first = idx * kLeafFloats;
            const int64_t left = nfloat - first;
            const int W = (int)(left < kLeafFloats ? (left > 0 ? left : 0) : kLeafFloats);
            LeafWords lw{C, first, N, ldc, ldc == N};
            sha256_prefixed(0x00u, W, lw, h);
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
    int cur = 0;
    int64_t width = kHashThreads;
    for (int level = 0; level < 4 && n > 1; ++level) {
        const int64_t nn = (n + 3) / 4;
        const int64_t nbase = lbase / 4;
        width /= 4;
        if (t < width) {
            const int64_t node = nbase + t;
            if (node < nn) {
                const int64_t first = node * 4;
                const int g = (int)(n - first < 4 ? n - first : 4);
                SmemWords sw{&dig[cur][first - lbase][0]};
                sha256_prefixed(0x01u, 8 * g, sw, h);
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
}

__global__ void digest_to_bytes_kernel(const uint32_t *__restrict__ d, uint8_t *__restrict__ out) {
    const int t = threadIdx.x;
    if (t < 32) out[t] = (uint8_t)(d[t >> 2] >> (24 - 8 * (t & 3)));
}

int64_t levels_after(int64_t n) {
    for (int l = 0; l < 4 && n > 1; ++l) n = (n + 3) / 4;
    return n;
}

}  // namespace

cudaError_t launch_probe_fill(uint64_t seed, int64_t M, int64_t N, int64_t K, float *A,
                              float *B, cudaStream_t st) {
    const int64_t total = M * K + K * N;
    const int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    probe_fill_kernel<<<(int)(blocks < cap ? blocks : cap), 256, 0, st>>>(seed, M * K, K * N, A, B);
    count_launches(1);
    return cudaGetLastError();
}

static int64_t num_leaves(int64_t M, int64_t N) {
    const int64_t nf = M * N;
    return nf <= 0 ? 1 : (nf + kLeafFloats - 1) / kLeafFloats;
}

size_t hash_workspace_bytes(int64_t M, int64_t N) {
    const int64_t n1 = (num_leaves(M, N) + kHashThreads - 1) / kHashThreads;
    return (size_t)round_up(2 * n1 * 32 + 64, 256);
}

cudaError_t launch_hash_f32(const float *C, int64_t M, int64_t N, int64_t ldc, uint8_t *out32,
                            void *ws, cudaStream_t st) {
    int64_t count = num_leaves(M, N);
    const int64_t n1cap = (count + kHashThreads - 1) / kHashThreads;
    uint32_t *bufs[2] = {static_cast<uint32_t *>(ws), static_cast<uint32_t *>(ws) + n1cap * 8};
    int which = 0;
    int nlaunch = 2;  // leaves + digest bytes
    int64_t blocks = (count + kHashThreads - 1) / kHashThreads;
    hash_level_kernel<true><<<(int)blocks, kHashThreads, 0, st>>>(C, M, N, ldc, nullptr, count,
                                                                   bufs[which]);
    count = levels_after(count);
    while (count > 1) {
        blocks = (count + kHashThreads - 1) / kHashThreads;
        hash_level_kernel<false><<<(int)blocks, kHashThreads, 0, st>>>(
            nullptr, 0, 0, 0, bufs[which], count, bufs[which ^ 1]);
        which ^= 1;
        count = levels_after(count);
        ++nlaunch;
    }
    digest_to_bytes_kernel<<<1, 32, 0, st>>>(bufs[which], out32);
    count_launches(nlaunch);
    return cudaGetLastError();
}

}  // namespace bsg
