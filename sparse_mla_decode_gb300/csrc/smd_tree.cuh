// The fixed summation tree of a row's split partials.
//
// A row's keys are cut by list position into leaves. Every kernel forms a
// leaf's FP32 sums (P V over the leaf's keys on the tensor cores, and the sum
// of its unquantized P) from zero in one fixed order, and combines the leaves
// as a complete binary tree over positions 0, 1, 2, ..., padded with absent
// leaves: a node is the FP32 sum of its two children, an absent child is the
// identity. A plan (cluster size, spread over the grid, CTAs per row, tiles,
// exchange path) only decides which CTA evaluates which subtree, so a row's
// bits depend on its count and keys and the kernel family alone.
//
// FP32 addition is commutative, so swapping the children of any node leaves
// its value unchanged: pushing positions in the order k -> j XOR k (an owner
// that starts with its own partial and then takes its partners), or in
// reverse order (a CTA walking its chunks downwards), evaluates the same tree.
//
// Leaves: 512 keys on the tcgen05 kernels (the keys one CTA's TMEM holds
// logits for); on the warp-MMA kernels 64 * ceil(n / 1024) keys for a row of
// n keys, so at most 16 leaves (every CTA then holds an aligned block of a
// power of two of them, at most 16, whatever the split).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace smd {

constexpr int kTcLeaf = 512;
constexpr int kMmaMaxLeaves = 16;

__host__ __device__ inline int pow2_ceil(int x) {
    int p = 1;
    while (p < x) p *= 2;
    return p;
}

__host__ __device__ inline int log2_exact(int x) {
    int d = 0;
    while ((1 << d) < x) ++d;
    return d;
}

// Keys per leaf of the warp-MMA kernels for a row of n keys: the smallest
// multiple of 64 that cuts the row into at most kMmaMaxLeaves leaves.
__host__ __device__ inline int mma_leaf(int n) {
    const int chunks = (n + 64 * kMmaMaxLeaves - 1) / (64 * kMmaMaxLeaves);
    return 64 * (chunks > 1 ? chunks : 1);
}

// Leaves of a row of n keys on the warp-MMA kernels.
__host__ __device__ inline int mma_leaves(int n) {
    const int leaf = mma_leaf(n);
    return (n + leaf - 1) / leaf;
}

// Leaves per CTA when a row of n keys is spread over S CTAs (S a power of
// two): CTA s holds leaves [s * lpc, s * lpc + lpc).
__host__ __device__ inline int mma_leaves_per_cta(int n, int S) {
    return pow2_ceil((mma_leaves(n) + S - 1) / S);
}

// Keys of the CTA holding the most, over rows of at most W keys (the count is
// non-decreasing in n, so the row of W keys decides).
__host__ __device__ inline int mma_cta_keys(int W, int S) {
    const int k = mma_leaves_per_cta(W, S) * mma_leaf(W);
    return k < W ? k : W;
}

// x (+) y where either may be absent (the identity).
__device__ __forceinline__ float tree_add(float x, bool px, float y, bool py) {
    return px ? (py ? x + y : x) : y;
}

__device__ __forceinline__ float tree_plus(float a, float b) { return a + b; }
__device__ __forceinline__ float4 tree_plus(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// The tree over positions [OFF + LO, OFF + LO + N) of a unit whose position k
// holds leaf j ^ k (j: the evaluating owner; j = 0 gives list order), leaf
// src present iff src < np; `load(k)` gives position k's value and is called
// for present leaves only. Evaluated depth first, so at most log2 N + 1
// partial sums are live; N is a compile-time power of two, so the tree
// unrolls. *pres: some leaf below is present (else 0 is returned).
template <int LO, int N, typename T, typename F>
__device__ __forceinline__ T tree_xor(F&& load, int j, int np, int off, bool* pres) {
    if constexpr (N == 1) {
        *pres = (j ^ (off + LO)) < np;
        return *pres ? load(off + LO) : T{};
    } else {
        bool pa, pb;
        const T a = tree_xor<LO, N / 2, T>(load, j, np, off, &pa);
        const T b = tree_xor<LO + N / 2, N / 2, T>(load, j, np, off, &pb);
        *pres = pa || pb;
        return pa ? (pb ? tree_plus(a, b) : a) : b;
    }
}

// tree_xor over positions 0 .. n - 1, n a power of two (at most 32) chosen at
// run time. Units of 16 or 32 positions are taken as blocks of 8 (subtrees of
// the same tree) whose results are then combined, which keeps the unrolled
// code and its registers small.
template <typename T, typename F>
__device__ __forceinline__ T tree_xor_n(int n, F&& load, int j, int np) {
    bool p;
    switch (n) {
        case 1: return tree_xor<0, 1, T>(load, j, np, 0, &p);
        case 2: return tree_xor<0, 2, T>(load, j, np, 0, &p);
        case 4: return tree_xor<0, 4, T>(load, j, np, 0, &p);
        case 8: return tree_xor<0, 8, T>(load, j, np, 0, &p);
        default: break;
    }
    T blk[4];
    bool pb[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        pb[b] = false;
        blk[b] = T{};
        if (8 * b < n) blk[b] = tree_xor<0, 8, T>(load, j, np, 8 * b, &pb[b]);
    }
    const T lo = pb[0] ? (pb[1] ? tree_plus(blk[0], blk[1]) : blk[0]) : blk[1];
    if (n == 16) return lo;
    const bool plo = pb[0] || pb[1];
    const T hi = pb[2] ? (pb[3] ? tree_plus(blk[2], blk[3]) : blk[2]) : blk[3];
    return plo ? ((pb[2] || pb[3]) ? tree_plus(lo, hi) : lo) : hi;
}

// ---- the subtree stack of the warp-MMA kernels ---------------------------------
// Those kernels hold a leaf's P V partial in registers (acc[T][4][4]: 16 T
// floats a thread) and keep the subtrees of the leaves already done in TMEM,
// which they otherwise leave unused: warp w owns TMEM lane quarter w % 4 and
// columns 128 (w / 4) .. + 127, level d of its 16 T floats at column
// 128 (w / 4) + 16 T d (T = 1, 2: at least the 4 levels 16 leaves need).

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld8_raw(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Stores the partial acc[T][4][4] at TMEM column address `at` (16 T columns).
template <int T>
__device__ __forceinline__ void stash_store(uint32_t at, const float (&acc)[T][4][4]) {
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
        for (int jj = 0; jj < 4; jj += 2) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[e] = acc[t][jj][e];
                v[4 + e] = acc[t][jj + 1][e];
            }
            tmem_st8(at + 16 * t + 4 * jj, v);
        }
    tmem_st_wait();
}

// acc = stored + acc, element by element (the stored subtree is the left child).
template <int T>
__device__ __forceinline__ void stash_add(uint32_t at, float (&acc)[T][4][4]) {
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
        for (int jj = 0; jj < 4; jj += 2) {
            float v[8];
            tmem_ld8_raw(at + 16 * t + 4 * jj, v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[t][jj][e] = v[e] + acc[t][jj][e];
                acc[t][jj + 1][e] = v[4 + e] + acc[t][jj + 1][e];
            }
        }
}

}  // namespace smd
