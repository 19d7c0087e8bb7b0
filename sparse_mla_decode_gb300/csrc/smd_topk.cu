// Top-k select over bf16 logits, one GPU: the select of the topk_exchange
// page's push_local_topk (its radix histogram passes, threshold and tie rule),
// producing the decode's index list and count on the device.
//
// Per row (one 512-thread CTA): the logits are valid unless NaN; each maps to
// an unsigned 16-bit key whose order is the value order (positive sign:
// bits | 0x8000; negative: ~bits; NaN: 0). Pass 1 streams the row from HBM,
// keeps the keys in shared memory when they fit, and counts the keys' high 9
// bits (512 bins);
// scanning the bins from the top finds the bin b1 holding the K-th largest
// key and the count above it. Pass 2 counts the low 7 bits of the keys in b1,
// which gives the K-th largest key v and the count c_gt of keys above v.
// Pass 3 writes every index with key > v at [0, c_gt) and the first
// K - c_gt indices with key == v after them, both in index order: warp w
// owns a contiguous part of the row, the warps' counts are scanned, and
// within a warp ballots and shuffles give each element its position.
// Rows with fewer than K valid logits return all of them (in index order).
// Each warp counts into its own histogram, and the 16 are summed after the
// pass: bf16 logits concentrate in a few
// exponent bins, where one shared histogram would serialize the warps.
#include <cstdint>

#include "smd.h"
#include "smd_internal.h"
#include "smd_ptx.cuh"

namespace smd {
namespace {

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkCacheElems = 98304;  // rows up to this many logits keep their keys in shared memory
constexpr int kTkUnroll = 8;          // 16-byte loads in flight per thread in pass 1
constexpr int kOffCache = 0;
constexpr int kOffWHist = kTkCacheElems * 2;                // [16][512] per-warp bins
constexpr int kOffHist = kOffWHist + kTkWarps * 512 * 4;    // [512] bins
constexpr int kOffWarp = kOffHist + 512 * 4;                // [16] scan totals; [16][2] counts
constexpr int kOffScal = kOffWarp + kTkWarps * 4 + kTkWarps * 8;
constexpr int kTkSmemBytes = kOffScal + 8 * 4;
static_assert(kTkSmemBytes <= 227 * 1024, "shared memory");

struct TopkParams {
    const uint16_t* logits;
    int64_t stride;            // elements between rows (>= L)
    const int32_t* row_ends;   // may be null
    int32_t B, L, K;
    int32_t* indices;          // [B, K]
    int32_t* counts;           // [B]
};

// The keys of a 16-byte vector of logits starting at element e0, as four
// pairs (element e0 + 2i in the low half of kp[i], e0 + 2i + 1 in the high
// half); keys of NaNs and of elements at or past `end` are 0. Both halves at
// once: positive sign -> bits | 0x8000, negative -> ~bits.
__device__ __forceinline__ void keys4x2(uint4 v, int e0, int end, uint32_t (&kp)[4]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = w[i];
        const uint32_t flip = ((x >> 15) & 0x00010001u) * 0xFFFFu;  // 0xFFFF in negative halves
        uint32_t key = x ^ (flip | 0x80008000u);
        const int e = e0 + 2 * i;
        const bool lo_ok = e < end && (x & 0x7FFFu) <= 0x7F80u;
        const bool hi_ok = e + 1 < end && ((x >> 16) & 0x7FFFu) <= 0x7F80u;
        key &= (lo_ok ? 0x0000FFFFu : 0u) | (hi_ok ? 0xFFFF0000u : 0u);
        kp[i] = key;
    }
}

// Vector vi (logits 8 vi .. 8 vi + 7) of a row: one 16-byte load when the
// rows are 16-byte aligned with a stride that is a multiple of 8 (then the
// row holds round_up(end, 8) readable logits), else 2-byte loads of the
// logits before `end` only.
__device__ __forceinline__ uint4 load_vec(const uint16_t* row, int vi, int end, bool vec) {
    if (vec) return __ldg(reinterpret_cast<const uint4*>(row) + vi);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = 8 * vi + 2 * i;
        const uint32_t lo = e < end ? __ldg(row + e) : 0u;
        const uint32_t hi = e + 1 < end ? __ldg(row + e + 1) : 0u;
        w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Inclusive sum over the block (every thread passes v); wtot: kTkWarps ints.
__device__ __forceinline__ int block_scan_incl(int v, int* wtot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kTkWarps ? wtot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kTkWarps) wtot[lane] = w;
    }
    __syncthreads();
    const int r = x + (warp > 0 ? wtot[warp - 1] : 0);
    __syncthreads();  // wtot is reused by the next scan
    return r;
}

// Exclusive sum over the 32 lanes, and the warp's total.
__device__ __forceinline__ int warp_scan_excl(int v, int& total) {
    const int lane = threadIdx.x & 31;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    total = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
}

__global__ void __launch_bounds__(kTkThreads, 1) topk_select_kernel(const TopkParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint4* cache = reinterpret_cast<uint4*>(smem + kOffCache);
    int* hist = reinterpret_cast<int*>(smem + kOffHist);
    int* wtot = reinterpret_cast<int*>(smem + kOffWarp);
    int* wcnt = wtot + kTkWarps;  // [16][2]: the warps' counts of keys > v and == v
    int* scal = reinterpret_cast<int*>(smem + kOffScal);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int* wh_all = reinterpret_cast<int*>(smem + kOffWHist);
    int* whist = wh_all + warp * 512;  // this warp's bins
    const int row = blockIdx.x;
    const int K = p.K;
    int end = p.L;
    if (p.row_ends != nullptr) end = max(0, min(p.L, p.row_ends[row]));
    const uint16_t* src = p.logits + static_cast<int64_t>(row) * p.stride;
    const bool vec = (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0 && (p.stride & 7) == 0;
    const bool cached = end <= kTkCacheElems;
    const int nvec = (end + 7) / 8;
    // Passes 2 and 3 read the cached keys, or the row again from global memory.
    auto fetch_keys = [&](int vi, uint32_t (&kp)[4]) {
        if (vi >= nvec) {
            kp[0] = kp[1] = kp[2] = kp[3] = 0u;
        } else if (cached) {
            const uint4 c = cache[vi];
            kp[0] = c.x;
            kp[1] = c.y;
            kp[2] = c.z;
            kp[3] = c.w;
        } else {
            keys4x2(load_vec(src, vi, end, vec), 8 * vi, end, kp);
        }
    };

    // ---- pass 1: the high 9 bits, caching the row ------------------------------
    for (int i = tid; i < kTkWarps * 512; i += kTkThreads) wh_all[i] = 0;
    if (tid == 0) scal[0] = -1;
    __syncthreads();
    for (int base = warp * 32; base < nvec; base += kTkThreads * kTkUnroll) {
        uint4 v[kTkUnroll];
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
            const int vi = base + lane + u * kTkThreads;
            v[u] = vi < nvec ? load_vec(src, vi, end, vec) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kTkUnroll; ++u) {
            const int vi = base + lane + u * kTkThreads;
            uint32_t kp[4];
            keys4x2(v[u], 8 * vi, vi < nvec ? end : 0, kp);
            if (cached && vi < nvec) cache[vi] = make_uint4(kp[0], kp[1], kp[2], kp[3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = kp[i] & 0xFFFFu, hi = kp[i] >> 16;
                if (lo) atomicAdd(whist + (lo >> 7), 1);
                if (hi) atomicAdd(whist + (hi >> 7), 1);
            }
        }
    }
    __syncthreads();
    {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kTkWarps; ++w) c += wh_all[w * 512 + tid];
        hist[tid] = c;
    }
    __syncthreads();
    // Bins from the top: thread t holds bin 511 - t.
    {
        const int c = hist[511 - tid];
        const int incl = block_scan_incl(c, wtot);
        if (c > 0 && incl >= K && incl - c < K) {
            scal[0] = 511 - tid;
            scal[1] = incl - c;
        }
        if (tid == kTkThreads - 1) scal[4] = incl;  // all valid logits
    }
    __syncthreads();
    const int b1 = scal[0];
    const int valid = scal[4];
    uint32_t v_key = 0;  // the K-th largest key (0: every valid logit is taken)
    int c_gt = 0;
    if (b1 >= 0) {
        // ---- pass 2: the low 7 bits inside bin b1 ---------------------------------
        const int above = scal[1];
        for (int i = tid; i < kTkWarps * 128; i += kTkThreads) wh_all[i] = 0;
        __syncthreads();
        int* wh2 = wh_all + warp * 128;
        const uint32_t ub1 = static_cast<uint32_t>(b1);
        for (int vi = warp * 32 + lane; vi < nvec; vi += kTkThreads) {
            uint32_t kp[4];
            fetch_keys(vi, kp);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // keys in bin b1 (a key of 0 is in bin 0, which holds no valid key
                // when it is b1's: b1 has the K-th largest valid key)
                const uint32_t lo = kp[i] & 0xFFFFu, hi = kp[i] >> 16;
                if (lo && (lo >> 7) == ub1) atomicAdd(wh2 + (lo & 127u), 1);
                if (hi && (hi >> 7) == ub1) atomicAdd(wh2 + (hi & 127u), 1);
            }
        }
        __syncthreads();
        if (tid < 128) {
            int c = 0;
#pragma unroll
            for (int w = 0; w < kTkWarps; ++w) c += wh_all[w * 128 + tid];
            hist[tid] = c;
        }
        __syncthreads();
        const int c = tid < 128 ? hist[127 - tid] : 0;
        const int incl = block_scan_incl(c, wtot);
        const int need = K - above;
        if (tid < 128 && c > 0 && incl >= need && incl - c < need) {
            scal[2] = 127 - tid;
            scal[3] = above + incl - c;
        }
        __syncthreads();
        v_key = (static_cast<uint32_t>(b1) << 7) | static_cast<uint32_t>(scal[2]);
        c_gt = scal[3];
    }
    const int count = b1 >= 0 ? K : valid;
    const int take_eq = K - c_gt;  // ties taken (only when b1 >= 0)
    // Ties only when a threshold exists (v_key > 0 then, so a key of 0 never ties).
    const uint32_t v_eq = b1 >= 0 ? v_key : 0x10000u;

    // ---- pass 3: compaction in index order ------------------------------------------
    // Warp w owns vectors [w * seg, w * seg + seg), seg a multiple of 32.
    const int seg = ((nvec + kTkWarps - 1) / kTkWarps + 31) & ~31;
    const int v0 = warp * seg, v1 = min(nvec, v0 + seg);
    int n_gt = 0, n_eq = 0;
    for (int vi = v0 + lane; vi < v0 + seg; vi += 32) {
        uint32_t kp[4];
        fetch_keys(vi < v1 ? vi : nvec, kp);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = kp[i] & 0xFFFFu, hi = kp[i] >> 16;
            n_gt += (lo > v_key) + (hi > v_key);
            n_eq += (lo == v_eq) + (hi == v_eq);
        }
    }
    n_gt = __reduce_add_sync(0xffffffffu, n_gt);
    n_eq = __reduce_add_sync(0xffffffffu, n_eq);
    if (lane == 0) {
        wcnt[2 * warp] = n_gt;
        wcnt[2 * warp + 1] = n_eq;
    }
    __syncthreads();
    int gt_run = 0, eq_run = 0;  // keys > v and == v in the warps before this one
    for (int w = 0; w < warp; ++w) {
        gt_run += wcnt[2 * w];
        eq_run += wcnt[2 * w + 1];
    }
    int32_t* out = p.indices + static_cast<int64_t>(row) * K;
    for (int vi = v0 + lane; vi < v0 + seg; vi += 32) {
        uint32_t kp[4];
        fetch_keys(vi < v1 ? vi : nvec, kp);
        uint32_t gm = 0, em = 0;  // bit j: element 8 vi + j is above v / equal to v
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = kp[i] & 0xFFFFu, hi = kp[i] >> 16;
            gm |= ((lo > v_key) ? 1u : 0u) << (2 * i) | ((hi > v_key) ? 2u : 0u) << (2 * i);
            em |= ((lo == v_eq) ? 1u : 0u) << (2 * i) | ((hi == v_eq) ? 2u : 0u) << (2 * i);
        }
        int g_tot, e_tot;
        int gpos = gt_run + warp_scan_excl(__popc(gm), g_tot);
        int epos = eq_run + warp_scan_excl(__popc(em), e_tot);
        while (gm) {
            const int j = __ffs(gm) - 1;
            gm &= gm - 1;
            out[gpos++] = 8 * vi + j;
        }
        while (em && epos < take_eq) {
            const int j = __ffs(em) - 1;
            em &= em - 1;
            out[c_gt + epos++] = 8 * vi + j;
        }
        gt_run += g_tot;
        eq_run += e_tot;
    }
    for (int i = count + tid; i < K; i += kTkThreads) out[i] = -1;
    if (tid == 0) p.counts[row] = count;
}

}  // namespace

int launch_topk(const uint16_t* logits, int64_t stride, const int32_t* row_ends, int32_t B,
                int32_t L, int32_t K, int32_t* indices, int32_t* counts, cudaStream_t stream) {
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kTkSmemBytes) != cudaSuccess) {
            (void)cudaGetLastError();
            return SMD_ERR_LAUNCH;
        }
        attr = true;
    }
    TopkParams p{logits, stride, row_ends, B, L, K, indices, counts};
    topk_select_kernel<<<B, kTkThreads, kTkSmemBytes, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return SMD_ERR_LAUNCH;
    return SMD_OK;
}

}  // namespace smd
