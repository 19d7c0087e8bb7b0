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
#include <atomic>
#include <cstdint>

#include "smd.h"
#include "smd_internal.h"
#include "smd_ptx.cuh"

namespace smd {
namespace {

constexpr int kMaxDevicesTk = 64;
constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkCacheElems = 16384;  // parts of up to this many logits keep their keys in shared memory
constexpr int kTkMaxCluster = 8;
constexpr int kTkUnroll = 8;          // 16-byte loads in flight per thread in pass 1
constexpr int kOffCache = 0;
constexpr int kOffWHist = kTkCacheElems * 2;                // [16][512] per-warp bins
constexpr int kWStride = 520;                               // per-warp bins + a spare one
constexpr int kOffHist = kOffWHist + kTkWarps * kWStride * 4;  // [512] bins
constexpr int kOffWarp = kOffHist + 512 * 4;                // [16] scan totals; [16][2] counts
constexpr int kOffScal = kOffWarp + kTkWarps * 4 + kTkWarps * 8;
constexpr int kOffIn1 = kOffScal + 8 * 4;                        // [C][512] peers' bins
constexpr int kOffIn2 = kOffIn1 + kTkMaxCluster * 512 * 4;       // [C][128]
constexpr int kOffIn3 = kOffIn2 + kTkMaxCluster * 128 * 4;       // [C][2]
constexpr int kOffBars = kOffIn3 + kTkMaxCluster * 2 * 4;        // 3 mbarriers
constexpr int kTkSmemBytes = kOffBars + 3 * 8;
static_assert(kOffBars % 8 == 0, "mbarrier alignment");
static_assert(kTkSmemBytes <= 227 * 1024, "shared memory");

struct TopkParams {
    const uint16_t* logits;
    int64_t stride;            // elements between rows (>= L)
    const int32_t* row_ends;   // may be null
    int32_t B, L, K;
    int32_t* indices;          // [B, K]
    int32_t* counts;           // [B]
    int32_t C;                 // CTAs per row (a cluster)
    int32_t* status;           // may be null
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

// Waits for the peers' pushes on `bar` (C > 1): warp 0 waits, the others
// wait at the block barrier (spinning threads would take issue slots from the
// warps still working).
__device__ __forceinline__ void wait_peers(uint32_t bar, int C, bool& ok, int32_t* status) {
    if (C > 1) {
        if ((threadIdx.x >> 5) == 0) mbar_wait(bar, 0, ok, status, kWaitBudgetNs, /*always=*/true);
        __syncthreads();
    }
}

// Sums bins [0, nbins) of this CTA's `local` histogram with the peers' (their
// pushes landed in `inbox`, [C][nbins], once `bar` completed): thread t < nbins
// returns bin t, summed in rank order.
__device__ __forceinline__ int cluster_bins(const int* local, const int* inbox, int nbins, int C,
                                            int rank, uint32_t bar, bool& ok, int32_t* status,
                                            int t) {
    wait_peers(bar, C, ok, status);
    if (t >= nbins) return 0;
    int c = 0;
    for (int r = 0; r < C; ++r) c += (r == rank) ? local[t] : inbox[r * nbins + t];
    return c;
}

__global__ void __launch_bounds__(kTkThreads, 2) topk_select_kernel(const TopkParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_entry();
    uint4* cache = reinterpret_cast<uint4*>(smem + kOffCache);
    int* hist = reinterpret_cast<int*>(smem + kOffHist);
    int* wtot = reinterpret_cast<int*>(smem + kOffWarp);
    int* wcnt = wtot + kTkWarps;  // [16][2]: the warps' counts of keys > v and == v
    int* scal = reinterpret_cast<int*>(smem + kOffScal);
    int* in1 = reinterpret_cast<int*>(smem + kOffIn1);  // [C][512] the peers' pass-1 bins
    int* in2 = reinterpret_cast<int*>(smem + kOffIn2);  // [C][128] the peers' pass-2 bins
    int* in3 = reinterpret_cast<int*>(smem + kOffIn3);  // [C][2] the peers' counts
    const uint32_t bars = smem_addr(smem + kOffBars);   // three exchange barriers
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int* wh_all = reinterpret_cast<int*>(smem + kOffWHist);
    const int C = p.C;
    const int rank = C > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int row = blockIdx.x / C;
    const int K = p.K;
    bool ok = true;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(bars + 8 * i, 1);
        fence_mbar_init();
        if (C > 1) {
            mbar_arrive_expect_tx(bars, (C - 1) * 512 * 4);
            mbar_arrive_expect_tx(bars + 8, (C - 1) * 128 * 4);
            mbar_arrive_expect_tx(bars + 16, (C - 1) * 2 * 4);
        }
    }
    // Every CTA's barriers are armed before a peer pushes (waited below).
    if (C > 1) cluster_arrive_relaxed();

    int end = p.L;
    if (p.row_ends != nullptr) end = max(0, min(p.L, p.row_ends[row]));
    const uint16_t* src = p.logits + static_cast<int64_t>(row) * p.stride;
    const bool vec = (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0 && (p.stride & 7) == 0;
    const int nvec = (end + 7) / 8;
    // This CTA's part of the row: vectors [cv0, cv1).
    const int per = (nvec + C - 1) / C;
    const int cv0 = min(nvec, rank * per), cv1 = min(nvec, cv0 + per);
    const bool cached = cv1 - cv0 <= kTkCacheElems / 8;
    // Passes 2 and 3 read the cached keys, or the row again from global memory.
    auto fetch_keys = [&](int vi, uint32_t (&kp)[4]) {
        if (vi < cv0 || vi >= cv1) {
            kp[0] = kp[1] = kp[2] = kp[3] = 0u;
        } else if (cached) {
            const uint4 c = cache[vi - cv0];
            kp[0] = c.x;
            kp[1] = c.y;
            kp[2] = c.z;
            kp[3] = c.w;
        } else {
            keys4x2(load_vec(src, vi, end, vec), 8 * vi, end, kp);
        }
    };
    // Pushes this CTA's n ints at `local` into every peer's inbox row `rank`.
    auto push = [&](const int* local, int* inbox, int n, uint32_t bar) {
        if (C == 1) return;
        for (int i = tid; i < n; i += kTkThreads)
            for (int r = 0; r < C; ++r)
                if (r != rank)
                    st_async_b32(mapa(smem_addr(inbox + rank * n + i), r),
                                 static_cast<uint32_t>(local[i]), mapa(bar, r));
    };

    // ---- pass 1: the high 9 bits, caching the keys -----------------------------
    for (int i = tid; i < kTkWarps * kWStride; i += kTkThreads) wh_all[i] = 0;
    if (tid == 0) scal[0] = -1;
    __syncthreads();
    {
        int* whist = wh_all + warp * kWStride;  // this warp's bins; NaNs and padding count in bin 512
        for (int base = cv0 + warp * 32; base < cv1; base += kTkThreads * kTkUnroll) {
            uint4 v[kTkUnroll];
#pragma unroll
            for (int u = 0; u < kTkUnroll; ++u) {
                const int vi = base + lane + u * kTkThreads;
                v[u] = vi < cv1 ? load_vec(src, vi, end, vec) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kTkUnroll; ++u) {
                const int vi = base + lane + u * kTkThreads;
                uint32_t kp[4];
                keys4x2(v[u], 8 * vi, vi < cv1 ? end : 0, kp);
                if (cached && vi < cv1) cache[vi - cv0] = make_uint4(kp[0], kp[1], kp[2], kp[3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t lo = kp[i] & 0xFFFFu, hi = kp[i] >> 16;
                    atomicAdd(whist + (lo ? lo >> 7 : 512u), 1);
                    atomicAdd(whist + (hi ? hi >> 7 : 512u), 1);
                }
            }
        }
    }
    __syncthreads();
    {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kTkWarps; ++w) c += wh_all[w * kWStride + tid];
        hist[tid] = c;
    }
    __syncthreads();
    if (C > 1) cluster_wait();  // the peers' barriers are armed
    push(hist, in1, 512, bars);
    // Bins from the top over the whole row: thread t holds bin 511 - t.
    {
        const int c = cluster_bins(hist, in1, 512, C, rank, bars, ok, p.status, 511 - tid);
        const int incl = block_scan_incl(c, wtot);
        if (c > 0 && incl >= K && incl - c < K) {
            scal[0] = 511 - tid;
            scal[1] = incl - c;
        }
        if (tid == kTkThreads - 1) scal[4] = incl;  // all valid logits of the row
    }
    __syncthreads();
    const int b1 = scal[0];
    const int valid = scal[4];
    uint32_t v_key = 0;  // the K-th largest key (0: every valid logit is taken)
    int c_gt = 0;
    int* hist2 = hist + 512 - 128;  // pass 2's local bins (pass 1's are still pushed from hist)
    if (b1 >= 0) {
        // ---- pass 2: the low 7 bits inside bin b1 ---------------------------------
        const int above = scal[1];
        for (int i = tid; i < kTkWarps * 128; i += kTkThreads) wh_all[i] = 0;
        __syncthreads();
        int* wh2 = wh_all + warp * 128;
        const uint32_t ub1 = static_cast<uint32_t>(b1);
        for (int vi = cv0 + warp * 32 + lane; vi < cv1; vi += kTkThreads) {
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
            hist2[tid] = c;
        }
        __syncthreads();
        push(hist2, in2, 128, bars + 8);
        const int c = cluster_bins(hist2, in2, 128, C, rank, bars + 8, ok, p.status, 127 - tid);
        const int incl = block_scan_incl(c, wtot);
        const int need = K - above;
        if (tid < 128 && c > 0 && incl >= need && incl - c < need) {
            scal[2] = 127 - tid;
            scal[3] = above + incl - c;
        }
        __syncthreads();
        v_key = (static_cast<uint32_t>(b1) << 7) | static_cast<uint32_t>(scal[2]);
        c_gt = scal[3];
    }  // (b1 is the same in every CTA of the cluster: all or none run pass 2)
    const int count = b1 >= 0 ? K : valid;
    const int take_eq = K - c_gt;  // ties taken (only when b1 >= 0)
    // Ties only when a threshold exists (v_key > 0 then, so a key of 0 never ties).
    const uint32_t v_eq = b1 >= 0 ? v_key : 0x10000u;

    // ---- pass 3: compaction in index order ------------------------------------------
    // Warp w owns vectors [v0, v0 + seg) of this CTA's part, seg a multiple of 32.
    const int seg = ((cv1 - cv0 + kTkWarps - 1) / kTkWarps + 31) & ~31;
    const int v0 = cv0 + warp * seg, v1 = min(cv1, v0 + seg);
    int n_gt = 0, n_eq = 0;
    for (int vi = v0 + lane; vi < v0 + seg; vi += 32) {
        uint32_t kp[4];
        fetch_keys(vi < v1 ? vi : cv1, kp);
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
    if (tid == 0) {
        int g = 0, e = 0;
        for (int w = 0; w < kTkWarps; ++w) {
            g += wcnt[2 * w];
            e += wcnt[2 * w + 1];
        }
        scal[5] = g;
        scal[6] = e;
    }
    __syncthreads();
    push(scal + 5, in3, 2, bars + 16);
    wait_peers(bars + 16, C, ok, p.status);
    // Keys > v and == v before this warp: the lower ranks', then this CTA's warps'.
    int gt_run = 0, eq_run = 0;
    for (int r = 0; r < rank; ++r) {
        gt_run += in3[2 * r];
        eq_run += in3[2 * r + 1];
    }
    for (int w = 0; w < warp; ++w) {
        gt_run += wcnt[2 * w];
        eq_run += wcnt[2 * w + 1];
    }
    int32_t* out = p.indices + static_cast<int64_t>(row) * K;
    for (int vi = v0 + lane; vi < v0 + seg; vi += 32) {
        uint32_t kp[4];
        fetch_keys(vi < v1 ? vi : cv1, kp);
        uint32_t gm = 0, em = 0;  // bit j: element 8 vi + j is above v / equal to v
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = kp[i] & 0xFFFFu, hi = kp[i] >> 16;
            gm |= ((lo > v_key) ? 1u : 0u) << (2 * i) | ((hi > v_key) ? 2u : 0u) << (2 * i);
            em |= ((lo == v_eq) ? 1u : 0u) << (2 * i) | ((hi == v_eq) ? 2u : 0u) << (2 * i);
        }
        // one scan of both counts (each at most 8 a lane)
        int tot;
        const int ex = warp_scan_excl(__popc(gm) | (__popc(em) << 16), tot);
        int gpos = gt_run + (ex & 0xFFFF);
        int epos = eq_run + (ex >> 16);
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
        gt_run += tot & 0xFFFF;
        eq_run += tot >> 16;
    }
    if (rank == 0) {
        for (int i = count + tid; i < K; i += kTkThreads) out[i] = -1;
        if (tid == 0) p.counts[row] = count;
    }
    // Every push into this CTA landed before its waits above ended, so no
    // peer writes into it after it exits.
}

}  // namespace

int launch_topk(const uint16_t* logits, int64_t stride, const int32_t* row_ends, int32_t B,
                int32_t L, int32_t K, int32_t* indices, int32_t* counts, int32_t* status,
                int C, cudaStream_t stream) {
    static std::atomic<int> attr_set[kMaxDevicesTk];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesTk) return SMD_ERR_DEVICE;
    if (!attr_set[dev].load()) {
        if (cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kTkSmemBytes) != cudaSuccess) {
            (void)cudaGetLastError();
            return SMD_ERR_LAUNCH;
        }
        attr_set[dev].store(1);
    }
    if (C < 1 || C > kTkMaxCluster || (C & (C - 1)) != 0) return SMD_ERR_PLAN;
    TopkParams p{logits, stride, row_ends, B, L, K, indices, counts, C, status};
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(C), 1, 1);
    lc.blockDim = dim3(kTkThreads, 1, 1);
    lc.dynamicSmemBytes = static_cast<size_t>(kTkSmemBytes);
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    // Programmatic dependent launch: this grid may be scheduled while the
    // kernel before it finishes (pdl_entry waits for that kernel's completion).
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    lc.numAttrs = 2;
    if (cudaLaunchKernelEx(&lc, topk_select_kernel, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return SMD_ERR_LAUNCH;
    }
    return SMD_OK;
}

}  // namespace smd
