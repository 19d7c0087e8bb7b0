// Sparse MLA decode for groups of query rows that share one index list, on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// The rows of a group (the causal verify rows of a multi-token decode step:
// row i of a request sees its first L - G + 1 + i tokens) read prefixes of one
// list, so one CTA takes all H heads of all G rows of the group - L = G * H of
// the 128 TMEM lanes, L = 32 or 64; the other lanes are padding whose results
// are never stored - and each cache row is gathered once for the whole group.
// The S CTAs of a cluster (S <= 16, so rows of up to 16 x 512 keys) split the
// group's longest list as the attn_sparse page's SparseDcpDecode splits a
// row's keys, at the 512-key leaf boundaries of smd_tree.cuh (CTA s takes
// keys [512 s, 512 s + 512)); lane l masks the keys past its own row's count,
// so each row sees exactly its own leaves.
//
// Per CTA the pipeline is the tcgen05 kernel's (TMA tile::gather4 of 128-key
// chunks into a two-slot ring, S = Q K^T into TMEM, the row maximum, P in E4M3
// straight into the swizzled operand layout on all 16 warps, O = P V into
// TMEM). Two exchanges differ, because up to 15 peers would not fit the
// per-peer arrays in shared memory: each CTA leaves its maxima in its own
// shared memory and reads its peers' after a cluster barrier, and after a
// second cluster barrier (every peer's tiles are then dead) each CTA pushes
// its FP32 partials of the other owners' columns, with its sums, into their
// inboxes over the dead tiles; the merge is the pairwise tree in the order
// own, split ^ 1, split ^ 2, ..., a CTA past a lane's own count absent for it.
//
// Contract (checked): every row of a group reads a prefix of the list of the
// group's row with the largest clamped count (the first such); a CTA that
// finds a mismatch in the keys it reads writes SMD_ERR_GROUP to the status.
#include <cuda.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "smd.h"
#include "smd_internal.h"
#include "smd_ptx.cuh"
#include "smd_tc_common.cuh"
#include "smd_tree.cuh"

namespace smd {
namespace {

using tcc::kBlock;
using tcc::kTile;
constexpr int kOffQP = 0;           // query tile, later the P tiles (4 x 16 KB)
constexpr int kOffRing = kTile;     // two chunk slots
constexpr int kDead = 3 * kTile;    // [0, kDead): inboxes and the output stage after PV
constexpr int kMaxLanes = 64;
constexpr int kOffMyMax = kDead;                       // [64] this CTA's maxima (read by peers)
constexpr int kOffRowMax = kOffMyMax + kMaxLanes * 4;  // [64] the row maxima
constexpr int kOffNrow = kOffRowMax + kMaxLanes * 4;   // [8] the group's clamped counts
constexpr int kOffIdx = kOffNrow + 32;                 // [512] this CTA's key indices
constexpr int kOffLsum = kOffIdx + kTcMaxKeys * 4;     // [4][64] sums of P per 32-key group
constexpr int kOffBars = kOffLsum + 4 * kMaxLanes * 4;
constexpr int kNumBars = 16;
constexpr int kOffTmem = kOffBars + 8 * kNumBars;
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // + alignment of the dynamic base to 1 KB

constexpr int kBarQ = 0, kBarFull = 1, kBarEmpty = 3, kBarS = 5, kBarP = 9, kBarO = 10,
              kBarFreeB = 11,  // [2] pass-B "slot free" (after PV)
              kBarIn = 13;     // every peer's partial of this CTA's columns and its sums

constexpr int kProducerThreads = 256;

struct TcgMaps {
    CUtensorMap q, q_tail, kv, kv_tail;
};

struct TcgParams {
    CallArgs a;
    int32_t split, G, lanes;
    float log2_448;
    uint64_t budget_ns;
    int32_t inject_stall;
};

struct Keys {
    int first, mine, nch;
};

// Bytes of one peer's inbox: its partial of this CTA's columns (lanes x CW
// floats) and its sums (lanes floats), rounded to 16.
__device__ __forceinline__ int inbox_bytes(int lanes, int CW) {
    return (lanes * CW * 4 + lanes * 4 + 15) & ~15;
}

// The shared-memory addresses and barriers of the chunk pipeline.
__device__ __forceinline__ tcc::Pipe pipe_of(const TcgParams& p, uint32_t base, uint32_t bars,
                                             const uint8_t* smem) {
    tcc::Pipe pp;
    pp.q = base + kOffQP;
    pp.q_lo = 0u;  // the query is one E4M3 tile
    pp.ring = base + kOffRing;
    pp.full = bars + 8 * kBarFull;
    pp.empty = bars + 8 * kBarEmpty;
    pp.free_b = bars + 8 * kBarFreeB;
    pp.s = bars + 8 * kBarS;
    pp.bar_q = bars + 8 * kBarQ;
    pp.bar_p = bars + 8 * kBarP;
    pp.bar_o = bars + 8 * kBarO;
    pp.idx = reinterpret_cast<const int32_t*>(smem + kOffIdx);
    pp.status = p.a.status;
    pp.budget_ns = p.budget_ns;
    return pp;
}

// The contract, on the keys this CTA reads: every other row of the group
// agrees with the staged list on its first count entries (warps 0-7, once the
// first chunks' gathers are in flight; a mismatch only sets the status).
__device__ __forceinline__ void check_contract(const TcgParams& p, const uint8_t* smem, int b0,
                                               int ref, const Keys& k) {
    const int t = threadIdx.x;
    const int32_t* idx_s = reinterpret_cast<const int32_t*>(smem + kOffIdx);
    const int32_t* nrow = reinterpret_cast<const int32_t*>(smem + kOffNrow);
    bool bad = false;
    for (int r = 0; r < p.G; ++r) {
        if (r == ref) continue;
        const int32_t* row_idx = p.a.indices + static_cast<int64_t>(b0 + r) * p.a.W + k.first;
        const int lim = min(k.mine, nrow[r] - k.first);
        int v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = t + u * kProducerThreads;
            v[u] = (i < lim) ? row_idx[i] : 0;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = t + u * kProducerThreads;
            if (i < lim && v[u] != idx_s[i]) bad = true;
        }
    }
    if (bad && p.a.status != nullptr) atomicCAS(p.a.status, 0, SMD_ERR_GROUP);
}

// ---- warps 0-7: TMA producers -------------------------------------------------
// Pass A: the query tile was issued at setup; here the CTA's indices (from the
// group's longest list) are staged, the first two chunks gathered, the
// contract checked (off the gathers' path) and the other chunks gathered.
__device__ __forceinline__ void producer_a(const TcgMaps& maps, const TcgParams& p,
                                           const tcc::Pipe& pp, uint8_t* smem, int b0, int ref,
                                           const Keys& k, bool& ok) {
    const int t = threadIdx.x;
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + kOffIdx);
    const int32_t* ref_idx = p.a.indices + static_cast<int64_t>(b0 + ref) * p.a.W + k.first;
    for (int i = t; i < kTcMaxKeys; i += kProducerThreads) idx_s[i] = (i < k.mine) ? ref_idx[i] : 0;
    asm volatile("bar.sync 1, %0;" ::"r"(kProducerThreads) : "memory");
    uint32_t seen[2] = {0u, 0u};
    const int head = min(k.nch, 2);
    tcc::gather_pass_a(maps.kv, maps.kv_tail, pp, 0, head, seen, ok);
    check_contract(p, smem, b0, ref, k);
    tcc::gather_pass_a(maps.kv, maps.kv_tail, pp, head, k.nch, seen, ok);
}

// ---- warps 12-13: this CTA's maxima (thread = lane = TMEM lane h < L) ----------
// Key k of the CTA (k < mine) counts for lane h if first + k < n(row of h).
__device__ __forceinline__ void local_max(const TcgParams& p, uint8_t* smem, uint32_t bars,
                                         uint32_t tmem, const Keys& k, bool& ok) {
    const int h = threadIdx.x & 127;
    if (h >= p.lanes) return;  // whole padding warps
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * ((threadIdx.x >> 5) & 3)) << 16);
    const int n = reinterpret_cast<const int32_t*>(smem + kOffNrow)[h / p.a.H];
    const int lim_row = n - k.first;  // keys of this CTA that row h reads
    const float lam = p.a.scale_log2;
    float m = -INFINITY;
    for (int c = 0; c < k.nch; ++c) {
        mbar_wait(bars + 8 * (kBarS + c), 0, ok, p.a.status, p.budget_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const int cnt = min(kTcChunk, k.mine - kTcChunk * c);
        for (int q = 0; 32 * q < cnt; ++q) {
            float v[32];
            tmem_ld32(lane_base + kTcChunk * c + 32 * q, v);
            const int lim = min(cnt, lim_row - kTcChunk * c) - 32 * q;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < lim) m = fmaxf(m, lam * v[j]);
        }
    }
    reinterpret_cast<float*>(smem + kOffMyMax)[h] = m;
}

// ---- all 16 warps: P (warp w: lane quarter w % 4, keys 32j .. 32j + 31 of every
// chunk, j = w / 4; padding quarters skip) -----------------------------------------
__device__ __forceinline__ void p_phase(const TcgParams& p, uint8_t* smem, uint32_t bars,
                                        uint32_t tmem, const Keys& k, bool ok) {
    const int warp = threadIdx.x >> 5;
    const int h = 32 * (warp & 3) + (threadIdx.x & 31);
    const int j = warp >> 2;
    if (h < p.lanes) {
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        const int n = reinterpret_cast<const int32_t*>(smem + kOffNrow)[h / p.a.H];
        const int lim_row = n - k.first;
        const float lam = p.a.scale_log2;
        const float bias = reinterpret_cast<const float*>(smem + kOffRowMax)[h] - p.log2_448;
        float l = 0.f;
        for (int c = 0; c < k.nch && ok; ++c) {
            const int cnt = min(kTcChunk, k.mine - kTcChunk * c);
            if (32 * j >= cnt) continue;  // warp-uniform
            const int lim = min(cnt, lim_row - kTcChunk * c) - 32 * j;
            uint8_t* row = smem + kOffQP + c * kBlock + (h >> 3) * 1024 + (h & 7) * 128;
            float v[32];
            tmem_ld32(lane_base + kTcChunk * c + 32 * j, v);
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float pr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kk = 4 * i + e;
                    pr[e] = (kk < lim) ? ex2_approx(lam * v[kk] - bias) : 0.f;
                    l += pr[e];
                }
                w[i] = static_cast<uint32_t>(e4m3x2(pr[0], pr[1])) |
                       (static_cast<uint32_t>(e4m3x2(pr[2], pr[3])) << 16);
            }
            *reinterpret_cast<uint4*>(row + (((2 * j) ^ (h & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(row + (((2 * j + 1) ^ (h & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        reinterpret_cast<float*>(smem + kOffLsum)[j * kMaxLanes + h] = l;
    }
    fence_proxy_async();  // P (generic stores) -> the tensor core's reads
    tc_fence_before();    // every logit read is complete
    mbar_arrive_local(bars + 8 * kBarP);
}

// BF16(v * inv) of 8 columns of lane h at column `col` of the staging tile
// (rows of row_bytes; 16-byte chunk c of row h at chunk c ^ (h & mask)).
__device__ __forceinline__ void stage8(uint8_t* stage, int row_bytes, int mask, int h, int col,
                                       const float (&v)[8], float inv) {
    const uint4 w = make_uint4(bf16x2(v[0] * inv, v[1] * inv), bf16x2(v[2] * inv, v[3] * inv),
                               bf16x2(v[4] * inv, v[5] * inv), bf16x2(v[6] * inv, v[7] * inv));
    *reinterpret_cast<uint4*>(stage + h * row_bytes + (((col >> 3) ^ (h & mask)) << 4)) = w;
}

// The first `rows` lanes of the staging tile to out (rows kLatent BF16 apart),
// whole rows per warp-wide store. The caller syncs before.
__device__ __forceinline__ void flush(const uint8_t* stage, int row_bytes, int mask, int rows,
                                      uint16_t* dst) {
    const int chunks = row_bytes >> 4;
    for (int e = threadIdx.x; e < rows * chunks; e += kTcThreads) {
        const int r = e / chunks, c = e - r * chunks;
        const uint4 v = *reinterpret_cast<const uint4*>(stage + r * row_bytes + ((c ^ (r & mask)) << 4));
        *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(r) * kLatent + c * 8) = v;
    }
}

// ---- all 16 warps: exchange, merge, output ---------------------------------------
// Warp w serves lane quarter w % 4 and column group cg = w / 4 (GW = CW / 4
// columns of every owner's CW) of every column range it handles.
__device__ __forceinline__ void finish(const TcgParams& p, uint8_t* smem, uint32_t base,
                                       uint32_t bars, uint32_t tmem, int b0, int split,
                                       const Keys& k, bool& ok) {
    const int warp = threadIdx.x >> 5;
    const int h = 32 * (warp & 3) + (threadIdx.x & 31);
    const int cg = warp >> 2;
    const int S = p.split, L = p.lanes;
    const int CW = kLatent / S, GW = CW / 4;
    const bool real = h < L;  // warp-uniform (L is a multiple of 32)
    const bool have_o = ok && k.mine > 0;  // O in TMEM is defined only if PV ran
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const float* lsum = reinterpret_cast<const float*>(smem + kOffLsum);
    const float l = real ? ((lsum[h] + lsum[kMaxLanes + h]) + lsum[2 * kMaxLanes + h]) +
                               lsum[3 * kMaxLanes + h]
                         : 0.f;
    const float m = real ? reinterpret_cast<const float*>(smem + kOffRowMax)[h] : 0.f;
    uint16_t* oblock = p.a.out + static_cast<int64_t>(b0) * p.a.H * kLatent;  // lane l: out row b0*H + l
    float* lse = p.a.lse + static_cast<int64_t>(b0) * p.a.H + h;
    const int mask = min(CW / 8, 8) - 1;

    if (S == 1) {
        if (ok) {  // uniform: set by the barrier before the finish
            const float total = l;
            const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
            if (real) {
                for (int q = 0; q < GW / 8; ++q) {
                    const int col = cg * GW + 8 * q;
                    float v[8];
                    if (have_o)
                        tmem_ld8(lane_base + col, v);
                    else
#pragma unroll
                        for (int i = 0; i < 8; ++i) v[i] = 0.f;
                    stage8(smem, CW * 2, mask, h, col, v, inv);
                }
                if (cg == 0)
                    *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f
                                       : -INFINITY;
            }
            __syncthreads();
            flush(smem, CW * 2, mask, L, oblock);
        }
        return;
    }

    // Every CTA of the cluster is past its PV: all tiles are dead and every
    // inbox may be written.
    cluster_arrive_release();
    cluster_wait();
    const int ib = inbox_bytes(L, CW);
    if (real) {
        for (int kk = 1; kk < S; ++kk) {
            const int pr = split ^ kk;
            const uint32_t dst = mapa(base + (kk - 1) * ib, pr);
            const uint32_t rin = mapa(bars + 8 * kBarIn, pr);
            for (int q = 0; q < GW / 8; ++q) {
                float v[8];
                if (have_o)
                    tmem_ld8(lane_base + pr * CW + cg * GW + 8 * q, v);
                else
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = 0.f;
                const int u = cg * (GW / 4) + 2 * q;  // 16-byte units, lane innermost
                st_async_v4(dst + (u * L + h) * 16, make_float4(v[0], v[1], v[2], v[3]), rin);
                st_async_v4(dst + ((u + 1) * L + h) * 16, make_float4(v[4], v[5], v[6], v[7]), rin);
            }
            if (cg == 0) st_async_b32(dst + L * CW * 4 + h * 4, __float_as_uint(l), rin);
        }
    }
    mbar_wait(bars + 8 * kBarIn, 0, ok, p.a.status, p.budget_ns, /*always=*/true);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) return;
    uint8_t* stage = smem + (S - 1) * ib;  // after the inboxes
    if (real) {
        // The pairwise tree in the order own, split ^ 1, split ^ 2, ...; CTA
        // src is absent for lane h when its leaf lies past h's own count.
        const int n_lane = reinterpret_cast<const int32_t*>(smem + kOffNrow)[h / p.a.H];
        const int np = (n_lane + kTcLeaf - 1) / kTcLeaf;  // CTAs 0 .. np - 1 hold keys of h's row
        const float total = tree_xor_n<float>(S, [&](int kk) {
            return kk == 0 ? l : *reinterpret_cast<const float*>(smem + (kk - 1) * ib + L * CW * 4 + h * 4);
        }, split, np);
        const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
        for (int q = 0; q < GW / 8; ++q) {
            const int u = cg * (GW / 4) + 2 * q;
            float own[8];
            if (have_o)
                tmem_ld8(lane_base + split * CW + cg * GW + 8 * q, own);
            else
#pragma unroll
                for (int i = 0; i < 8; ++i) own[i] = 0.f;
            float acc[8];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const float4 r = tree_xor_n<float4>(S, [&](int kk) {
                    if (kk == 0)
                        return make_float4(own[4 * half], own[4 * half + 1], own[4 * half + 2],
                                           own[4 * half + 3]);
                    return reinterpret_cast<const float4*>(smem + (kk - 1) * ib)[(u + half) * L + h];
                }, split, np);
                acc[4 * half] = r.x;
                acc[4 * half + 1] = r.y;
                acc[4 * half + 2] = r.z;
                acc[4 * half + 3] = r.w;
            }
            stage8(stage, CW * 2, mask, h, cg * GW + 8 * q, acc, inv);
        }
        if (split == 0 && cg == 0)
            *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f : -INFINITY;
    }
    __syncthreads();
    flush(stage, CW * 2, mask, L, oblock + split * CW);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    tcg_decode_kernel(const __grid_constant__ TcgMaps maps, const TcgParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    pdl_entry();
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_addr(smem);
    const uint32_t bars = base + kOffBars;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.split, L = p.lanes, G = p.G;
    const int split = static_cast<int>(cluster_ctarank());
    const int b0 = blockIdx.y * G;
    bool ok = true;

    // The group's counts first: their round trip overlaps the setup.
    const int cnt_raw = (threadIdx.x < G) ? p.a.counts[b0 + threadIdx.x] : 0;

    if (threadIdx.x == 0) {
        mbar_init(bars + 8 * kBarQ, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars + 8 * (kBarFull + i), 1);
            mbar_init(bars + 8 * (kBarEmpty + i), 1);
            mbar_init(bars + 8 * (kBarFreeB + i), 1);
        }
        for (int c = 0; c < 4; ++c) mbar_init(bars + 8 * (kBarS + c), 1);
        mbar_init(bars + 8 * kBarP, kTcThreads);
        mbar_init(bars + 8 * kBarO, 1);
        mbar_init(bars + 8 * kBarIn, 1);
        fence_mbar_init();
        // (inject_stall: the query barrier also expects 16 bytes nobody sends,
        // so its bounded wait runs out; a test hook for the timeout path.)
        mbar_arrive_expect_tx(bars + 8 * kBarQ, kTile + (p.inject_stall ? 16 : 0));
        const int CW = kLatent / S;
        mbar_arrive_expect_tx(bars + 8 * kBarIn, (S - 1) * (L * CW * 4 + L * 4));
        // The query rows b0*H .. b0*H + 127 (the group's L, then padding).
        const int y = b0 * p.a.H;
        for (int j = 0; j < 4; ++j)
            tma_load_2d(base + kOffQP + j * kBlock, &maps.q, 128 * j, y, bars + 8 * kBarQ);
        tma_load_2d(base + kOffQP + 4 * kBlock, &maps.q_tail, 512, y, bars + 8 * kBarQ);
    }
    if (threadIdx.x < G)
        reinterpret_cast<int32_t*>(smem + kOffNrow)[threadIdx.x] = max(min(cnt_raw, p.a.W), 0);
    if (warp == 8) tmem_alloc(base + kOffTmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmem);

    // The group's longest list and this CTA's share of it.
    const int32_t* nrow = reinterpret_cast<const int32_t*>(smem + kOffNrow);
    int ref = 0, nmax = -1;
    for (int r = 0; r < G; ++r)
        if (nrow[r] > nmax) {
            nmax = nrow[r];
            ref = r;
        }
    Keys k;
    k.first = min(nmax, split * kTcLeaf);
    k.mine = min(nmax - k.first, kTcLeaf);
    k.nch = (k.mine + kTcChunk - 1) / kTcChunk;

    const tcc::Pipe pp = pipe_of(p, base, bars, smem);
    uint32_t full_seen[2] = {0u, 0u};
    if (warp < 8) {
        producer_a(maps, p, pp, smem, b0, ref, k, ok);
    } else if (warp == 8) {
        if (lane == 0) tcc::mma_qk(pp, tmem, k.nch, full_seen, ok);
        __syncwarp();
    } else if (warp >= 12) {
        local_max(p, smem, bars, tmem, k, ok);
    }
    // The row maximum: every CTA of the cluster has left its maxima in its
    // shared memory; the max warps read the peers' there.
    if (S > 1) {
        cluster_arrive_release();
        cluster_wait();
    }
    if (warp >= 12) {
        const int h = threadIdx.x & 127;
        if (h < L) {
            const float* my_max = reinterpret_cast<const float*>(smem + kOffMyMax);
            float m = my_max[h];
            const uint32_t a = smem_addr(my_max + h);
            for (int pr = 0; pr < S; ++pr)
                if (pr != split) m = fmaxf(m, ld_shared_cluster_f32(mapa(a, pr)));
            reinterpret_cast<float*>(smem + kOffRowMax)[h] = m;
        }
    }
    ok = __syncthreads_and(ok) != 0;  // every QK is complete; the row maxima are here
    tc_fence_after();
    p_phase(p, smem, bars, tmem, k, ok);
    if (warp < 8) {
        tcc::gather_pass_b(maps.kv, pp, k.nch, ok);
    } else if (warp == 8) {
        if (lane == 0) tcc::mma_pv(pp, tmem, k.nch, k.mine, full_seen, ok);
        __syncwarp();
    }
    mbar_wait(bars + 8 * kBarO, 0, ok, p.a.status, p.budget_ns);
    tc_fence_after();
    ok = __syncthreads_and(ok) != 0;  // the partial sums of P are visible; one verdict
    finish(p, smem, base, bars, tmem, b0, split, k, ok);
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_free(tmem, 512);
    }
}

constexpr int kMaxDevices = 64;

}  // namespace

int tcg_smem_bytes() { return kSmemBytes; }

int launch_tcg(const CallArgs& a, const TcgConfig& cfg, cudaStream_t stream) {
    TcgMaps maps;
    const uint64_t qrows = static_cast<uint64_t>(a.B) * static_cast<uint64_t>(a.H);
    if (!encode_row_map(&maps.q, a.q, qrows, 128, kTcHeads) ||
        !encode_row_map(&maps.q_tail, a.q, qrows, 64, kTcHeads) ||
        !encode_row_map(&maps.kv, a.kv, static_cast<uint64_t>(a.N), 128, 1) ||
        !encode_row_map(&maps.kv_tail, a.kv, static_cast<uint64_t>(a.N), 64, 1))
        return SMD_ERR_LAUNCH;
    TcgParams prm{};
    prm.a = a;
    prm.split = cfg.split;
    prm.G = cfg.G;
    prm.lanes = cfg.G * a.H;
    prm.log2_448 = static_cast<float>(std::log2(448.0));
    prm.budget_ns = cfg.wait_budget_ns;
    prm.inject_stall = cfg.inject_stall;

    static std::atomic<int> smem_set[kMaxDevices];
    static std::atomic<int> np_set[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMD_ERR_DEVICE;
    if (!smem_set[dev].load()) {
        if (cudaFuncSetAttribute(tcg_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess)
            return SMD_ERR_LAUNCH;
        smem_set[dev].store(1);
    }
    if (cfg.split > 8 && !np_set[dev].load()) {
        if (cudaFuncSetAttribute(tcg_decode_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                 1) != cudaSuccess)
            return SMD_ERR_LAUNCH;
        np_set[dev].store(1);
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(cfg.split), static_cast<unsigned>(a.B / cfg.G), 1);
    lc.blockDim = dim3(kTcThreads, 1, 1);
    lc.dynamicSmemBytes = static_cast<size_t>(kSmemBytes);
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cfg.split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    // Programmatic dependent launch: this grid may be scheduled while the
    // kernel before it finishes (pdl_entry waits for that kernel's completion).
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    lc.numAttrs = 2;
    if (cudaLaunchKernelEx(&lc, tcg_decode_kernel, maps, prm) != cudaSuccess) {
        (void)cudaGetLastError();
        return SMD_ERR_LAUNCH;
    }
    return SMD_OK;
}

}  // namespace smd
