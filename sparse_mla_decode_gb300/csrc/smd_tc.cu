// Sparse MLA decode on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA takes (query row b, a group of 128 heads, one 512-key leaf of the
// row's keys); the S CTAs of a cluster (S <= 4) split the row's keys as the
// attn_sparse page's SparseDcpDecode does, with the split points fixed at
// multiples of 512 (CTA s takes keys [512 s, 512 s + 512) clamped to n), and
// merge their FP32 partials by the fixed pairwise tree of smd_tree.cuh (the
// page's merge method, column ownership and FP32 sums, in an order that does
// not depend on S). The P anchor is the maximum over the
// whole row: every CTA first computes the logits of all its keys, the CTAs
// exchange their maxima, and only then is P formed (P = 2^(s - m + log2 448),
// E4M3, FP32 sums of the unquantized P) and multiplied with V.
//
// All 128 heads of the group live in one CTA, so every gathered cache row is
// read into shared memory once and used by all heads (M = 128 MMAs).
//
// Warp roles (512 threads):
//   warps 0-7   producers: the row's count and key range, the query tile (2D
//               TMA, 128-byte swizzle + 64-byte-swizzle tail) and 128-key
//               chunks of cache rows (TMA tile::gather4, same swizzles, one
//               issue per thread) into a two-slot ring; in pass B they gather
//               again the V columns of chunks no longer resident.
//   warp 8      MMA issuer: per chunk S = Q K^T (18 x M128 N128 K32 E4M3 MMAs)
//               into TMEM columns 128c..128c+127; after P is ready, O = P V
//               (M128 N256 K32 MMAs, V read MN-major from the same gathered
//               tile) into TMEM columns 0..511, which the logits no longer need.
//   warps 12-15 row maximum, thread h = head h = TMEM lane h, as the QK
//               chunks complete (cluster exchange over DSMEM).
//   all warps   then P, written straight into the K-major swizzled operand
//               layout over the dead query tile (four warps per TMEM lane
//               quarter, 32 keys of every chunk each);
//               once O is complete: the partials of O go to their column
//               owners over DSMEM and are merged in CTA order into BF16 out
//               and the LSE (four warps per TMEM lane quarter).
// Every wait on a copy, the tensor core or a peer is bounded.
#include <cuda.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "smd.h"
#include "smd_internal.h"
#include "smd_ptx.cuh"
#include "smd_tc_common.cuh"
#include "smd_trace.cuh"
#include "smd_tree.cuh"

namespace smd {
namespace {

using tcc::kBlock;
using tcc::kTile;
constexpr int kOffQP = 0;           // query tile, later the P tiles (4 x 16 KB)
constexpr int kOffRing = kTile;     // two chunk slots
constexpr int kOffMax = 3 * kTile;  // [S][128] maxima
constexpr int kOffSums = kOffMax + 4 * 128 * 4;  // [S][128] sums
constexpr int kOffRowMax = kOffSums + 4 * 128 * 4;  // [128] the row maxima
constexpr int kOffSmid = kOffRowMax + 128 * 4;       // [4] SM ids of the cluster's CTAs
constexpr int kOffIdx = kOffSmid + 16;               // [512] this CTA's key indices
constexpr int kOffLsum = kOffIdx + kTcMaxKeys * 4;   // [4][128] sums of P per 32-key group
constexpr int kOffFlags = kOffLsum + 4 * 128 * 4;    // [4] words the partners' "free" signals write
constexpr int kOffBars = kOffFlags + 16;
constexpr int kNumBars = 24;
constexpr int kOffTmem = kOffBars + 8 * kNumBars;
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // + alignment of the dynamic base to 1 KB

// barrier indices. A slot's "free" signals of pass A (after QK) and of pass B
// (after PV) use separate barriers, so that no barrier can complete twice
// before the thread that waits on it has seen the first completion.
constexpr int kBarQ = 0, kBarFull = 1, kBarEmpty = 3, kBarS = 5, kBarP = 9, kBarO = 10,
              kBarMax = 11, kBarIn = 13, kBarFreeB = 14, kBarDataReady = 16,
              kBarReadersDone = 17,
              kBarRoundFree = 18,  // [3]: k - 1: partner split ^ k's inbox is free
              kBarRoundFull = 21;  // [3]: k - 1: partner split ^ k's partial has landed here

struct TcMaps {
    CUtensorMap q, q_tail, kv, kv_tail;
};

// Tracing build: phase ends of CTA blockIdx.y * gridDim.x + blockIdx.x
// (stamps 0 entry, 1 keys staged, 2 own maximum, 3 row maximum, 4 P, 5 O,
// 6 partials pushed, 7 partials in, 8 merged, 9 end).
SMD_TRACE_TABLE(g_trace_tc);

__device__ __forceinline__ int trace_row() { return static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x); }

struct TcParams {
    CallArgs a;
    int32_t split;
    float log2_448;
    uint64_t budget_ns;
    int32_t inject_stall;
    float* ws;          // L2 exchange workspace (ws_slots SM slots), or null: DSMEM exchange
    int32_t ws_slots;   // SM-id slots the workspace holds
    int32_t lanes;      // heads a CTA computes (min(H, 128)); the other TMEM lanes are padding
};

__device__ __forceinline__ uint32_t sm_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

__device__ __forceinline__ float4 ld_global_cg(const float* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_global_v4(float* p, float4 v) {
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

struct Range {
    int n, first, mine, nch;
};

// CTA `split` holds leaf `split`: keys [512 split, 512 split + 512) of the row
// (the plan's S * 512 >= W).
__device__ __forceinline__ Range key_range(const TcParams& p, int b, int split) {
    Range r;
    int n = p.a.counts[b];
    n = max(min(n, p.a.W), 0);
    r.n = n;
    r.first = min(n, split * kTcLeaf);
    r.mine = min(n - r.first, kTcLeaf);
    r.nch = (r.mine + kTcChunk - 1) / kTcChunk;
    return r;
}

// Leaf `rank` of a row of n keys holds at least one key.
__device__ __forceinline__ bool leaf_present(int rank, int n) { return rank * kTcLeaf < n; }

// The shared-memory addresses and barriers of the chunk pipeline.
__device__ __forceinline__ tcc::Pipe pipe_of(const TcParams& p, uint32_t base, uint32_t bars,
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

// ---- warps 0-7: TMA producers -------------------------------------------------
// One TMA issue per thread per chunk: a single warp issuing all of a chunk's
// 160 gathers is limited by the issue rate (well below HBM bandwidth).
constexpr int kProducerThreads = 256;

// Entries of the row's index list each producer thread loads at kernel entry.
constexpr int kSpecPer = kTcMaxSplit * kTcMaxKeys / kProducerThreads;

// Pass A: this CTA's key indices are staged (from the row's list, loaded at
// kernel entry; entries past its keys name pool row 0, a real row: finite
// bytes, and its P is zero), then every chunk is gathered.
__device__ __forceinline__ void producer_a(const TcMaps& maps, const tcc::Pipe& pp, uint8_t* smem,
                                           const Range& r, const int32_t (&spec)[kSpecPer],
                                           bool& ok) {
    const int t = threadIdx.x;
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + kOffIdx);
#pragma unroll
    for (int k = 0; k < kSpecPer; ++k) {
        const int i = t + k * kProducerThreads - r.first;
        if (i >= 0 && i < r.mine) idx_s[i] = spec[k];
    }
    for (int i = r.mine + t; i < kTcMaxKeys; i += kProducerThreads) idx_s[i] = 0;
    asm volatile("bar.sync 1, %0;" ::"r"(kProducerThreads) : "memory");
    if (t == 0) SMD_STAMP(g_trace_tc, trace_row(), 1);
    uint32_t seen[2] = {0u, 0u};
    tcc::gather_pass_a(maps.kv, maps.kv_tail, pp, 0, r.nch, seen, ok);
}

__device__ __forceinline__ void zero32(float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
}

// ---- warps 12-15: row maximum (thread h = head h = TMEM lane h) ------------------
// The maximum of the CTA's logits as the QK chunks complete, then the maximum
// over the row (cluster exchange over DSMEM), left in shared memory.
__device__ __forceinline__ void row_max(const TcParams& p, uint8_t* smem, uint32_t bars,
                                        uint32_t tmem, int b, int split, bool& ok) {
    const int h = threadIdx.x & 127;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * ((threadIdx.x >> 5) & 3)) << 16);
    const Range r = key_range(p, b, split);
    const int S = p.split;
    const float lam = p.a.scale_log2;
    float* maxima = reinterpret_cast<float*>(smem + kOffMax);
    float* rowmax = reinterpret_cast<float*>(smem + kOffRowMax);
    int32_t* status = p.a.status;

    float m = -INFINITY;
    for (int c = 0; c < r.nch; ++c) {
        mbar_wait(bars + 8 * (kBarS + c), 0, ok, status, p.budget_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const int cnt = min(kTcChunk, r.mine - kTcChunk * c);
        for (int q = 0; 32 * q < cnt; ++q) {
            float v[32];
            tmem_ld32(lane_base + kTcChunk * c + 32 * q, v);
            const int lim = cnt - 32 * q;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < lim) m = fmaxf(m, lam * v[j]);
        }
    }
    if (h == 0) SMD_STAMP(g_trace_tc, trace_row(), 2);
    if (S > 1) {
        cluster_wait();  // every peer's barriers are initialised
        maxima[split * 128 + h] = m;
        const uint32_t slot = smem_addr(maxima + split * 128 + h);
        for (int pr = 0; pr < S; ++pr)
            if (pr != split) st_async_b32(mapa(slot, pr), __float_as_uint(m), mapa(bars + 8 * kBarMax, pr));
        if (h == 0) {  // this CTA's SM id, for the L2 exchange workspace
            uint32_t* smids = reinterpret_cast<uint32_t*>(smem + kOffSmid);
            const uint32_t me = sm_id();
            smids[split] = me;
            for (int pr = 0; pr < S; ++pr)
                if (pr != split) st_async_b32(mapa(smem_addr(smids + split), pr), me, mapa(bars + 8 * kBarMax, pr));
        }
        mbar_wait(bars + 8 * kBarMax, 0, ok, status, p.budget_ns, /*always=*/true);
        ok = __all_sync(0xffffffffu, ok);
        for (int pr = 0; pr < S; ++pr) m = fmaxf(m, maxima[pr * 128 + h]);
    }
    rowmax[h] = m;
    if (h == 0) SMD_STAMP(g_trace_tc, trace_row(), 3);
}

// ---- all 16 warps: P ---------------------------------------------------------------
// Warp w takes TMEM lane quarter w % 4 (thread = head h) and keys 32j..32j+31,
// j = w / 4, of every chunk: P = 2^(s - m + log2 448) in E4M3 into the K-major
// 128-byte-swizzled A operand (row h, 16-byte chunk k stored at chunk
// k ^ (h & 7)), and the FP32 sum of the unquantized P of its keys, chunks in
// ascending order, into lsum[j][h]. The exp2 unit bounds this phase, so it
// runs on every warp.
__device__ __forceinline__ void p_phase(const TcParams& p, uint8_t* smem, uint32_t bars,
                                        uint32_t tmem, int b, int split, bool ok) {
    const int warp = threadIdx.x >> 5;
    const int h = 32 * (warp & 3) + (threadIdx.x & 31);
    const int j = warp >> 2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const Range r = key_range(p, b, split);
    const float lam = p.a.scale_log2;
    const float bias = reinterpret_cast<const float*>(smem + kOffRowMax)[h] - p.log2_448;
    float l = 0.f;
    for (int c = 0; c < r.nch && ok; ++c) {
        const int lim = min(kTcChunk, r.mine - kTcChunk * c) - 32 * j;
        if (lim <= 0) continue;  // warp-uniform
        uint8_t* row = smem + kOffQP + c * kBlock + (h >> 3) * 1024 + (h & 7) * 128;
        float v[32];
        tmem_ld32(lane_base + kTcChunk * c + 32 * j, v);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float pr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = 4 * i + e;
                pr[e] = (k < lim) ? ex2_approx(lam * v[k] - bias) : 0.f;
                l += pr[e];
            }
            w[i] = static_cast<uint32_t>(e4m3x2(pr[0], pr[1])) |
                   (static_cast<uint32_t>(e4m3x2(pr[2], pr[3])) << 16);
        }
        *reinterpret_cast<uint4*>(row + (((2 * j) ^ (h & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(row + (((2 * j + 1) ^ (h & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    reinterpret_cast<float*>(smem + kOffLsum)[j * 128 + h] = l;
    fence_proxy_async();  // P (generic stores) -> the tensor core's reads
    tc_fence_before();    // every logit read is complete
    mbar_arrive_local(bars + 8 * kBarP);
}

// BF16(v * inv) of 32 columns of head h, starting at column `col` of the
// staging tile (128 rows of row_bytes; 16-byte chunk c of row h is stored at
// chunk c ^ (h & 7), so that 32 heads' stores spread over the banks).
__device__ __forceinline__ void stage_bf16x32(uint8_t* stage, int row_bytes, int h, int col,
                                              const float (&v)[32], float inv) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = bf16x2(v[2 * i] * inv, v[2 * i + 1] * inv);
    uint8_t* row = stage + h * row_bytes;
    const int c0 = col >> 3;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4*>(row + (((c0 + i) ^ (h & 7)) << 4)) =
            make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// The first `rows` heads of the staged tile to out (dst = head 0's first
// column; rows kLatent BF16 apart), every warp-wide store covering whole rows
// of the tile. The caller makes the staged tile visible to all threads first.
__device__ __forceinline__ void flush_tile(const uint8_t* stage, int row_bytes, int rows,
                                           uint16_t* dst) {
    const int chunks = row_bytes >> 4;
    for (int e = threadIdx.x; e < rows * chunks; e += kTcThreads) {
        const int r = e / chunks, c = e - r * chunks;
        const uint4 v = *reinterpret_cast<const uint4*>(stage + r * row_bytes + ((c ^ (r & 7)) << 4));
        *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(r) * kLatent + c * 8) = v;
    }
}

// a (+) b of 32 floats, either operand possibly absent.
__device__ __forceinline__ void tree_add32(float (&a)[32], bool pa, const float (&b)[32], bool pb) {
#pragma unroll
    for (int j = 0; j < 32; ++j) a[j] = tree_add(a[j], pa, b[j], pb);
}

// The four 8-float4 pieces of a partial in an inbox or workspace block (unit
// i of 32 columns at src[i * stride]).
template <typename LD>
__device__ __forceinline__ void load32(LD ld, float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 x = ld(i);
        v[4 * i] = x.x;
        v[4 * i + 1] = x.y;
        v[4 * i + 2] = x.z;
        v[4 * i + 3] = x.w;
    }
}

// DSMEM exchange and merge of one CTA's columns; NP = 32-column pieces per
// thread (2 for a 2-way split, 1 for a 4-way split). This CTA holds one inbox
// per partner: inbox k - 1 receives partner split ^ k's partial of this CTA's
// columns (128 x CW floats in 16-byte units: unit u of head h's columns in
// column group cg at (cg * GW / 4 + u) * 128 + h, so that one warp-wide
// 16-byte store of 32 heads covers 512 contiguous bytes). The pushes go out
// back to back, partner split ^ 1 first, each once that partner's tiles are
// dead. The merge is the pairwise tree in the order own, split ^ 1, split ^ 2,
// split ^ 3: (own + x1) as soon as round 1 has landed, then + (x2 + x3).
template <int NP>
__device__ __forceinline__ void exchange_dsmem(const TcParams& p, uint8_t* smem, uint32_t bars,
                                               uint32_t lane_base, uint16_t* oblock, float* lse,
                                               float m, int h, int cg, int split, int n,
                                               bool have_o, bool& ok) {
    const int S = p.split;
    const int CW = kLatent / S, GW = CW / 4;
    const int units = 128 * CW / 4;  // 16-byte units per inbox
    float4* inbox = reinterpret_cast<float4*>(smem);
    const float* sums = reinterpret_cast<const float*>(smem + kOffSums);
    int32_t* status = p.a.status;
    for (int k = 1; k < S; ++k) {
        const int pr = split ^ k;
        mbar_wait(bars + 8 * (kBarRoundFree + k - 1), 0, ok, status, p.budget_ns, /*always=*/true);
        const uint32_t rfull = mapa(bars + 8 * (kBarRoundFull + k - 1), pr);
        const uint32_t dst = mapa(smem_addr(inbox + (k - 1) * units + cg * (GW / 4) * 128 + h), pr);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            float v[32];
            if (have_o)
                tmem_ld32(lane_base + pr * CW + cg * GW + 32 * q, v);
            else
                zero32(v);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                st_async_v4(dst + (8 * q + i) * 128 * 16,
                            make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]), rfull);
        }
    }
    if (threadIdx.x == 0) SMD_STAMP(g_trace_tc, trace_row(), 6);
    const bool p0 = leaf_present(split, n), p1 = leaf_present(split ^ 1, n);
    float acc[NP][32];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        if (have_o)
            tmem_ld32(lane_base + split * CW + cg * GW + 32 * q, acc[q]);
        else
            zero32(acc[q]);
    }
    auto inbox_ld = [&](int k, int q) {
        const float4* src = inbox + (k - 1) * units + (cg * (GW / 4) + 8 * q) * 128 + h;
        return [src](int i) { return src[i * 128]; };
    };
    mbar_wait(bars + 8 * kBarRoundFull, 0, ok, status, p.budget_ns, /*always=*/true);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        float x[32];
        load32(inbox_ld(1, q), x);
        tree_add32(acc[q], p0, x, p1);
    }
    bool pa = p0 || p1;
    if (S == 4) {
        const bool p2 = leaf_present(split ^ 2, n), p3 = leaf_present(split ^ 3, n);
        mbar_wait(bars + 8 * (kBarRoundFull + 1), 0, ok, status, p.budget_ns, /*always=*/true);
        mbar_wait(bars + 8 * (kBarRoundFull + 2), 0, ok, status, p.budget_ns, /*always=*/true);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            float x[32], y[32];
            load32(inbox_ld(2, q), x);
            load32(inbox_ld(3, q), y);
            tree_add32(x, p2, y, p3);
            tree_add32(acc[q], pa, x, p2 || p3);
        }
        pa = pa || p2 || p3;
    }
    if (threadIdx.x == 0) SMD_STAMP(g_trace_tc, trace_row(), 7);
    mbar_wait(bars + 8 * kBarIn, 0, ok, status, p.budget_ns, /*always=*/true);
    ok = __syncthreads_and(ok) != 0;  // also: every inbox is consumed
    if (!ok) return;
    if (threadIdx.x == 0) SMD_STAMP(g_trace_tc, trace_row(), 8);
    // The sums by the same tree.
    float total = tree_add(sums[split * 128 + h], p0, sums[(split ^ 1) * 128 + h], p1);
    if (S == 4) {
        const bool p2 = leaf_present(split ^ 2, n), p3 = leaf_present(split ^ 3, n);
        total = tree_add(total, p0 || p1,
                         tree_add(sums[(split ^ 2) * 128 + h], p2, sums[(split ^ 3) * 128 + h], p3),
                         p2 || p3);
    }
    if (!pa) total = 0.f;
    const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        if (!pa) zero32(acc[q]);
        stage_bf16x32(smem, CW * 2, h, cg * GW + 32 * q, acc[q], inv);
    }
    if (split == 0 && cg == 0 && h < p.lanes)
        *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f : -INFINITY;
    __syncthreads();
    flush_tile(smem, CW * 2, p.lanes, oblock);
}

// ---- all 16 warps: partial exchange, merge and output -----------------------------
// Warp w serves TMEM lane quarter w % 4 (heads 32(w % 4) .. +31) and column
// group w / 4 of every column range it handles.
__device__ __forceinline__ void finish(const TcParams& p, uint8_t* smem, uint32_t bars,
                                       uint32_t tmem, int b, int group, int split, bool& ok) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = 32 * (warp & 3) + lane;
    const int cg = warp >> 2;  // column group 0..3
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const Range r = key_range(p, b, split);
    const int S = p.split;
    float* sums = reinterpret_cast<float*>(smem + kOffSums);
    const float m = reinterpret_cast<const float*>(smem + kOffRowMax)[h];
    // This CTA's sum of P: its four key groups in a fixed order.
    const float* lsum = reinterpret_cast<const float*>(smem + kOffLsum);
    const float l = ((lsum[h] + lsum[128 + h]) + lsum[256 + h]) + lsum[384 + h];
    if (cg == 0) sums[split * 128 + h] = l;  // read after the barriers below
    int32_t* status = p.a.status;
    const bool have_o = ok && r.mine > 0;  // O in TMEM is defined only if PV ran
    // Head 0 of the group; this CTA writes columns [split * CW, split * CW + CW).
    uint16_t* oblock = p.a.out + (static_cast<int64_t>(b) * p.a.H + group * kTcHeads) * kLatent;
    float* lse = p.a.lse + static_cast<int64_t>(b) * p.a.H + group * kTcHeads + h;

    if (S == 1) {
        if (ok) {  // uniform: set by the barrier before the finish
            const float total = l;
            const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
            for (int q = 0; q < kLatent / 128; ++q) {
                const int col = cg * (kLatent / 4) + 32 * q;
                float v[32];
                if (have_o)
                    tmem_ld32(lane_base + col, v);
                else
                    zero32(v);
                stage_bf16x32(smem, kLatent * 2, h, col, v, inv);
            }
            if (cg == 0 && h < p.lanes)
                *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f
                                   : -INFINITY;
            __syncthreads();
            flush_tile(smem, kLatent * 2, p.lanes, oblock);
        }
        return;
    }

    const int CW = kLatent / S;       // columns per owner
    const int GW = CW / 4;            // columns per column group
    if (p.ws != nullptr) {
        // ---- L2 exchange: every CTA writes its partials of the other owners'
        // columns into its SM's workspace slot; each owner reads the peers'
        // slots (bypassing L1) and merges them by the tree. A slot stays valid
        // until the peers have read it (the readers-done handshake), so the
        // next CTA on the same SM cannot overwrite it early.
        const uint32_t* smids = reinterpret_cast<const uint32_t*>(smem + kOffSmid);
        bool slots_ok = true;
        for (int rk = 0; rk < S; ++rk) slots_ok = slots_ok && smids[rk] < static_cast<uint32_t>(p.ws_slots);
        if (!slots_ok && threadIdx.x == 0 && status != nullptr) atomicCAS(status, 0, SMD_ERR_DEVICE);
        const bool write = ok && slots_ok;
        float* mine_ws = p.ws + static_cast<size_t>(slots_ok ? smids[split] : 0) * kTcWsSlotFloats;
        const uint32_t sum_slot = smem_addr(sums + split * 128 + h);
        for (int k = 1; k < S; ++k) {
            const int pr = split ^ k;
            if (cg == 0) st_async_b32(mapa(sum_slot, pr), __float_as_uint(l), mapa(bars + 8 * kBarIn, pr));
            if (!write) continue;
            const int blk = (split + S - pr - 1) % S;  // this CTA's block for owner pr
            // 16-byte unit u of head h's columns in group cg at (cg * GW / 4 + u) * 128 + h
            float* dst = mine_ws + static_cast<size_t>(blk) * 128 * CW + (cg * (GW / 4) * 128 + h) * 4;
            for (int q = 0; q < GW / 32; ++q) {
                float v[32];
                if (have_o)
                    tmem_ld32(lane_base + pr * CW + cg * GW + 32 * q, v);
                else
                    zero32(v);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    st_global_v4(dst + (8 * q + i) * 128 * 4,
                                 make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
            }
        }
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0)
            for (int pr = 0; pr < S; ++pr)
                if (pr != split) mbar_arrive_remote(mapa(bars + 8 * kBarDataReady, pr));
        mbar_wait(bars + 8 * kBarDataReady, 0, ok, status, p.budget_ns, /*always=*/true);
        mbar_wait(bars + 8 * kBarIn, 0, ok, status, p.budget_ns, /*always=*/true);
        const bool go = __syncthreads_and(ok && slots_ok) != 0;
        if (go) {
            // The pairwise tree in the order own, split ^ 1, split ^ 2, split ^ 3
            // (the DSMEM path's sums, bit for bit).
            auto present = [&](int k) { return leaf_present(split ^ k, r.n); };
            auto ws_ld = [&](int k, int q) {
                const int rk = split ^ k;
                const int blk = (rk + S - split - 1) % S;  // rk's block for this owner
                const float* src = p.ws + static_cast<size_t>(smids[rk]) * kTcWsSlotFloats +
                                   static_cast<size_t>(blk) * 128 * CW +
                                   ((cg * (GW / 4) + 8 * q) * 128 + h) * 4;
                return [src](int i) { return ld_global_cg(src + i * 128 * 4); };
            };
            float total = tree_add(sums[split * 128 + h], present(0), sums[(split ^ 1) * 128 + h],
                                   present(1));
            bool pa = present(0) || present(1);
            if (S == 4) {
                total = tree_add(total, pa,
                                 tree_add(sums[(split ^ 2) * 128 + h], present(2),
                                          sums[(split ^ 3) * 128 + h], present(3)),
                                 present(2) || present(3));
                pa = pa || present(2) || present(3);
            }
            if (!pa) total = 0.f;
            const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
            for (int q = 0; q < GW / 32; ++q) {
                const int col = split * CW + cg * GW + 32 * q;
                float acc[32], x[32];
                if (have_o)
                    tmem_ld32(lane_base + col, acc);
                else
                    zero32(acc);
                load32(ws_ld(1, q), x);
                tree_add32(acc, present(0), x, present(1));
                if (S == 4) {
                    float y[32];
                    load32(ws_ld(2, q), x);
                    load32(ws_ld(3, q), y);
                    tree_add32(x, present(2), y, present(3));
                    tree_add32(acc, present(0) || present(1), x, present(2) || present(3));
                }
                if (!pa) zero32(acc);
                stage_bf16x32(smem, CW * 2, h, col - split * CW, acc, inv);
            }
            if (split == 0 && cg == 0 && h < p.lanes)
                *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f
                                   : -INFINITY;
            __syncthreads();
            flush_tile(smem, CW * 2, p.lanes, oblock + split * CW);
        }
        __syncthreads();  // every read of the peers' slots is done
        if (threadIdx.x == 0)
            for (int pr = 0; pr < S; ++pr)
                if (pr != split) mbar_arrive_remote(mapa(bars + 8 * kBarReadersDone, pr));
        mbar_wait(bars + 8 * kBarReadersDone, 0, ok, status, p.budget_ns, /*always=*/true);
        return;
    }

    // ---- DSMEM exchange: one inbox per partner over this CTA's dead tiles
    // (P and the ring); partner split ^ k pushes into inbox k - 1.
    if (cg == 0)
        for (int k = 1; k < S; ++k) {
            const int pr = split ^ k;
            st_async_b32(mapa(smem_addr(sums + split * 128 + h), pr), __float_as_uint(l),
                         mapa(bars + 8 * kBarIn, pr));
        }
    // This CTA's tiles are dead: every partner may push into its inbox here.
    // The signal is a 4-byte st.async completing on the partner's barrier (a
    // cluster-scope release arrive costs about 3 us here).
    if (threadIdx.x == 0)
        for (int k = 1; k < S; ++k) {
            const int pr = split ^ k;
            st_async_b32(mapa(smem_addr(smem + kOffFlags + 4 * k), pr), 1u,
                         mapa(bars + 8 * (kBarRoundFree + k - 1), pr));
        }
    if (S == 2)
        exchange_dsmem<2>(p, smem, bars, lane_base, oblock + split * CW, lse, m, h, cg, split, r.n,
                          have_o, ok);
    else
        exchange_dsmem<1>(p, smem, bars, lane_base, oblock + split * CW, lse, m, h, cg, split, r.n,
                          have_o, ok);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_decode_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    pdl_entry();
    if (threadIdx.x == 0) {
        SMD_STAMP(g_trace_tc, trace_row(), 0);
        SMD_TRACE_SM(g_trace_tc, trace_row());
    }
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_addr(smem);
    const uint32_t bars = base + kOffBars;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.split;
    const int split = static_cast<int>(cluster_ctarank());
    const int group = blockIdx.x / S;
    const int b = blockIdx.y;
    bool ok = true;

    // The row's count (read again later from L1) and whole index list
    // (W <= 2048) are loaded first: their round trip overlaps the setup.
    int32_t spec[kSpecPer];
    {
        const int n_early = p.a.counts[b];
        const int32_t* row_idx = p.a.indices + static_cast<int64_t>(b) * p.a.W;
        const int lim = min(p.a.W, max(n_early, 0));
#pragma unroll
        for (int k = 0; k < kSpecPer; ++k) {
            const int i = threadIdx.x + k * kProducerThreads;
            spec[k] = (warp < 8 && i < lim) ? row_idx[i] : 0;
        }
    }

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
        mbar_init(bars + 8 * kBarMax, 1);
        mbar_init(bars + 8 * kBarIn, 1);
        for (int k = 0; k < 3; ++k) {
            mbar_init(bars + 8 * (kBarRoundFree + k), 1);
            mbar_init(bars + 8 * (kBarRoundFull + k), 1);
        }
        mbar_init(bars + 8 * kBarDataReady, S > 1 ? S - 1 : 1);
        mbar_init(bars + 8 * kBarReadersDone, S > 1 ? S - 1 : 1);
        fence_mbar_init();
        const int CW = kLatent / S;
        // (inject_stall: the query barrier also expects 16 bytes nobody sends,
        // so its bounded wait runs out; a test hook for the timeout path.)
        mbar_arrive_expect_tx(bars + 8 * kBarQ, kTile + (p.inject_stall ? 16 : 0));
        // The query tile depends on nothing: it goes before the rest of the setup.
        const int y = b * p.a.H + group * kTcHeads;
        for (int j = 0; j < 4; ++j)
            tma_load_2d(base + kOffQP + j * kBlock, &maps.q, 128 * j, y, bars + 8 * kBarQ);
        tma_load_2d(base + kOffQP + 4 * kBlock, &maps.q_tail, 512, y, bars + 8 * kBarQ);
        mbar_arrive_expect_tx(bars + 8 * kBarMax, (S - 1) * (128 * 4 + 4));
        // The peers' sums; on the DSMEM path, round k's partial of this CTA's columns.
        mbar_arrive_expect_tx(bars + 8 * kBarIn, (S - 1) * 128 * 4);
        if (p.ws == nullptr)
            for (int k = 1; k < S; ++k) {
                mbar_arrive_expect_tx(bars + 8 * (kBarRoundFree + k - 1), 4);
                mbar_arrive_expect_tx(bars + 8 * (kBarRoundFull + k - 1), 128 * CW * 4);
            }
    }
    if (warp == 8) tmem_alloc(base + kOffTmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmem);
    if (S > 1) cluster_arrive_relaxed();

    const tcc::Pipe pp = pipe_of(p, base, bars, smem);
    uint32_t full_seen[2] = {0u, 0u};
    const Range r = key_range(p, b, split);
    if (warp < 8) {
        producer_a(maps, pp, smem, r, spec, ok);
    } else if (warp == 8) {
        if (lane == 0) tcc::mma_qk(pp, tmem, r.nch, full_seen, ok);
        __syncwarp();
    } else if (warp >= 12) {
        row_max(p, smem, bars, tmem, b, split, ok);
    }
    if (S > 1 && warp < 12) cluster_wait();  // the max warps waited before their exchange
    // Every QK is complete and the row maxima are in shared memory; one verdict.
    ok = __syncthreads_and(ok) != 0;
    tc_fence_after();
    p_phase(p, smem, bars, tmem, b, split, ok);
    if (threadIdx.x == 0) SMD_STAMP(g_trace_tc, trace_row(), 4);
    if (warp < 8) {
        tcc::gather_pass_b(maps.kv, pp, r.nch, ok);
    } else if (warp == 8) {
        if (lane == 0) tcc::mma_pv(pp, tmem, r.nch, r.mine, full_seen, ok);
        __syncwarp();
    }
    // Every warp: O is complete in TMEM; then the exchange and the merge.
    mbar_wait(bars + 8 * kBarO, 0, ok, p.a.status, p.budget_ns);
    tc_fence_after();
    ok = __syncthreads_and(ok) != 0;  // the partial sums of P are visible; one verdict
    if (threadIdx.x == 0) SMD_STAMP(g_trace_tc, trace_row(), 5);
    finish(p, smem, bars, tmem, b, group, split, ok);
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) SMD_STAMP(g_trace_tc, trace_row(), 9);
    if (warp == 8) {
        tc_fence_after();
        tmem_free(tmem, 512);
    }
}

// ---- host ------------------------------------------------------------------------

// A few encoded tensor maps, keyed by (tensor base, rows, box): encoding is a
// host call of about a microsecond, and the cache pool / query buffers of a
// decode loop do not move.
struct MapEntry {
    const void* ptr;
    uint64_t rows;
    uint32_t box_cols, box_rows;
    CUtensorMap map;
};

std::mutex g_map_mu;
MapEntry g_maps[16];
int g_map_n = 0, g_map_next = 0;

// cuTensorMapEncodeTiled, looked up through the runtime (the library does not
// link the driver library, so it loads on machines without one).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

bool encode_map(CUtensorMap* out, const void* ptr, uint64_t rows, uint32_t box_cols,
                uint32_t box_rows) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_map_n; ++i) {
        const MapEntry& e = g_maps[i];
        if (e.ptr == ptr && e.rows == rows && e.box_cols == box_cols && e.box_rows == box_rows) {
            *out = e.map;
            return true;
        }
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRow), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRow)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle swz =
        box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    EncodeTiledFn encode = encode_fn();
    if (encode == nullptr) return false;
    CUtensorMap m;
    const CUresult r = encode(
        &m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    MapEntry& e = g_maps[g_map_next];
    e.ptr = ptr;
    e.rows = rows;
    e.box_cols = box_cols;
    e.box_rows = box_rows;
    e.map = m;
    g_map_next = (g_map_next + 1) % 16;
    if (g_map_n < 16) ++g_map_n;
    *out = m;
    return true;
}

constexpr int kMaxDevices = 64;

}  // namespace

SMD_TRACE_COPY_FN(tc_trace_copy, g_trace_tc)

int tc_smem_bytes() { return kSmemBytes; }

int tc_resident_clusters(int split) {
    static std::atomic<int> cached[kMaxDevices][kTcMaxSplit + 1];
    int dev = 0;
    if (split < 1 || split > kTcMaxSplit || cudaGetDevice(&dev) != cudaSuccess || dev < 0 ||
        dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return 0;
    }
    int v = cached[dev][split].load();
    if (v > 0) return v;
    if (cudaFuncSetAttribute(tc_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(split), 1, 1);
    lc.blockDim = dim3(kTcThreads, 1, 1);
    lc.dynamicSmemBytes = static_cast<size_t>(kSmemBytes);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_decode_kernel, &lc) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 0;
    }
    cached[dev][split].store(n);
    return n;
}

bool encode_row_map(CUtensorMap* out, const void* ptr, uint64_t rows, uint32_t box_cols,
                    uint32_t box_rows) {
    return encode_map(out, ptr, rows, box_cols, box_rows);
}

// ---- the exchange scratch of smd_sparse_mla_decode_noalloc --------------------------
// A file-scope device array: every GPU that loads the library holds these
// kStaticScratchSlots x 192 KiB (30 MiB) until the process exits. Host code
// must not pass the symbol itself to a kernel (in host code it names a host-
// side stand-in); static_scratch() looks up its device address once per
// device, with that device current.
static __device__ __align__(256) float g_exchange_scratch[static_cast<size_t>(kStaticScratchSlots) *
                                                           kTcWsSlotFloats];

float* static_scratch(int* rc) {
    static std::mutex mu;
    static float* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *rc = SMD_ERR_DEVICE;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_exchange_scratch) != cudaSuccess || ptr == nullptr) {
            (void)cudaGetLastError();
            *rc = SMD_ERR_DEVICE;
            return nullptr;
        }
        addr[dev] = static_cast<float*>(ptr);
    }
    *rc = SMD_OK;
    return addr[dev];
}

int launch_tc(const CallArgs& a, const TcConfig& cfg, cudaStream_t stream) {
    TcMaps maps;
    const uint64_t qrows = static_cast<uint64_t>(a.B) * static_cast<uint64_t>(a.H);
    if (!encode_map(&maps.q, a.q, qrows, 128, kTcHeads) ||
        !encode_map(&maps.q_tail, a.q, qrows, 64, kTcHeads) ||
        !encode_map(&maps.kv, a.kv, static_cast<uint64_t>(a.N), 128, 1) ||
        !encode_map(&maps.kv_tail, a.kv, static_cast<uint64_t>(a.N), 64, 1))
        return SMD_ERR_LAUNCH;
    TcParams prm{};
    prm.a = a;
    prm.split = cfg.split;
    prm.log2_448 = static_cast<float>(std::log2(448.0));
    prm.budget_ns = cfg.wait_budget_ns;
    prm.inject_stall = cfg.inject_stall;
    prm.ws = cfg.split > 1 ? cfg.ws : nullptr;
    prm.ws_slots = cfg.ws_slots > 0 ? cfg.ws_slots : kTcWsSlots;
    prm.lanes = a.H < kTcHeads ? a.H : kTcHeads;

    static std::atomic<int> attr_set[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMD_ERR_DEVICE;
    if (!attr_set[dev].load()) {
        if (cudaFuncSetAttribute(tc_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess)
            return SMD_ERR_LAUNCH;
        attr_set[dev].store(1);
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>((a.H + kTcHeads - 1) / kTcHeads * cfg.split),
                      static_cast<unsigned>(a.B), 1);
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
    if (cudaLaunchKernelEx(&lc, tc_decode_kernel, maps, prm) != cudaSuccess) {
        (void)cudaGetLastError();
        return SMD_ERR_LAUNCH;
    }
    return SMD_OK;
}

}  // namespace smd
