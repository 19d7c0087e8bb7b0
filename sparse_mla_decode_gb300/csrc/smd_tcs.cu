// Sparse MLA decode on the tcgen05 tensor cores with a row's keys spread over
// any CTAs of the grid (not one cluster): the split-KV pattern of the
// attn_sparse page's SparseDcpDecode carried across clusters, with the FP32
// partials and the per-row counter in global memory as the page's P3 split
// variant does (its "cross-cluster merge through a global workspace").
//
// Work items. A unit is (query row b, group of 128 heads); a unit whose row
// holds n > 0 keys (n = clamp(counts[b], 0, W)) becomes s = ceil(n / 512)
// items of at most 512 keys each: piece j takes the 512-key leaf
// [512 j, 512 j + 512) clamped to n, the split points of the cluster kernel,
// so that both evaluate the same summation tree (smd_tree.cuh). Every CTA
// reads the counts and lays the items out the same way:
// a prefix sum over units numbers them, and item i runs on CTA i % grid in
// round i / grid. The grid is launched cooperatively (every CTA resident), so
// a CTA that waits for a peer item of its unit always waits for a CTA that is
// running: the peer's earlier rounds never wait on later items.
//
// Per item the pipeline is the tcgen05 kernel's (TMA tile::gather4 of 128-key
// chunks into a two-slot ring, S = Q K^T into TMEM, P in E4M3 straight into
// the swizzled operand layout, O = P V into TMEM). The row maximum and the
// partials go through global memory (L2):
//   1. each item publishes its 128 maxima, each as a 64-bit word tagged with
//      the call (so the value and its readiness arrive in one load), and
//      takes the maximum over the unit's items as their tags appear;
//   2. after PV it writes its FP32 partials of the other items' columns
//      (owner j of s owns columns [16 floor(32 j / s), 16 floor(32 (j+1) / s)))
//      and its sums, and raises one flag per owner;
//   3. each owner waits for its flags, merges the pieces by the pairwise tree
//      (its own partial first, then pieces j ^ 1, j ^ 2, ...), and writes BF16
//      out (and LSE, owner 0).
// A flag holds the call's 64-bit token (a maximum's word its low half), so
// stale words from earlier calls never pass; the reader of a flag zeroes it
// once it is consumed, an item its maxima once every peer has read them.
// Every wait (copies, tensor core, peer flags) is bounded.
#include <cuda.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>

#include "smd.h"
#include "smd_internal.h"
#include "smd_ptx.cuh"
#include "smd_qsplit.cuh"
#include "smd_tc_common.cuh"
#include "smd_trace.cuh"
#include "smd_tree.cuh"

namespace smd {
namespace {

using tcc::kBlock;
using tcc::kTile;

constexpr int kOffQP = 0;                                 // query tile, later the P tiles
constexpr int kOffRing = kTile;                           // two chunk slots; the output stage after PV
constexpr int kOffPrefix = 3 * kTile;                     // [units + 1] first item of each unit
constexpr int kOffRowMax = kOffPrefix + (kTcsMaxUnits + 1) * 4 + 12;  // [128]
constexpr int kOffLsum = kOffRowMax + 128 * 4;            // [4][128] sums of P per 32-key group
constexpr int kOffIdx = kOffLsum + 4 * 128 * 4;           // [512] this item's key indices
constexpr int kOffWarpSum = kOffIdx + kTcMaxKeys * 4;     // [16] block scan
constexpr int kOffBars = kOffWarpSum + 16 * 4;
constexpr int kNumBars = 14;
constexpr int kOffTmem = kOffBars + 8 * kNumBars;
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // + alignment of the dynamic base to 1 KB
static_assert(kOffRowMax % 16 == 0 && kOffBars % 8 == 0, "layout alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

constexpr int kBarQ = 0, kBarFull = 1, kBarEmpty = 3, kBarFreeB = 5, kBarS = 7, kBarP = 11,
              kBarO = 12, kBarLand = 13;  // the staged merge's bulk copies

constexpr int kProducerThreads = 256;

// Tracing build: phase ends of round r < 4 of CTA blockIdx.x, row 4 blockIdx.x
// + r (stamps 0 item start, 1 keys staged, 2 own maximum, 3 row maximum over
// the unit's pieces, 4 P, 5 O, 6 partials written, 7 partials in, 8 end; and
// within the merge, 9 sums merged, 10 columns merged, 11 output staged).
SMD_TRACE_TABLE(g_trace_tcs);

__device__ __forceinline__ int trace_row(int item, int grid) {
    const int r = item / grid;
    return r < 4 ? static_cast<int>(blockIdx.x) * 4 + r : -1;
}

struct TcsMaps {
    CUtensorMap q, q_tail, kv, kv_tail;
    CUtensorMap q_lo, q_lo_tail;  // the split query's lo rows (unused otherwise)
};

struct TcsParams {
    CallArgs a;
    int32_t HG;      // head groups per row (ceil(H / 128); 1 for row groups)
    int32_t G;       // rows per unit: 1, or the row group (rows sharing one index list)
    int32_t lanes;   // query rows a unit computes (min(H, 128), or G * H); the rest is padding
    int32_t units;   // B / G * HG
    int32_t grid;    // CTAs
    float log2_448;
    uint64_t budget_ns;
    int32_t inject_stall;
    uint64_t token;  // this call's flag value (never 0)
    TcsWorkspace ws;
    uint8_t* ws_base;
    const float* lamh;  // the split query's per-row logit scales [B * H], or null
};

// A unit is G consecutive query rows b0 .. b0 + G - 1 (G = 1: one row) and
// head group g; its TMEM lane h (h < lanes) is query row (b0 H + g 128 + h) of
// the [B * H, 576] query, whose own key count is that of row b0 + h / H. Its
// keys are the list of its row with the most keys (`ref`, the first such);
// the other rows read prefixes of it (the row-group contract).
struct Item {
    int b0, g, s, j, item0;  // first row, head group, items of the unit, this piece, its first item
    int ref, n;              // the row (0 .. G - 1) whose list the unit reads, and its count
    int first, mine, nch;    // keys of this piece
    int64_t row0;            // the unit's first query row (b0 * H + g * 128)
};

// The logit scale of lane h of the unit at query row row0.
__device__ __forceinline__ float lam_of(const TcsParams& p, int64_t row0, int h) {
    if (p.lamh == nullptr) return p.a.scale_log2;
    return h < p.lanes ? p.lamh[row0 + h] : 0.f;
}


__device__ __forceinline__ float4 ld_cg_v4(const float* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_cg_f32(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(float* p, float4 v) {
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// The tag a maximum's word carries: the low half of the call's token, never 0
// (a consumed word is zeroed).
__device__ __forceinline__ uint32_t max_tag(uint64_t token) { return static_cast<uint32_t>(token) | 1u; }

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Waits (bounded) until *flag holds the call's token; on expiry the status
// gets SMD_ERR_TIMEOUT and ok is cleared.
__device__ __forceinline__ void wait_flag(const uint64_t* flag, uint64_t token, bool& ok,
                                          int32_t* status, uint64_t budget_ns) {
    if (ld_acquire_u64(flag) == token) return;
    const uint64_t t0 = globaltimer();
    while (ld_acquire_u64(flag) != token) {
        if (globaltimer() - t0 > budget_ns) {
            if (status != nullptr) atomicCAS(status, 0, kStatusTimeout);
            ok = false;
            return;
        }
    }
}

// First column of owner j's slice when a unit has s items (a multiple of 16).
__device__ __forceinline__ int slice_begin(int j, int s) { return 16 * ((32 * j) / s); }

__device__ __forceinline__ int clamped_count(const TcsParams& p, int b) {
    return max(min(p.a.counts[b], p.a.W), 0);
}

__device__ __forceinline__ int pieces_of(int n) { return (n + kTcMaxKeys - 1) / kTcMaxKeys; }

// The most keys any row of unit u holds, and the first row holding them.
__device__ __forceinline__ int unit_count(const TcsParams& p, int u, int* ref = nullptr) {
    const int b0 = (u / p.HG) * p.G;
    int n = -1, r0 = 0;
    for (int r = 0; r < p.G; ++r) {
        const int c = clamped_count(p, b0 + r);
        if (c > n) {
            n = c;
            r0 = r;
        }
    }
    if (ref != nullptr) *ref = r0;
    return n;
}

// Keys lane h of the item reads: those of its own row (padding lanes: none).
__device__ __forceinline__ int lane_count(const TcsParams& p, int b0, int h) {
    return h < p.lanes ? clamped_count(p, b0 + h / p.a.H) : 0;
}

// The shared-memory addresses and barriers of the chunk pipeline.
__device__ __forceinline__ tcc::Pipe pipe_of(const TcsParams& p, uint32_t base, uint32_t bars,
                                             const uint8_t* smem) {
    tcc::Pipe pp;
    pp.q = base + kOffQP;
    pp.q_lo = p.lamh != nullptr ? base + kOffRing + kTile : 0u;
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

// ---- setup: the item layout ----------------------------------------------------------
// pre[u] = first item of unit u (exclusive prefix sum of the units' item
// counts), pre[units] = all items. Two units per thread (units <= 1024).
__device__ __forceinline__ void scan_units(const TcsParams& p, uint8_t* smem) {
    int32_t* pre = reinterpret_cast<int32_t*>(smem + kOffPrefix);
    int32_t* wsum = reinterpret_cast<int32_t*>(smem + kOffWarpSum);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int u0 = 2 * t, u1 = 2 * t + 1;
    const int s0 = u0 < p.units ? pieces_of(unit_count(p, u0)) : 0;
    const int s1 = u1 < p.units ? pieces_of(unit_count(p, u1)) : 0;
    const int v = s0 + s1;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kTcThreads / 32 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kTcThreads / 32) wsum[lane] = w;
    }
    __syncthreads();
    const int excl = x - v + (warp > 0 ? wsum[warp - 1] : 0);
    if (u0 < p.units) pre[u0] = excl;
    if (u1 < p.units) pre[u1] = excl + s0;
    if (t == 0) pre[p.units] = wsum[kTcThreads / 32 - 1];
    __syncthreads();
}

// Item i (< all items): its unit (binary search over pre) and keys.
__device__ __forceinline__ Item item_of(const TcsParams& p, const uint8_t* smem, int i) {
    const int32_t* pre = reinterpret_cast<const int32_t*>(smem + kOffPrefix);
    int lo = 0, hi = p.units - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= i)
            lo = mid;
        else
            hi = mid - 1;
    }
    Item it;
    it.b0 = (lo / p.HG) * p.G;
    it.g = lo % p.HG;
    it.row0 = static_cast<int64_t>(it.b0) * p.a.H + it.g * kTcHeads;
    it.item0 = pre[lo];
    it.s = pre[lo + 1] - pre[lo];
    it.j = i - it.item0;
    const int n = unit_count(p, lo, &it.ref);
    it.n = n;
    it.first = min(n, it.j * kTcLeaf);
    it.mine = min(n - it.first, kTcLeaf);
    it.nch = (it.mine + kTcChunk - 1) / kTcChunk;
    return it;
}

// Units without keys assigned to this CTA (unit u on CTA u % grid): zero
// output and LSE -inf. Run by `nthreads` threads starting at thread t0.
__device__ __forceinline__ void zero_empty_units(const TcsParams& p, const uint8_t* smem, int t0,
                                                 int nthreads) {
    const int32_t* pre = reinterpret_cast<const int32_t*>(smem + kOffPrefix);
    const int t = threadIdx.x - t0;
    for (int u = blockIdx.x; u < p.units; u += p.grid) {
        if (pre[u + 1] != pre[u]) continue;
        const int64_t row0 = static_cast<int64_t>((u / p.HG) * p.G) * p.a.H + (u % p.HG) * kTcHeads;
        uint4* dst = reinterpret_cast<uint4*>(p.a.out + row0 * kLatent);
        for (int e = t; e < p.lanes * (kLatent / 8); e += nthreads) dst[e] = make_uint4(0u, 0u, 0u, 0u);
        for (int h = t; h < p.lanes; h += nthreads) p.a.lse[row0 + h] = -INFINITY;
    }
}

// (Re)initialises the pipeline barriers (thread 0). Before the second and
// later items every barrier is idle: all copies have landed and every MMA
// has completed (O is complete).
__device__ __forceinline__ void init_bars(uint32_t bars, bool again) {
    if (again)
        for (int i = 0; i < kNumBars; ++i)
            asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bars + 8 * i) : "memory");
    mbar_init(bars + 8 * kBarQ, 1);
    for (int i = 0; i < 2; ++i) {
        mbar_init(bars + 8 * (kBarFull + i), 1);
        mbar_init(bars + 8 * (kBarEmpty + i), 1);
        mbar_init(bars + 8 * (kBarFreeB + i), 1);
    }
    for (int c = 0; c < 4; ++c) mbar_init(bars + 8 * (kBarS + c), 1);
    mbar_init(bars + 8 * kBarP, kTcThreads);
    mbar_init(bars + 8 * kBarO, 1);
    mbar_init(bars + 8 * kBarLand, 1);
    fence_mbar_init();
}

// ---- warps 0-7: this item's key indices, then pass A's gathers -------------------
// Entries past its keys name pool row 0 (a real row: finite bytes; its P is 0).
// This item's key indices, two per producer thread (entries past its keys: 0).
__device__ __forceinline__ void load_idx(const TcsParams& p, const Item& it, int32_t (&v)[2]) {
    const int32_t* row_idx = p.a.indices + static_cast<int64_t>(it.b0 + it.ref) * p.a.W + it.first;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int i = threadIdx.x + u * kProducerThreads;
        v[u] = (i < it.mine) ? row_idx[i] : 0;
    }
}

// The row-group contract on this piece's keys: every other row of the unit
// agrees with the staged list on its own first count entries; a mismatch
// writes SMD_ERR_GROUP to the status (producer threads).
__device__ __forceinline__ void check_contract(const TcsParams& p, const int32_t* idx_s,
                                               const Item& it) {
    const int t = threadIdx.x;
    bool bad = false;
    for (int r = 0; r < p.G; ++r) {
        if (r == it.ref) continue;
        const int lim = min(it.mine, clamped_count(p, it.b0 + r) - it.first);
        const int32_t* row_idx = p.a.indices + static_cast<int64_t>(it.b0 + r) * p.a.W + it.first;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = t + u * kProducerThreads;
            if (i < lim && row_idx[i] != idx_s[i]) bad = true;
        }
    }
    if (bad && p.a.status != nullptr) atomicCAS(p.a.status, 0, SMD_ERR_GROUP);
}

// `pre` holds this item's indices when `have` (loaded early for the first item).
__device__ __forceinline__ void producer_a(const TcsMaps& maps, const TcsParams& p,
                                           const tcc::Pipe& pp, uint8_t* smem, const Item& it,
                                           const int32_t (&pre)[2], bool have, bool& ok) {
    const int t = threadIdx.x;
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + kOffIdx);
    int32_t v[2] = {pre[0], pre[1]};
    if (!have) load_idx(p, it, v);
    idx_s[t] = v[0];
    idx_s[t + kProducerThreads] = v[1];
    asm volatile("bar.sync 1, %0;" ::"r"(kProducerThreads) : "memory");
    if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(it.item0 + it.j, p.grid), 1);
    uint32_t seen[2] = {0u, 0u};
    if (p.G == 1) {
        tcc::gather_pass_a(maps.kv, maps.kv_tail, pp, 0, it.nch, seen, ok);
        return;
    }
    // Row groups: the contract is checked once the first chunks' gathers are
    // in flight (it changes nothing but the status).
    const int head = min(it.nch, pp.q_lo ? 1 : 2);
    tcc::gather_pass_a(maps.kv, maps.kv_tail, pp, 0, head, seen, ok);
    check_contract(p, idx_s, it);
    tcc::gather_pass_a(maps.kv, maps.kv_tail, pp, head, it.nch, seen, ok);
}

// ---- warps 12-15: the row maximum (thread h = head h = TMEM lane h) ---------------
// This item's maximum as the QK chunks complete; for a unit of several items
// it is published (global memory + the item's flag) and the maximum over the
// unit's items is taken once every flag is up.
__device__ __forceinline__ void row_max(const TcsParams& p, uint8_t* smem, uint32_t bars,
                                        uint32_t tmem, const Item& it, int item, bool& ok) {
    const int h = threadIdx.x & 127;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * ((threadIdx.x >> 5) & 3)) << 16);
    const float lam = lam_of(p, it.row0, h);
    const int lim_row = lane_count(p, it.b0, h) - it.first;  // this lane's keys in the piece
    float m = -INFINITY;
    for (int c = 0; c < it.nch; ++c) {
        mbar_wait(bars + 8 * (kBarS + c), 0, ok, p.a.status, p.budget_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const int cnt = min(kTcChunk, it.mine - kTcChunk * c);
        for (int q = 0; 32 * q < cnt; ++q) {  // warp-uniform; lanes mask their own keys
            float v[32];
            tmem_ld32(lane_base + kTcChunk * c + 32 * q, v);
            const int lim = min(cnt, lim_row - kTcChunk * c) - 32 * q;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < lim) m = fmaxf(m, lam * v[j]);
        }
    }
    float* rowmax = reinterpret_cast<float*>(smem + kOffRowMax);
    if (h == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 2);
    if (it.s == 1) {
        rowmax[h] = m;
        if (h == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 3);
        return;
    }
    // Head h's maximum as one 64-bit word: the tag and the value's bits, so a
    // reader that sees the tag sees the value (one single-copy-atomic store,
    // no fence, no separate flag); published even after a failure. Then
    // every other item's word for head h, taken as its tag appears (bounded).
    uint64_t* ws_max = reinterpret_cast<uint64_t*>(p.ws_base + p.ws.max);
    const uint32_t tag = max_tag(p.token);
    st_relaxed_u64(ws_max + static_cast<int64_t>(item) * kTcHeads + h,
                   (static_cast<uint64_t>(tag) << 32) | __float_as_uint(m));
    float mr = m;
    uint32_t pending = (it.s >= 32 ? 0xffffffffu : ((1u << it.s) - 1u)) & ~(1u << it.j);
    const uint64_t t0 = globaltimer();
    while (pending != 0u && ok) {
        for (uint32_t rest = pending; rest != 0u; rest &= rest - 1u) {
            const int jj = __ffs(rest) - 1;
            const uint64_t w = ld_relaxed_u64(ws_max + static_cast<int64_t>(it.item0 + jj) * kTcHeads + h);
            if (static_cast<uint32_t>(w >> 32) == tag) {
                mr = fmaxf(mr, __uint_as_float(static_cast<uint32_t>(w)));
                pending &= ~(1u << jj);
            }
        }
        if (pending != 0u && globaltimer() - t0 > p.budget_ns) {
            if (p.a.status != nullptr) atomicCAS(p.a.status, 0, kStatusTimeout);
            ok = false;
        }
    }
    rowmax[h] = mr;
    if (h == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 3);
}

// ---- all 16 warps: P ---------------------------------------------------------------
// Warp w: TMEM lane quarter w % 4 (thread = head h), keys 32j .. 32j + 31 of
// every chunk, j = w / 4; P = 2^(s - m + log2 448) in E4M3 into the K-major
// 128-byte-swizzled A operand, and the FP32 sum of the unquantized P of those
// keys (chunks ascending) into lsum[j][h].
__device__ __forceinline__ void p_phase(const TcsParams& p, uint8_t* smem, uint32_t bars,
                                        uint32_t tmem, const Item& it, bool ok) {
    const int warp = threadIdx.x >> 5;
    const int h = 32 * (warp & 3) + (threadIdx.x & 31);
    const int j = warp >> 2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const float lam = lam_of(p, it.row0, h);
    const float bias = reinterpret_cast<const float*>(smem + kOffRowMax)[h] - p.log2_448;
    const int lim_row = lane_count(p, it.b0, h) - it.first;  // this lane's keys in the piece
    float l = 0.f;
    for (int c = 0; c < it.nch && ok; ++c) {
        const int cnt = min(kTcChunk, it.mine - kTcChunk * c);
        if (32 * j >= cnt) continue;  // warp-uniform
        const int lim = min(cnt, lim_row - kTcChunk * c) - 32 * j;  // per lane
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

// BF16(v * inv) of 16 columns of head h at column `col` of the staging tile
// (rows of row_bytes; 16-byte chunk c of row h at chunk c ^ (h & mask)).
__device__ __forceinline__ void stage16(uint8_t* stage, int row_bytes, int mask, int h, int col,
                                        const float (&v)[16], float inv) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = bf16x2(v[2 * i] * inv, v[2 * i + 1] * inv);
    uint8_t* row = stage + h * row_bytes;
    const int c0 = col >> 3;
    *reinterpret_cast<uint4*>(row + ((c0 ^ (h & mask)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (h & mask)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// The first `rows` heads of the staging tile to out (rows kLatent BF16 apart),
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

// XOR mask of the staging swizzle for rows of `chunks` 16-byte chunks: the
// largest power of two (at most 8) that divides chunks, minus one.
__device__ __forceinline__ int stage_mask(int chunks) { return min(chunks & -chunks, 8) - 1; }

// One owner's 16 columns at `col` of a unit: the pairwise tree over positions
// k = 0 .. P - 1 (piece j ^ k; P = the unit's pieces rounded up to a power of
// two), pieces src >= np absent (np: the pieces holding keys of lane h's own
// row; all of the unit's pieces unless row groups), 4 columns at a time; L:
// the partials' row stride (part_stride).
template <bool kNarrow>
__device__ __forceinline__ void merge_cols(const float* part, int64_t item0, int j, int P, int np,
                                           int L, int h, int col, const float (&own)[16],
                                           float (&out)[16]) {
    constexpr int64_t kPartFloats = static_cast<int64_t>(kTcHeads) * kLatent;
#pragma unroll
    for (int c0 = 0; c0 < 16; c0 += 4) {
        const float4 r = tree_xor_n<float4>(P, [&](int k) {
            if (k == 0) return make_float4(own[c0], own[c0 + 1], own[c0 + 2], own[c0 + 3]);
            return ld_cg_v4(part + (item0 + (j ^ k)) * kPartFloats +
                            (((col + c0) >> 2) * (kNarrow ? L : kTcHeads) + h) * 4);
        }, j, np);
        out[c0] = r.x;
        out[c0 + 1] = r.y;
        out[c0 + 2] = r.z;
        out[c0 + 3] = r.w;
    }
}

// Groups of cp.async copies (16-byte global -> shared, through the load/store
// unit): close the group this thread has issued since the last commit; wait
// until at most N of its groups are still in flight.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 4 consecutive TMEM columns of this thread's lane (warp-wide).
__device__ __forceinline__ float4 tmem_ld4(uint32_t taddr) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    return make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]),
                       __uint_as_float(r[3]));
}

// ---- all 16 warps: exchange, merge, output ---------------------------------------
// Warp w serves TMEM lane quarter w % 4 (thread = head h) and column group
// cg = w / 4.
// kNarrow: units of at most 64 lanes (row groups, H <= 64), whose partials
// take the lanes as their row stride and whose merge lands every peer's slice
// at once; wider units keep the stride of 128 (the launch picks the kernel
// by the units' lanes).
template <bool kNarrow>
__device__ __forceinline__ void finish(const TcsParams& p, uint8_t* smem, uint32_t tmem,
                                       const Item& it, int item, bool& ok) {
    const int warp = threadIdx.x >> 5;
    const int h = 32 * (warp & 3) + (threadIdx.x & 31);
    const int cg = warp >> 2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const float* lsum = reinterpret_cast<const float*>(smem + kOffLsum);
    const float l = ((lsum[h] + lsum[128 + h]) + lsum[256 + h]) + lsum[384 + h];
    const float m = reinterpret_cast<const float*>(smem + kOffRowMax)[h];
    const bool have_o = ok && it.mine > 0;  // O in TMEM is defined only if PV ran
    const int64_t row0 = it.row0;
    uint16_t* oblock = p.a.out + row0 * kLatent;
    float* lse = p.a.lse + row0 + h;
    uint8_t* stage = smem + kOffRing;  // the ring is dead once O is complete

    if (it.s == 1) {
        if (ok) {  // uniform: set by the barrier before the finish
            const float total = l;
            const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
            for (int q = 0; q < 8; ++q) {
                const int col = cg * 128 + 16 * q;
                float v[16];
                if (have_o) {
                    tmem_ld16(lane_base + col, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                }
                stage16(stage, kLatent * 2, 7, h, col, v, inv);
            }
            if (cg == 0 && h < p.lanes)
                *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f
                                   : -INFINITY;
            __syncthreads();
            flush(stage, kLatent * 2, 7, p.lanes, oblock);
        }
        return;
    }

    const int s = it.s, j = it.j;
    const int c0 = slice_begin(j, s), c1 = slice_begin(j + 1, s), CW = c1 - c0;
    constexpr int64_t kPartFloats = static_cast<int64_t>(kTcHeads) * kLatent;
    float* part = reinterpret_cast<float*>(p.ws_base + p.ws.part);
    float* sums = reinterpret_cast<float*>(p.ws_base + p.ws.sum);
    uint64_t* fpart = reinterpret_cast<uint64_t*>(p.ws_base + p.ws.flag_part);
    uint64_t* ws_max = reinterpret_cast<uint64_t*>(p.ws_base + p.ws.max);

    // 1. This item's partials of the other owners' columns (16-byte unit u of
    // lane h at (u * stride + h), stride = the lanes (narrow units) or 128:
    // one warp-wide store covers 512 contiguous bytes, and an owner's slice
    // from one piece is contiguous), and its sums; then one flag per owner.
    // (Every SM exchanges at once here, so the phase is bound by L2
    // bandwidth; all 16 warps write.)
    const int stride = kNarrow ? p.lanes : kTcHeads;
    float* mine_part = part + static_cast<int64_t>(item) * kPartFloats;
    for (int q = 0; q < 8; ++q) {
        const int col = 128 * cg + 16 * q;
        if (col >= c0 && col < c1) continue;  // warp-uniform: the own slice
        float v[16];
        if (have_o) {
            tmem_ld16(lane_base + col, v);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
        if (h >= p.lanes) continue;  // padding lanes are never merged
        float* dst = mine_part + ((col >> 2) * stride + h) * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            st_v4(dst + i * stride * 4, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
    }
    if (cg == 0) sums[static_cast<int64_t>(item) * kTcHeads + h] = l;
    __syncthreads();
    const int t = threadIdx.x;
    if (t < s && t != j) {
        __threadfence();  // after the barrier: orders every thread's stores above
        st_release_u64(fpart + static_cast<int64_t>(item) * kTcsMaxPieces + t, p.token);
    }
    if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 6);

    // 2. The other items' partials of this slice (each flag is read here only,
    // so it is zeroed once seen).
    if (t < s && t != j) {
        uint64_t* f = fpart + static_cast<int64_t>(it.item0 + t) * kTcsMaxPieces + j;
        wait_flag(f, p.token, ok, p.a.status, p.budget_ns);
        *f = 0ull;
    }
    ok = __syncthreads_and(ok) != 0;
    if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 7);
    // Every item of the unit has read the maxima (it raised its flags for the
    // owners after that): this item's maxima are consumed.
    if (t < kTcHeads) ws_max[static_cast<int64_t>(item) * kTcHeads + t] = 0ull;
    if (!ok) return;

    // 3. Merge: the pairwise tree over the unit's pieces in the order j ^ k.
    const int n_lane = lane_count(p, it.b0, h);
    const int P = pow2_ceil(s);
    const int np = min(s, (n_lane + kTcLeaf - 1) / kTcLeaf);  // pieces holding keys of h's row
    const float total = tree_xor_n<float>(P, [&](int k) {
        return k == 0 ? l : ld_cg_f32(sums + static_cast<int64_t>(it.item0 + (j ^ k)) * kTcHeads + h);
    }, j, np);
    const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
    if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 9);
    if (s <= 4) {
        // Up to four pieces: each thread's 16-column pieces, the peers' values
        // loaded into registers (at most three loads per four columns), the
        // BF16 tile staged in the dead ring and stored by whole rows.
        const int mask = stage_mask(CW / 8);
        for (int q = cg; 16 * q < CW; q += 4) {
            const int col = c0 + 16 * q;
            float own[16], acc[16];
            if (have_o) {
                tmem_ld16(lane_base + col, own);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) own[i] = 0.f;
            }
            if (h < p.lanes) {
                merge_cols<kNarrow>(part, it.item0, j, P, np, stride, h, col, own, acc);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.f;  // padding lanes are never stored
            }
            stage16(stage, CW * 2, mask, h, col - c0, acc, inv);
        }
        if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 10);
        if (j == 0 && cg == 0 && h < p.lanes)
            *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f : -INFINITY;
        __syncthreads();
        if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 11);
        flush(stage, CW * 2, mask, p.lanes, oblock + c0);
        return;
    }
    // More pieces (narrow slices, many loads per column): the peers' slices
    // come into shared memory first, into the dead query, P tiles and ring,
    // and the tree reads them from there. Where every peer's slice fits at
    // once (units of at most 64 lanes), each comes by one bulk copy (it is
    // contiguous in the workspace); otherwise in batches of BC columns over
    // two buffers by cp.async (which holds no register while in flight), a
    // whole batch in flight at once. The BF16 tile is staged behind the
    // buffers and stored by whole rows (out may be mapped host memory).
    constexpr int kStageMax = kTcHeads * 112 * 2;  // the widest slice of 5 or more pieces
    constexpr int kLandBytes = (3 * kTile - kStageMax) / 2 / 16 * 16;  // one of the two buffers
    uint8_t* tile = smem + 2 * kLandBytes;
    const int mask = stage_mask(CW / 8);
    const int peers = s - 1;
    // Only the lanes of real query rows are copied (the peers never write the
    // padding lanes' partials, so those lines are not in L2) and landed, so
    // a batch holds 128 / lanes times the columns of a full tile. The
    // batches are of equal width (a multiple of 4 columns).
    const int lanes = p.lanes;
    const int bc_max = (kLandBytes / (peers * lanes * 16)) * 4;  // columns a buffer holds
    const int nbatch = (CW + bc_max - 1) / bc_max;
    const int BC = (CW + 4 * nbatch - 1) / (4 * nbatch) * 4;
    const uint32_t land0 = smem_addr(smem);
    // Thread t copies lane hh of the (peer slot, 4-column group) pairs
    // q = q0, q0 + R, ...: lanes rounded up to a power of two threads per
    // pair, R pairs at once (the pair is stepped, not divided out per copy).
    int lanes_p2 = 16;
    while (lanes_p2 < lanes) lanes_p2 <<= 1;
    const int R = kTcThreads / lanes_p2, hh = t & (lanes_p2 - 1), q0 = t / lanes_p2;
    auto issue = [&](int bt) {
        const int cb = bt * BC, g4 = min(BC, CW - cb) / 4;  // 4-column units of the batch
        const uint32_t dst0 = land0 + (bt & 1) * kLandBytes;
        if (hh < lanes) {
            int slot = q0 / g4, g = q0 - slot * g4;
            for (int q = q0; q < peers * g4; q += R) {
                const int src = slot < j ? slot : slot + 1;
                const float* from = part + (it.item0 + src) * kPartFloats +
                                    ((((c0 + cb) >> 2) + g) * stride + hh) * 4;
                cp_async16(dst0 + (q * lanes + hh) * 16, from);
                for (g += R; g >= g4; g -= g4) ++slot;
            }
        }
        cp_async_commit();
    };
    const int units = CW / 4;  // 4-column groups of the slice
    const uint32_t slice_bytes = static_cast<uint32_t>(units * lanes * 16);
    if (kNarrow && static_cast<int64_t>(peers) * slice_bytes <= 2 * static_cast<int64_t>(kLandBytes)) {
        const uint32_t bar = smem_addr(smem) + kOffBars + 8 * kBarLand;
        if (t < 32) {
            fence_proxy_async_global();  // the peers' partials (acquired above) -> the copy engine
            if (t == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(peers) * slice_bytes);
            __syncwarp();
            for (int slot = t; slot < peers; slot += 32) {
                const int src = slot < j ? slot : slot + 1;
                bulk_g2s(land0 + slot * slice_bytes,
                         part + (it.item0 + src) * kPartFloats + (c0 >> 2) * lanes * 4, slice_bytes, bar);
            }
        }
        bool landed = true;
        mbar_wait(bar, 0, landed, p.a.status, p.budget_ns);
        landed = __all_sync(0xffffffffu, landed);  // the TMEM loads below are warp-wide
        const float4* land = reinterpret_cast<const float4*>(smem);
        for (int g = cg; g < units && landed; g += 4) {  // warp-uniform
            const int col = c0 + 4 * g;
            const float4 own = have_o ? tmem_ld4(lane_base + col) : make_float4(0.f, 0.f, 0.f, 0.f);
            if (h >= p.lanes) continue;  // padding lanes are never stored
            const float4 acc = tree_xor_n<float4>(P, [&](int k) {
                if (k == 0) return own;
                const int src = j ^ k;
                return land[((src < j ? src : src - 1) * units + g) * lanes + h];
            }, j, np);
            const int cs = col - c0;
            *reinterpret_cast<uint2*>(tile + h * (CW * 2) + ((((cs >> 3) ^ (h & mask))) << 4) +
                                      ((cs >> 2) & 1) * 8) =
                make_uint2(bf16x2(acc.x * inv, acc.y * inv), bf16x2(acc.z * inv, acc.w * inv));
        }
        __syncthreads();  // the tile is staged
        if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 10);
        if (j == 0 && cg == 0 && h < p.lanes)
            *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f : -INFINITY;
        if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 11);
        flush(tile, CW * 2, mask, p.lanes, oblock + c0);
        return;
    }
    issue(0);
    if (nbatch > 1) issue(1);
    for (int bt = 0; bt < nbatch; ++bt) {
        if (bt + 1 < nbatch)
            cp_async_wait_group<1>();
        else
            cp_async_wait_group<0>();
        __syncthreads();  // batch bt has landed for every thread
        const int cb = bt * BC, g4 = min(BC, CW - cb) / 4;
        const float4* land = reinterpret_cast<const float4*>(smem + (bt & 1) * kLandBytes);
        for (int g = cg; g < g4; g += 4) {  // warp-uniform
            const int col = c0 + cb + 4 * g;
            const float4 own = have_o ? tmem_ld4(lane_base + col) : make_float4(0.f, 0.f, 0.f, 0.f);
            if (h >= p.lanes) continue;  // padding lanes are never stored
            const float4 acc = tree_xor_n<float4>(P, [&](int k) {
                if (k == 0) return own;
                const int src = j ^ k;
                return land[((src < j ? src : src - 1) * g4 + g) * lanes + h];
            }, j, np);
            const int cs = col - c0;  // column in the slice: half (cs >> 2) & 1 of chunk cs >> 3
            *reinterpret_cast<uint2*>(tile + h * (CW * 2) + ((((cs >> 3) ^ (h & mask))) << 4) +
                                      ((cs >> 2) & 1) * 8) =
                make_uint2(bf16x2(acc.x * inv, acc.y * inv), bf16x2(acc.z * inv, acc.w * inv));
        }
        __syncthreads();  // buffer bt & 1 is free (after the last batch: the tile is staged)
        if (bt + 2 < nbatch) issue(bt + 2);
    }
    if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 10);
    if (j == 0 && cg == 0 && h < p.lanes)
        *lse = total > 0.f ? (m - p.log2_448 + log2f(total)) * 0.69314718055994530942f : -INFINITY;
    if (t == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 11);
    flush(tile, CW * 2, mask, p.lanes, oblock + c0);
}

template <bool kNarrow>
__global__ void __launch_bounds__(kTcThreads, 1)
    tcs_decode_kernel(const __grid_constant__ TcsMaps maps, const TcsParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_addr(smem);
    const uint32_t bars = base + kOffBars;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    bool ok = true;

    scan_units(p, smem);
    const int total = reinterpret_cast<const int32_t*>(smem + kOffPrefix)[p.units];
    // The first item's indices are loaded now: their round trip overlaps the setup.
    int32_t idx0[2] = {0, 0};
    if (warp < 8 && static_cast<int>(blockIdx.x) < total)
        load_idx(p, item_of(p, smem, blockIdx.x), idx0);
    if (threadIdx.x == 0) init_bars(bars, false);
    if (warp == 8) tmem_alloc(base + kOffTmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmem);
    const tcc::Pipe pp = pipe_of(p, base, bars, smem);
    // Warps 9-11 have nothing to do until P: the empty units go now.
    if (warp >= 9 && warp < 12) zero_empty_units(p, smem, 9 * 32, 3 * 32);

    for (int r = 0;; ++r) {
        const int item = blockIdx.x + r * p.grid;
        if (item >= total) break;  // uniform
        const Item it = item_of(p, smem, item);
        if (r > 0) {
            if (threadIdx.x == 0) init_bars(bars, true);
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 0);
            SMD_TRACE_SM(g_trace_tcs, trace_row(item, p.grid));
        }
        if (threadIdx.x == 0) {
            // (inject_stall: the query barrier also expects 16 bytes nobody
            // sends, so its bounded wait runs out; a test hook.)
            const bool split = p.lamh != nullptr;
            mbar_arrive_expect_tx(bars + 8 * kBarQ, (split ? 2 : 1) * kTile + (p.inject_stall ? 16 : 0));
            const int y = static_cast<int>(it.row0);
            for (int c = 0; c < 4; ++c)
                tma_load_2d(base + kOffQP + c * kBlock, &maps.q, 128 * c, y, bars + 8 * kBarQ);
            tma_load_2d(base + kOffQP + 4 * kBlock, &maps.q_tail, 512, y, bars + 8 * kBarQ);
            if (split) {  // the lo rows into ring slot 1, free until QK is done
                const uint32_t lo = base + kOffRing + kTile;
                for (int c = 0; c < 4; ++c)
                    tma_load_2d(lo + c * kBlock, &maps.q_lo, 128 * c, y, bars + 8 * kBarQ);
                tma_load_2d(lo + 4 * kBlock, &maps.q_lo_tail, 512, y, bars + 8 * kBarQ);
            }
        }
        uint32_t full_seen[2] = {0u, 0u};
        if (warp < 8) {
            producer_a(maps, p, pp, smem, it, idx0, r == 0, ok);
        } else if (warp == 8) {
            if (lane == 0) tcc::mma_qk(pp, tmem, it.nch, full_seen, ok);
            __syncwarp();
        } else if (warp >= 12) {
            row_max(p, smem, bars, tmem, it, item, ok);
        }
        ok = __syncthreads_and(ok) != 0;  // every QK is complete; the row maxima are here
        tc_fence_after();
        p_phase(p, smem, bars, tmem, it, ok);
        if (threadIdx.x == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 4);
        if (warp < 8) {
            tcc::gather_pass_b(maps.kv, pp, it.nch, ok);
        } else if (warp == 8) {
            if (lane == 0) tcc::mma_pv(pp, tmem, it.nch, it.mine, full_seen, ok);
            __syncwarp();
        }
        mbar_wait(bars + 8 * kBarO, 0, ok, p.a.status, p.budget_ns);
        tc_fence_after();
        ok = __syncthreads_and(ok) != 0;  // the partial sums of P are visible; one verdict
        if (threadIdx.x == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 5);
        finish<kNarrow>(p, smem, tmem, it, item, ok);
        tc_fence_before();  // every TMEM read of this item precedes the next item's MMAs
        __syncthreads();
        if (threadIdx.x == 0) SMD_STAMP(g_trace_tcs, trace_row(item, p.grid), 8);
    }
    if (warp == 8) {
        tc_fence_after();
        tmem_free(tmem, 512);
    }
}

// The split query into the workspace (smd_qsplit.cuh): one warp per query row.
__global__ void __launch_bounds__(256) tcs_qsplit_kernel(const uint16_t* q16, int64_t rows,
                                                         float lam0, uint8_t* q_hi, uint8_t* q_lo,
                                                         float* lamh) {
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;  // warp-uniform
    const float lam = split_query_row(q16 + r * kRow, q_hi + r * kRow, q_lo + r * kRow, lam0);
    if ((threadIdx.x & 31) == 0) lamh[r] = lam;
}

}  // namespace

// ---- host ------------------------------------------------------------------------

SMD_TRACE_COPY_FN(tcs_trace_copy, g_trace_tcs)

int tcs_smem_bytes() { return kSmemBytes; }

namespace {

constexpr int kMaxDevices = 64;

// A flag token for each call: a counter run through a 64-bit mixer (splitmix64)
// from a per-process seed, so that words left by another process or an
// earlier call that stopped early do not match; never 0.
uint64_t next_token() {
    static std::atomic<uint64_t> counter{0};
    static const uint64_t seed = [] {
        uint64_t x = reinterpret_cast<uintptr_t>(&counter);
        x ^= static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count());
        return x;
    }();
    uint64_t z = seed + 0x9E3779B97F4A7C15ull * (counter.fetch_add(1) + 1);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z == 0 ? 1 : z;
}

}  // namespace

int tcs_max_grid() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int v = cached[dev].load();
    if (v > 0) return v;
    if (cudaFuncSetAttribute(tcs_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(tcs_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    int per_sm = 0, sms = 0, per_sm_narrow = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tcs_decode_kernel<false>, kTcThreads,
                                                      kSmemBytes) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_narrow, tcs_decode_kernel<true>,
                                                      kTcThreads, kSmemBytes) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    v = std::min(per_sm, per_sm_narrow) * sms;
    cached[dev].store(v);
    return v;
}

int launch_tcs(const CallArgs& a, const TcsConfig& cfg, cudaStream_t stream) {
    TcsMaps maps{};
    const uint64_t qrows = static_cast<uint64_t>(a.B) * static_cast<uint64_t>(a.H);
    const TcsWorkspace ws = tcs_workspace(cfg.items_cap, cfg.qsplit ? static_cast<int64_t>(qrows) : 0);
    uint8_t* base = static_cast<uint8_t*>(cfg.ws);
    const uint8_t* q = a.q;
    if (cfg.qsplit) {
        // The bf16 rows split into E4M3 hi and lo rows and their logit scales, in the workspace.
        if (a.q16 == nullptr) return SMD_ERR_NULL;
        const unsigned blocks = static_cast<unsigned>((qrows + 7) / 8);
        tcs_qsplit_kernel<<<blocks, 256, 0, stream>>>(a.q16, static_cast<int64_t>(qrows),
                                                      a.scale_log2, base + ws.q_hi, base + ws.q_lo,
                                                      reinterpret_cast<float*>(base + ws.lamh));
        if (cudaGetLastError() != cudaSuccess) return SMD_ERR_LAUNCH;
        q = base + ws.q_hi;
        if (!encode_row_map(&maps.q_lo, base + ws.q_lo, qrows, 128, kTcHeads) ||
            !encode_row_map(&maps.q_lo_tail, base + ws.q_lo, qrows, 64, kTcHeads))
            return SMD_ERR_LAUNCH;
    }
    if (!encode_row_map(&maps.q, q, qrows, 128, kTcHeads) ||
        !encode_row_map(&maps.q_tail, q, qrows, 64, kTcHeads) ||
        !encode_row_map(&maps.kv, a.kv, static_cast<uint64_t>(a.N), 128, 1) ||
        !encode_row_map(&maps.kv_tail, a.kv, static_cast<uint64_t>(a.N), 64, 1))
        return SMD_ERR_LAUNCH;
    const int max_grid = tcs_max_grid();
    if (max_grid <= 0 || cfg.grid > max_grid) return SMD_ERR_LAUNCH;
    TcsParams prm{};
    prm.a = a;
    prm.G = cfg.G > 1 ? cfg.G : 1;
    prm.HG = prm.G > 1 ? 1 : (a.H + kTcHeads - 1) / kTcHeads;
    prm.lanes = prm.G > 1 ? prm.G * a.H : (a.H < kTcHeads ? a.H : kTcHeads);
    prm.units = a.B / prm.G * prm.HG;
    prm.grid = cfg.grid;
    prm.log2_448 = static_cast<float>(std::log2(448.0));
    prm.budget_ns = cfg.wait_budget_ns;
    prm.inject_stall = cfg.inject_stall;
    prm.token = next_token();
    prm.ws = ws;
    prm.ws_base = base;
    prm.lamh = cfg.qsplit ? reinterpret_cast<const float*>(base + ws.lamh) : nullptr;

    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(cfg.grid), 1, 1);
    lc.blockDim = dim3(kTcThreads, 1, 1);
    lc.dynamicSmemBytes = static_cast<size_t>(kSmemBytes);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: peers' waits end
    attr[0].val.cooperative = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const cudaError_t e = prm.lanes <= 64 ? cudaLaunchKernelEx(&lc, tcs_decode_kernel<true>, maps, prm)
                                          : cudaLaunchKernelEx(&lc, tcs_decode_kernel<false>, maps, prm);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return SMD_ERR_LAUNCH;
    }
    return SMD_OK;
}

}  // namespace smd
