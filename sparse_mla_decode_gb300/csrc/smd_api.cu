// C ABI of the sparse MLA decode library: argument checks, the launch plan
// (split / tile / window choice keyed on heads, top-k width and batch) and
// dispatch to the kernels. Host code only.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cuda_runtime.h>

#include "smd.h"
#include "smd_internal.h"
#include "smd_trace.cuh"
#include "smd_ptx.cuh"
#include "smd_tree.cuh"

namespace smd {
namespace {

constexpr int kMaxSmemBytes = 227 * 1024;  // dynamic shared memory per CTA on sm_103

struct DeviceInfo {
    int sm_count = 0;
    int major = 0, minor = 0;
    int smem_optin = 0;
    bool ok = false;
};

DeviceInfo query_device() {
    DeviceInfo d;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return d;
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    d.ok = true;
    return d;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

bool is_split(int s) { return s == 1 || s == 2 || s == 4 || s == 8 || s == 16; }

// Most keys one CTA can hold logits for with `tiles` 16-head tiles, a
// `window`-key buffer and `idx_cap` staged indices, under the shared-memory
// limit.
int key_cap_limit(int tiles, int split, int window, int idx_cap, bool qsplit) {
    // The layout grows by (16*tiles + 1) * 4 bytes per key of capacity.
    const int base = mma_layout(tiles, split, window, 0, idx_cap, qsplit).total;
    const int per_key = (kHeadsPerTile * tiles + 1) * 4;
    int cap = std::max(0, (kMaxSmemBytes - base) / per_key) / kChunk * kChunk;
    while (cap > 0 && mma_layout(tiles, split, window, cap, idx_cap, qsplit).total > kMaxSmemBytes)
        cap -= kChunk;
    return cap;
}

// Fills the MMA kernel's plan. `force` fields that are non-zero override the
// automatic choice. Returns an smd_status.
int plan_mma(int B, int H, int W, int sm_count, const smd_plan_t* force, smd_plan_t* out,
             MmaConfig* cfg, bool qsplit = false) {
    // One 16-head tile per CTA by default: on GB300 the second tile's KV reuse
    // is worth less than the extra cluster exchange and registers it costs.
    int tiles = 1;
    if (force && force->tiles) tiles = force->tiles;
    if (tiles != 1 && tiles != 2) return SMD_ERR_PLAN;
    if (H % (kHeadsPerTile * tiles) != 0) return SMD_ERR_PLAN;
    const int units = B * (H / (kHeadsPerTile * tiles));
    const int window_req = (force && force->window) ? force->window : 128;
    if (window_req % kChunk != 0 || window_req < kChunk || window_req > 2048) return SMD_ERR_PLAN;
    // Rows up to kSpecIdxMaxW wide have their whole index list staged.
    const int spec = (W <= kSpecIdxMaxW) ? W : 0;

    // A CTA takes an aligned block of the row's leaves (smd_tree.cuh); the
    // CTA holding the most holds mma_cta_keys(W, split) keys.
    int split = 0;
    if (force && force->split) {
        split = force->split;
        if (!is_split(split)) return SMD_ERR_PLAN;
    } else {
        // Smallest split whose per-CTA share fits; then wider while the grid is
        // under one wave and every CTA still gets a leaf of the widest row. A
        // wider split shortens each CTA's gather but adds a cluster exchange of
        // FP32 partials, which is slow on this part (tens of GB/s per SM).
        for (int s = 1; s <= 16; s *= 2) {
            const int per = mma_cta_keys(std::max(W, 1), s);
            const int win = std::min(window_req, std::max(kChunk, ceil_div(per, kChunk) * kChunk));
            if (per <= key_cap_limit(tiles, s, win, spec, qsplit)) {
                split = s;
                break;
            }
        }
        if (split == 0) return SMD_ERR_SHAPE;
        while (split < 16 && units * split < sm_count && split * 2 <= mma_leaves(W)) split *= 2;
    }
    const int per = mma_cta_keys(std::max(W, 1), split);
    const int window = std::min(window_req, std::max(kChunk, ceil_div(per, kChunk) * kChunk));
    const int key_cap = std::max(kChunk, ceil_div(per, kChunk) * kChunk);
    const MmaLayout L = mma_layout(tiles, split, window, key_cap, spec, qsplit);
    if (L.total > kMaxSmemBytes) return (force && (force->split || force->window)) ? SMD_ERR_PLAN
                                                                                  : SMD_ERR_SHAPE;
    cfg->tiles = tiles;
    cfg->wait_budget_ns = (force && force->wait_budget_us > 0)
                              ? static_cast<uint64_t>(force->wait_budget_us) * 1000ull
                              : kWaitBudgetNs;
    cfg->inject_stall = (force && force->inject_stall) ? 1 : 0;
    cfg->spec_idx = spec > 0 ? 1 : 0;
    cfg->qsplit = qsplit ? 1 : 0;
    // Some row of at most W keys has more leaves than CTAs: its CTAs keep a
    // subtree stack (the widest rows have min(16, ceil(W / 64)) leaves).
    cfg->tree_tmem = std::min(kMmaMaxLeaves, ceil_div(W, kChunk)) > split ? 1 : 0;
    cfg->split = split;
    cfg->window = window;
    cfg->key_cap = key_cap;
    cfg->layout = L;
    out->kernel = SMD_KERNEL_MMA;
    out->split = split;
    out->tiles = tiles;
    out->window = window;
    out->key_cap = key_cap;
    out->grid_x = H / (kHeadsPerTile * tiles) * split;
    out->grid_y = B;
    out->cluster_x = split;
    out->threads = kMmaThreads;
    out->smem_bytes = L.total;
    return SMD_OK;
}

// The tcgen05 kernel takes 128 heads per CTA, or all H < 128 heads of a row
// (the remaining TMEM lanes are padding that is computed and not stored).
bool tc_fits(int H, int W) {
    return (H % kTcHeads == 0 || H < kTcHeads) && W >= 1 && W <= kTcMaxSplit * kTcMaxKeys;
}

// The tcgen05 kernel's plan: the smallest cluster whose CTAs hold at most
// kTcMaxKeys keys each (all of them resident in TMEM as logits).
int plan_tc(int B, int H, int W, const smd_plan_t* force, smd_plan_t* out, TcConfig* cfg) {
    if (!tc_fits(H, W)) return SMD_ERR_PLAN;
    const int lanes = std::min(H, kTcHeads);
    if (force && ((force->tiles && force->tiles != lanes / kHeadsPerTile) ||
                  (force->window && force->window != kTcChunk)))
        return SMD_ERR_PLAN;
    int split = 1;
    while (ceil_div(W, split) > kTcMaxKeys) split *= 2;
    if (force && force->split) {
        if (force->split != 1 && force->split != 2 && force->split != 4) return SMD_ERR_PLAN;
        if (ceil_div(W, force->split) > kTcMaxKeys) return SMD_ERR_PLAN;
        split = force->split;
    }
    cfg->split = split;
    cfg->wait_budget_ns = (force && force->wait_budget_us > 0)
                              ? static_cast<uint64_t>(force->wait_budget_us) * 1000ull
                              : kWaitBudgetNs;
    cfg->inject_stall = (force && force->inject_stall) ? 1 : 0;
    out->kernel = SMD_KERNEL_TC;
    out->split = split;
    out->tiles = lanes / kHeadsPerTile;
    out->window = kTcChunk;
    out->key_cap = kTcMaxKeys;
    out->grid_x = ceil_div(H, kTcHeads) * split;
    out->grid_y = B;
    out->cluster_x = split;
    out->threads = kTcThreads;
    out->smem_bytes = tc_smem_bytes();
    return SMD_OK;
}

// The row-group kernel's plan: the smallest cluster whose CTAs stage at most
// kGroupMaxKeys indices each, then wider while the grid is under one wave and
// every CTA keeps >= 64 keys; a ring of two 64-key slots unless forced.
bool tcg_fits(int H, int W, int G) {
    const int lanes = G * H;
    return (lanes == 32 || lanes == 64) && W >= 1 && W <= kTcgMaxSplit * kTcMaxKeys;
}

// The tcgen05 row-group plan: the smallest cluster whose CTAs hold at most
// kTcMaxKeys keys of the group's longest list each.
int plan_tcg(int B, int H, int W, int G, const smd_plan_t* force, smd_plan_t* out, TcgConfig* cfg) {
    if (!tcg_fits(H, W, G)) return SMD_ERR_PLAN;
    if ((force && force->tiles && force->tiles != G * H / kHeadsPerTile) ||
        (force && force->window && force->window != kTcChunk))
        return SMD_ERR_PLAN;
    int split = 1;
    while (ceil_div(W, split) > kTcMaxKeys) split *= 2;
    if (force && force->split) {
        if (!is_split(force->split) || ceil_div(W, force->split) > kTcMaxKeys) return SMD_ERR_PLAN;
        split = force->split;
    }
    cfg->G = G;
    cfg->split = split;
    cfg->wait_budget_ns = (force && force->wait_budget_us > 0)
                              ? static_cast<uint64_t>(force->wait_budget_us) * 1000ull
                              : kWaitBudgetNs;
    cfg->inject_stall = (force && force->inject_stall) ? 1 : 0;
    out->kernel = SMD_KERNEL_TC_GROUP;
    out->split = split;
    out->tiles = G * H / kHeadsPerTile;
    out->window = kTcChunk;
    out->key_cap = kTcMaxKeys;
    out->grid_x = split;
    out->grid_y = B / G;
    out->cluster_x = split;
    out->threads = kTcThreads;
    out->smem_bytes = 0;  // filled by the caller
    return SMD_OK;
}

int plan_group(int B, int H, int W, int G, int sm_count, const smd_plan_t* force, smd_plan_t* out,
               GroupConfig* cfg) {
    if ((G != 2 && G != 4) || B % G != 0) return SMD_ERR_SHAPE;
    if (force && force->tiles && force->tiles != G) return SMD_ERR_PLAN;
    if (force && force->kernel && force->kernel != SMD_KERNEL_GROUP) return SMD_ERR_PLAN;
    const int units = B / G * (H / kHeadsPerTile);
    // A CTA takes an aligned block of leaves of the group's longest list
    // (smd_tree.cuh): at most kGroupMaxKeys staged indices, and at most as
    // many leaves as the TMEM subtree stack holds levels for (128 columns a
    // warp, 16 G a level: 2^(128 / (16 G)) leaves).
    const int max_lpc = 1 << (128 / (kHeadsPerTile * G));
    auto fits = [&](int s) {
        return mma_cta_keys(std::max(W, 1), s) <= kGroupMaxKeys &&
               mma_leaves_per_cta(std::max(W, 1), s) <= max_lpc;
    };
    int split = 1;
    while (split < kGroupMaxSplit && !fits(split)) split *= 2;
    if (!fits(split)) return SMD_ERR_SHAPE;
    if (force && force->split) {
        if (!is_split(force->split) || !fits(force->split)) return SMD_ERR_PLAN;
        split = force->split;
    } else {
        while (split < kGroupMaxSplit && units * split < sm_count && split * 2 <= mma_leaves(W))
            split *= 2;
    }
    int nslots = 2;
    if (force && force->window) {
        if (force->window % kChunk != 0 || force->window < kChunk || force->window > 8 * kChunk)
            return SMD_ERR_PLAN;
        nslots = force->window / kChunk;
    }
    const int key_cap =
        std::max(kChunk, ceil_div(mma_cta_keys(std::max(W, 1), split), kChunk) * kChunk);
    const GroupLayout L = group_layout(G, split, nslots, key_cap);
    if (L.total > kMaxSmemBytes) return SMD_ERR_PLAN;
    cfg->tree_tmem = std::min(kMmaMaxLeaves, ceil_div(W, kChunk)) > split ? 1 : 0;
    cfg->G = G;
    cfg->split = split;
    cfg->nslots = nslots;
    cfg->key_cap = key_cap;
    cfg->layout = L;
    cfg->wait_budget_ns = (force && force->wait_budget_us > 0)
                              ? static_cast<uint64_t>(force->wait_budget_us) * 1000ull
                              : kWaitBudgetNs;
    cfg->inject_stall = (force && force->inject_stall) ? 1 : 0;
    out->kernel = SMD_KERNEL_GROUP;
    out->split = split;
    out->tiles = G;
    out->window = nslots * kChunk;
    out->key_cap = key_cap;
    out->grid_x = H / kHeadsPerTile * split;
    out->grid_y = B / G;
    out->cluster_x = split;
    out->threads = kMmaThreads;
    out->smem_bytes = L.total;
    return SMD_OK;
}

// The spread kernel: 128 heads per CTA (or all H < 128), or all H heads of a
// group of G rows (G * H <= 128 lanes); pieces of at most kTcMaxKeys keys, at
// most kTcsMaxPieces pieces per unit.
int64_t tcs_units(int B, int H, int G) {
    return G > 1 ? B / G : static_cast<int64_t>(B) * ceil_div(H, kTcHeads);
}

bool tcs_fits(int B, int H, int W, int G = 1) {
    const bool lanes_ok = G > 1 ? (B % G == 0 && G * H <= kTcHeads)
                                : (H % kTcHeads == 0 || H < kTcHeads);
    return lanes_ok && W >= 1 && W <= kTcsMaxPieces * kTcMaxKeys &&
           tcs_units(B, H, G) <= kTcsMaxUnits;
}

int64_t tcs_items_cap(int B, int H, int W, int G = 1) {
    return tcs_units(B, H, G) * ceil_div(W, kTcMaxKeys);
}

// The spread kernel's plan: one CTA per resident slot, no more than there can
// be pieces (a forced grid_x caps it).
int plan_tcs(int B, int H, int W, int sm_count, const smd_plan_t* force, smd_plan_t* out,
             TcsConfig* cfg, int G = 1) {
    if (!tcs_fits(B, H, W, G)) return SMD_ERR_PLAN;
    const int lanes = G > 1 ? G * H : std::min(H, kTcHeads);
    if (force && ((force->tiles && force->tiles != lanes / kHeadsPerTile) ||
                  (force->window && force->window != kTcChunk) || force->split))
        return SMD_ERR_PLAN;
    // Resident CTAs (one per SM); without a device, planning assumes one per SM.
    int max_grid = tcs_max_grid();
    if (max_grid <= 0) max_grid = sm_count;
    const int64_t items = tcs_items_cap(B, H, W, G);
    int grid = static_cast<int>(std::min<int64_t>(max_grid, items));
    if (force && force->grid_x) {
        if (force->grid_x < 1 || force->grid_x > max_grid) return SMD_ERR_PLAN;
        // every piece of a row must find a CTA of its own
        if (force->grid_x < std::min(kTcsMaxPieces, ceil_div(W, kTcMaxKeys))) return SMD_ERR_PLAN;
        grid = std::min<int64_t>(force->grid_x, items);
    }
    cfg->G = G;
    cfg->grid = grid;
    cfg->items_cap = static_cast<int>(items);
    cfg->wait_budget_ns = (force && force->wait_budget_us > 0)
                              ? static_cast<uint64_t>(force->wait_budget_us) * 1000ull
                              : kWaitBudgetNs;
    cfg->inject_stall = (force && force->inject_stall) ? 1 : 0;
    cfg->ws = nullptr;
    out->kernel = SMD_KERNEL_TC_SPREAD;
    out->split = ceil_div(W, kTcMaxKeys);  // the most pieces a row can have
    out->tiles = lanes / kHeadsPerTile;
    out->window = kTcChunk;
    out->key_cap = kTcMaxKeys;
    out->grid_x = grid;
    out->grid_y = 1;
    out->cluster_x = 1;
    out->threads = kTcThreads;
    out->smem_bytes = tcs_smem_bytes();
    return SMD_OK;
}

// Row groups with a workspace run on the spread kernel wherever it takes
// them. Its pieces are the group's 512-key leaves laid out over the whole
// grid, while the row-group cluster kernel gives every group a cluster of
// ceil(W / 512) CTAs, of which a group with a shorter list leaves the rest
// idle (dense-as-sparse: 125 against 139 us).
bool grouped_spread(int B, int H, int W, int G) { return tcs_fits(B, H, W, G); }

int64_t grouped_workspace_bytes(int B, int H, int W, int G) {
    return grouped_spread(B, H, W, G) ? tcs_workspace(tcs_items_cap(B, H, W, G)).total : 0;
}

// With a workspace, the spread kernel takes rows longer than a cluster holds
// and, for rows longer than one CTA holds, batches whose pieces fill at most
// two waves (the cluster kernel would leave SMs idle or run a second wave of
// whole rows).
bool prefer_spread(int B, int H, int W, int sm_count) {
    if (H % kTcHeads != 0 || !tcs_fits(B, H, W) || W <= kTcMaxKeys) return false;
    return W > kTcMaxSplit * kTcMaxKeys || tcs_items_cap(B, H, W) <= 2 * sm_count;
}

// The split query on the spread kernel: 128-head groups and rows it takes.
bool bf16q_spread_fits(int B, int H, int W) { return H % kTcHeads == 0 && tcs_fits(B, H, W); }

int64_t bf16q_workspace_bytes(int B, int H, int W) {
    if (!bf16q_spread_fits(B, H, W)) return 0;
    return tcs_workspace(tcs_items_cap(B, H, W), static_cast<int64_t>(B) * H).total;
}

struct AnyConfig {
    int kernel;
    MmaConfig mma;
    TcConfig tc;
    TcsConfig tcs;
};

// ws_bytes: >= 0 when the caller passes a workspace (its size is checked by
// the caller of make_plan), -1 when there is none.
int make_plan(int B, int H, int W, const smd_plan_t* force, smd_plan_t* out, AnyConfig* cfg,
              int64_t ws_bytes = -1) {
    if (B < 0 || W < 0 || H <= 0 || H % kHeadsPerTile != 0) return SMD_ERR_SHAPE;
    static std::once_flag once;
    static DeviceInfo info;
    std::call_once(once, [] { info = query_device(); });
    const int sm_count = info.ok ? info.sm_count : 152;
    int kernel = (force && force->kernel) ? force->kernel : SMD_KERNEL_AUTO;
    if (kernel == SMD_KERNEL_AUTO) {
        if (ws_bytes >= 0 && prefer_spread(B, H, W, sm_count))
            kernel = SMD_KERNEL_TC_SPREAD;
        else
            kernel = (H % kTcHeads == 0 && tc_fits(H, W)) ? SMD_KERNEL_TC : SMD_KERNEL_MMA;
    }
    cfg->kernel = kernel;
    if (kernel == SMD_KERNEL_MMA) return plan_mma(B, H, W, sm_count, force, out, &cfg->mma);
    if (kernel == SMD_KERNEL_TC) return plan_tc(B, H, W, force, out, &cfg->tc);
    if (kernel == SMD_KERNEL_TC_SPREAD) return plan_tcs(B, H, W, sm_count, force, out, &cfg->tcs);
    return SMD_ERR_PLAN;
}

float scale_log2_of(float sm, float qs, float ks) {
    const double v = static_cast<double>(sm) * static_cast<double>(qs) * static_cast<double>(ks);
    return static_cast<float>(v * 1.4426950408889634073599246810019);
}

int64_t workspace_for(const AnyConfig& cfg) {
    if (cfg.kernel == SMD_KERNEL_TC_SPREAD) return tcs_workspace(cfg.tcs.items_cap).total;
    return (cfg.kernel == SMD_KERNEL_TC && cfg.tc.split > 1) ? kTcWsBytes : 0;
}

int sm_count_of_device() {
    static std::once_flag once;
    static DeviceInfo info;
    std::call_once(once, [] { info = query_device(); });
    return info.ok ? info.sm_count : 152;
}

int decode(const uint8_t* q, const uint8_t* kv_pool, int64_t N, const int32_t* indices, int32_t W,
           const int32_t* counts, int32_t B, int32_t H, float sm_scale, float q_scale,
           float k_scale, uint16_t* out, float* lse, int32_t* status, void* workspace,
           int64_t workspace_bytes, smd_stream_t stream, const smd_plan_t* force,
           bool library_scratch = false, int row_group = 1, const uint16_t* q16 = nullptr,
           smd_plan_t* dry = nullptr) {
    // dry != nullptr: no launch and no pointer checks; the plan the call would
    // run is written to *dry (a workspace of any size counts as given).
    if (B < 0 || W < 0 || N < 0 || H <= 0 || H % kHeadsPerTile != 0) return SMD_ERR_SHAPE;
    if (row_group != 1 && ((row_group != 2 && row_group != 4) || B % row_group != 0))
        return SMD_ERR_SHAPE;
    if (N >= (int64_t(1) << 31)) return SMD_ERR_SHAPE;
    if (dry == nullptr) {
        if (B == 0) return SMD_OK;
        if (!q || !out || !lse || !counts) return SMD_ERR_NULL;
        if (W > 0 && (!indices || !kv_pool)) return SMD_ERR_NULL;
        if (W > 0 && N == 0) return SMD_ERR_SHAPE;
        if (!aligned(q, 16) || !aligned(out, 16) || (kv_pool && !aligned(kv_pool, 16)))
            return SMD_ERR_ALIGN;
        if ((indices && !aligned(indices, 4)) || !aligned(counts, 4) || !aligned(lse, 4) ||
            (status && !aligned(status, 4)))
            return SMD_ERR_ALIGN;
    }

    if (row_group > 1) {
        if (B % row_group != 0) return SMD_ERR_SHAPE;
        if (workspace != nullptr && !aligned(workspace, 16)) return SMD_ERR_WORKSPACE;
        const int want = (force && force->kernel) ? force->kernel
                         : (workspace != nullptr && grouped_spread(B, H, W, row_group)) ? SMD_KERNEL_TC_SPREAD
                         : tcg_fits(H, W, row_group) ? SMD_KERNEL_TC_GROUP
                                                     : SMD_KERNEL_GROUP;
        if (want == SMD_KERNEL_TC_SPREAD) {
            smd_plan_t plan{};
            TcsConfig scfg{};
            const int rc = plan_tcs(B, H, W, sm_count_of_device(), force, &plan, &scfg, row_group);
            if (rc != SMD_OK) return rc;
            if (dry != nullptr) {
                *dry = plan;
                return SMD_OK;
            }
            if (workspace == nullptr || workspace_bytes < tcs_workspace(scfg.items_cap).total)
                return SMD_ERR_WORKSPACE;
            scfg.ws = workspace;
            CallArgs a{};
            a.q = q;
            a.kv = kv_pool;
            a.N = N;
            a.indices = indices;
            a.W = W;
            a.counts = counts;
            a.B = B;
            a.H = H;
            a.scale_log2 = scale_log2_of(sm_scale, q_scale, k_scale);
            a.k_scale = k_scale;
            a.out = out;
            a.lse = lse;
            a.status = status;
            return launch_tcs(a, scfg, reinterpret_cast<cudaStream_t>(stream));
        }
        smd_plan_t plan{};
        GroupConfig gcfg{};
        TcgConfig tcfg{};
        const int rc = want == SMD_KERNEL_TC_GROUP
                           ? plan_tcg(B, H, W, row_group, force, &plan, &tcfg)
                           : plan_group(B, H, W, row_group, sm_count_of_device(), force, &plan, &gcfg);
        if (rc != SMD_OK) return rc;
        if (dry != nullptr) {
            if (want == SMD_KERNEL_TC_GROUP) plan.smem_bytes = tcg_smem_bytes();
            *dry = plan;
            return SMD_OK;
        }
        CallArgs a{};
        a.q = q;
        a.kv = kv_pool;
        a.N = N;
        a.indices = indices;
        a.W = W;
        a.counts = counts;
        a.B = B;
        a.H = H;
        a.scale_log2 = scale_log2_of(sm_scale, q_scale, k_scale);
        a.k_scale = k_scale;
        a.out = out;
        a.lse = lse;
        a.status = status;
        if (want == SMD_KERNEL_TC_GROUP) return launch_tcg(a, tcfg, reinterpret_cast<cudaStream_t>(stream));
        return launch_group(a, gcfg, reinterpret_cast<cudaStream_t>(stream));
    }

    if (q16 != nullptr) {
        // The split query: on the spread tcgen05 kernel when a workspace is
        // given and the shapes fit it, else on the warp-MMA kernel.
        const int fk = (force && force->kernel) ? force->kernel : SMD_KERNEL_AUTO;
        if (fk != SMD_KERNEL_AUTO && fk != SMD_KERNEL_MMA && fk != SMD_KERNEL_TC_SPREAD)
            return SMD_ERR_PLAN;
        if (workspace != nullptr && !aligned(workspace, 16)) return SMD_ERR_WORKSPACE;
        const bool spread = fk == SMD_KERNEL_TC_SPREAD ||
                            (fk == SMD_KERNEL_AUTO && workspace != nullptr && bf16q_spread_fits(B, H, W));
        smd_plan_t plan{};
        MmaConfig mcfg{};
        TcsConfig tcfg{};
        const int rc = spread ? plan_tcs(B, H, W, sm_count_of_device(), force, &plan, &tcfg)
                              : plan_mma(B, H, W, sm_count_of_device(), force, &plan, &mcfg, true);
        if (rc != SMD_OK) return rc;
        if (dry != nullptr) {
            *dry = plan;
            return SMD_OK;
        }
        if (spread) {
            const int64_t need = tcs_workspace(tcfg.items_cap, static_cast<int64_t>(B) * H).total;
            if (workspace == nullptr || workspace_bytes < need) return SMD_ERR_WORKSPACE;
            tcfg.qsplit = 1;
            tcfg.ws = workspace;
        }
        CallArgs a{};
        a.q = nullptr;
        a.q16 = q16;
        a.kv = kv_pool;
        a.N = N;
        a.indices = indices;
        a.W = W;
        a.counts = counts;
        a.B = B;
        a.H = H;
        a.scale_log2 = scale_log2_of(sm_scale, 1.0f, k_scale);  // 2^-k per head on the GPU
        a.k_scale = k_scale;
        a.out = out;
        a.lse = lse;
        a.status = status;
        if (spread) return launch_tcs(a, tcfg, reinterpret_cast<cudaStream_t>(stream));
        return launch_mma(a, mcfg, reinterpret_cast<cudaStream_t>(stream));
    }

    smd_plan_t plan{};
    AnyConfig cfg{};
    if (workspace != nullptr && !aligned(workspace, 16)) return SMD_ERR_WORKSPACE;
    const int rc = make_plan(B, H, W, force, &plan, &cfg, workspace != nullptr ? 0 : -1);
    if (rc != SMD_OK) return rc;
    if (dry != nullptr) {
        *dry = plan;
        return SMD_OK;
    }
    if (cfg.kernel == SMD_KERNEL_TC_SPREAD) {
        if (workspace == nullptr || workspace_bytes < workspace_for(cfg)) return SMD_ERR_WORKSPACE;
        cfg.tcs.ws = workspace;
    } else if (workspace != nullptr && force != nullptr) {
        // A forced plan with a workspace: a cluster plan's partials go through
        // it (L2). The automatic plan keeps the on-chip exchange, which is the
        // faster one on GB300.
        if (workspace_bytes < workspace_for(cfg)) return SMD_ERR_WORKSPACE;
        if (workspace_for(cfg) > 0) cfg.tc.ws = static_cast<float*>(workspace);
    } else if (library_scratch && workspace_for(cfg) > 0) {
        // The library's own static scratch: one slot per SM id.
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SMD_ERR_DEVICE;
        if (sms > kStaticScratchSlots) return SMD_ERR_WORKSPACE;
        int src = SMD_OK;
        float* scratch = static_scratch(&src);
        if (src != SMD_OK) return src;
        cfg.tc.ws = scratch;
        cfg.tc.ws_slots = kStaticScratchSlots;
    }

    CallArgs a{};
    a.q = q;
    a.kv = kv_pool;
    a.N = N;
    a.indices = indices;
    a.W = W;
    a.counts = counts;
    a.B = B;
    a.H = H;
    a.scale_log2 = scale_log2_of(sm_scale, q_scale, k_scale);
    a.k_scale = k_scale;
    a.out = out;
    a.lse = lse;
    a.status = status;
    if (cfg.kernel == SMD_KERNEL_TC) return launch_tc(a, cfg.tc, reinterpret_cast<cudaStream_t>(stream));
    if (cfg.kernel == SMD_KERNEL_TC_SPREAD)
        return launch_tcs(a, cfg.tcs, reinterpret_cast<cudaStream_t>(stream));
    return launch_mma(a, cfg.mma, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace smd

extern "C" {

int smd_sparse_mla_decode(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                          const int32_t* indices, int32_t W, const int32_t* counts, int32_t B,
                          int32_t H, float sm_scale, float q_scale, float k_scale, uint16_t* out,
                          float* lse, int32_t* status, smd_stream_t stream) {
    return smd::decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out,
                       lse, status, nullptr, 0, stream, nullptr);
}

int smd_sparse_mla_decode_ws(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                             const int32_t* indices, int32_t W, const int32_t* counts, int32_t B,
                             int32_t H, float sm_scale, float q_scale, float k_scale,
                             uint16_t* out, float* lse, int32_t* status, void* workspace,
                             int64_t workspace_bytes, smd_stream_t stream) {
    return smd::decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out,
                       lse, status, workspace, workspace_bytes, stream, nullptr);
}

int smd_sparse_mla_decode_ex(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                             const int32_t* indices, int32_t W, const int32_t* counts, int32_t B,
                             int32_t H, float sm_scale, float q_scale, float k_scale,
                             uint16_t* out, float* lse, int32_t* status, void* workspace,
                             int64_t workspace_bytes, smd_stream_t stream,
                             const smd_plan_t* force) {
    return smd::decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out,
                       lse, status, workspace, workspace_bytes, stream, force);
}

int smd_sparse_mla_decode_bf16q(const uint16_t* q, const uint8_t* kv_pool, int64_t N,
                                const int32_t* indices, int32_t W, const int32_t* counts,
                                int32_t B, int32_t H, float sm_scale, float k_scale,
                                uint16_t* out, float* lse, int32_t* status, smd_stream_t stream) {
    return smd::decode(reinterpret_cast<const uint8_t*>(q), kv_pool, N, indices, W, counts, B, H,
                       sm_scale, 1.0f, k_scale, out, lse, status, nullptr, 0, stream, nullptr,
                       false, 1, q);
}

int smd_sparse_mla_decode_bf16q_ws(const uint16_t* q, const uint8_t* kv_pool, int64_t N,
                                   const int32_t* indices, int32_t W, const int32_t* counts,
                                   int32_t B, int32_t H, float sm_scale, float k_scale,
                                   uint16_t* out, float* lse, int32_t* status, void* workspace,
                                   int64_t workspace_bytes, smd_stream_t stream) {
    return smd::decode(reinterpret_cast<const uint8_t*>(q), kv_pool, N, indices, W, counts, B, H,
                       sm_scale, 1.0f, k_scale, out, lse, status, workspace, workspace_bytes,
                       stream, nullptr, false, 1, q);
}

int smd_sparse_mla_decode_bf16q_ex(const uint16_t* q, const uint8_t* kv_pool, int64_t N,
                                   const int32_t* indices, int32_t W, const int32_t* counts,
                                   int32_t B, int32_t H, float sm_scale, float k_scale,
                                   uint16_t* out, float* lse, int32_t* status, void* workspace,
                                   int64_t workspace_bytes, smd_stream_t stream,
                                   const smd_plan_t* force) {
    return smd::decode(reinterpret_cast<const uint8_t*>(q), kv_pool, N, indices, W, counts, B, H,
                       sm_scale, 1.0f, k_scale, out, lse, status, workspace, workspace_bytes,
                       stream, force, false, 1, q);
}

}  // extern "C"

namespace smd {
namespace {

// The variant an options struct names (NULL: the defaults); SMD_OK or the
// status of an invalid combination.
int check_options(const smd_options_t* opt) {
    if (opt == nullptr) return SMD_OK;
    if (opt->reserved != 0) return SMD_ERR_SHAPE;
    if (opt->query_type != SMD_QUERY_E4M3 && opt->query_type != SMD_QUERY_BF16) return SMD_ERR_SHAPE;
    const int G = opt->row_group == 0 ? 1 : opt->row_group;
    if (G != 1 && G != 2 && G != 4) return SMD_ERR_SHAPE;
    if (opt->query_type == SMD_QUERY_BF16 && G != 1) return SMD_ERR_PLAN;
    if (opt->library_scratch &&
        (opt->workspace != nullptr || G != 1 || opt->query_type == SMD_QUERY_BF16))
        return SMD_ERR_PLAN;
    return SMD_OK;
}

int decode_opts(const void* q, const uint8_t* kv_pool, int64_t N, const int32_t* indices,
                int32_t W, const int32_t* counts, int32_t B, int32_t H, float sm_scale,
                float q_scale, float k_scale, uint16_t* out, float* lse,
                const smd_options_t* opt, smd_stream_t stream, smd_plan_t* dry) {
    const int rc = check_options(opt);
    if (rc != SMD_OK) return rc;
    const smd_options_t o = opt ? *opt : smd_options_t{};
    const int G = o.row_group == 0 ? 1 : o.row_group;
    const bool bf16 = o.query_type == SMD_QUERY_BF16;
    void* ws = o.workspace;
    int64_t ws_bytes = o.workspace_bytes;
    // A plan query passes no pointers: a stand-in marks "a workspace is
    // given" and "the query is bf16" (neither is read).
    alignas(16) static unsigned char token[16];
    if (dry != nullptr && ws == nullptr && ws_bytes > 0) ws = token;
    if (dry != nullptr && q == nullptr) q = token;
    const uint8_t* q8 = static_cast<const uint8_t*>(q);
    return decode(q8, kv_pool, N, indices, W, counts, B, H, sm_scale, bf16 ? 1.0f : q_scale, k_scale,
                  out, lse, o.status, ws, ws_bytes, stream, o.force, o.library_scratch != 0, G,
                  bf16 ? static_cast<const uint16_t*>(q) : nullptr, dry);
}

}  // namespace
}  // namespace smd

extern "C" {

int smd_decode(const void* q, const uint8_t* kv_pool, int64_t N, const int32_t* indices, int32_t W,
               const int32_t* counts, int32_t B, int32_t H, float sm_scale, float q_scale,
               float k_scale, uint16_t* out, float* lse, const smd_options_t* options,
               smd_stream_t stream) {
    return smd::decode_opts(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out,
                            lse, options, stream, nullptr);
}

int smd_decode_plan(int32_t B, int32_t H, int32_t W, const smd_options_t* options,
                    smd_plan_t* plan) {
    if (!plan) return SMD_ERR_NULL;
    smd_plan_t p{};
    const int rc = smd::decode_opts(nullptr, nullptr, 1, nullptr, W, nullptr, B, H, 1.f, 1.f, 1.f,
                                    nullptr, nullptr, options, nullptr, &p);
    if (rc == SMD_OK) *plan = p;
    return rc;
}

int64_t smd_decode_workspace_bytes(int32_t B, int32_t H, int32_t W, const smd_options_t* options) {
    if (smd::check_options(options) != SMD_OK) return 0;
    const int G = options && options->row_group ? options->row_group : 1;
    if (options && options->query_type == SMD_QUERY_BF16) return smd_workspace_bytes_bf16q(B, H, W);
    if (G > 1) return smd_workspace_bytes_grouped(B, H, W, G);
    if (options && options->force) return smd_workspace_bytes_ex(B, H, W, options->force);
    return smd_workspace_bytes(B, H, W);
}

int64_t smd_workspace_bytes_bf16q(int32_t B, int32_t H, int32_t W) {
    if (B < 0 || W < 0 || H <= 0 || H % smd::kHeadsPerTile != 0) return 0;
    return smd::bf16q_workspace_bytes(B, H, W);
}

int smd_plan_bf16q(int32_t B, int32_t H, int32_t W, int64_t workspace_bytes, smd_plan_t* plan) {
    if (!plan) return SMD_ERR_NULL;
    if (B < 0 || W < 0 || H <= 0 || H % smd::kHeadsPerTile != 0) return SMD_ERR_SHAPE;
    smd_plan_t p{};
    int rc;
    if (workspace_bytes > 0 && smd::bf16q_spread_fits(B, H, W)) {
        smd::TcsConfig cfg{};
        rc = smd::plan_tcs(B, H, W, smd::sm_count_of_device(), nullptr, &p, &cfg);
    } else {
        smd::MmaConfig cfg{};
        rc = smd::plan_mma(B, H, W, smd::sm_count_of_device(), nullptr, &p, &cfg, true);
    }
    if (rc == SMD_OK) *plan = p;
    return rc;
}

int smd_sparse_mla_decode_noalloc(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                                  const int32_t* indices, int32_t W, const int32_t* counts,
                                  int32_t B, int32_t H, float sm_scale, float q_scale,
                                  float k_scale, uint16_t* out, float* lse, int32_t* status,
                                  smd_stream_t stream) {
    return smd::decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out,
                       lse, status, nullptr, 0, stream, nullptr, /*library_scratch=*/true);
}

int64_t smd_workspace_bytes(int32_t B, int32_t H, int32_t W) {
    smd::AnyConfig cfg{};
    smd_plan_t p{};
    if (smd::make_plan(B, H, W, nullptr, &p, &cfg, 0) != SMD_OK) return 0;
    return cfg.kernel == SMD_KERNEL_TC_SPREAD ? smd::workspace_for(cfg) : 0;
}

int64_t smd_workspace_bytes_ex(int32_t B, int32_t H, int32_t W, const smd_plan_t* force) {
    smd::AnyConfig cfg{};
    smd_plan_t p{};
    if (smd::make_plan(B, H, W, force, &p, &cfg, 0) != SMD_OK) return 0;
    return smd::workspace_for(cfg);
}

int smd_plan_ws(int32_t B, int32_t H, int32_t W, smd_plan_t* plan) {
    if (!plan) return SMD_ERR_NULL;
    smd::AnyConfig cfg{};
    smd_plan_t p{};
    const int rc = smd::make_plan(B, H, W, nullptr, &p, &cfg, 0);
    if (rc == SMD_OK) *plan = p;
    return rc;
}

int smd_plan(int32_t B, int32_t H, int32_t W, smd_plan_t* plan) {
    if (!plan) return SMD_ERR_NULL;
    smd::AnyConfig cfg{};
    smd_plan_t p{};
    const int rc = smd::make_plan(B, H, W, nullptr, &p, &cfg);
    if (rc == SMD_OK) *plan = p;
    return rc;
}

int smd_sparse_mla_decode_grouped(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                                  const int32_t* indices, int32_t W, const int32_t* counts,
                                  int32_t B, int32_t H, int32_t row_group, float sm_scale,
                                  float q_scale, float k_scale, uint16_t* out, float* lse,
                                  int32_t* status, smd_stream_t stream) {
    return smd::decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out,
                       lse, status, nullptr, 0, stream, nullptr, false, row_group);
}

int smd_sparse_mla_decode_grouped_ws(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                                     const int32_t* indices, int32_t W, const int32_t* counts,
                                     int32_t B, int32_t H, int32_t row_group, float sm_scale,
                                     float q_scale, float k_scale, uint16_t* out, float* lse,
                                     int32_t* status, void* workspace, int64_t workspace_bytes,
                                     smd_stream_t stream) {
    return smd::decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out,
                       lse, status, workspace, workspace_bytes, stream, nullptr, false, row_group);
}

int smd_sparse_mla_decode_grouped_ex(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                                     const int32_t* indices, int32_t W, const int32_t* counts,
                                     int32_t B, int32_t H, int32_t row_group, float sm_scale,
                                     float q_scale, float k_scale, uint16_t* out, float* lse,
                                     int32_t* status, void* workspace, int64_t workspace_bytes,
                                     smd_stream_t stream, const smd_plan_t* force) {
    return smd::decode(q, kv_pool, N, indices, W, counts, B, H, sm_scale, q_scale, k_scale, out,
                       lse, status, workspace, workspace_bytes, stream, force, false, row_group);
}

int64_t smd_workspace_bytes_grouped(int32_t B, int32_t H, int32_t W, int32_t row_group) {
    if (row_group == 1) return smd_workspace_bytes(B, H, W);
    if (B < 0 || W < 0 || H <= 0 || H % smd::kHeadsPerTile != 0) return 0;
    if ((row_group != 2 && row_group != 4) || B % row_group != 0) return 0;
    return smd::grouped_workspace_bytes(B, H, W, row_group);
}

int smd_plan_grouped(int32_t B, int32_t H, int32_t W, int32_t row_group, int64_t workspace_bytes,
                     smd_plan_t* plan) {
    if (!plan) return SMD_ERR_NULL;
    if (row_group == 1)
        return workspace_bytes > 0 ? smd_plan_ws(B, H, W, plan) : smd_plan(B, H, W, plan);
    if (B < 0 || W < 0 || H <= 0 || H % smd::kHeadsPerTile != 0) return SMD_ERR_SHAPE;
    if ((row_group != 2 && row_group != 4) || B % row_group != 0) return SMD_ERR_SHAPE;
    smd_plan_t p{};
    int rc;
    if (workspace_bytes > 0 && smd::grouped_spread(B, H, W, row_group)) {
        smd::TcsConfig cfg{};
        rc = smd::plan_tcs(B, H, W, smd::sm_count_of_device(), nullptr, &p, &cfg, row_group);
    } else if (smd::tcg_fits(H, W, row_group)) {
        smd::TcgConfig cfg{};
        rc = smd::plan_tcg(B, H, W, row_group, nullptr, &p, &cfg);
        p.smem_bytes = smd::tcg_smem_bytes();
    } else {
        smd::GroupConfig cfg{};
        rc = smd::plan_group(B, H, W, row_group, smd::sm_count_of_device(), nullptr, &p, &cfg);
    }
    if (rc == SMD_OK) *plan = p;
    return rc;
}

int smd_topk_select_ex(const uint16_t* logits, int64_t row_stride, const int32_t* row_ends,
                       int32_t B, int32_t L, int32_t K, int32_t* indices, int32_t* counts,
                       int32_t* status, smd_stream_t stream, int32_t cluster) {
    if (B < 0 || L < 0 || K < 1 || row_stride < L) return SMD_ERR_SHAPE;
    if (cluster < 0 || cluster > 8 || (cluster & (cluster - 1)) != 0) return SMD_ERR_PLAN;
    if (B == 0) return SMD_OK;
    if (!indices || !counts || (L > 0 && !logits)) return SMD_ERR_NULL;
    if ((logits && !smd::aligned(logits, 2)) || !smd::aligned(indices, 4) ||
        !smd::aligned(counts, 4) || (row_ends && !smd::aligned(row_ends, 4)) ||
        (status && !smd::aligned(status, 4)))
        return SMD_ERR_ALIGN;
    int C = cluster;
    if (C == 0) {
        // CTAs per row (a power of two, at most 8): parts whose keys stay in
        // shared memory (16384 logits) while the CTAs fit the device at once
        // (two per SM), then more while the SMs are not all busy.
        const int slots = 2 * smd::sm_count_of_device();
        C = 1;
        while (C < 8 && (L + C - 1) / C > 16384 && static_cast<int64_t>(B) * C * 2 <= slots) C *= 2;
        while (C < 8 && static_cast<int64_t>(B) * C * 2 <= slots / 2 && C * 4096 < L) C *= 2;
    }
    return smd::launch_topk(logits, row_stride, row_ends, B, L, K, indices, counts, status, C,
                            reinterpret_cast<cudaStream_t>(stream));
}

int smd_topk_select(const uint16_t* logits, int64_t row_stride, const int32_t* row_ends,
                    int32_t B, int32_t L, int32_t K, int32_t* indices, int32_t* counts,
                    int32_t* status, smd_stream_t stream) {
    return smd_topk_select_ex(logits, row_stride, row_ends, B, L, K, indices, counts, status,
                              stream, 0);
}

float smd_scale_log2(float sm_scale, float q_scale, float k_scale) {
    return smd::scale_log2_of(sm_scale, q_scale, k_scale);
}

const char* smd_status_str(int status) {
    switch (status) {
        case SMD_OK:
            return "ok";
        case SMD_ERR_NULL:
            return "a required pointer is NULL";
        case SMD_ERR_SHAPE:
            return "invalid shape (H must be a positive multiple of 16; B, W, N >= 0; N >= 1 "
                   "when B*W > 0; N < 2^31; the top-k width must fit the plan)";
        case SMD_ERR_ALIGN:
            return "misaligned pointer (q, kv_pool, out: 16 bytes; indices, counts, lse, "
                   "status: 4 bytes)";
        case SMD_ERR_LAUNCH:
            return "CUDA launch failed";
        case SMD_ERR_TIMEOUT:
            return "a bounded device wait ran out (device status)";
        case SMD_ERR_PLAN:
            return "the forced plan is invalid for these shapes";
        case SMD_ERR_DEVICE:
            return "no usable CUDA device (or an SM id beyond the exchange workspace)";
        case SMD_ERR_WORKSPACE:
            return "workspace smaller than smd_workspace_bytes() or not 16-byte aligned";
        case SMD_ERR_GROUP:
            return "rows of a group do not share their index list (device status)";
        case SMD_ERR_INDEX:
            return "a valid entry of the index list lies outside [0, N) (device status)";
        default:
            return "unknown status";
    }
}

int smd_version(void) { return 100; }

int smd_trace_enabled(void) {
#ifdef SMD_TRACE
    return 1;
#else
    return 0;
#endif
}

static int trace_copy(int32_t kernel, uint64_t* host, int32_t n, bool clear) {
    if (!clear && host == nullptr) return SMD_ERR_NULL;
    if (!clear && (n < 0 || n > smd::kTraceRows * smd::kTraceSlots)) return SMD_ERR_SHAPE;
    switch (kernel) {
        case SMD_KERNEL_MMA: return smd::mma_trace_copy(host, n, clear);
        case SMD_KERNEL_TC: return smd::tc_trace_copy(host, n, clear);
        case SMD_KERNEL_TC_SPREAD: return smd::tcs_trace_copy(host, n, clear);
        default: return SMD_ERR_PLAN;
    }
}

int smd_trace_read(int32_t kernel, uint64_t* host, int32_t n) { return trace_copy(kernel, host, n, false); }

int smd_trace_clear(int32_t kernel) { return trace_copy(kernel, nullptr, 0, true); }

}  // extern "C"
