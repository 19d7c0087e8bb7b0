// Internal declarations shared by the C ABI layer and the kernels.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "smd.h"

namespace smd {

constexpr int kRow = 576;        // bytes of a cache / query row
constexpr int kLatent = 512;     // columns read by PV
constexpr int kHeadsPerTile = 16;
constexpr int kRowPitch = 592;   // shared-memory pitch of a 576-byte row (bank spread)
constexpr int kChunk = 64;       // keys per gather barrier
constexpr int kSpecIdxMaxW = 2048;  // widest row whose index list the warp-MMA kernel loads up front
constexpr int kMmaThreads = 512; // 16 warps; PV warp w owns latent columns 32w..32w+31

// Everything a kernel needs to know about one call.
struct CallArgs {
    const uint8_t* q;
    const uint8_t* kv;
    int64_t N;
    const int32_t* indices;
    int32_t W;
    const int32_t* counts;
    int32_t B, H;
    float scale_log2;  // fp32(sm * q_s * k_s * log2 e)
    float k_scale;
    uint16_t* out;
    float* lse;
    int32_t* status;
    const uint16_t* q16;  // bf16 query [B, H, 576] (the split-query call), else null
};

// Shared-memory carve-up of the warp-MMA kernel (byte offsets).
struct MmaLayout {
    int32_t kv, q, logits, probs, idx, inbox, sums, maxima, wmax, lsum, rowmax, lamh, lstk, tslot,
        bars;
    int32_t logit_pitch;  // floats per logits row
    int32_t prob_pitch;   // bytes per P8 row
    int32_t total;
};

__host__ __device__ inline int32_t align_up(int32_t x, int32_t a) { return (x + a - 1) / a * a; }

// idx_cap: int32 entries of the index staging area (the CTA's keys, or the
// row's whole list when it is loaded speculatively). qsplit: the query is
// held as two E4M3 tiles (hi, then lo) with a logit scale per head.
__host__ __device__ inline MmaLayout mma_layout(int tiles, int split, int window, int key_cap,
                                                int idx_cap, bool qsplit = false) {
    MmaLayout L{};
    const int ch = kHeadsPerTile * tiles;
    int32_t o = 0;
    L.kv = o;
    o += window * kRowPitch;
    o = align_up(o, 128);
    L.q = o;
    o += ch * kRowPitch * (qsplit ? 2 : 1);
    o = align_up(o, 16);
    L.logit_pitch = key_cap + 8;  // rows 8 banks apart for the float2 stores
    L.logits = o;
    o += ch * L.logit_pitch * 4;
    o = align_up(o, 16);
    L.prob_pitch = window + 16;
    L.probs = o;
    o += ch * L.prob_pitch;
    o = align_up(o, 16);
    L.idx = o;
    o += (idx_cap > key_cap ? idx_cap : key_cap) * 4;
    o = align_up(o, 16);
    L.inbox = o;  // [split][ch][512/split] fp32: every CTA's partial of my columns
    o += ch * kLatent * 4;
    L.sums = o;   // [split][ch] fp32
    o += split * ch * 4;
    L.maxima = o; // [split][ch] fp32
    o += split * ch * 4;
    L.wmax = o;   // [4 key groups][ch] fp32: the QK jobs' maxima
    o += 4 * ch * 4;
    L.lsum = o;   // [ch] running sums of P
    o += ch * 4;
    L.rowmax = o; // [ch] the row maximum
    o += ch * 4;
    L.lamh = o;   // [ch] per-head logit scale (split query)
    o += ch * 4;
    L.lstk = o;   // [4 levels][ch] the sums' subtree stack (the leaf tree)
    o += 4 * ch * 4;
    L.tslot = o;  // the TMEM address of the partials' subtree stack
    o += 16;
    o = align_up(o, 8);
    L.bars = o;   // window/64 gather barriers, q, maxima, inbound
    o += 8 * (window / kChunk + 3);
    L.total = align_up(o, 128);
    (void)split;
    return L;
}

struct MmaConfig {
    int tiles, split, window, key_cap;
    MmaLayout layout;
    uint64_t wait_budget_ns;
    int inject_stall;
    int spec_idx;
    int qsplit;     // 1: bf16 query (CallArgs::q16), split into E4M3 hi + lo
    int tree_tmem;  // 1: some CTA holds several leaves (the subtree stack lives in TMEM)
};

// Launches the warp-MMA kernel; returns an smd_status.
int launch_mma(const CallArgs& a, const MmaConfig& cfg, cudaStream_t stream);

// tcgen05 kernel: a CTA holds all heads of a 128-head group and at most
// kTcMaxKeys keys of a row (their logits fill the 512 TMEM columns).
constexpr int kTcHeads = 128;
constexpr int kTcChunk = 128;    // keys per gathered chunk
constexpr int kTcMaxKeys = 512;  // keys per CTA
constexpr int kTcMaxSplit = 4;   // CTAs per cluster (the merge inbox must fit)
constexpr int kTcThreads = 512;

// L2 exchange workspace of the tcgen05 kernel: one slot per SM id (%smid <
// kTcWsSlots), each holding a CTA's FP32 partials of the other owners'
// columns: (split - 1) x 128 heads x (512 / split) floats, at most 3 x 128 x 128.
constexpr int kTcWsSlots = 256;
constexpr int kTcWsSlotFloats = 3 * 128 * 128;
constexpr int64_t kTcWsBytes = static_cast<int64_t>(kTcWsSlots) * kTcWsSlotFloats * 4;

struct TcConfig {
    int split;
    uint64_t wait_budget_ns;
    int inject_stall;
    float* ws;     // exchange workspace or null (on-chip exchange)
    int ws_slots;  // SM-id slots in ws (0: kTcWsSlots)
};

// Row-group warp-MMA kernel: G consecutive rows that share one index list
// (each reads a prefix of it) go through one gather; a CTA takes 16 heads of
// each of the G rows (G tiles) and its share of the group's longest list.
constexpr int kGroupMaxSplit = 16;
constexpr int kGroupMaxKeys = 2048;  // keys per CTA (index staging)

struct GroupLayout {
    int32_t ring, q, lg, probs, overlay_end;  // inbox of the partials overlays [0, overlay_end)
    int32_t idx, sums, maxima, wmax, lsum, rowmax, nrow, flags, lstk, tslot, bars;
    int32_t total;
};

// lg: logits of the current chunk, [16 G][72] fp32; probs: its E4M3 P, [16 G][80].
__host__ __device__ inline GroupLayout group_layout(int G, int split, int nslots, int key_cap) {
    GroupLayout L{};
    const int ch = kHeadsPerTile * G;
    int32_t o = 0;
    L.ring = o;
    o += nslots * kChunk * kRowPitch;
    L.q = o;
    o += ch * kRowPitch;
    L.lg = o;
    o += ch * (kChunk + 8) * 4;
    L.probs = o;
    o += ch * (kChunk + 16);
    o = align_up(o, 16);
    const int32_t inbox = ch * kLatent * 4;  // split x ch x (512 / split) fp32
    L.overlay_end = o > inbox ? o : inbox;
    o = L.overlay_end;
    L.idx = o;
    o += key_cap * 4;
    L.sums = o;    // [split][ch]
    o += split * ch * 4;
    L.maxima = o;  // [split][ch]
    o += split * ch * 4;
    L.wmax = o;    // [4 key groups][ch]
    o += 4 * ch * 4;
    L.lsum = o;
    o += ch * 4;
    L.rowmax = o;
    o += ch * 4;
    L.nrow = o;    // [G] clamped counts
    o += 16;
    L.flags = o;   // words the peers' "free" signals write
    o += 16;
    L.lstk = o;    // [4 levels][ch] the sums' subtree stack (the leaf tree)
    o += 4 * ch * 4;
    L.tslot = o;   // the TMEM address of the partials' subtree stack
    o += 16;
    o = align_up(o, 8);
    L.bars = o;    // ring slots, q, maxima, inbound, peers free
    o += 8 * (nslots + 4);
    L.total = align_up(o, 128);
    return L;
}

struct GroupConfig {
    int G, split, nslots, key_cap;
    GroupLayout layout;
    uint64_t wait_budget_ns;
    int inject_stall;
    int tree_tmem;  // 1: some CTA holds several leaves (the subtree stack lives in TMEM)
};

// Launches the row-group kernel; returns an smd_status.
int launch_group(const CallArgs& a, const GroupConfig& cfg, cudaStream_t stream);

// Row groups on the tcgen05 kernel: a CTA takes all H heads of the G rows
// (G * H = 32 or 64 TMEM lanes) and at most 512 keys of the group's longest
// list; clusters of up to 16 CTAs.
constexpr int kTcgMaxSplit = 16;

struct TcgConfig {
    int G, split;
    uint64_t wait_budget_ns;
    int inject_stall;
};

int launch_tcg(const CallArgs& a, const TcgConfig& cfg, cudaStream_t stream);

// Dynamic shared memory of the tcgen05 row-group kernel (bytes).
int tcg_smem_bytes();

// tcgen05 kernel with a row's keys spread over any CTAs of a cooperative grid:
// a unit (row, 128-head group) of n keys becomes ceil(n / 512) items; maxima
// and FP32 partials are exchanged through a global workspace.
constexpr int kTcsMaxUnits = 1024;  // B * ceil(H / 128)
constexpr int kTcsMaxPieces = 32;   // items per unit: W <= 32 * 512

// Byte offsets of the workspace parts for `items` item slots.
struct TcsWorkspace {
    int64_t flag_part;  // [items][kTcsMaxPieces] u64: its partial for owner j is written
    int64_t max;        // [items][128] u64: the call's tag (high half) and an fp32 maximum (low)
    int64_t sum;        // [items][128] fp32
    int64_t part;       // [items][128 x 512] fp32 partials, 16-byte units head-innermost
    int64_t q_hi, q_lo; // [qrows][576] E4M3: the split bf16 query (qrows = B * H, else 0)
    int64_t lamh;       // [qrows] fp32: each query row's logit scale
    int64_t total;
};

__host__ __device__ inline int64_t align_up64(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline TcsWorkspace tcs_workspace(int64_t items, int64_t qrows = 0) {
    TcsWorkspace w{};
    int64_t o = 0;
    w.flag_part = o;
    o = align_up64(o + items * kTcsMaxPieces * 8, 256);
    w.max = o;
    o = align_up64(o + items * 128 * 8, 256);
    w.sum = o;
    o = align_up64(o + items * 128 * 4, 256);
    w.part = o;
    o = align_up64(o + items * 128 * kLatent * 4, 256);
    w.q_hi = o;
    o = align_up64(o + qrows * kRow, 256);
    w.q_lo = o;
    o = align_up64(o + qrows * kRow, 256);
    w.lamh = o;
    o = align_up64(o + qrows * 4, 256);
    w.total = o;
    return w;
}

struct TcsConfig {
    int G;          // rows per unit (row groups sharing one index list; 1 = per row)
    int grid;       // CTAs (at most the resident CTAs of the device)
    int items_cap;  // item slots in the workspace: units * ceil(W / 512)
    int qsplit;     // 1: bf16 query (CallArgs::q16), split into the workspace first
    uint64_t wait_budget_ns;
    int inject_stall;
    void* ws;
};

int launch_tcs(const CallArgs& a, const TcsConfig& cfg, cudaStream_t stream);

// Dynamic shared memory of the spread kernel (bytes).
int tcs_smem_bytes();

// CTAs of the spread kernel the current device holds at once (0 on failure).
int tcs_max_grid();

// Top-k select over bf16 logits (a cluster of C CTAs per row, C a power of
// two <= 8); returns an smd_status.
int launch_topk(const uint16_t* logits, int64_t stride, const int32_t* row_ends, int32_t B,
                int32_t L, int32_t K, int32_t* indices, int32_t* counts, int32_t* status,
                int C, cudaStream_t stream);

// SM-id slots of the library's own static exchange scratch (GB300: 152 SMs).
constexpr int kStaticScratchSlots = 160;

// Device address of the static exchange scratch on the current device (looked
// up once per device); null with *rc set on failure.
float* static_scratch(int* rc);

// Dynamic shared memory of the tcgen05 kernel (bytes).
int tc_smem_bytes();
// Copies (or zeroes, `clear`) a kernel's phase-stamp table of a tracing build
// (smd_trace.cuh); SMD_ERR_PLAN in the normal build.
int mma_trace_copy(uint64_t* host, int n, bool clear);
int tc_trace_copy(uint64_t* host, int n, bool clear);
int tcs_trace_copy(uint64_t* host, int n, bool clear);
// Clusters of `split` tcgen05 CTAs (one per SM) the current device holds at
// once; 0 when the query fails (no device).
int tc_resident_clusters(int split);

// A 2D tensor map over rows of 576 bytes (query or cache rows) with a box of
// box_cols x box_rows (128 columns: 128-byte swizzle; 64: 64-byte swizzle),
// from a small cache keyed by (ptr, rows, box). False if encoding failed.
bool encode_row_map(CUtensorMap* out, const void* ptr, uint64_t rows, uint32_t box_cols,
                    uint32_t box_rows);

// Launches the tcgen05 kernel; returns an smd_status.
int launch_tc(const CallArgs& a, const TcConfig& cfg, cudaStream_t stream);

}  // namespace smd
