// The chunk pipeline shared by the tcgen05 kernels (per row and per row
// group): a CTA holds up to 128 TMEM lanes (heads) and at most 512 keys; its
// keys pass through a two-slot ring of 128-key chunks gathered by TMA
// tile::gather4 (four 128-byte column blocks in the 128-byte swizzle plus the
// 64-byte tail in the 64-byte swizzle), S = Q K^T goes to TMEM columns
// 128c .. 128c + 127, and after P is formed O = P V goes to TMEM columns
// 0 .. 511, V read MN-major from the gathered tiles (chunks that left the ring
// are gathered again, V columns only).
#pragma once

#include <cuda.h>

#include <cstdint>

#include "smd_internal.h"
#include "smd_ptx.cuh"

namespace smd {
namespace tcc {

constexpr int kBlock = 16384;              // one 128-byte-wide column block of 128 rows (SW128)
constexpr int kTail = 8192;                // the 64-byte tail block of 128 rows (SW64)
constexpr int kTile = 4 * kBlock + kTail;  // 576 columns x 128 rows

// Shared-memory addresses and barriers of one CTA's pipeline.
//
// Split query (q_lo != 0): the query's hi tile is at q and its lo tile fills
// ring slot 1 until QK is done, so pass A gathers every chunk into slot 0
// (one chunk in flight) and QK adds the lo products; pass B finds chunk
// nch - 1 resident in slot 0 and brings the others back into slot
// (nch - 1 - c) & 1. Otherwise chunk c uses slot c & 1 in both passes and
// the last two chunks are resident after pass A.
struct Pipe {
    uint32_t q;       // the query tile, later the P tiles (chunk c at q + c * kBlock)
    uint32_t q_lo;    // the split query's lo tile (ring slot 1), or 0
    uint32_t ring;    // two chunk slots of kTile bytes
    uint32_t full;    // [2] a slot's gathers have landed
    uint32_t empty;   // [2] pass A: QK has left a slot
    uint32_t free_b;  // [2] pass B: PV has left a slot
    uint32_t s;       // [4] QK of chunk c is complete
    uint32_t bar_q, bar_p, bar_o;  // query tile landed; P formed; O complete
    const int32_t* idx;            // this CTA's keys (entries past them name pool row 0)
    int32_t* status;
    uint64_t budget_ns;
};

// Waits for the next completion of a barrier whose completions this thread
// counts in `seen`.
__device__ __forceinline__ void wait_next(uint32_t bar, uint32_t& seen, bool& ok, int32_t* status,
                                          uint64_t budget) {
    mbar_wait(bar, seen & 1u, ok, status, budget);
    ++seen;
}

// Slot of chunk c in pass A and in pass B (see Pipe).
__device__ __forceinline__ int slot_a(const Pipe& pp, int c) { return pp.q_lo ? 0 : (c & 1); }
__device__ __forceinline__ int slot_b(const Pipe& pp, int c, int nch) {
    return pp.q_lo ? ((nch - 1 - c) & 1) : (c & 1);
}
// Chunks pass B finds resident (the last ones gathered in pass A).
__device__ __forceinline__ int resident_b(const Pipe& pp) { return pp.q_lo ? 1 : 2; }

// The producers are warps 0-7 (256 threads). A warp's TMA issues run one
// after another, so a chunk's gathers are spread over all eight warps: lanes
// 0..P-1 of warp w issue ops P w .. P w + P - 1 (P = 20 in pass A, 16 in
// pass B).
constexpr int kIssueA = 20;  // 160 gather4 ops per 128-key chunk (32 row quads x 5 pieces)
constexpr int kIssueB = 16;  // 128 ops per chunk in pass B (32 row quads x 4 V blocks)

// Producer warps, pass A, chunks [c_begin, c_end): chunk c goes to its slot
// once QK of the chunk before it in that slot has left; op o < 160 is
// piece o % 5 of rows 4g .. 4g + 3, g = o / 5. `seen` counts the "empty"
// completions.
__device__ __forceinline__ void gather_pass_a(const CUtensorMap& kv, const CUtensorMap& kv_tail,
                                              const Pipe& pp, int c_begin, int c_end,
                                              uint32_t (&seen)[2], bool& ok) {
    const int t = threadIdx.x;
    const int lane = t & 31, o = kIssueA * (t >> 5) + lane;
    for (int c = c_begin; c < c_end && ok; ++c) {
        const int s = slot_a(pp, c);
        const uint32_t need = static_cast<uint32_t>(pp.q_lo ? c : (c >> 1));
        while (seen[s] < need) wait_next(pp.empty + 8 * s, seen[s], ok, pp.status, pp.budget_ns);
        if (!ok) break;
        const uint32_t slot = pp.ring + s * kTile;
        const uint32_t full = pp.full + 8 * s;
        if (t == 0) mbar_arrive_expect_tx(full, kTile);
        if (lane < kIssueA) {
            const int g = o / 5, j = o % 5;
            const int32_t* rw = pp.idx + kTcChunk * c + 4 * g;
            if (j < 4)
                tma_gather4(slot + j * kBlock + 4 * g * 128, &kv, 128 * j, rw[0], rw[1], rw[2], rw[3], full);
            else
                tma_gather4(slot + 4 * kBlock + 4 * g * 64, &kv_tail, 512, rw[0], rw[1], rw[2], rw[3], full);
        }
    }
}

// Producer warps, pass B: chunks in descending order; the resident ones stay,
// the others come back (V columns only) into their slot once PV of the chunk
// two above has released it (a slot that held no chunk is free at once).
__device__ __forceinline__ void gather_pass_b(const CUtensorMap& kv, const Pipe& pp, int nch,
                                              bool& ok) {
    const int t = threadIdx.x;
    const int lane = t & 31, o = kIssueB * (t >> 5) + lane;
    uint32_t seen_b[2] = {0u, 0u};  // completions of the pass-B "slot free" barriers seen
    for (int c = nch - 1 - resident_b(pp); c >= 0 && ok; --c) {
        const int s = slot_b(pp, c, nch);
        int freed = 0;  // pass-B completions on slot s up to PV(c + 2), its previous chunk
        for (int c2 = nch - 1; c2 >= c + 2; --c2) freed += (slot_b(pp, c2, nch) == s);
        const uint32_t need = static_cast<uint32_t>(freed);
        while (seen_b[s] < need) wait_next(pp.free_b + 8 * s, seen_b[s], ok, pp.status, pp.budget_ns);
        if (!ok) break;
        const uint32_t slot = pp.ring + s * kTile;
        const uint32_t full = pp.full + 8 * s;
        if (t == 0) mbar_arrive_expect_tx(full, 4 * kBlock);
        if (lane < kIssueB) {
            const int g = o / 4, j = o % 4;
            const int32_t* rw = pp.idx + kTcChunk * c + 4 * g;
            tma_gather4(slot + j * kBlock + 4 * g * 128, &kv, 128 * j, rw[0], rw[1], rw[2], rw[3], full);
        }
    }
}

// MMA issuer (one lane), pass A: S_c = Q K_c^T into TMEM columns 128c .. + 127
// (18 x M128 N128 K32 E4M3 MMAs; 36 with the split query's lo tile),
// committing to "QK done" and "slot empty". `full_seen` counts the slots'
// "full" completions (pass B continues it).
__device__ __forceinline__ void mma_qk(const Pipe& pp, uint32_t tmem, int nch,
                                       uint32_t (&full_seen)[2], bool& ok) {
    mbar_wait(pp.bar_q, 0, ok, pp.status, pp.budget_ns);
    tc_fence_after();
    constexpr uint32_t kIdQK = umma_idesc_e4m3(128, kTcChunk, 0);
    for (int c = 0; c < nch && ok; ++c) {
        const int s = slot_a(pp, c);
        wait_next(pp.full + 8 * s, full_seen[s], ok, pp.status, pp.budget_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t slot = pp.ring + s * kTile;
        const uint32_t d = tmem + kTcChunk * c;
        uint32_t acc = 0;
        for (int part = 0; part < (pp.q_lo ? 2 : 1); ++part) {  // hi, then the split query's lo
            const uint32_t qa = part ? pp.q_lo : pp.q;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    umma_e4m3(d, umma_desc(qa + j * kBlock + 32 * kk, 16, 1024, 2),
                              umma_desc(slot + j * kBlock + 32 * kk, 16, 1024, 2), kIdQK, acc);
                    acc = 1;
                }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
                umma_e4m3(d, umma_desc(qa + 4 * kBlock + 32 * kk, 16, 512, 4),
                          umma_desc(slot + 4 * kBlock + 32 * kk, 16, 512, 4), kIdQK, 1);
        }
        umma_commit(pp.s + 8 * c);
        umma_commit(pp.empty + 8 * s);
    }
}

// MMA issuer, pass B, once P is formed: O = sum_c P_c V_c, chunks in
// descending order, into TMEM columns 0..511 (two N = 256 halves). V is the
// MN-major operand: 128-byte latent chunks one column block (16 KB) apart,
// 8-key groups 1 KB apart.
__device__ __forceinline__ void mma_pv(const Pipe& pp, uint32_t tmem, int nch, int mine,
                                       uint32_t (&full_seen)[2], bool& ok) {
    constexpr uint32_t kIdPV = umma_idesc_e4m3(128, 256, 1);
    mbar_wait(pp.bar_p, 0, ok, pp.status, pp.budget_ns);
    tc_fence_after();
    for (int c = nch - 1; c >= 0 && ok; --c) {
        const int s = slot_b(pp, c, nch);
        if (c < nch - resident_b(pp)) {
            wait_next(pp.full + 8 * s, full_seen[s], ok, pp.status, pp.budget_ns);
            if (!ok) break;
            tc_fence_after();
        }
        const uint32_t slot = pp.ring + s * kTile;
        const uint32_t p_tile = pp.q + c * kBlock;
        const int cnt = min(kTcChunk, mine - kTcChunk * c);
        const int ksteps = (cnt + 31) / 32;
        for (int ks = 0; ks < ksteps; ++ks) {
            const uint32_t acc = (c == nch - 1 && ks == 0) ? 0u : 1u;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                umma_e4m3(tmem + 256 * h, umma_desc(p_tile + 32 * ks, 16, 1024, 2),
                          umma_desc(slot + 2 * h * kBlock + ks * 4096, kBlock, 1024, 2), kIdPV, acc);
        }
        umma_commit(pp.free_b + 8 * s);
    }
    umma_commit(pp.bar_o);
}

}  // namespace tcc
}  // namespace smd
