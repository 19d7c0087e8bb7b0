// Sparse MLA decode, warp-level FP8 tensor-core kernel (sm_103a).
//
// One CTA takes (query row b, 16*T heads, its share of the row's keys); the
// S CTAs of a thread-block cluster split the row's keys as the attn_sparse
// page's SparseDcpDecode does, with the split points at leaf boundaries: the
// row's keys form leaves of 64 * ceil(n / 1024) keys (at most 16) and CTA s takes
// an aligned block of a power of two of them (smd_tree.cuh). The partials
// merge over distributed shared memory in FP32 (the page's merge method:
// column ownership), by the fixed pairwise tree over the leaves, so that the
// bits do not depend on S: each leaf's P V and sums of P are formed from
// zero, the subtrees of the leaves a CTA has done wait in TMEM (which this
// kernel does not otherwise use), and the owner adds the CTAs' subtrees by
// the same tree.
//
// Precision follows the page's "Precision" paragraph with the P anchor at the
// maximum over the WHOLE row: the CTAs first compute all their logits (pass
// A), exchange their maxima across the cluster, and only then form
// P = 2^(s - m + log2 448) in E4M3 and run PV (pass B). Per head, every
// reduction runs in a fixed order that depends neither on timing nor on the
// number of 16-head tiles a CTA takes.
//
// The keys pass through a ring of 64-key slots. Pass A per chunk: the
// 576-byte cache rows come into shared memory as 16-byte cp.async copies
// spread over all threads (one mbarrier per slot, one arrival per thread),
// issued a ring's length ahead of their use; QK is mma.sync m16n8k32 E4M3 x
// E4M3 -> FP32 over the 576 columns (a warp job is 16 heads x 16 keys, two
// accumulation chains per 8 keys over the 18 k-steps); the scaled logits go
// to shared memory. Pass B per chunk, descending: P for 64 keys of a
// head per warp (lane: a key pair, stored as an E4M3 pair), the FP32 sum of
// the unquantized P by a fixed butterfly, then PV: warp w owns latent columns
// 32w..32w+31, V read as words and byte-transposed in registers into the MMA's
// B fragments. Rows past the count up to the 32-key step are zeroed so that a
// zero P never meets a NaN byte pattern.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "smd_internal.h"
#include "smd_ptx.cuh"
#include "smd_qsplit.cuh"
#include "smd_trace.cuh"
#include "smd_tree.cuh"

namespace smd {

namespace {

constexpr int kMaxDevices = 64;

struct MmaParams {
    CallArgs a;
    int32_t split, window, key_cap;
    MmaLayout L;
    float log2_448;
    uint64_t budget_ns;  // bound of every wait
    int32_t inject_stall;
    int32_t spec_idx;    // 1: load the row's whole index list with the count
    int32_t tree_tmem;   // 1: a CTA may hold several leaves (TMEM subtree stack)
};

// Issues the gathers of one chunk of `cnt` <= 64 keys (`keys`: their pool
// rows) into a ring slot: `bytes` of each row (576 for QK + PV, 512 when only
// V is needed), as 16-byte copies spread over all threads. Every thread
// arrives on the slot's barrier once its copies have landed. Rows
// [cnt, roundup32(cnt)) are zeroed.
__device__ __forceinline__ void gather_chunk(const MmaParams& p, uint32_t slot_s,
                                             const int32_t* keys, uint32_t bar, int cnt,
                                             uint32_t bytes) {
    // Warp w copies rows w, w + 16, ...; lane l the row's 16-byte pieces l
    // and l + 32 (36 pieces per 576-byte row, 32 per 512-byte V row).
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per_row = static_cast<int>(bytes) / 16;
    for (int r = warp; r < cnt; r += kMmaThreads / 32) {
        const uint8_t* src = p.a.kv + static_cast<int64_t>(keys[r]) * kRow;
        const uint32_t dst = slot_s + r * kRowPitch;
        cp_async16(dst + 16 * lane, src + 16 * lane);
        if (lane + 32 < per_row) cp_async16(dst + 16 * (lane + 32), src + 16 * (lane + 32));
    }
    cp_async_arrive(bar);
    const int span = (cnt + 31) & ~31;
    for (int e = cnt * (kRow / 16) + threadIdx.x; e < span * (kRow / 16); e += kMmaThreads) {
        const int r = e / (kRow / 16), c16 = e % (kRow / 16);
        sts_zero16(slot_s + r * kRowPitch + 16 * c16);
    }
}

// The split query: warp w takes heads w, w + 16, ... of the CTA's CH into the
// two query tiles (rows kRowPitch apart) and their logit scales.
template <int CH>
__device__ __forceinline__ void split_query(const MmaParams& p, int b, int head0, uint8_t* q_hi,
                                            uint8_t* q_lo, float* lamh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int hh = warp; hh < CH; hh += kMmaThreads / 32) {
        const float lam = split_query_row(p.a.q16 + (static_cast<int64_t>(b) * p.a.H + head0 + hh) * kRow,
                                          q_hi + hh * kRowPitch, q_lo + hh * kRowPitch,
                                          p.a.scale_log2);
        if (lane == 0) lamh[hh] = lam;
    }
}

// Frees the subtree stack's TMEM once every thread is past its last use
// (warp 0 allocated it).
__device__ __forceinline__ void release_tmem(uint32_t tbase) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        tc_fence_after();
        tmem_free(tbase, 512);
    }
}

SMD_TRACE_TABLE(g_trace_mma);

// TR: some CTA of the plan holds several leaves (p.tree_tmem), so the kernel
// keeps a subtree stack in TMEM; without it every CTA's keys form one leaf and
// no TMEM is touched.
template <int T, bool QS, bool TR>
__global__ void __launch_bounds__(kMmaThreads, 1) mma_decode_kernel(const MmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_entry();
    // Tracing build: phase ends of CTA `trow` (stamps 0 entry, 1 keys staged,
    // 2 query landed, 3 logits, 4 row maximum, 5 PV, 6 partials in, 7 end).
    const int trow = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x);
    if (threadIdx.x == 0) {
        SMD_STAMP(g_trace_mma, trow, 0);
        SMD_TRACE_SM(g_trace_mma, trow);
    }
    constexpr int CH = kHeadsPerTile * T;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, qd = lane & 3;
    const int S = p.split;
    const int split = static_cast<int>(cluster_ctarank());
    const int tile_group = blockIdx.x / S;
    const int b = blockIdx.y;
    const int head0 = tile_group * CH;

    const uint32_t base = smem_addr(smem);
    const uint32_t kv_s = base + p.L.kv;
    const uint32_t q_s = base + p.L.q;
    const uint32_t prob_s = base + p.L.probs;
    float* logits = reinterpret_cast<float*>(smem + p.L.logits);
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + p.L.idx);
    float* inbox = reinterpret_cast<float*>(smem + p.L.inbox);
    float* sums = reinterpret_cast<float*>(smem + p.L.sums);
    float* maxima = reinterpret_cast<float*>(smem + p.L.maxima);
    float* wmax = reinterpret_cast<float*>(smem + p.L.wmax);
    float* lsum = reinterpret_cast<float*>(smem + p.L.lsum);
    float* rowmax = reinterpret_cast<float*>(smem + p.L.rowmax);
    float* lstk = reinterpret_cast<float*>(smem + p.L.lstk);
    const int nchunk_bars = p.window / kChunk;
    const uint32_t bars = base + p.L.bars;
    const uint32_t q_bar = bars + 8 * nchunk_bars;
    const uint32_t max_bar = q_bar + 8;
    const uint32_t in_bar = q_bar + 16;
    const int LP = p.L.logit_pitch, PP = p.L.prob_pitch;
    const int CW = kLatent / S;  // latent columns this CTA merges

    bool ok = true;
    int32_t* status = p.a.status;

    // The row's count and (when the row is at most kSpecIdxMaxW wide) its whole
    // index list are loaded first, in one round trip that the setup below
    // overlaps; the loads do not depend on each other.
    const int W = p.a.W;
    const int32_t* row_idx = p.a.indices + static_cast<int64_t>(b) * W;
    int n = p.a.counts[b];
    constexpr int kSpecPerThread = kSpecIdxMaxW / kMmaThreads;
    int32_t spec[kSpecPerThread];
#pragma unroll
    for (int k = 0; k < kSpecPerThread; ++k) {
        const int i = tid + k * kMmaThreads;
        spec[k] = (p.spec_idx && i < W) ? row_idx[i] : 0;
    }

    if (tid == 0) {
        for (int c = 0; c < nchunk_bars; ++c) mbar_init(bars + 8 * c, kMmaThreads);
        // E4M3 query: every thread's 16-byte copies arrive, and thread 0's
        // expect-tx below (0 bytes, or the stall hook's 16).
        mbar_init(q_bar, QS ? 1 : 1 + kMmaThreads);
        mbar_init(max_bar, 1);
        mbar_init(in_bar, 1);
        fence_mbar_init();
        // Bytes the peers will push into this CTA: their maxima, and their
        // partials of this CTA's columns plus their sums.
        mbar_arrive_expect_tx(max_bar, (S - 1) * CH * 4);
        mbar_arrive_expect_tx(in_bar, (S - 1) * (CH * CW * 4 + CH * 4));
        // (inject_stall: the barrier also expects 16 bytes nobody sends, so
        // the bounded wait below runs out; a test hook for the timeout path.)
        mbar_arrive_expect_tx(q_bar, p.inject_stall ? 16 : 0);
    }
    for (int h = tid; h < CH; h += kMmaThreads) lsum[h] = 0.f;
    uint32_t tbase = 0u;
    if constexpr (TR) {
        if (warp == 0) tmem_alloc(base + p.L.tslot, 512);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tbase = *reinterpret_cast<volatile uint32_t*>(smem + p.L.tslot);
    } else {
        __syncthreads();
    }
    // Every CTA's barriers are armed before any peer pushes (waited below).
    if (S > 1) cluster_arrive_relaxed();

    // The query rows depend on nothing: their copies go first.
    float* lamh = reinterpret_cast<float*>(smem + p.L.lamh);
    if constexpr (QS) {
        split_query<CH>(p, b, head0, smem + p.L.q, smem + p.L.q + CH * kRowPitch, lamh);
    } else {
        // 16-byte copies through the load/store unit (the query may be mapped
        // host memory), spread over all threads; each thread arrives once its
        // own have landed.
        const uint8_t* src = p.a.q + (static_cast<int64_t>(b) * p.a.H + head0) * kRow;
        for (int e = tid; e < CH * (kRow / 16); e += kMmaThreads) {
            const int r = e / (kRow / 16), c16 = e - r * (kRow / 16);
            cp_async16(q_s + r * kRowPitch + 16 * c16, src + r * kRow + 16 * c16);
        }
        cp_async_arrive(q_bar);
    }

    // ---- this CTA's keys: [first, first + mine) of the row ------------------
    // With spec_idx the index list came with the count, so the gathers wait
    // for one DRAM latency instead of two.
    if (p.spec_idx) {
#pragma unroll
        for (int k = 0; k < kSpecPerThread; ++k) {
            const int i = tid + k * kMmaThreads;
            if (i < W) idx_s[i] = spec[k];
        }
    }
    n = max(min(n, W), 0);
    const int leaf = mma_leaf(n);
    const int lpc = mma_leaves_per_cta(n, S);
    const int first = min(n, split * lpc * leaf);
    const int mine = min(n - first, lpc * leaf);
    if (!p.spec_idx)
        for (int i = tid; i < mine; i += kMmaThreads) idx_s[i] = row_idx[first + i];
    const int32_t* my_idx = idx_s + (p.spec_idx ? first : 0);
    __syncthreads();
    if (tid == 0) SMD_STAMP(g_trace_mma, trow, 1);

    const float neg_inf = -INFINITY;
    const float lam = p.a.scale_log2;
    // The KV buffer is a ring of NS slots of 64 keys; chunk c (keys
    // 64c .. 64c + 63 of this CTA) goes to slot c % NS.
    const int NS = p.window / kChunk;
    const int nch = (mine + kChunk - 1) / kChunk;
    // Parity of the next completion of each slot's barrier (bit s: slot s).
    uint32_t phase_bits = 0;

    // ldmatrix lane addressing: A (16 rows x 32 B), B (8 keys x 64 B).
    const int a_row = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int a_col = 16 * (lane >> 4);

    mbar_wait(q_bar, 0, ok, status, p.budget_ns);
    if (tid == 0) SMD_STAMP(g_trace_mma, trow, 2);

    // The maximum of each QK job's logits (heads g and g + 8 of its tile over
    // its keys), kept as the logits are written; warp w has job w (4T <= 16).
    float jmax[2] = {-INFINITY, -INFINITY};

    // ================================ pass A: logits =========================
    // The gather of chunk c + NS is issued as soon as QK of chunk c has left
    // its slot, so copies and QK overlap.
    for (int c = 0; c < min(NS, nch); ++c)
        gather_chunk(p, kv_s + c * kChunk * kRowPitch, my_idx + c * kChunk, bars + 8 * c,
                     min(kChunk, mine - c * kChunk), kRow);
    for (int c = 0; c < nch; ++c) {
        const int s = c % NS;
        const int cnt = min(kChunk, mine - c * kChunk);
        const uint32_t slot_s = kv_s + s * kChunk * kRowPitch;
        mbar_wait(bars + 8 * s, (phase_bits >> s) & 1u, ok, status, p.budget_ns);
        phase_bits ^= 1u << s;
        // Warp job: 16 heads (tile t) x 16 keys (two 8-key n-tiles), so each
        // query fragment read from shared memory serves two MMAs; per n-tile
        // two accumulation chains (the two 32-byte halves of every 64-byte
        // k-step), added once at the end.
        for (int job = warp; job < 4 * T; job += kMmaThreads / 32) {
            const int t = job >> 2, kg = job & 3;
            if (16 * kg >= cnt) continue;
            float c0[2][4] = {}, c1[2][4] = {};
            const uint32_t kaddr = slot_s + (16 * kg + (lane & 7)) * kRowPitch + 16 * (lane >> 3);
            const uint32_t qaddr = q_s + (16 * t + a_row) * kRowPitch + a_col;
#pragma unroll
            for (int kp = 0; kp < kRow / 64; ++kp) {
                uint32_t kb0[4], kb1[4], qa[4], qb[4];
                ldsm_x4(qaddr + 64 * kp, qa);
                ldsm_x4(qaddr + 64 * kp + 32, qb);
                ldsm_x4(kaddr + 64 * kp, kb0);
                ldsm_x4(kaddr + 8 * kRowPitch + 64 * kp, kb1);
                mma_e4m3(c0[0], qa, kb0[0], kb0[1]);
                mma_e4m3(c1[0], qb, kb0[2], kb0[3]);
                mma_e4m3(c0[1], qa, kb1[0], kb1[1]);
                mma_e4m3(c1[1], qb, kb1[2], kb1[3]);
                if constexpr (QS) {  // the lo tile into the same accumulators
                    ldsm_x4(qaddr + CH * kRowPitch + 64 * kp, qa);
                    ldsm_x4(qaddr + CH * kRowPitch + 64 * kp + 32, qb);
                    mma_e4m3(c0[0], qa, kb0[0], kb0[1]);
                    mma_e4m3(c1[0], qb, kb0[2], kb0[3]);
                    mma_e4m3(c0[1], qa, kb1[0], kb1[1]);
                    mma_e4m3(c1[1], qb, kb1[2], kb1[3]);
                }
            }
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int kk = 16 * kg + 8 * n + 2 * qd;  // within the chunk
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float lr = QS ? lamh[16 * t + g + 8 * r] : lam;
                    const float s0 = (kk < cnt) ? lr * (c0[n][2 * r] + c1[n][2 * r]) : neg_inf;
                    const float s1 =
                        (kk + 1 < cnt) ? lr * (c0[n][2 * r + 1] + c1[n][2 * r + 1]) : neg_inf;
                    float2* dst = reinterpret_cast<float2*>(
                        logits + (16 * t + g + 8 * r) * LP + c * kChunk + kk);
                    *dst = make_float2(s0, s1);
                    jmax[r] = fmaxf(jmax[r], fmaxf(s0, s1));
                }
            }
        }
        // The slot is free; a failed CTA issues no more copies.
        if (!__syncthreads_and(ok)) break;
        if (c + NS < nch)
            gather_chunk(p, slot_s, my_idx + (c + NS) * kChunk, bars + 8 * s,
                         min(kChunk, mine - (c + NS) * kChunk), kRow);
    }

    // ---- the row maximum over the cluster ------------------------------------
    if (tid == 0) SMD_STAMP(g_trace_mma, trow, 3);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        jmax[r] = fmaxf(jmax[r], __shfl_xor_sync(0xffffffffu, jmax[r], 1));
        jmax[r] = fmaxf(jmax[r], __shfl_xor_sync(0xffffffffu, jmax[r], 2));
    }
    if (warp < 4 * T && qd == 0) {
        const int t = warp >> 2, kg = warp & 3;
        wmax[kg * CH + 16 * t + g] = jmax[0];
        wmax[kg * CH + 16 * t + g + 8] = jmax[1];
    }
    __syncthreads();
    for (int h = tid; h < CH; h += kMmaThreads)
        maxima[split * CH + h] =
            fmaxf(fmaxf(wmax[h], wmax[CH + h]), fmaxf(wmax[2 * CH + h], wmax[3 * CH + h]));
    __syncthreads();
    if (S > 1) {
        cluster_wait();  // peers' barriers are initialised
        if (tid < CH) {
            const uint32_t v = __float_as_uint(maxima[split * CH + tid]);
            const uint32_t slot = smem_addr(maxima + split * CH + tid);
            for (int pr = 0; pr < S; ++pr)
                if (pr != split) st_async_b32(mapa(slot, pr), v, mapa(max_bar, pr));
        }
        mbar_wait(max_bar, 0, ok, status, p.budget_ns, /*always=*/true);
    }
    if (tid == 0) SMD_STAMP(g_trace_mma, trow, 4);
    for (int h = tid; h < CH; h += kMmaThreads) {
        float m = neg_inf;
        for (int pr = 0; pr < S; ++pr) m = fmaxf(m, maxima[pr * CH + h]);
        rowmax[h] = m;
    }
    __syncthreads();

    // ================================ pass B: P and PV =======================
    float acc[T][4][4];
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[t][j][e] = 0.f;

    // Chunks in descending order, so every row's chunks are summed in one
    // global order whatever the ring size: the last NS chunks are still
    // resident; chunk c - NS comes back (V columns only) into the slot of
    // chunk c once PV of chunk c has left it.
    //
    // Leaves: slot l of this CTA is chunks [l cpl, l cpl + cpl) of its keys,
    // walked downwards (the mirror of the tree, same bits). A leaf's P V is
    // summed from zero in acc and its sums of P in lsum; at its end it is
    // pushed: the stored subtrees along the binary counter's carry are added
    // (TMEM levels for acc, lstk for the sums), and the result is stored at the
    // first free level unless it is this CTA's root, which stays in acc / lsum.
    const int cpl = leaf / kChunk;
    int tcnt = nch > 0 ? lpc - 1 - (nch - 1) / cpl : lpc;  // leaves pushed: the absent slots
    uint32_t tpres = 0u;  // bit d: stack level d holds a subtree
    const uint32_t tcol = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 128u * (warp >> 2);
    for (int c = nch - 1; c >= 0; --c) {
        const int s = c % NS;
        const int cnt = min(kChunk, mine - c * kChunk);
        const uint32_t slot_s = kv_s + s * kChunk * kRowPitch;
        if (c < nch - NS) {
            mbar_wait(bars + 8 * s, (phase_bits >> s) & 1u, ok, status, p.budget_ns);
            phase_bits ^= 1u << s;
        }
        // V of the chunk, byte-transposed into MMA fragments, before P (it
        // does not depend on P): latent columns 32*warp + 4*g + (0..3).
        const int span = (cnt + 31) & ~31;
        uint32_t vb[kChunk / 32][2][4];
#pragma unroll
        for (int ks = 0; ks < kChunk / 32; ++ks) {
            if (32 * ks >= span) break;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int key = 32 * ks + 16 * hf + 4 * qd + i;
                    w[i] = lds_u32(slot_s + key * kRowPitch + 32 * warp + 4 * g);
                }
                byte_transpose4(w[0], w[1], w[2], w[3], vb[ks][hf]);
            }
        }
        // P of 64 keys x this warp's heads; lane: keys 2*lane, 2*lane + 1.
#pragma unroll
        for (int i = 0; i < T; ++i) {
            const int h = warp + 16 * i;
            const float bias = rowmax[h] - p.log2_448;
            const int kk = 2 * lane;
            const float2 sv = *reinterpret_cast<const float2*>(logits + h * LP + c * kChunk + kk);
            const float p0 = (kk < cnt) ? ex2_approx(sv.x - bias) : 0.f;
            const float p1 = (kk + 1 < cnt) ? ex2_approx(sv.y - bias) : 0.f;
            sts_u16(prob_s + h * PP + kk, e4m3x2(p0, p1));
            const float tot = warp_sum(p0 + p1);
            if (lane == 0) lsum[h] += tot;
        }
        __syncthreads();
        // PV: latent columns 32*warp + 4*g + (0..3), every tile.
#pragma unroll
        for (int ks = 0; ks < kChunk / 32; ++ks) {
            if (32 * ks >= span) break;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                uint32_t pa[4];
                ldsm_x4(prob_s + (16 * t + a_row) * PP + 32 * ks + a_col, pa);
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_e4m3(acc[t][j], pa, vb[ks][0][j], vb[ks][1][j]);
            }
        }
        if (TR && c % cpl == 0) {  // leaf c / cpl is complete (uniform)
            int d = 0;
            while ((tcnt >> d) & 1) {
                if ((tpres >> d) & 1u) {
                    stash_add<T>(tcol + 16u * T * d, acc);
                    if (lane == 0)
#pragma unroll
                        for (int i = 0; i < T; ++i) {
                            const int h = warp + 16 * i;
                            lsum[h] = lstk[d * CH + h] + lsum[h];
                        }
                }
                ++d;
            }
            tpres &= ~((1u << d) - 1u);
            if (++tcnt < lpc) {  // not the root: keep the subtree, start the next leaf at zero
                stash_store<T>(tcol + 16u * T * d, acc);
                if (lane == 0)
#pragma unroll
                    for (int i = 0; i < T; ++i) {
                        const int h = warp + 16 * i;
                        lstk[d * CH + h] = lsum[h];
                        lsum[h] = 0.f;
                    }
                tpres |= 1u << d;
#pragma unroll
                for (int t = 0; t < T; ++t)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[t][j][e] = 0.f;
            }
        }
        // The slot and P are free; a failed CTA issues no more copies.
        if (!__syncthreads_and(ok)) break;
        if (c - NS >= 0)
            gather_chunk(p, slot_s, my_idx + (c - NS) * kChunk, bars + 8 * s, kChunk, kLatent);
    }

    if (tid == 0) SMD_STAMP(g_trace_mma, trow, 5);
    if (S == 1) {
        // No peers: BF16(acc * k_scale / total) straight from the registers
        // (the same operations as the merge below with one partial).
        if (ok) {
#pragma unroll
            for (int t = 0; t < T; ++t) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = 16 * t + g + 8 * (e >> 1);
                    const int col = 32 * warp + 8 * qd + 4 * (e & 1);
                    const float total = lsum[h];
                    const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
                    uint2 packed;
                    packed.x = bf16x2(acc[t][0][e] * inv, acc[t][1][e] * inv);
                    packed.y = bf16x2(acc[t][2][e] * inv, acc[t][3][e] * inv);
                    uint16_t* dst =
                        p.a.out + (static_cast<int64_t>(b) * p.a.H + head0 + h) * kLatent + col;
                    *reinterpret_cast<uint2*>(dst) = packed;
                }
            }
            for (int h = tid; h < CH; h += kMmaThreads) {
                const float total = lsum[h];
                p.a.lse[static_cast<int64_t>(b) * p.a.H + head0 + h] =
                    total > 0.f ? (rowmax[h] - p.log2_448 + log2f(total)) * 0.69314718055994530942f
                                : -INFINITY;
            }
        }
        cp_async_wait_all();  // after a failed wait, no copy may land once the CTA is gone
        if constexpr (TR) release_tmem(tbase);
        if (tid == 0) SMD_STAMP(g_trace_mma, trow, 7);
        return;
    }

    // ---- partials to the column owners (FP32 bits over DSMEM) ----------------
    // acc[t][j][e]: head 16t + g + 8(e>>1), column 32*warp + 8*qd + 4*(e&1) + j.
    // The inbox holds 16-byte units (columns j = 0..3 of one (t, e, lane)):
    // unit ((((src * WPO + wl) * T + t) * 4 + e) * 32 + lane) for the partial
    // of CTA src from warp wl of the owner's WPO = CW / 32 column warps, so one
    // warp-wide store covers 512 contiguous bytes.
    const int WPO = CW / 32;
    {
        const int owner = warp / WPO;
        const int wl = warp - owner * WPO;
        const uint32_t inbox_s = smem_addr(inbox);
#pragma unroll
        for (int t = 0; t < T; ++t) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 v = make_float4(acc[t][0][e], acc[t][1][e], acc[t][2][e], acc[t][3][e]);
                const uint32_t dst = inbox_s + (((((split * WPO + wl) * T + t) * 4 + e) * 32) + lane) * 16;
                if (owner == split)
                    sts_v4(dst, v);
                else
                    st_async_v4(mapa(dst, owner), v, mapa(in_bar, owner));
            }
        }
        if (tid < CH) {
            const float l = lsum[tid];
            sums[split * CH + tid] = l;
            const uint32_t slot = smem_addr(sums + split * CH + tid);
            for (int pr = 0; pr < S; ++pr)
                if (pr != split) st_async_b32(mapa(slot, pr), __float_as_uint(l), mapa(in_bar, pr));
        }
    }
    mbar_wait(in_bar, 0, ok, status, p.budget_ns, /*always=*/true);
    __syncthreads();  // this CTA's own partial (plain stores)
    if (tid == 0) SMD_STAMP(g_trace_mma, trow, 6);

    // ---- merge by the leaf tree; BF16(sum * k_scale / total) -----------------
    // CTA src holds the subtree of leaves [src lpc, src lpc + lpc): absent if
    // they lie past the row's count.
    if (ok) {
        const int units = WPO * T * 128;  // 16-byte units of one CTA's partial of my columns
        const float4* in4 = reinterpret_cast<const float4*>(inbox);
        const int np = (mma_leaves(n) + lpc - 1) / lpc;  // CTAs 0 .. np - 1 hold keys
        for (int u = tid; u < units; u += kMmaThreads) {
            const int ln = u & 31, e = (u >> 5) & 3, t = (u >> 7) % T, wl = (u >> 7) / T;
            const int h = 16 * t + (ln >> 2) + 8 * (e >> 1);
            const int c = 32 * wl + 8 * (ln & 3) + 4 * (e & 1);
            const float4 m = tree_xor_n<float4>(S, [&](int k) { return in4[k * units + u]; }, 0, np);
            const float total = tree_xor_n<float>(S, [&](int k) { return sums[k * CH + h]; }, 0, np);
            const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
            uint2 packed;
            packed.x = bf16x2(m.x * inv, m.y * inv);
            packed.y = bf16x2(m.z * inv, m.w * inv);
            uint16_t* dst = p.a.out + (static_cast<int64_t>(b) * p.a.H + head0 + h) * kLatent +
                            split * CW + c;
            *reinterpret_cast<uint2*>(dst) = packed;
        }
        if (split == 0) {
            for (int h = tid; h < CH; h += kMmaThreads) {
                const float total =
                    tree_xor_n<float>(S, [&](int k) { return sums[k * CH + h]; }, 0, np);
                const float lse2 =
                    total > 0.f ? rowmax[h] - p.log2_448 + log2f(total) : neg_inf;
                p.a.lse[static_cast<int64_t>(b) * p.a.H + head0 + h] =
                    total > 0.f ? lse2 * 0.69314718055994530942f : neg_inf;
            }
        }
    }
    cp_async_wait_all();
    if constexpr (TR) release_tmem(tbase);
    if (tid == 0) SMD_STAMP(g_trace_mma, trow, 7);
}

// Function attributes are set once per device and kernel (and again only when
// a launch needs more shared memory than was granted before).
template <int T, bool QS, bool TR>
int ensure_attributes(int smem_bytes, bool nonportable) {
    static std::atomic<int> smem_set[kMaxDevices];
    static std::atomic<int> np_set[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMD_ERR_DEVICE;
    auto kern = mma_decode_kernel<T, QS, TR>;
    if (smem_bytes > smem_set[dev].load()) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
            cudaSuccess)
            return SMD_ERR_LAUNCH;
        smem_set[dev].store(smem_bytes);
    }
    if (nonportable && !np_set[dev].load()) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
            return SMD_ERR_LAUNCH;
        np_set[dev].store(1);
    }
    return SMD_OK;
}

template <int T, bool QS, bool TR>
int launch_t(const MmaParams& prm, const MmaConfig& cfg, const CallArgs& a, cudaStream_t stream) {
    auto kern = mma_decode_kernel<T, QS, TR>;
    const int rc = ensure_attributes<T, QS, TR>(cfg.layout.total, cfg.split > 8);
    if (rc != SMD_OK) return rc;
    cudaError_t err;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(a.H / (kHeadsPerTile * T) * cfg.split),
                      static_cast<unsigned>(a.B), 1);
    lc.blockDim = dim3(kMmaThreads, 1, 1);
    lc.dynamicSmemBytes = static_cast<size_t>(cfg.layout.total);
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
    err = cudaLaunchKernelEx(&lc, kern, prm);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return SMD_ERR_LAUNCH;
    }
    return SMD_OK;
}

}  // namespace

SMD_TRACE_COPY_FN(mma_trace_copy, g_trace_mma)

int launch_mma(const CallArgs& a, const MmaConfig& cfg, cudaStream_t stream) {
    MmaParams prm{};
    prm.a = a;
    prm.split = cfg.split;
    prm.window = cfg.window;
    prm.key_cap = cfg.key_cap;
    prm.L = cfg.layout;
    prm.log2_448 = static_cast<float>(std::log2(448.0));
    prm.budget_ns = cfg.wait_budget_ns;
    prm.inject_stall = cfg.inject_stall;
    prm.spec_idx = cfg.spec_idx;
    prm.tree_tmem = cfg.tree_tmem;
    if (cfg.qsplit && a.q16 == nullptr) return SMD_ERR_NULL;
    switch (cfg.tiles * 4 + (cfg.qsplit ? 2 : 0) + (cfg.tree_tmem ? 1 : 0)) {
        case 4:
            return launch_t<1, false, false>(prm, cfg, a, stream);
        case 5:
            return launch_t<1, false, true>(prm, cfg, a, stream);
        case 6:
            return launch_t<1, true, false>(prm, cfg, a, stream);
        case 7:
            return launch_t<1, true, true>(prm, cfg, a, stream);
        case 8:
            return launch_t<2, false, false>(prm, cfg, a, stream);
        case 9:
            return launch_t<2, false, true>(prm, cfg, a, stream);
        case 10:
            return launch_t<2, true, false>(prm, cfg, a, stream);
        case 11:
            return launch_t<2, true, true>(prm, cfg, a, stream);
        default:
            return SMD_ERR_PLAN;
    }
}

}  // namespace smd
