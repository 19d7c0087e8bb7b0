// Sparse MLA decode for groups of query rows that share one index list
// (warp-level FP8 tensor cores, sm_103a).
//
// The rows of a multi-token decode step (the attn_sparse page's verify rows;
// the dense-as-sparse workload's causal rows of one request) read prefixes of
// one index list: row i of a request sees its first L - qlen + 1 + i tokens.
// Gathering the list once for the whole group instead of once per row is the
// point of this kernel. A CTA takes 16 heads of each of the G rows of a group
// (G tiles of 16 heads) and its share of the group's longest list; the S CTAs
// of a cluster split that list as the page's SparseDcpDecode splits a row's
// keys, at the leaf boundaries of smd_tree.cuh (leaves of 64 * ceil(n / 1024)
// keys of the group's longest list, at most 16; CTA s takes an aligned block of a
// power of two of them), and tile t masks the keys past its own row's count.
//
// The arithmetic per (row, head) is the warp-MMA kernel's: logits by
// mma.sync m16n8k32 E4M3 (two accumulation chains per 8 keys), the P anchor at
// the maximum over the whole row (cluster exchange of the CTAs' maxima),
// P = 2^(s - m + log2 448) in E4M3, FP32 sums of the unquantized P, PV (each
// leaf from zero, the subtrees of a CTA's finished leaves waiting in TMEM),
// and the FP32 merge of the split partials by the leaf tree, so that the bits
// do not depend on the split. Two things differ so that
// G = 4 tiles fit in shared memory: the logits are not kept between the two
// passes (pass A only tracks the maximum; pass B gathers each chunk again and
// recomputes its logits, which the same MMA sequence reproduces bit for bit),
// and the inbox of the split partials lies over the dead key ring once every
// peer has signalled that its own ring is dead.
//
// Contract (checked): for every row r of a group and i < count(r),
// indices[r][i] equals indices[r*][i], r* the group's row with the largest
// clamped count (the first such). A CTA that finds a mismatch in the keys it
// reads writes SMD_ERR_GROUP to the status word; that group's outputs are then
// unspecified.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "smd_internal.h"
#include "smd_ptx.cuh"
#include "smd_tree.cuh"

namespace smd {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kLgPitch = kChunk + 8;   // floats per row of the chunk's logits
constexpr int kPPitch = kChunk + 16;   // bytes per row of the chunk's P

struct GroupParams {
    CallArgs a;
    int32_t split, nslots, key_cap;
    GroupLayout L;
    float log2_448;
    uint64_t budget_ns;
    int32_t inject_stall;
    int32_t tree_tmem;  // 1: a CTA may hold several leaves (TMEM subtree stack)
};

// Frees the subtree stack's TMEM once every thread is past its last use
// (warp 0 allocated it).
__device__ __forceinline__ void release_tmem(int tree_tmem, uint32_t tbase) {
    tc_fence_before();
    __syncthreads();
    if (tree_tmem && (threadIdx.x >> 5) == 0) {
        tc_fence_after();
        tmem_free(tbase, 512);
    }
}

// The gathers of one chunk of `cnt` <= 64 keys (`keys`: their pool rows) into
// a ring slot, all 576 bytes of each row, as 16-byte cp.async copies: warp w
// copies rows w, w + 16, ...; lane l the row's pieces l and l + 32. Every
// thread arrives on the slot's barrier once its copies have landed. Rows
// [cnt, roundup32(cnt)) are zeroed (PV reads them with P = 0).
__device__ __forceinline__ void gather_rows(const GroupParams& p, uint32_t slot_s,
                                            const int32_t* keys, uint32_t bar, int cnt) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < cnt; r += kMmaThreads / 32) {
        const uint8_t* src = p.a.kv + static_cast<int64_t>(keys[r]) * kRow;
        const uint32_t dst = slot_s + r * kRowPitch;
        cp_async16(dst + 16 * lane, src + 16 * lane);
        if (lane < kRow / 16 - 32) cp_async16(dst + 16 * (lane + 32), src + 16 * (lane + 32));
    }
    cp_async_arrive(bar);
    const int span = (cnt + 31) & ~31;
    for (int e = cnt * (kRow / 16) + threadIdx.x; e < span * (kRow / 16); e += kMmaThreads) {
        const int r = e / (kRow / 16), c16 = e % (kRow / 16);
        sts_zero16(slot_s + r * kRowPitch + 16 * c16);
    }
}

// QK of one 16-head x 16-key job of a chunk: heads of tile t, keys
// 16 kg .. 16 kg + 15 of the chunk in slot `slot_s`. Returns the two n-tiles'
// accumulators (c0: first 32 bytes of every 64-byte k-step, c1: second).
__device__ __forceinline__ void qk_job(uint32_t slot_s, uint32_t q_s, int t, int kg, int lane,
                                       float (&c0)[2][4], float (&c1)[2][4]) {
    const int a_row = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int a_col = 16 * (lane >> 4);
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) c0[n][e] = c1[n][e] = 0.f;
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
    }
}

template <int G>
__global__ void __launch_bounds__(kMmaThreads, 1) group_decode_kernel(const GroupParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_entry();
    constexpr int CH = kHeadsPerTile * G;  // tile t: heads head0 .. head0 + 15 of row b0 + t
    constexpr int kJobs = 4 * G;           // 16-key QK jobs per chunk, one per warp

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, qd = lane & 3;
    const int S = p.split;
    const int split = static_cast<int>(cluster_ctarank());
    const int head0 = (blockIdx.x / S) * kHeadsPerTile;
    const int b0 = blockIdx.y * G;
    const int W = p.a.W, H = p.a.H;

    const uint32_t base = smem_addr(smem);
    const uint32_t ring_s = base + p.L.ring;
    const uint32_t q_s = base + p.L.q;
    const uint32_t prob_s = base + p.L.probs;
    float* lg = reinterpret_cast<float*>(smem + p.L.lg);
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + p.L.idx);
    float* sums = reinterpret_cast<float*>(smem + p.L.sums);
    float* maxima = reinterpret_cast<float*>(smem + p.L.maxima);
    float* wmax = reinterpret_cast<float*>(smem + p.L.wmax);
    float* lsum = reinterpret_cast<float*>(smem + p.L.lsum);
    float* rowmax = reinterpret_cast<float*>(smem + p.L.rowmax);
    int32_t* nrow = reinterpret_cast<int32_t*>(smem + p.L.nrow);
    float* lstk = reinterpret_cast<float*>(smem + p.L.lstk);
    const int NS = p.nslots;
    const uint32_t bars = base + p.L.bars;
    const uint32_t q_bar = bars + 8 * NS;
    const uint32_t max_bar = q_bar + 8;
    const uint32_t in_bar = q_bar + 16;
    const uint32_t free_bar = q_bar + 24;
    const int CW = kLatent / S;  // latent columns this CTA merges

    bool ok = true;
    int32_t* status = p.a.status;

    // The group's counts first: their round trip overlaps the setup.
    const int cnt_raw = (tid < G) ? p.a.counts[b0 + tid] : 0;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bars + 8 * s, kMmaThreads);
        mbar_init(q_bar, 1);
        mbar_init(max_bar, 1);
        mbar_init(in_bar, 1);
        mbar_init(free_bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(max_bar, (S - 1) * CH * 4);
        mbar_arrive_expect_tx(in_bar, (S - 1) * (CH * CW * 4 + CH * 4));
        mbar_arrive_expect_tx(free_bar, (S - 1) * 4);
        // (inject_stall: the barrier also expects 16 bytes nobody sends, so
        // the bounded wait below runs out; a test hook for the timeout path.)
        mbar_arrive_expect_tx(q_bar, CH * kRow + (p.inject_stall ? 16 : 0));
    }
    for (int h = tid; h < CH; h += kMmaThreads) lsum[h] = 0.f;
    if (tid < G) nrow[tid] = max(min(cnt_raw, W), 0);
    if (p.tree_tmem && warp == 0) tmem_alloc(base + p.L.tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = p.tree_tmem ? *reinterpret_cast<volatile uint32_t*>(smem + p.L.tslot) : 0u;
    // Every CTA's barriers are armed before any peer pushes (waited below).
    if (S > 1) cluster_arrive_relaxed();

    // The query rows: head head0 + (i % 16) of row b0 + i / 16.
    if (tid < CH) {
        const uint8_t* src =
            p.a.q + (static_cast<int64_t>(b0 + tid / kHeadsPerTile) * H + head0 + tid % kHeadsPerTile) * kRow;
        bulk_g2s(q_s + tid * kRowPitch, src, kRow, q_bar);
    }

    // ---- the group's list and this CTA's share of it -------------------------
    int nt[G];
    int ref = 0, nmax = -1;
#pragma unroll
    for (int t = 0; t < G; ++t) {
        nt[t] = nrow[t];
        if (nt[t] > nmax) {
            nmax = nt[t];
            ref = t;
        }
    }
    const int leaf = mma_leaf(nmax);
    const int lpc = mma_leaves_per_cta(nmax, S);
    const int first = min(nmax, split * lpc * leaf);
    const int mine = min(nmax - first, lpc * leaf);
    const int32_t* ref_idx = p.a.indices + static_cast<int64_t>(b0 + ref) * W + first;
    for (int i = tid; i < mine; i += kMmaThreads) idx_s[i] = ref_idx[i];
    // The contract: the other rows' lists agree with it on the keys they read.
    bool bad = false;
#pragma unroll
    for (int t = 0; t < G; ++t) {
        if (t == ref) continue;
        const int32_t* row_idx = p.a.indices + static_cast<int64_t>(b0 + t) * W + first;
        const int lim = min(mine, nt[t] - first);
        for (int i = tid; i < lim; i += kMmaThreads) bad = bad || (row_idx[i] != ref_idx[i]);
    }
    if (__syncthreads_or(bad) && tid == 0 && status != nullptr) atomicCAS(status, 0, SMD_ERR_GROUP);

    const float neg_inf = -INFINITY;
    const float lam = p.a.scale_log2;
    const int nch = (mine + kChunk - 1) / kChunk;
    uint32_t phase_bits = 0;  // parity of each ring slot's next completion
    // This warp's QK job, the same in both passes: tile jt, keys 16 jkg .. + 15.
    const bool has_job = warp < kJobs;
    const int jt = warp >> 2, jkg = warp & 3;
    const int njt = has_job ? nrow[jt] : 0;

    // ================================ pass A: the maximum =====================
    for (int c = 0; c < min(NS, nch); ++c)
        gather_rows(p, ring_s + c * kChunk * kRowPitch, idx_s + c * kChunk, bars + 8 * c,
                    min(kChunk, mine - c * kChunk));
    mbar_wait(q_bar, 0, ok, status, p.budget_ns);
    float mx[2] = {neg_inf, neg_inf};  // heads g and g + 8 of tile jt, this warp's keys
    for (int c = 0; c < nch; ++c) {
        const int s = c % NS;
        const int cnt = min(kChunk, mine - c * kChunk);
        const uint32_t slot_s = ring_s + s * kChunk * kRowPitch;
        mbar_wait(bars + 8 * s, (phase_bits >> s) & 1u, ok, status, p.budget_ns);
        phase_bits ^= 1u << s;
        if (has_job && 16 * jkg < cnt) {
            float c0[2][4], c1[2][4];
            qk_job(slot_s, q_s, jt, jkg, lane, c0, c1);
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int kk = 16 * jkg + 8 * n + 2 * qd;
                const int key = first + c * kChunk + kk;  // in the group's list
                const bool v0 = kk < cnt && key < njt, v1 = kk + 1 < cnt && key + 1 < njt;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float s0 = v0 ? lam * (c0[n][2 * r] + c1[n][2 * r]) : neg_inf;
                    const float s1 = v1 ? lam * (c0[n][2 * r + 1] + c1[n][2 * r + 1]) : neg_inf;
                    mx[r] = fmaxf(mx[r], fmaxf(s0, s1));
                }
            }
        }
        // The slot is free; a failed CTA issues no more copies.
        if (!__syncthreads_and(ok)) break;
        if (c + NS < nch)
            gather_rows(p, slot_s, idx_s + (c + NS) * kChunk, bars + 8 * s,
                        min(kChunk, mine - (c + NS) * kChunk));
    }

    // ---- the row maximum over the cluster ------------------------------------
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    if (has_job && qd == 0) {
        wmax[jkg * CH + 16 * jt + g] = mx[0];
        wmax[jkg * CH + 16 * jt + g + 8] = mx[1];
    }
    __syncthreads();
    for (int h = tid; h < CH; h += kMmaThreads)
        maxima[split * CH + h] = fmaxf(fmaxf(wmax[h], wmax[CH + h]), fmaxf(wmax[2 * CH + h], wmax[3 * CH + h]));
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
    for (int h = tid; h < CH; h += kMmaThreads) {
        float m = neg_inf;
        for (int pr = 0; pr < S; ++pr) m = fmaxf(m, maxima[pr * CH + h]);
        rowmax[h] = m;
    }
    __syncthreads();

    // ================================ pass B: P and PV ========================
    // Chunks in descending order; the last NS are still resident, the others
    // come back (whole rows: their logits are computed again) into the slot of
    // the chunk NS above once PV of that chunk has left it.
    const int a_row = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int a_col = 16 * (lane >> 4);
    float acc[G][4][4];
#pragma unroll
    for (int t = 0; t < G; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[t][j][e] = 0.f;

    // Leaves (as in the warp-MMA kernel): slot l of this CTA is chunks
    // [l cpl, l cpl + cpl), walked downwards; each leaf is summed from zero and
    // pushed into the subtree stack at its end (acc: TMEM levels of 16 G
    // floats; the sums of P: lstk).
    const int cpl = leaf / kChunk;
    int tcnt = nch > 0 ? lpc - 1 - (nch - 1) / cpl : lpc;  // leaves pushed: the absent slots
    uint32_t tpres = 0u;  // bit d: stack level d holds a subtree
    const uint32_t tcol = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 128u * (warp >> 2);
    for (int c = nch - 1; c >= 0; --c) {
        const int s = c % NS;
        const int cnt = min(kChunk, mine - c * kChunk);
        const uint32_t slot_s = ring_s + s * kChunk * kRowPitch;
        if (c < nch - NS) {
            mbar_wait(bars + 8 * s, (phase_bits >> s) & 1u, ok, status, p.budget_ns);
            phase_bits ^= 1u << s;
        }
        // The chunk's logits, by the same MMAs as in pass A.
        if (has_job && 16 * jkg < cnt) {
            float c0[2][4], c1[2][4];
            qk_job(slot_s, q_s, jt, jkg, lane, c0, c1);
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int kk = 16 * jkg + 8 * n + 2 * qd;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float2* dst = reinterpret_cast<float2*>(lg + (16 * jt + g + 8 * r) * kLgPitch + kk);
                    *dst = make_float2(lam * (c0[n][2 * r] + c1[n][2 * r]),
                                       lam * (c0[n][2 * r + 1] + c1[n][2 * r + 1]));
                }
            }
        }
        __syncthreads();
        // P of 64 keys: warp w takes head w of every tile; lane: keys 2*lane, 2*lane + 1.
#pragma unroll
        for (int t = 0; t < G; ++t) {
            const int h = 16 * t + warp;
            const float bias = rowmax[h] - p.log2_448;
            const int kk = 2 * lane;
            const int key = first + c * kChunk + kk;
            const float2 sv = *reinterpret_cast<const float2*>(lg + h * kLgPitch + kk);
            const float p0 = (kk < cnt && key < nt[t]) ? ex2_approx(sv.x - bias) : 0.f;
            const float p1 = (kk + 1 < cnt && key + 1 < nt[t]) ? ex2_approx(sv.y - bias) : 0.f;
            sts_u16(prob_s + h * kPPitch + kk, e4m3x2(p0, p1));
            const float tot = warp_sum(p0 + p1);
            if (lane == 0) lsum[h] += tot;
        }
        __syncthreads();
        // PV: latent columns 32*warp + 4*g + (0..3) of every tile.
        const int span = (cnt + 31) & ~31;
#pragma unroll
        for (int ks = 0; ks < kChunk / 32; ++ks) {
            if (32 * ks >= span) break;
            uint32_t vb[2][4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int key = 32 * ks + 16 * hf + 4 * qd + i;
                    w[i] = lds_u32(slot_s + key * kRowPitch + 32 * warp + 4 * g);
                }
                byte_transpose4(w[0], w[1], w[2], w[3], vb[hf]);
            }
#pragma unroll
            for (int t = 0; t < G; ++t) {
                uint32_t pa[4];
                ldsm_x4(prob_s + (16 * t + a_row) * kPPitch + 32 * ks + a_col, pa);
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_e4m3(acc[t][j], pa, vb[0][j], vb[1][j]);
            }
        }
        if (c % cpl == 0) {  // leaf c / cpl is complete (uniform)
            int d = 0;
            while ((tcnt >> d) & 1) {
                if ((tpres >> d) & 1u) {
                    stash_add<G>(tcol + 16u * G * d, acc);
                    if (lane == 0)
#pragma unroll
                        for (int t = 0; t < G; ++t) {
                            const int h = 16 * t + warp;
                            lsum[h] = lstk[d * CH + h] + lsum[h];
                        }
                }
                ++d;
            }
            tpres &= ~((1u << d) - 1u);
            if (++tcnt < lpc) {  // not the root: keep the subtree, start the next leaf at zero
                stash_store<G>(tcol + 16u * G * d, acc);
                if (lane == 0)
#pragma unroll
                    for (int t = 0; t < G; ++t) {
                        const int h = 16 * t + warp;
                        lstk[d * CH + h] = lsum[h];
                        lsum[h] = 0.f;
                    }
                tpres |= 1u << d;
#pragma unroll
                for (int t = 0; t < G; ++t)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[t][j][e] = 0.f;
            }
        }
        // The slot, the logits and P are free; a failed CTA issues no more copies.
        if (!__syncthreads_and(ok)) break;
        if (c - NS >= 0) gather_rows(p, slot_s, idx_s + (c - NS) * kChunk, bars + 8 * s, kChunk);
    }
    cp_async_wait_all();  // no copy into the ring is in flight from here on
    __syncthreads();      // ... from any thread of this CTA

    if (S == 1) {
        // No peers: BF16(acc * k_scale / total) straight from the registers.
        if (ok) {
#pragma unroll
            for (int t = 0; t < G; ++t) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int hh = g + 8 * (e >> 1);
                    const int col = 32 * warp + 8 * qd + 4 * (e & 1);
                    const float total = lsum[16 * t + hh];
                    const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
                    uint2 packed;
                    packed.x = bf16x2(acc[t][0][e] * inv, acc[t][1][e] * inv);
                    packed.y = bf16x2(acc[t][2][e] * inv, acc[t][3][e] * inv);
                    uint16_t* dst =
                        p.a.out + (static_cast<int64_t>(b0 + t) * H + head0 + hh) * kLatent + col;
                    *reinterpret_cast<uint2*>(dst) = packed;
                }
            }
            for (int h = tid; h < CH; h += kMmaThreads) {
                const float total = lsum[h];
                p.a.lse[static_cast<int64_t>(b0 + h / kHeadsPerTile) * H + head0 + h % kHeadsPerTile] =
                    total > 0.f ? (rowmax[h] - p.log2_448 + log2f(total)) * 0.69314718055994530942f
                                : -INFINITY;
            }
        }
        release_tmem(p.tree_tmem, tbase);
        return;
    }

    // ---- partials to the column owners (FP32 bits over DSMEM) ----------------
    // The inbox lies over this CTA's ring, query tile, logits and P: every
    // peer is told that they are dead (a 4-byte st.async completing on the
    // peer's barrier), and nothing is pushed before every peer has said so.
    if (tid == 0) {
        const uint32_t flag = smem_addr(smem + p.L.flags + 4 * (split & 3));
        for (int pr = 0; pr < S; ++pr)
            if (pr != split) st_async_b32(mapa(flag, pr), 1u, mapa(free_bar, pr));
    }
    mbar_wait(free_bar, 0, ok, status, p.budget_ns, /*always=*/true);
    // acc[t][j][e]: head 16t + g + 8(e>>1), column 32*warp + 8*qd + 4*(e&1) + j.
    // Inbox unit ((((src * WPO + wl) * G + t) * 4 + e) * 32 + lane) holds the
    // partial of CTA src from warp wl of the owner's WPO = CW / 32 column warps.
    const int WPO = CW / 32;
    {
        const int owner = warp / WPO;
        const int wl = warp - owner * WPO;
        const uint32_t inbox_s = base;
#pragma unroll
        for (int t = 0; t < G; ++t) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 v = make_float4(acc[t][0][e], acc[t][1][e], acc[t][2][e], acc[t][3][e]);
                const uint32_t dst = inbox_s + (((((split * WPO + wl) * G + t) * 4 + e) * 32) + lane) * 16;
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

    // ---- merge by the leaf tree; BF16(sum * k_scale / total) -----------------
    // CTA src holds the subtree of leaves [src lpc, src lpc + lpc) of the
    // group's list: absent if they lie past its longest count.
    if (ok) {
        const int units = WPO * G * 128;  // 16-byte units of one CTA's partial of my columns
        const float4* in4 = reinterpret_cast<const float4*>(smem);
        const int np = (mma_leaves(nmax) + lpc - 1) / lpc;  // CTAs 0 .. np - 1 hold keys
        for (int u = tid; u < units; u += kMmaThreads) {
            const int ln = u & 31, e = (u >> 5) & 3, t = (u >> 7) % G, wl = (u >> 7) / G;
            const int hh = (ln >> 2) + 8 * (e >> 1);
            const int h = 16 * t + hh;
            const int c = 32 * wl + 8 * (ln & 3) + 4 * (e & 1);
            const float4 m = tree_xor_n<float4>(S, [&](int k) { return in4[k * units + u]; }, 0, np);
            const float total = tree_xor_n<float>(S, [&](int k) { return sums[k * CH + h]; }, 0, np);
            const float inv = total > 0.f ? p.a.k_scale / total : 0.f;
            uint2 packed;
            packed.x = bf16x2(m.x * inv, m.y * inv);
            packed.y = bf16x2(m.z * inv, m.w * inv);
            uint16_t* dst = p.a.out + (static_cast<int64_t>(b0 + t) * H + head0 + hh) * kLatent +
                            split * CW + c;
            *reinterpret_cast<uint2*>(dst) = packed;
        }
        if (split == 0) {
            for (int h = tid; h < CH; h += kMmaThreads) {
                const float total =
                    tree_xor_n<float>(S, [&](int k) { return sums[k * CH + h]; }, 0, np);
                p.a.lse[static_cast<int64_t>(b0 + h / kHeadsPerTile) * H + head0 + h % kHeadsPerTile] =
                    total > 0.f ? (rowmax[h] - p.log2_448 + log2f(total)) * 0.69314718055994530942f
                                : -INFINITY;
            }
        }
    }
    release_tmem(p.tree_tmem, tbase);
}

// Shared-memory size and (for clusters above 8) the non-portable cluster
// attribute, set once per device and kernel.
template <int G>
int ensure_group_attributes(int smem_bytes, bool nonportable) {
    static std::atomic<int> smem_set[kMaxDevices];
    static std::atomic<int> np_set[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMD_ERR_DEVICE;
    auto kern = group_decode_kernel<G>;
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

template <int G>
int launch_g(const GroupParams& prm, const GroupConfig& cfg, const CallArgs& a, cudaStream_t stream) {
    const int rc = ensure_group_attributes<G>(cfg.layout.total, cfg.split > 8);
    if (rc != SMD_OK) return rc;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(a.H / kHeadsPerTile * cfg.split),
                      static_cast<unsigned>(a.B / G), 1);
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
    if (cudaLaunchKernelEx(&lc, group_decode_kernel<G>, prm) != cudaSuccess) {
        (void)cudaGetLastError();
        return SMD_ERR_LAUNCH;
    }
    return SMD_OK;
}

}  // namespace

int launch_group(const CallArgs& a, const GroupConfig& cfg, cudaStream_t stream) {
    GroupParams prm{};
    prm.a = a;
    prm.split = cfg.split;
    prm.nslots = cfg.nslots;
    prm.key_cap = cfg.key_cap;
    prm.L = cfg.layout;
    prm.log2_448 = static_cast<float>(std::log2(448.0));
    prm.budget_ns = cfg.wait_budget_ns;
    prm.inject_stall = cfg.inject_stall;
    prm.tree_tmem = cfg.tree_tmem;
    switch (cfg.G) {
        case 2:
            return launch_g<2>(prm, cfg, a, stream);
        case 4:
            return launch_g<4>(prm, cfg, a, stream);
        default:
            return SMD_ERR_PLAN;
    }
}

}  // namespace smd
