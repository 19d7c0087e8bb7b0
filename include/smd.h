/*
 * smd.h -- sparse MLA decode over an FP8 (E4M3) latent KV cache, for GB300
 * (sm_103a). C ABI of libsmd.so.
 *
 * The operation (the "attn_sparse" page, SparseDcpDecode: module docstring
 * paragraphs "Per CTA", "Precision" and "Rows of count 0"; run_sparse's
 * argument list): for each query row b and head h, over the row's first
 * n_b = clamp(counts[b], 0, W) key indices j_i = indices[b, i],
 *
 *   s_i  = fp32(lambda * fp32(sum_{c<576} q8[b,h,c] * kv8[j_i,c]))
 *          lambda = fp32(sm_scale * q_scale * k_scale * log2(e))
 *   m    = max_i s_i                       (the row maximum over ALL n_b keys)
 *   P_i  = 2^(s_i - m + log2 448)          (fp32; P of the max key is 448)
 *   P8_i = E4M3(P_i), round to nearest even, saturating
 *   T    = sum_i P_i                       (fp32, unquantized P)
 *   out[b,h,c] = BF16(k_scale * sum_i P8_i * kv8[j_i,c] / T),   c < 512
 *   lse[b,h]   = ln 2 * (m - log2 448 + log2 T)                 (natural log)
 *
 * and rows with n_b = 0 write zeros and lse = -inf. The 576-byte cache row
 * holds 512 latent columns (read by both products) followed by 64 columns
 * read by the logits only. The keys of a row are split over the CTAs of a
 * thread-block cluster; their partial sums merge in FP32 over distributed
 * shared memory. The anchor m is the maximum over the whole row, exchanged
 * across the cluster before any P is formed, so the result does not depend
 * on the order of a row's indices beyond FP32 summation order.
 *
 * Memory: every pointer argument is DEVICE memory owned by the caller
 * (cudaMalloc / torch), except the *_host arguments of
 * smd_sparse_mla_decode_host. The library allocates nothing per call and
 * keeps no per-call state (that call keeps two copy streams and a few
 * events per device, created on its first use); all calls are asynchronous
 * on `stream`.
 *
 * Errors: argument and launch problems are returned synchronously as a
 * negative smd_status (nothing is launched). Problems only the GPU can see
 * (a bounded wait that ran out) are written to the optional device word
 * `status` (left untouched on success; the caller zeroes it beforehand).
 * Indices of valid entries must lie in [0, N); the decode does not check
 * them (smd_validate_indices does, as a separate call).
 */
#ifndef SMD_H
#define SMD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st* smd_stream_t;

typedef enum {
    SMD_OK = 0,
    SMD_ERR_NULL = -1,    /* a required pointer is NULL                       */
    SMD_ERR_SHAPE = -2,   /* H not a positive multiple of 16, B/W/N negative,
                             N == 0 while B*W > 0, or W beyond the plan limit  */
    SMD_ERR_ALIGN = -3,   /* q, kv_pool, out not 16-byte aligned; indices,
                             counts, lse, status not 4-byte aligned            */
    SMD_ERR_LAUNCH = -4,  /* the CUDA launch failed (cudaGetLastError)        */
    SMD_ERR_TIMEOUT = -5, /* device status: a bounded wait ran out            */
    SMD_ERR_PLAN = -6,    /* a forced plan is invalid for these shapes        */
    SMD_ERR_DEVICE = -7,  /* no usable sm_103 device / attribute query failed;
                             device status: an SM id beyond the workspace    */
    SMD_ERR_WORKSPACE = -8, /* workspace given but smaller than
                             smd_workspace_bytes() or not 16-byte aligned    */
    SMD_ERR_GROUP = -9,   /* device status: rows of a group do not share their
                             index list (smd_sparse_mla_decode_grouped)      */
    SMD_ERR_INDEX = -10   /* device status: a valid entry of the index list
                             lies outside [0, N) (smd_validate_indices)      */
} smd_status;

/* Kernel families. */
enum {
    SMD_KERNEL_AUTO = 0,
    SMD_KERNEL_MMA = 1,  /* warp-level FP8 MMA (mma.sync), 16-head tiles       */
    SMD_KERNEL_TC = 2,   /* tcgen05 + TMEM, 128 heads per CTA (or all H < 128
                            heads of a row), TMA gather4; 1 <= W <= 2048     */
    SMD_KERNEL_GROUP = 3,   /* warp-level FP8 MMA over groups of rows sharing
                               one index list (smd_sparse_mla_decode_grouped) */
    SMD_KERNEL_TC_GROUP = 4, /* tcgen05 over such groups: G * H = 32 or 64 TMEM
                               lanes, W <= 16 * 512, clusters of up to 16     */
    SMD_KERNEL_TC_SPREAD = 5 /* tcgen05 with a row's keys spread over any CTAs
                               of a cooperative grid (pieces of <= 512 keys,
                               as many as the row's count needs); maxima and
                               FP32 partials through the caller's workspace;
                               H % 128 == 0 or H < 128, 1 <= W <= 32 * 512,
                               B * ceil(H / 128) <= 1024                      */
};

/* A launch plan: how the work is laid out. `split` decides which keys each
 * CTA sums (and so the FP32 summation grouping); `tiles` and `window` only
 * decide layout, and plans that differ only in them give identical bits. */
typedef struct {
    int32_t kernel;      /* SMD_KERNEL_* */
    int32_t split;       /* CTAs per cluster sharing one row: 1, 2, 4, 8, 16
                            (SMD_KERNEL_TC: 1, 2, 4)                         */
    int32_t tiles;       /* 16-head tiles per CTA (1 or 2; TC: 8, fixed)     */
    int32_t window;      /* keys resident in shared memory per pass (64k;
                            TC: 128-key chunks, fixed)                       */
    /* testing hooks (0 = off); only smd_sparse_mla_decode_ex reads them:    */
    int32_t wait_budget_us; /* bound of every device wait (default 200 ms)   */
    int32_t inject_stall;   /* 1: the query barrier expects 16 bytes that no
                               copy delivers, so its wait runs out and the
                               call reports SMD_ERR_TIMEOUT in `status`      */
    /* filled in by smd_plan / smd_sparse_mla_decode_ex:                     */
    int32_t key_cap;     /* most keys one CTA holds logits for               */
    int32_t grid_x, grid_y, cluster_x, threads, smem_bytes;
                         /* (SMD_KERNEL_TC_SPREAD: a non-zero grid_x in a
                            forced plan caps the grid; it only lays work out,
                            so every grid gives identical bits)             */
} smd_plan_t;

/*
 * The decode.
 *   q        [B, H, 576] uint8 E4M3 codes, row-major (head stride 576 B,
 *            row stride H*576 B). 16-byte aligned.
 *   kv_pool  [N, 576] uint8 E4M3 codes (row stride 576 B). 16-byte aligned.
 *   N        rows in kv_pool (>= 1 when B*W > 0; < 2^31).
 *   indices  [B, W] int32, row-major; entries [0, counts[b]) of row b are
 *            its keys (duplicates count twice); the rest are not read.
 *   W        width of the index array (the top-k), >= 0.
 *   counts   [B] int32; clamped to [0, W].
 *   B, H     rows and heads; H a positive multiple of 16. B == 0 is a no-op.
 *   sm_scale, q_scale, k_scale   softmax scale and the per-tensor E4M3
 *            scales of q and of the cache.
 *   out      [B, H, 512] bfloat16 (raw 16-bit storage). 16-byte aligned.
 *   lse      [B, H] float32, natural log; -inf for empty rows.
 *   status   optional device int32; a device-side failure writes an
 *            smd_status there. May be NULL.
 *   stream   CUDA stream the work is queued on.
 * Returns SMD_OK or a negative smd_status.
 */
int smd_sparse_mla_decode(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                          const int32_t* indices, int32_t W, const int32_t* counts,
                          int32_t B, int32_t H,
                          float sm_scale, float q_scale, float k_scale,
                          uint16_t* out, float* lse, int32_t* status,
                          smd_stream_t stream);

/* The plan smd_sparse_mla_decode would use for (B, H, W) on the current
 * device. Host only; touches no device memory. */
int smd_plan(int32_t B, int32_t H, int32_t W, smd_plan_t* plan);

/* Bytes of workspace smd_sparse_mla_decode_ws can use for (B, H, W): the
 * size SMD_KERNEL_TC_SPREAD wants when smd_plan_ws would choose it (one slot
 * per possible piece, B * ceil(H / 128) * ceil(W / 512) slots of about
 * 257 KiB), else 0 (the plan merges on chip: no workspace needed). Host only. */
int64_t smd_workspace_bytes(int32_t B, int32_t H, int32_t W);

/* Bytes of workspace the plan forced by `force` (as smd_sparse_mla_decode_ex
 * reads it; NULL = automatic) can use: the spread kernel's slots, or a
 * cluster plan's L2 exchange slots (which smd_sparse_mla_decode_ex uses when
 * it is given a workspace). Host only. */
int64_t smd_workspace_bytes_ex(int32_t B, int32_t H, int32_t W, const smd_plan_t* force);

/* The plan smd_sparse_mla_decode_ws uses for (B, H, W) given a workspace:
 * with H % 128 == 0, B * ceil(H / 128) <= 1024 and W > 512 it is
 * SMD_KERNEL_TC_SPREAD when the rows are longer than one cluster holds
 * (W > 2048) or when the at most B * ceil(H / 128) * ceil(W / 512) pieces
 * fill no more than two waves of the device; otherwise the plan of smd_plan.
 * Host only. */
int smd_plan_ws(int32_t B, int32_t H, int32_t W, smd_plan_t* plan);

/* As smd_sparse_mla_decode, with a caller-owned device workspace, in the
 * plan of smd_plan_ws. SMD_KERNEL_TC_SPREAD exchanges the row maxima and the
 * FP32 partials of a row's pieces through it. workspace may be NULL (the plan of
 * smd_plan is used); otherwise it must be 16-byte aligned and at least
 * smd_workspace_bytes(B, H, W) long (else SMD_ERR_WORKSPACE); plans other
 * than the spread kernel leave it untouched. Its contents need no initialisation: the
 * spread kernel's flags hold a per-call 64-bit token and are zeroed as they
 * are consumed. Calls that overlap on the GPU must not share one workspace;
 * after a call that reported a device error, zero the workspace before a
 * CUDA graph replays a captured call on it. */
int smd_sparse_mla_decode_ws(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                             const int32_t* indices, int32_t W, const int32_t* counts,
                             int32_t B, int32_t H,
                             float sm_scale, float q_scale, float k_scale,
                             uint16_t* out, float* lse, int32_t* status,
                             void* workspace, int64_t workspace_bytes,
                             smd_stream_t stream);

/* As smd_sparse_mla_decode_ws, with the plan fields kernel/split/tiles/window
 * (and the testing hooks) taken from `force` (0 = the automatic choice for
 * that field). Used by the tests to run every variant; `force` and
 * `workspace` may be NULL. Given a workspace (smd_workspace_bytes_ex bytes),
 * a forced cluster plan of the tcgen05 kernel exchanges its partials through
 * it (L2) instead of distributed shared memory. */
int smd_sparse_mla_decode_ex(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                             const int32_t* indices, int32_t W, const int32_t* counts,
                             int32_t B, int32_t H,
                             float sm_scale, float q_scale, float k_scale,
                             uint16_t* out, float* lse, int32_t* status,
                             void* workspace, int64_t workspace_bytes,
                             smd_stream_t stream, const smd_plan_t* force);

/* As smd_sparse_mla_decode, for callers that cannot allocate device memory:
 * a plug-in living inside a host framework that owns every device buffer
 * and hands it only its inputs and outputs, or a serving loop whose memory
 * is reserved up front so that no call can fail for lack of it or stall in
 * the allocator. The attn_sparse page has no counterpart of this call.
 *
 * It allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine). When the plan splits rows over a cluster of tcgen05 CTAs, their
 * FP32 partials go through scratch that the library itself holds: a
 * file-scope device array of 160 SM slots of 192 KiB (30 MiB), which every
 * GPU that loads the library keeps until the process exits. Other plans need
 * no scratch and run as smd_sparse_mla_decode does.
 *
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture on the device.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents; nothing in it needs to start at zero (each call writes
 *     every value it reads). Calls whose kernels overlap on the GPU race on
 *     it: queue them on one stream or order them by events.
 *   - A device with more than 160 SMs is rejected (SMD_ERR_WORKSPACE); a CTA
 *     on an SM id beyond the array writes SMD_ERR_DEVICE to `status` and
 *     leaves the array untouched. That row's out and lse are then not
 *     written although the call returned SMD_OK: pass a `status` word and
 *     read it after the call, as for any device-side error.
 * Arguments, layouts, ownership and the other errors are those of
 * smd_sparse_mla_decode. */
int smd_sparse_mla_decode_noalloc(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                                  const int32_t* indices, int32_t W, const int32_t* counts,
                                  int32_t B, int32_t H,
                                  float sm_scale, float q_scale, float k_scale,
                                  uint16_t* out, float* lse, int32_t* status,
                                  smd_stream_t stream);

/* The decode with a BF16 query, without its per-tensor E4M3 rounding (the
 * mla_attn page: "q_split", the bf16 Q rows to "E4M3 hi, lo of q 2^k", and
 * "fp8_split4", x ~ hi + lo). Each (row, head) query row is scaled by 2^k,
 * the largest power of two with max|q| 2^k <= 448 (k = 0 for a zero row,
 * k clamped to [-32, 32]), and split into hi = E4M3(q 2^k) and
 * lo = E4M3(q 2^k - hi), both round-to-nearest-even and saturating; hi + lo
 * is q 2^k exactly wherever |q 2^k| >= 2^-2. The logit is
 *   s_i = fp32(lambda_h * fp32(sum_c (hi_c + lo_c) * kv8[j_i, c])),
 *   lambda_h = fp32(sm_scale * 2^-k * k_scale * log2 e)
 * and everything after the logits is as in smd_sparse_mla_decode. QK costs
 * twice the MMAs. This call runs on the warp-MMA kernel (any H multiple of 16),
 * which splits the query itself.
 *   q   [B, H, 576] bfloat16 (raw 16-bit storage), row-major, 16-byte
 *       aligned, finite. There is no q_scale: the split finds its own scale.
 * The other arguments, layouts, ownership and errors are those of
 * smd_sparse_mla_decode. */
int smd_sparse_mla_decode_bf16q(const uint16_t* q, const uint8_t* kv_pool, int64_t N,
                                const int32_t* indices, int32_t W, const int32_t* counts,
                                int32_t B, int32_t H, float sm_scale, float k_scale,
                                uint16_t* out, float* lse, int32_t* status, smd_stream_t stream);

/* As smd_sparse_mla_decode_bf16q with a caller-owned device workspace of at
 * least smd_workspace_bytes_bf16q(B, H, W) bytes (16-byte aligned; else
 * SMD_ERR_WORKSPACE): when H % 128 == 0, B * H / 128 <= 1024 and W <= 16384
 * the query is split by a first kernel into E4M3 hi and lo rows and logit
 * scales in the workspace, and the decode runs on the spread tcgen05 kernel
 * (SMD_KERNEL_TC_SPREAD: its query tile holds hi, its second ring slot holds
 * lo until QK is done, so its gathers run one chunk deep). Other shapes run
 * as smd_sparse_mla_decode_bf16q. The workspace needs no initialisation
 * (see smd_sparse_mla_decode_ws). */
int smd_sparse_mla_decode_bf16q_ws(const uint16_t* q, const uint8_t* kv_pool, int64_t N,
                                   const int32_t* indices, int32_t W, const int32_t* counts,
                                   int32_t B, int32_t H, float sm_scale, float k_scale,
                                   uint16_t* out, float* lse, int32_t* status, void* workspace,
                                   int64_t workspace_bytes, smd_stream_t stream);

/* Bytes of workspace smd_sparse_mla_decode_bf16q_ws uses for (B, H, W): the
 * spread kernel's slots and the split query (2 x 576 + 4 bytes per query
 * row), or 0 where it runs on the warp-MMA kernel. Host only. */
int64_t smd_workspace_bytes_bf16q(int32_t B, int32_t H, int32_t W);

/* As smd_sparse_mla_decode_bf16q_ws with plan fields (kernel SMD_KERNEL_MMA,
 * SMD_KERNEL_TC_SPREAD or 0, split, tiles, window, grid_x, the testing hooks)
 * taken from `force` (may be NULL); workspace may be NULL unless the plan is
 * the spread kernel. For the tests. */
int smd_sparse_mla_decode_bf16q_ex(const uint16_t* q, const uint8_t* kv_pool, int64_t N,
                                   const int32_t* indices, int32_t W, const int32_t* counts,
                                   int32_t B, int32_t H, float sm_scale, float k_scale,
                                   uint16_t* out, float* lse, int32_t* status, void* workspace,
                                   int64_t workspace_bytes, smd_stream_t stream,
                                   const smd_plan_t* force);

/* The plan of the bf16-query call with a workspace of workspace_bytes (0:
 * smd_sparse_mla_decode_bf16q's). Host only. */
int smd_plan_bf16q(int32_t B, int32_t H, int32_t W, int64_t workspace_bytes, smd_plan_t* plan);

/* Top-k select over bf16 logits, producing the decode's index list and
 * count on the device (the topk_exchange page: the select of
 * push_local_topk, its radix passes, threshold and tie rule, for one GPU).
 * For row r, over its first end = clamp(row_ends[r], 0, L) logits (all L when
 * row_ends is NULL):
 *   a logit is valid unless it is a NaN; its key is the bf16 bit pattern
 *   mapped to an unsigned 16-bit number in value order (bits | 0x8000 for a
 *   positive sign, ~bits for a negative one, so -0 sorts just below +0);
 *   v = the K-th largest key among the valid logits;
 *   indices[r] = every position with key > v in ascending order, then the
 *   positions with key == v in ascending order until K are taken;
 *   a row with fewer than K valid logits gets all of them in ascending order;
 *   counts[r] = min(K, valid logits); indices[r][counts[r] .. K) = -1.
 * A row is split over a cluster of up to 8 CTAs; a part of up to 16384
 * logits is read from HBM once (longer parts are read again from L2).
 *   logits     [B, row_stride] bf16 bits, row_stride >= L, 2-byte aligned.
 *              Read only. With 16-byte aligned rows (logits 16-byte aligned,
 *              row_stride a multiple of 8) the rows are read in 16-byte
 *              pieces, up to round_up(L, 8) logits a row.
 *   row_ends   [B] int32 or NULL.
 *   indices    [B, K] int32 (row stride K); counts [B] int32. Written.
 *   status     optional device int32: a bounded wait on a peer CTA that ran
 *              out writes SMD_ERR_TIMEOUT there.
 * B >= 0 (0: no-op), L >= 0, K >= 1; otherwise SMD_ERR_SHAPE. All pointers
 * are caller-owned device memory; asynchronous on `stream`. */
int smd_topk_select(const uint16_t* logits, int64_t row_stride, const int32_t* row_ends,
                    int32_t B, int32_t L, int32_t K, int32_t* indices, int32_t* counts,
                    int32_t* status, smd_stream_t stream);

/* As smd_topk_select with the CTAs per row forced (`cluster` 1, 2, 4 or 8;
 * 0 = automatic; else SMD_ERR_PLAN). The split only lays work out: every
 * value gives the same indices and counts. For the tests. */
int smd_topk_select_ex(const uint16_t* logits, int64_t row_stride, const int32_t* row_ends,
                       int32_t B, int32_t L, int32_t K, int32_t* indices, int32_t* counts,
                       int32_t* status, smd_stream_t stream, int32_t cluster);

/* The decode for rows that come in groups sharing one index list: the
 * verify rows of a multi-token decode step, where row i of a request sees the
 * first L - G + 1 + i tokens of its cache (the attn_sparse page's verify rows;
 * the dense-as-sparse workload). The result is that of smd_sparse_mla_decode
 * on the same arguments, up to FP32 summation order (the keys are split over
 * a cluster by the group's longest list instead of by each row's own); the
 * cache rows a group reads are gathered once for all its rows.
 *   row_group  G: 1 (same as smd_sparse_mla_decode), 2 or 4; B % G == 0.
 *              Rows g*G .. g*G + G - 1 form group g.
 * Contract: within a group, let r* be the row with the largest clamped count
 * (the first such); every row r of the group reads a prefix of r*'s list:
 * indices[r][i] == indices[r*][i] for i < clamp(counts[r], 0, W). The kernel
 * checks this for the keys it reads and writes SMD_ERR_GROUP to `status` on
 * a mismatch (the outputs of that group are then unspecified).
 * The other arguments, layouts, ownership and errors are those of
 * smd_sparse_mla_decode; B % G != 0 or another G is SMD_ERR_SHAPE. */
int smd_sparse_mla_decode_grouped(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                                  const int32_t* indices, int32_t W, const int32_t* counts,
                                  int32_t B, int32_t H, int32_t row_group,
                                  float sm_scale, float q_scale, float k_scale,
                                  uint16_t* out, float* lse, int32_t* status,
                                  smd_stream_t stream);

/* The plan of the grouped call with a workspace of workspace_bytes (0: the
 * plan of smd_sparse_mla_decode_grouped: G > 1: kernel SMD_KERNEL_TC_GROUP
 * when G * H is 32 or 64 and W <= 8192, else SMD_KERNEL_GROUP with tiles = G
 * and window = keys of its ring of 64-key slots; with a workspace the spread
 * kernel where smd_sparse_mla_decode_grouped_ws takes it). Host only. */
int smd_plan_grouped(int32_t B, int32_t H, int32_t W, int32_t row_group, int64_t workspace_bytes,
                     smd_plan_t* plan);

/* As smd_sparse_mla_decode_grouped, with a caller-owned device workspace of
 * at least smd_workspace_bytes_grouped(B, H, W, row_group) bytes (16-byte
 * aligned; else SMD_ERR_WORKSPACE). When G * H <= 128, B / G <= 1024 and
 * W <= 16384 and the row-group tcgen05 kernel does not take the shapes
 * (W > 8192, or G * H other than 32 and 64) the groups run on the spread
 * tcgen05 kernel
 * (SMD_KERNEL_TC_SPREAD): a group (all H heads of its G rows, G * H TMEM
 * lanes) of n keys (its longest list) becomes ceil(n / 512) pieces over a
 * cooperative grid, each lane masking the keys past its own row's count, the
 * contract checked as in smd_sparse_mla_decode_grouped. Other shapes run as
 * smd_sparse_mla_decode_grouped. The workspace needs no initialisation. */
int smd_sparse_mla_decode_grouped_ws(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                                     const int32_t* indices, int32_t W, const int32_t* counts,
                                     int32_t B, int32_t H, int32_t row_group,
                                     float sm_scale, float q_scale, float k_scale,
                                     uint16_t* out, float* lse, int32_t* status,
                                     void* workspace, int64_t workspace_bytes,
                                     smd_stream_t stream);

/* Bytes of workspace smd_sparse_mla_decode_grouped_ws uses (0 where it runs
 * the cluster kernels; row_group 1: smd_workspace_bytes). Host only. */
int64_t smd_workspace_bytes_grouped(int32_t B, int32_t H, int32_t W, int32_t row_group);

/* As smd_sparse_mla_decode_grouped_ws, with kernel (SMD_KERNEL_GROUP,
 * SMD_KERNEL_TC_GROUP or SMD_KERNEL_TC_SPREAD), split, window, grid_x and the
 * testing hooks taken from `force` (0 = automatic; may be NULL); workspace
 * may be NULL unless the plan is the spread kernel. For the tests. */
int smd_sparse_mla_decode_grouped_ex(const uint8_t* q, const uint8_t* kv_pool, int64_t N,
                                     const int32_t* indices, int32_t W, const int32_t* counts,
                                     int32_t B, int32_t H, int32_t row_group,
                                     float sm_scale, float q_scale, float k_scale,
                                     uint16_t* out, float* lse, int32_t* status,
                                     void* workspace, int64_t workspace_bytes,
                                     smd_stream_t stream, const smd_plan_t* force);

/* ---- one call for every device-memory variant ------------------------------------
 *
 * smd_decode runs the decode of smd_sparse_mla_decode with the variant an
 * options struct names; options == NULL (or all fields zero) is
 * smd_sparse_mla_decode itself. Each specialised entry point above equals
 * smd_decode with these options, bit for bit (they stay for existing callers):
 *   _ws                    workspace, workspace_bytes
 *   _ex                    workspace, workspace_bytes, force
 *   _bf16q / _bf16q_ws / _bf16q_ex   query_type = SMD_QUERY_BF16 (+ as above)
 *   _grouped / _grouped_ws / _grouped_ex   row_group = 2 or 4 (+ as above)
 *   _noalloc               library_scratch = 1
 * The fields:
 *   row_group        0 or 1: every row has its own index list; 2 or 4: rows
 *                    in consecutive groups sharing one list (the grouped calls).
 *   query_type       SMD_QUERY_E4M3: q is [B, H, 576] E4M3 codes with q_scale;
 *                    SMD_QUERY_BF16: q is [B, H, 576] bfloat16 and q_scale is
 *                    not used (the bf16q calls).
 *   library_scratch  nonzero: a split plan exchanges its partials through the
 *                    library's static scratch (smd_sparse_mla_decode_noalloc,
 *                    with its restrictions).
 *   reserved         must be 0.
 *   workspace, workspace_bytes   caller device workspace or NULL (its size
 *                    from smd_decode_workspace_bytes).
 *   status           optional device status word, as in smd_sparse_mla_decode.
 *   force            NULL: the automatic plan; else a forced plan (for tests).
 * Invalid combinations return, with nothing launched: SMD_ERR_SHAPE for a
 * nonzero `reserved`, an unknown query_type or a row_group other than
 * 0, 1, 2, 4; SMD_ERR_PLAN for a bf16 query with row groups, or
 * library_scratch with a workspace, row groups or a bf16 query. Otherwise
 * the return codes, ownership and ordering are those of the call the options
 * name. */
typedef enum { SMD_QUERY_E4M3 = 0, SMD_QUERY_BF16 = 1 } smd_query_type;

typedef struct {
    int32_t row_group;
    int32_t query_type;
    int32_t library_scratch;
    int32_t reserved;
    void* workspace;
    int64_t workspace_bytes;
    int32_t* status;
    const smd_plan_t* force;
} smd_options_t;

int smd_decode(const void* q, const uint8_t* kv_pool, int64_t N, const int32_t* indices,
               int32_t W, const int32_t* counts, int32_t B, int32_t H, float sm_scale,
               float q_scale, float k_scale, uint16_t* out, float* lse,
               const smd_options_t* options, smd_stream_t stream);

/* Bytes of workspace the workspace plan of these options wants (0 when that
 * plan needs none, or for invalid shapes or options): smd_workspace_bytes,
 * _ex (with force), _bf16q or _grouped. Host only. */
int64_t smd_decode_workspace_bytes(int32_t B, int32_t H, int32_t W, const smd_options_t* options);

/* The plan smd_decode would run for these shapes and options, written to
 * *plan (a workspace counts as given when options->workspace is non-NULL or
 * workspace_bytes > 0; its size is not checked here). Host only; pointers
 * are not needed. Returns SMD_OK or the status smd_decode would return for
 * the shapes and options. */
int smd_decode_plan(int32_t B, int32_t H, int32_t W, const smd_options_t* options,
                    smd_plan_t* plan);

/* ---- the decode from and to host memory ---------------------------------------
 *
 * Options of smd_sparse_mla_decode_host (all zero: E4M3 query, one row per
 * index list, the library's chunking).
 *   row_group   0 or 1: every row has its own index list (smd_sparse_mla_decode_ws);
 *               2 or 4: rows in groups sharing one list (smd_sparse_mla_decode_grouped_ws).
 *   bf16_query  0: q is [B, H, 576] E4M3 codes; 1: q is [B, H, 576] bfloat16
 *               (smd_sparse_mla_decode_bf16q_ws; q_scale is not used). Not
 *               with row_group > 1.
 *   chunks      0: the library's choice (smd_plan_host); 1..8: the rows are
 *               cut into that many consecutive chunks (whole row groups).
 *   copies      0: the library's choice; 1: always copy through the workspace
 *               (never read or write the host buffers from a kernel).
 */
typedef struct {
    int32_t row_group;
    int32_t bf16_query;
    int32_t chunks;
    int32_t copies;
} smd_host_opts_t;

/* The number of row chunks smd_sparse_mla_decode_host pipelines for these
 * shapes and options (opts may be NULL), written to *chunks. One chunk when
 * the call moves at most 16 MiB of host data (q, indices, counts, out, lse),
 * when the device call's plan is the spread kernel (a chunk of its rows would
 * leave SMs idle) or when it fills fewer than three waves of the device;
 * otherwise up to four, each still filling at least one and a half waves,
 * except on the tcgen05 cluster plan: there the rows are cut where the
 * kernel's waves end (rows per wave = the clusters the device holds at once
 * over the clusters a row takes; with no device, one cluster per `split`
 * SMs): one wave, then chunks of two waves (more when eight chunks would
 * not hold them), then the rows of the partial wave, if any; at most eight.
 * An explicit opts->chunks cuts the row groups evenly instead.
 * Host only. Returns SMD_OK or SMD_ERR_SHAPE / SMD_ERR_NULL / SMD_ERR_PLAN. */
int smd_plan_host(int32_t B, int32_t H, int32_t W, const smd_host_opts_t* opts, int32_t* chunks);

/* Bytes of device workspace smd_sparse_mla_decode_host needs (opts may be
 * NULL): staging for q, indices, counts, out and lse of all B rows, each
 * 256-byte aligned, plus the device call's own workspace for one chunk.
 * Negative (an smd_status) for invalid shapes or options. Host only. */
int64_t smd_workspace_bytes_host(int32_t B, int32_t H, int32_t W, const smd_host_opts_t* opts);

/* The decode with its inputs and outputs in host memory; the cache pool stays
 * in device memory (kv_pool as in smd_sparse_mla_decode).
 *   q_host        [B, H, 576] E4M3 codes, or bfloat16 with opts->bf16_query.
 *   indices_host  [B, W] int32; counts_host [B] int32.
 *   out_host      [B, H, 512] bfloat16 (raw 16-bit storage); lse_host [B, H] float32.
 *   workspace     device memory of at least smd_workspace_bytes_host bytes,
 *                 16-byte aligned (else SMD_ERR_WORKSPACE); no initialisation needed.
 * The rows are cut into chunks (smd_plan_host); every array moves with one
 * cudaMemcpyAsync per chunk. One chunk: copies in, decode and copies out are
 * queued on `stream` in that order. Several: chunk 0 moves in on `stream`,
 * the later chunks on the library's upload stream after it (while the earlier
 * chunks are decoded); each chunk is decoded on `stream` once it is in; every
 * chunk but the last moves out on the library's download stream while the
 * next one is decoded, the last on `stream`, which then waits for both copy
 * streams. (With mapped host buffers, chunk 0's q is pulled in by a copy
 * kernel and the last chunk's out and lse are written in place.) So the call is ordered on `stream` like a kernel launch (and can be
 * captured in a CUDA graph from `stream`). The call is asynchronous: host
 * buffers must stay valid, and the results are in out_host / lse_host once
 * `stream` has reached this point.
 * Host buffers should be page-locked (cudaHostAlloc, cudaHostRegister) for the
 * copies to overlap; pageable memory gives the same results, without overlap.
 * Direct access: with one chunk, and indices, counts, out and lse page-locked,
 * mapped into the device's address space (cudaPointerGetAttributes reports
 * host memory with a device pointer) and aligned as the device call wants
 * them, only q is copied: the kernel reads the index list and the counts from
 * host memory and writes out and lse there itself (every kernel reads and
 * writes them with plain loads and stores; copies = 1 turns this off). On
 * the warp-MMA plan (SMD_KERNEL_MMA), which loads q with 16-byte cp.async,
 * and for a bf16 query on the spread plan (read only by the split into E4M3
 * halves), a mapped q is read in place as well and nothing is copied; on the
 * other plans a mapped q is pulled into the workspace by a small copy kernel
 * (the SMs' loads read host memory faster than one copy-engine transfer).
 * The results are the same bits.
 * Each chunk is decoded by the device call for its rows, so chunks = 1 gives
 * the bits of that call on all B rows, and more chunks give the bits of the
 * device calls on the chunks' rows (with the workspace when the whole batch's
 * plan is the spread kernel, else without one: a chunk runs the kernel of the
 * whole batch). Calls of several chunks from several host threads are
 * serialised while they queue their work; such a call being captured into a
 * CUDA graph keeps the device's copy streams in that capture until it ends,
 * so no other thread may make one for the same device meanwhile. Returns SMD_OK or a
 * negative smd_status (argument errors before anything is queued). */
int smd_sparse_mla_decode_host(const void* q_host, const uint8_t* kv_pool, int64_t N,
                               const int32_t* indices_host, int32_t W, const int32_t* counts_host,
                               int32_t B, int32_t H,
                               float sm_scale, float q_scale, float k_scale,
                               uint16_t* out_host, float* lse_host, int32_t* status,
                               void* workspace, int64_t workspace_bytes,
                               const smd_host_opts_t* opts, smd_stream_t stream);

/* Bytes of device workspace smd_topk_select_host needs when it copies:
 * staging for the logits (rows padded to a multiple of 8), row ends,
 * indices and counts, each 256-byte aligned. Negative for invalid shapes.
 * Host only. */
int64_t smd_workspace_bytes_topk_host(int32_t B, int32_t L, int32_t K);

/* The top-k select with its inputs and outputs in host memory: logits_host
 * [B, row_stride] bf16 bits and row_ends_host [B] (or NULL) are read, and
 * indices_host [B, K] and counts_host [B] written, as by smd_topk_select
 * (same arguments, same results). When all of them are page-locked and
 * mapped into the device's address space (and copies == 0), the select reads
 * and writes them in place (its kernel uses plain loads and stores); the
 * workspace is then not touched and may be NULL. Otherwise the logits are
 * copied into the workspace (at least smd_workspace_bytes_topk_host bytes,
 * 16-byte aligned, else SMD_ERR_WORKSPACE) with rows padded to a multiple of
 * 8 logits, and the results are copied back, all on `stream` in order.
 * copies: 0 the library's choice, 1 always copy (other values SMD_ERR_PLAN).
 * Asynchronous on `stream`; the results are in the host buffers once `stream`
 * has reached this point. */
int smd_topk_select_host(const uint16_t* logits_host, int64_t row_stride,
                         const int32_t* row_ends_host, int32_t B, int32_t L, int32_t K,
                         int32_t* indices_host, int32_t* counts_host, int32_t* status,
                         void* workspace, int64_t workspace_bytes, int32_t copies,
                         smd_stream_t stream);

/* The base-2 logit scale the kernels use: fp32(sm*q_s*k_s*log2 e),
 * evaluated in double and rounded once. */
float smd_scale_log2(float sm_scale, float q_scale, float k_scale);

/* Range check of an index list before a decode: for every row b < B and
 * entry i < n_b = clamp(counts[b], 0, W), indices[b, i] must lie in [0, N).
 * The attn_sparse page's kernel gathers the rows an index list names without
 * such a check (SparseDcpDecode.kernel, the gather loop), and so do the
 * decode calls here, where an out-of-range entry reads outside the cache
 * pool; a caller that cannot vouch for its lists runs this first, reads
 * `status`, and decodes only if it is still SMD_OK.
 *   indices  [B, W] int32 device memory (4-byte aligned); entries past a
 *            row's count are not read.
 *   counts   [B] int32 device memory (4-byte aligned).
 *   N        rows of the cache pool the lists index.
 *   status   device int32 (4-byte aligned), required; the caller zeroes it
 *            beforehand. SMD_ERR_INDEX is written there (first writer wins)
 *            if any valid entry lies outside [0, N); it is left untouched
 *            otherwise.
 * Reads the counts and the valid entries only; no entry is used as an
 * address. Asynchronous on `stream`. Returns SMD_OK, or SMD_ERR_SHAPE (B, W
 * or N negative), SMD_ERR_NULL, SMD_ERR_ALIGN, SMD_ERR_DEVICE,
 * SMD_ERR_LAUNCH with nothing launched. B == 0 is a no-op. */
int smd_validate_indices(const int32_t* indices, int32_t W, const int32_t* counts, int32_t B,
                         int64_t N, int32_t* status, smd_stream_t stream);

/* Measurement aid, not part of the decode: the rate probe of the FP8 tensor
 * pipe that gives the tensor side of the decode's roofline its denominator
 * (the pages state no tensor peak for this part). Launches one CTA per SM,
 * each issuing `iters` tcgen05.mma.kind::f8f6f4 instructions (E4M3 x E4M3 ->
 * FP32, M = 128, N = 256, K = 32 as in the decode's PV; both operands K-major
 * in the 128-byte swizzle) back to back into one TMEM accumulator;
 * every instruction is 2 * 128 * 256 * 32 FLOPs. The caller times the
 * launch on `stream` (CUDA events) and divides. *ctas (optional, host
 * memory) receives the number of CTAs launched; `status` (optional device
 * int32) receives SMD_ERR_TIMEOUT if the completion wait (2 s) runs out.
 * Returns SMD_OK, SMD_ERR_SHAPE (iters < 1), SMD_ERR_ALIGN, SMD_ERR_DEVICE
 * or SMD_ERR_LAUNCH. */
int smd_fp8_mma_probe(int32_t iters, int32_t* status, smd_stream_t stream, int32_t* ctas);

/* Diagnostics of a tracing build (the library built with -DSMD_TRACE:
 * sparse_mla_decode_gb300.build.build(trace=True), loaded by the binding when
 * SMD_TRACE_BUILD=1; `python -m sparse_mla_decode_gb300.phases` prints the
 * timeline). Each traced kernel (SMD_KERNEL_MMA, SMD_KERNEL_TC,
 * SMD_KERNEL_TC_SPREAD) keeps a table of 8192 rows x 32 uint64 %globaltimer
 * readings (ns) in device memory: row = CTA (blockIdx.y * gridDim.x +
 * blockIdx.x; for the spread kernel 4 * blockIdx.x + round, rounds 0..3),
 * slot = the phase that just ended (the phase list is in the kernel's
 * source). A launch overwrites the stamps of the rows it runs.
 *   smd_trace_enabled  1 in a tracing build, else 0.
 *   smd_trace_read     copies the first n (<= 8192 * 32) stamps of `kernel`'s
 *                      table to host memory; synchronous.
 *   smd_trace_clear    zeroes the table; synchronous.
 * Both return SMD_OK, SMD_ERR_PLAN (not a tracing build, or a kernel without
 * a table), SMD_ERR_NULL, SMD_ERR_SHAPE or SMD_ERR_LAUNCH. */
int smd_trace_enabled(void);
int smd_trace_read(int32_t kernel, uint64_t* host, int32_t n);
int smd_trace_clear(int32_t kernel);

/* Static text for a status code. */
const char* smd_status_str(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int smd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SMD_H */
