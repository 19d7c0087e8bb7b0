// The decode and the top-k select from and to host memory
// (smd_sparse_mla_decode_host, smd_topk_select_host): the kernels read and
// write mapped page-locked host buffers in place where they can; otherwise
// the data is copied, for the decode in row chunks whose copies in, decode
// and copies out are pipelined over a few library-owned copy streams and the
// caller's stream. Host code only; every launch goes through the public
// device calls.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "smd.h"
#include "smd_internal.h"

namespace smd {
namespace {

constexpr int kMaxChunks = 8;
constexpr int kAutoChunks = 4;
constexpr int64_t kStageAlign = 256;
// Calls moving at most this much host data take one chunk (the decode reads
// and writes the host buffers in place when it can: that beat pipelined
// copies up to this size); larger ones are chunked when the device fills.
constexpr int64_t kOneChunkMaxBytes = int64_t(16) << 20;
constexpr int kHostMaxDevices = 64;
// Events a call takes: chunk 0's uploads done, one per later upload and per
// decode but the last, and the join.
constexpr int kEventsPerDevice = 2 + 2 * kMaxChunks;

int64_t round_up(int64_t x) { return (x + kStageAlign - 1) / kStageAlign * kStageAlign; }

bool is_aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

struct Opts {
    int G = 1;            // rows per group sharing one index list
    bool bf16 = false;    // the query is bfloat16
    int chunks = 0;       // 0: automatic
    bool copies = false;  // always copy through the workspace
};


int read_opts(const smd_host_opts_t* o, Opts* out) {
    Opts r;
    if (o != nullptr) {
        if ((o->bf16_query != 0 && o->bf16_query != 1) || (o->copies != 0 && o->copies != 1))
            return SMD_ERR_PLAN;
        r.G = o->row_group == 0 ? 1 : o->row_group;
        r.bf16 = o->bf16_query != 0;
        r.chunks = o->chunks;
        r.copies = o->copies != 0;
    }
    if (r.G != 1 && r.G != 2 && r.G != 4) return SMD_ERR_SHAPE;
    if (r.bf16 && r.G != 1) return SMD_ERR_PLAN;
    if (r.chunks < 0 || r.chunks > kMaxChunks) return SMD_ERR_PLAN;
    *out = r;
    return SMD_OK;
}

int host_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();  // no device here: plan for a GB300
        return 152;
    }
    return sms;
}

// Workspace bytes the device call wants for B rows (the spread kernel's), 0
// when its plan needs none.
int64_t device_ws(int B, int H, int W, const Opts& o) {
    if (o.bf16) return smd_workspace_bytes_bf16q(B, H, W);
    if (o.G > 1) return smd_workspace_bytes_grouped(B, H, W, o.G);
    return smd_workspace_bytes(B, H, W);
}

// The plan of the device call on all B rows given its workspace.
int whole_plan(int B, int H, int W, const Opts& o, smd_plan_t* p) {
    const int64_t ws = device_ws(B, H, W, o);
    if (o.bf16) return smd_plan_bf16q(B, H, W, ws, p);
    if (o.G > 1) return smd_plan_grouped(B, H, W, o.G, ws, p);
    return smd_plan_ws(B, H, W, p);
}

// Where the staging buffers sit in the workspace, and how the rows are cut.
struct Layout {
    int chunks = 1, rows = 0;  // chunk c holds rows r0[c] .. r0[c + 1] - 1; rows: the most in one
    int r0[kMaxChunks + 1] = {};
    int kernel = 0;            // the whole batch's plan (SMD_KERNEL_*)
    bool spread = false;       // the whole batch's plan is the spread kernel
    int64_t q_row = 0;         // bytes of one row of q
    int64_t off_q = 0, off_idx = 0, off_cnt = 0, off_out = 0, off_lse = 0, off_dws = 0;
    int64_t dws_bytes = 0, total = 0;
};

// Chunks cut at whole waves of the cluster kernel (rows per wave: the clusters
// the device holds at once over the clusters a row takes): a one-wave chunk
// first (its upload is short, so the first decode starts early), then
// chunks of two waves, then the rows of the last, partial wave (its output
// is small, so little is left to move out after the last decode). A chunk
// that ended inside a wave would cost that wave's whole duration again.
// Unchanged when fewer than three waves.
void wave_chunks(int B, int G, const smd_plan_t& p, Layout* r) {
    const int split = std::max(p.split, 1);
    int clusters = tc_resident_clusters(split);
    if (clusters <= 0) clusters = host_sm_count() / split;  // no device: every SM
    const int per_row = std::max(p.grid_x / split, 1);     // clusters a row takes
    const int rpw = clusters / per_row / G * G;              // rows per wave
    if (rpw <= 0) return;
    const int full = B / rpw, rem = B - full * rpw;
    if (full < 3) return;
    int w[kMaxChunks];  // waves per chunk (the partial wave apart)
    int n = 0;
    w[n++] = 1;
    const int slots = kMaxChunks - 1 - (rem > 0 ? 1 : 0);  // chunks left for the middle waves
    const int middle = full - 1;
    const int per_chunk = std::max(2, (middle + slots - 1) / slots);
    for (int left = middle; left > 0; left -= per_chunk) w[n++] = std::min(per_chunk, left);
    int row = 0;
    for (int c = 0; c < n; ++c) {
        r->r0[c] = row;
        row += w[c] * rpw;
    }
    r->chunks = n;
    if (rem > 0) r->r0[r->chunks++] = row;
    r->r0[r->chunks] = B;
}

int layout_of(int B, int H, int W, const Opts& o, Layout* L) {
    if (B < 0 || W < 0 || H <= 0 || H % 16 != 0) return SMD_ERR_SHAPE;
    if (B % o.G != 0) return SMD_ERR_SHAPE;
    Layout r;
    r.q_row = static_cast<int64_t>(H) * 576 * (o.bf16 ? 2 : 1);
    if (B > 0) {
        smd_plan_t p{};
        const int rc = whole_plan(B, H, W, o, &p);
        if (rc != SMD_OK) return rc;
        r.kernel = p.kernel;
        r.spread = p.kernel == SMD_KERNEL_TC_SPREAD;
        int chunks = o.chunks;
        if (chunks == 0) {
            // Chunks pay for large host data when each still fills the device:
            // at least three waves of CTAs in all, one and a half per chunk.
            const int64_t host_bytes =
                static_cast<int64_t>(B) * (r.q_row + static_cast<int64_t>(W) * 4 + 4 +
                                           static_cast<int64_t>(H) * (1024 + 4));
            const int64_t ctas = static_cast<int64_t>(std::max(p.grid_x, 1)) * std::max(p.grid_y, 1);
            const int64_t sms = host_sm_count();
            chunks = (host_bytes <= kOneChunkMaxBytes || r.spread || ctas < 3 * sms)
                         ? 1
                         : static_cast<int>(std::min<int64_t>(kAutoChunks, ctas * 2 / (3 * sms)));
        }
        const int groups = B / o.G;
        chunks = std::max(1, std::min(chunks, groups));
        const int per = (groups + chunks - 1) / chunks;  // groups per chunk
        r.chunks = (groups + per - 1) / per;
        for (int c = 0; c <= r.chunks; ++c) r.r0[c] = std::min(B, c * per * o.G);
        if (o.chunks == 0 && r.chunks > 1 && p.kernel == SMD_KERNEL_TC)
            wave_chunks(B, o.G, p, &r);
        for (int c = 0; c < r.chunks; ++c) r.rows = std::max(r.rows, r.r0[c + 1] - r.r0[c]);
        // A chunk is decoded by the device call the whole batch would use: with
        // the workspace when that is the spread kernel, else without one.
        r.dws_bytes = r.spread ? device_ws(r.rows, H, W, o) : 0;
        if (r.dws_bytes < 0) return SMD_ERR_SHAPE;
    }
    int64_t off = 0;
    r.off_q = off;
    off += round_up(static_cast<int64_t>(B) * r.q_row);
    r.off_idx = off;
    off += round_up(static_cast<int64_t>(B) * W * 4);
    r.off_cnt = off;
    off += round_up(static_cast<int64_t>(B) * 4);
    r.off_out = off;
    off += round_up(static_cast<int64_t>(B) * H * 512 * 2);
    r.off_lse = off;
    off += round_up(static_cast<int64_t>(B) * H * 4);
    r.off_dws = off;
    off += round_up(r.dws_bytes);
    r.total = off;
    *L = r;
    return SMD_OK;
}

// The device address of a page-locked host buffer mapped into the current
// device's address space, or null (pageable memory, device memory, unknown).
const void* mapped_host(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// A copy from mapped host memory into device memory by the SMs' own loads
// (16-byte pieces, grid-stride): over the C2C link these run faster than the
// copy engine does for a single copy.
__global__ void __launch_bounds__(256) host_to_device16(const uint4* __restrict__ src,
                                                        uint4* __restrict__ dst, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = __ldg(src + i);
}

// The library's copy streams and events of one device, created on first use
// (only calls of more than one chunk use them).
struct CopyEngine {
    std::once_flag once;
    std::mutex mu;  // held while a call queues its work
    bool ok = false;
    cudaStream_t up = nullptr;    // uploads of chunks 1 ..
    cudaStream_t down = nullptr;  // downloads of every chunk but the last
    cudaEvent_t ev[kEventsPerDevice] = {};
};

CopyEngine g_engines[kHostMaxDevices];

CopyEngine* engine_of_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kHostMaxDevices) return nullptr;
    CopyEngine& e = g_engines[dev];
    std::call_once(e.once, [&e] {
        bool ok = cudaStreamCreateWithFlags(&e.up, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&e.down, cudaStreamNonBlocking) == cudaSuccess;
        for (auto& v : e.ev) ok = ok && cudaEventCreateWithFlags(&v, cudaEventDisableTiming) == cudaSuccess;
        e.ok = ok;
    });
    return e.ok ? &e : nullptr;
}

}  // namespace
}  // namespace smd

extern "C" {

int smd_plan_host(int32_t B, int32_t H, int32_t W, const smd_host_opts_t* opts, int32_t* chunks) {
    if (chunks == nullptr) return SMD_ERR_NULL;
    smd::Opts o;
    int rc = smd::read_opts(opts, &o);
    if (rc != SMD_OK) return rc;
    smd::Layout L;
    rc = smd::layout_of(B, H, W, o, &L);
    if (rc != SMD_OK) return rc;
    *chunks = L.chunks;
    return SMD_OK;
}

int64_t smd_workspace_bytes_host(int32_t B, int32_t H, int32_t W, const smd_host_opts_t* opts) {
    smd::Opts o;
    int rc = smd::read_opts(opts, &o);
    if (rc != SMD_OK) return rc;
    smd::Layout L;
    rc = smd::layout_of(B, H, W, o, &L);
    return rc != SMD_OK ? rc : L.total;
}

int smd_sparse_mla_decode_host(const void* q_host, const uint8_t* kv_pool, int64_t N,
                               const int32_t* indices_host, int32_t W, const int32_t* counts_host,
                               int32_t B, int32_t H, float sm_scale, float q_scale, float k_scale,
                               uint16_t* out_host, float* lse_host, int32_t* status,
                               void* workspace, int64_t workspace_bytes,
                               const smd_host_opts_t* opts, smd_stream_t stream) {
    using namespace smd;
    Opts o;
    int rc = read_opts(opts, &o);
    if (rc != SMD_OK) return rc;
    Layout L;
    rc = layout_of(B, H, W, o, &L);
    if (rc != SMD_OK) return rc;
    if (N < 0 || N >= (int64_t(1) << 31)) return SMD_ERR_SHAPE;
    if (B == 0) return SMD_OK;
    // The argument checks of the device call, before anything is queued.
    if (!q_host || !counts_host || !out_host || !lse_host || !workspace) return SMD_ERR_NULL;
    if (W > 0 && (!indices_host || !kv_pool)) return SMD_ERR_NULL;
    if (W > 0 && N == 0) return SMD_ERR_SHAPE;
    if ((kv_pool && !is_aligned(kv_pool, 16)) || (status && !is_aligned(status, 4)))
        return SMD_ERR_ALIGN;
    if (!is_aligned(workspace, 16) || workspace_bytes < L.total) return SMD_ERR_WORKSPACE;
    // Direct access (one chunk): every kernel reads the index list and the
    // counts with plain loads and writes out and lse with plain stores (TMA
    // touches only the query and the cache pool), so when those four host
    // buffers are page-locked and mapped into the device's address space they
    // are handed to the device call as they are, and only q is copied. The
    // warp-MMA kernel (SMD_KERNEL_MMA) loads q with 16-byte cp.async, and a
    // bf16 query is read only by the split into E4M3 halves (plain loads, in
    // the warp-MMA kernel or in the split kernel before the spread kernel),
    // so there q is read in place too; the others bring it in by TMA or bulk
    // copies, which are kept to device memory. (With several chunks the copy
    // engines move the data faster than the kernels' own host-memory traffic:
    // throughput 325 against 418 us.)
    const int32_t* m_idx = nullptr;
    const int32_t* m_cnt = nullptr;
    uint16_t* m_out = nullptr;
    float* m_lse = nullptr;
    const uint8_t* q_mapped = nullptr;
    if (!o.copies) {
        if (W > 0 && is_aligned(indices_host, 4))
            m_idx = static_cast<const int32_t*>(mapped_host(indices_host));
        if (is_aligned(counts_host, 4)) m_cnt = static_cast<const int32_t*>(mapped_host(counts_host));
        if (is_aligned(out_host, 16))
            m_out = static_cast<uint16_t*>(const_cast<void*>(mapped_host(out_host)));
        if (is_aligned(lse_host, 4)) m_lse = static_cast<float*>(const_cast<void*>(mapped_host(lse_host)));
        if (is_aligned(q_host, 16)) q_mapped = static_cast<const uint8_t*>(mapped_host(q_host));
    }
    // One chunk: everything in place when indices, counts, out and lse are.
    const bool direct = L.chunks == 1 && (m_idx != nullptr || W == 0) && m_cnt && m_out && m_lse;
    const bool q_by_loads = L.kernel == SMD_KERNEL_MMA || (o.bf16 && L.kernel == SMD_KERNEL_TC_SPREAD);
    const uint8_t* m_q = (direct && q_by_loads) ? q_mapped : nullptr;
    // Otherwise a mapped q is pulled into the staging area by the SMs' loads:
    // on one chunk, and for chunk 0 of several (nothing is decoded yet then,
    // so the copy kernel has the SMs; later chunks' copies overlap decodes and
    // stay on the copy engine).
    const uint8_t* q_pull = m_q != nullptr ? nullptr : q_mapped;
    // Several chunks: the last chunk's out and lse go straight to host memory
    // when mapped (no download after the last decode).
    const bool last_in_place = L.chunks > 1 && m_out && m_lse;

    CopyEngine* eng = nullptr;
    if (L.chunks > 1) {
        eng = engine_of_current_device();
        if (eng == nullptr) return SMD_ERR_DEVICE;
    }

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint8_t* dq = m_q != nullptr ? const_cast<uint8_t*>(m_q) : ws + L.off_q;
    const int32_t* didx = direct ? m_idx : reinterpret_cast<const int32_t*>(ws + L.off_idx);
    const int32_t* dcnt = direct ? m_cnt : reinterpret_cast<const int32_t*>(ws + L.off_cnt);
    uint16_t* const sout = reinterpret_cast<uint16_t*>(ws + L.off_out);
    float* const slse = reinterpret_cast<float*>(ws + L.off_lse);
    void* dws = L.dws_bytes > 0 ? ws + L.off_dws : nullptr;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const int64_t out_row = static_cast<int64_t>(H) * 512 * 2, lse_row = static_cast<int64_t>(H) * 4;
    // Where chunk c's out and lse go: host memory (in place) or staging.
    auto in_place = [&](int c) { return direct || (last_in_place && c == L.chunks - 1); };

    std::unique_lock<std::mutex> lock;
    if (eng != nullptr) lock = std::unique_lock<std::mutex>(eng->mu);
    int next_ev = 0;
    auto take = [&]() { return eng->ev[next_ev++]; };
    bool cuda_ok = true;
    auto chk = [&](cudaError_t e) { cuda_ok = cuda_ok && e == cudaSuccess; };
    int result = SMD_OK;

    // Chunk c's copies in / out, queued on s. The counts of all rows go in
    // with chunk 0 and the LSE of the staged chunks comes back in one copy at
    // the end (both are small): fewer calls for the host to issue.
    auto upload = [&](int c, cudaStream_t s) {
        const int r0 = L.r0[c], nr = L.r0[c + 1] - r0;
        if (q_pull != nullptr && c == 0) {
            const int64_t n16 = nr * L.q_row / 16;  // q rows are multiples of 16 bytes
            const int blocks = static_cast<int>(std::min<int64_t>((n16 + 255) / 256, 4 * host_sm_count()));
            host_to_device16<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(q_pull + r0 * L.q_row),
                                                    reinterpret_cast<uint4*>(dq + r0 * L.q_row), n16);
            chk(cudaGetLastError());
        } else if (m_q == nullptr) {
            chk(cudaMemcpyAsync(dq + r0 * L.q_row, static_cast<const uint8_t*>(q_host) + r0 * L.q_row,
                                nr * L.q_row, cudaMemcpyHostToDevice, s));
        }
        if (direct) return;
        if (W > 0)
            chk(cudaMemcpyAsync(const_cast<int32_t*>(didx) + static_cast<int64_t>(r0) * W,
                                indices_host + static_cast<int64_t>(r0) * W,
                                static_cast<int64_t>(nr) * W * 4, cudaMemcpyHostToDevice, s));
        if (c == 0)
            chk(cudaMemcpyAsync(const_cast<int32_t*>(dcnt), counts_host, static_cast<int64_t>(B) * 4,
                                cudaMemcpyHostToDevice, s));
    };
    auto download = [&](int c, cudaStream_t s) {
        if (in_place(c)) return;  // the kernel wrote them in host memory
        const int r0 = L.r0[c], nr = L.r0[c + 1] - r0;
        chk(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(out_host) + r0 * out_row,
                            reinterpret_cast<const uint8_t*>(sout) + r0 * out_row, nr * out_row,
                            cudaMemcpyDeviceToHost, s));
    };
    // The LSE of every staged chunk, once they are all decoded (on `stream`).
    auto download_lse = [&]() {
        int staged = 0;  // chunks 0 .. staged - 1 are staged (only the last can be in place)
        while (staged < L.chunks && !in_place(staged)) ++staged;
        const int nr = L.r0[staged];
        if (nr > 0)
            chk(cudaMemcpyAsync(lse_host, slse, nr * lse_row, cudaMemcpyDeviceToHost, cs));
    };
    auto decode = [&](int c) {
        const int r0 = L.r0[c], nr = L.r0[c + 1] - r0;
        const int32_t* ci = didx + static_cast<int64_t>(r0) * W;
        uint16_t* co = (in_place(c) ? m_out : sout) + static_cast<int64_t>(r0) * H * 512;
        float* cl = (in_place(c) ? m_lse : slse) + static_cast<int64_t>(r0) * H;
        const int64_t dbytes = dws != nullptr ? L.dws_bytes : 0;
        if (o.bf16)
            return smd_sparse_mla_decode_bf16q_ws(reinterpret_cast<const uint16_t*>(dq + r0 * L.q_row),
                                                  kv_pool, N, ci, W, dcnt + r0, nr, H, sm_scale,
                                                  k_scale, co, cl, status, dws, dbytes, stream);
        if (o.G > 1)
            return smd_sparse_mla_decode_grouped_ws(dq + r0 * L.q_row, kv_pool, N, ci, W, dcnt + r0,
                                                    nr, H, o.G, sm_scale, q_scale, k_scale, co, cl,
                                                    status, dws, dbytes, stream);
        return smd_sparse_mla_decode_ws(dq + r0 * L.q_row, kv_pool, N, ci, W, dcnt + r0, nr, H,
                                        sm_scale, q_scale, k_scale, co, cl, status, dws, dbytes,
                                        stream);
    };

    // Chunk 0 moves in on `stream` itself and is decoded there at once; each
    // later chunk moves in on the upload stream (one after another, after
    // chunk 0: concurrent uploads would share the bandwidth chunk 0 needs
    // first) and is decoded on `stream` once it is in; every chunk but the
    // last goes back on the download stream while the next one is decoded,
    // the last on `stream`. The calls are issued in the order the device
    // needs them (decode c before upload c + 1), so that the device never
    // waits for the host to issue the next decode.
    upload(0, cs);
    if (L.chunks > 1) {
        const cudaEvent_t up0 = take();
        chk(cudaEventRecord(up0, cs));
        chk(cudaStreamWaitEvent(eng->up, up0, 0));
        chk(cudaStreamWaitEvent(eng->down, up0, 0));
    }
    cudaEvent_t up_done = nullptr;
    for (int c = 0; c < L.chunks && cuda_ok; ++c) {
        if (c > 0) chk(cudaStreamWaitEvent(cs, up_done, 0));
        if (!cuda_ok) break;
        rc = decode(c);
        if (rc != SMD_OK) {
            result = rc;
            break;
        }
        if (c + 1 < L.chunks) {
            upload(c + 1, eng->up);
            up_done = take();
            chk(cudaEventRecord(up_done, eng->up));
            const cudaEvent_t done = take();
            chk(cudaEventRecord(done, cs));
            chk(cudaStreamWaitEvent(eng->down, done, 0));
            download(c, eng->down);
        } else {
            download(c, cs);
        }
    }
    if (result == SMD_OK && cuda_ok && !direct) download_lse();
    // Join: `stream` continues after the download stream's last copy (every
    // upload was waited for before its chunk's decode on `stream`).
    if (L.chunks > 1) {
        const cudaEvent_t down_end = take();
        chk(cudaEventRecord(down_end, eng->down));
        chk(cudaStreamWaitEvent(cs, down_end, 0));
    }
    if (result == SMD_OK && !cuda_ok) result = SMD_ERR_LAUNCH;
    return result;
}

int64_t smd_workspace_bytes_topk_host(int32_t B, int32_t L, int32_t K) {
    using namespace smd;
    if (B < 0 || L < 0 || K < 1) return SMD_ERR_SHAPE;
    const int64_t pitch = (static_cast<int64_t>(L) + 7) / 8 * 8;  // staged rows: 16-byte pieces
    return round_up(B * pitch * 2) + round_up(static_cast<int64_t>(B) * 4) +
           round_up(static_cast<int64_t>(B) * K * 4) + round_up(static_cast<int64_t>(B) * 4);
}

int smd_topk_select_host(const uint16_t* logits_host, int64_t row_stride,
                         const int32_t* row_ends_host, int32_t B, int32_t L, int32_t K,
                         int32_t* indices_host, int32_t* counts_host, int32_t* status,
                         void* workspace, int64_t workspace_bytes, int32_t copies,
                         smd_stream_t stream) {
    using namespace smd;
    if (B < 0 || L < 0 || K < 1 || row_stride < L) return SMD_ERR_SHAPE;
    if (copies != 0 && copies != 1) return SMD_ERR_PLAN;
    if (B == 0) return SMD_OK;
    if (!indices_host || !counts_host || (L > 0 && !logits_host)) return SMD_ERR_NULL;
    if ((logits_host && !is_aligned(logits_host, 2)) || !is_aligned(indices_host, 4) ||
        !is_aligned(counts_host, 4) || (row_ends_host && !is_aligned(row_ends_host, 4)) ||
        (status && !is_aligned(status, 4)))
        return SMD_ERR_ALIGN;

    // Direct access: the select reads the logits and the row ends with plain
    // loads and writes the indices and counts with plain stores, so mapped
    // page-locked host buffers go to the device call as they are.
    if (!copies) {
        const void* ml = L > 0 ? mapped_host(logits_host) : nullptr;
        const void* me = row_ends_host ? mapped_host(row_ends_host) : nullptr;
        const void* mi = mapped_host(indices_host);
        const void* mc = mapped_host(counts_host);
        if ((ml || L == 0) && (me || !row_ends_host) && mi && mc)
            return smd_topk_select(static_cast<const uint16_t*>(ml), row_stride,
                                   static_cast<const int32_t*>(me), B, L, K,
                                   static_cast<int32_t*>(const_cast<void*>(mi)),
                                   static_cast<int32_t*>(const_cast<void*>(mc)), status, stream);
    }

    // Copies: the logits into rows of a multiple of 8 logits (so the select
    // reads them in 16-byte pieces), the select, the results back; all on
    // `stream` in order.
    const int64_t need = smd_workspace_bytes_topk_host(B, L, K);
    if (!workspace || !is_aligned(workspace, 16) || workspace_bytes < need) return SMD_ERR_WORKSPACE;
    const int64_t pitch = (static_cast<int64_t>(L) + 7) / 8 * 8;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint16_t* dx = reinterpret_cast<uint16_t*>(ws);
    int32_t* de = reinterpret_cast<int32_t*>(ws + round_up(B * pitch * 2));
    int32_t* di = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(de) + round_up(int64_t(B) * 4));
    int32_t* dc = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(di) +
                                             round_up(static_cast<int64_t>(B) * K * 4));
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    bool ok = true;
    if (L > 0)
        ok = cudaMemcpy2DAsync(dx, pitch * 2, logits_host, row_stride * 2, static_cast<size_t>(L) * 2,
                               B, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    if (ok && row_ends_host)
        ok = cudaMemcpyAsync(de, row_ends_host, static_cast<size_t>(B) * 4, cudaMemcpyHostToDevice,
                             cs) == cudaSuccess;
    if (!ok) return SMD_ERR_LAUNCH;
    const int rc = smd_topk_select(L > 0 ? dx : nullptr, pitch, row_ends_host ? de : nullptr, B, L,
                                   K, di, dc, status, stream);
    if (rc != SMD_OK) return rc;
    ok = cudaMemcpyAsync(indices_host, di, static_cast<size_t>(B) * K * 4, cudaMemcpyDeviceToHost,
                         cs) == cudaSuccess &&
         cudaMemcpyAsync(counts_host, dc, static_cast<size_t>(B) * 4, cudaMemcpyDeviceToHost, cs) ==
             cudaSuccess;
    return ok ? SMD_OK : SMD_ERR_LAUNCH;
}

}  // extern "C"
