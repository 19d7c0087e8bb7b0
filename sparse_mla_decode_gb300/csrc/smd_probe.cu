// Rate probe of the FP8 tensor pipe (smd_fp8_mma_probe): the denominator of
// the tensor side of the decode's roofline, measured on the GPU it runs on.
//
// One CTA per SM; one thread issues `iters` tcgen05.mma.cta_group::1
// .kind::f8f6f4 instructions back to back (E4M3 x E4M3 -> FP32, M = 128,
// N = 256, K = 32 as in the decode's PV products; both operands K-major in
// the 128-byte swizzle) from two zeroed shared-memory tiles into one TMEM
// accumulator, commits them to an mbarrier and waits for it (bounded). Each instruction is 2 * 128 * 256 * 32 FLOPs;
// the caller times the launch with CUDA events.
#include <cstdint>

#include "smd.h"
#include "smd_internal.h"
#include "smd_ptx.cuh"

namespace smd {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kTileA = 128 * 128;  // 128 rows x 128 bytes
constexpr int kTileB = 256 * 128;  // 256 rows x 128 bytes
// Dynamic shared memory asked for: the tiles fit in 48 KB; asking for more
// keeps one CTA per SM.
constexpr int kProbeSmem = 160 * 1024;

__global__ void __launch_bounds__(kProbeThreads, 1) fp8_mma_probe_kernel(int iters, int32_t* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t a = smem_addr(smem), b = a + kTileA;
    const uint32_t bar = b + kTileB, slot = bar + 8;
    for (int i = threadIdx.x; i < (kTileA + kTileB) / 16; i += kProbeThreads)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    fence_proxy_async();  // the zeroed tiles -> the tensor core's reads
    if ((threadIdx.x >> 5) == 0) tmem_alloc(slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTileA + kTileB + 8);
    if (threadIdx.x == 0) {
        constexpr uint32_t kId = umma_idesc_e4m3(128, 256, 0);
        for (int i = 0; i < iters; ++i) {
            const int kk = i & 3;
            umma_e4m3(tmem, umma_desc(a + 32 * kk, 16, 1024, 2), umma_desc(b + 32 * kk, 16, 1024, 2),
                      kId, i > 0 ? 1u : 0u);
        }
        umma_commit(bar);
    }
    bool ok = true;
    mbar_wait(bar, 0, ok, status, 2000000000ull);  // 2 s
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        tc_fence_after();
        tmem_free(tmem, 256);
    }
}

}  // namespace
}  // namespace smd

extern "C" int smd_fp8_mma_probe(int32_t iters, int32_t* status, smd_stream_t stream,
                                 int32_t* ctas) {
    if (iters < 1) return SMD_ERR_SHAPE;
    if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u)) return SMD_ERR_ALIGN;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SMD_ERR_DEVICE;
    if (cudaFuncSetAttribute(smd::fp8_mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smd::kProbeSmem) != cudaSuccess) {
        (void)cudaGetLastError();
        return SMD_ERR_LAUNCH;
    }
    smd::fp8_mma_probe_kernel<<<sms, smd::kProbeThreads, smd::kProbeSmem,
                                reinterpret_cast<cudaStream_t>(stream)>>>(iters, status);
    if (cudaGetLastError() != cudaSuccess) return SMD_ERR_LAUNCH;
    if (ctas != nullptr) *ctas = sms;
    return SMD_OK;
}
