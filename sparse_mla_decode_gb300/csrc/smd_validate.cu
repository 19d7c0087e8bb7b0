// Range check of a decode's index list (smd_validate_indices).
//
// The attn_sparse page's kernel reads a row's cache-row indices and gathers
// them without a range check (SparseDcpDecode.kernel, the gather loop), and
// so do the decode kernels here: an index outside [0, N) of a valid entry is
// the caller's error and would make the gather read outside the pool. This
// kernel is the check a caller can run first. It reads the counts and the
// first count entries of every row, compares each entry with [0, N), and
// writes SMD_ERR_INDEX to the status word when one lies outside; it never
// uses an index as an address.
#include <cstdint>

#include "smd.h"
#include "smd_internal.h"
#include "smd_ptx.cuh"

namespace smd {
namespace {

constexpr int kThreads = 256;

// Block r takes rows r, r + grid, ...; its threads read the row's valid
// entries with consecutive loads.
__global__ void __launch_bounds__(kThreads) validate_kernel(const int32_t* indices, int32_t W,
                                                            const int32_t* counts, int32_t B,
                                                            int64_t N, int32_t* status) {
    pdl_entry();
    bool bad = false;
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        const int n = max(min(counts[b], W), 0);
        const int32_t* row = indices + static_cast<int64_t>(b) * W;
        for (int i = threadIdx.x; i < n; i += kThreads) {
            const int32_t v = row[i];
            bad = bad || v < 0 || static_cast<int64_t>(v) >= N;
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicCAS(status, 0, SMD_ERR_INDEX);
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace smd

extern "C" int smd_validate_indices(const int32_t* indices, int32_t W, const int32_t* counts,
                                    int32_t B, int64_t N, int32_t* status, smd_stream_t stream) {
    if (B < 0 || W < 0 || N < 0) return SMD_ERR_SHAPE;
    if (status == nullptr) return SMD_ERR_NULL;
    if (B == 0) return SMD_OK;
    if (counts == nullptr || (W > 0 && indices == nullptr)) return SMD_ERR_NULL;
    if (!smd::aligned4(status) || !smd::aligned4(counts) || (indices && !smd::aligned4(indices)))
        return SMD_ERR_ALIGN;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SMD_ERR_DEVICE;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(B < 4 * sms ? B : 4 * sms), 1, 1);
    lc.blockDim = dim3(smd::kThreads, 1, 1);
    lc.stream = reinterpret_cast<cudaStream_t>(stream);
    // Programmatic dependent launch, as the other kernels of the library.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, smd::validate_kernel, indices, W, counts, B, N, status) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return SMD_ERR_LAUNCH;
    }
    return SMD_OK;
}
