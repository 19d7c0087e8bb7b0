// The bf16 query split into E4M3 hi + lo (the mla_attn page: "q_split", the
// bf16 Q rows to "E4M3 hi, lo of q 2^k"; "fp8_split4", x ~ hi + lo), one
// 576-column query row per warp. Per row the largest k with amax 2^k <= 448
// (k = 0 for a zero row; clamped to [-32, 32]), hi = E4M3(q 2^k) and
// lo = E4M3(q 2^k - hi), both round-to-nearest-even and saturating (q 2^k and
// q 2^k - hi are exact in fp32), and the row's logit scale lam0 2^-k.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "smd_internal.h"
#include "smd_ptx.cuh"

namespace smd {

// The E4M3 values of two codes (exact in f16, then f32).
__device__ __forceinline__ float2 e4m3x2_values(uint16_t codes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
    return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// Splits the bf16 row `src` (576 values, 16-byte aligned) into the E4M3 rows
// hi and lo (8-byte aligned); all 32 lanes of the warp take part. Returns
// lam0 2^-k (every lane).
__device__ __forceinline__ float split_query_row(const uint16_t* src, uint8_t* hi, uint8_t* lo,
                                                 float lam0) {
    const int lane = threadIdx.x & 31;
    constexpr int kPieces = kRow / 8;  // 16-byte pieces of a bf16 row
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4 v[3];
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int piece = lane + 32 * u;
        v[u] = piece < kPieces ? __ldg(s4 + piece) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                                     fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
    }
    amax = warp_max(amax);
    int k = 0;
    if (amax > 0.f) {
        int e = 0;
        const float m = frexpf(amax, &e);  // amax = m 2^e, m in [0.5, 1)
        k = (m <= 0.875f) ? 9 - e : 8 - e;
        k = max(-32, min(32, k));
    }
    const float up = __int_as_float((127 + k) << 23);  // 2^k
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int piece = lane + 32 * u;
        if (piece >= kPieces) continue;
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t hw[2], lw[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x0 = __uint_as_float(w[i] << 16) * up;
            const float x1 = __uint_as_float(w[i] & 0xFFFF0000u) * up;
            const uint16_t hc = e4m3x2(x0, x1);
            const float2 hv = e4m3x2_values(hc);
            const uint16_t lc = e4m3x2(x0 - hv.x, x1 - hv.y);
            if (i & 1) {
                hw[i >> 1] |= static_cast<uint32_t>(hc) << 16;
                lw[i >> 1] |= static_cast<uint32_t>(lc) << 16;
            } else {
                hw[i >> 1] = hc;
                lw[i >> 1] = lc;
            }
        }
        *reinterpret_cast<uint2*>(hi + 8 * piece) = make_uint2(hw[0], hw[1]);
        *reinterpret_cast<uint2*>(lo + 8 * piece) = make_uint2(lw[0], lw[1]);
    }
    return lam0 * __int_as_float((127 - k) << 23);
}

}  // namespace smd
