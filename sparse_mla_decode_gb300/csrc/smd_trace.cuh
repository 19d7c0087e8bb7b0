// Per-phase timestamps of the decode kernels, for a tracing build only.
//
// Built with -DSMD_TRACE (sparse_mla_decode_gb300.build, trace=True), each
// kernel file keeps one table of kTraceRows x kTraceSlots 64-bit %globaltimer
// readings in device memory and stamps the end of each of its phases into it
// (row = CTA, or CTA and round), and the SM the row ran on into its last slot;
// smd_trace_read / smd_trace_clear copy or zero a kernel's table. In the
// normal build the stamps compile to nothing and the tables do not exist, so
// the product kernels are unchanged.
#pragma once

#include <cstdint>

namespace smd {

constexpr int kTraceRows = 8192;  // CTAs (or CTA x round) a table holds
constexpr int kTraceSlots = 32;   // stamps per row

}  // namespace smd

#ifdef SMD_TRACE

#define SMD_TRACE_TABLE(name) __device__ unsigned long long name[smd::kTraceRows * smd::kTraceSlots]
#define SMD_STAMP(name, row, slot) smd::trace_stamp(name, (row), (slot))
#define SMD_TRACE_SM(name, row) smd::trace_sm(name, (row))

namespace smd {

__device__ __forceinline__ void trace_stamp(unsigned long long* table, int row, int slot) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (row >= 0 && row < kTraceRows && slot >= 0 && slot < kTraceSlots)
        table[row * kTraceSlots + slot] = t;
}

// The SM the row ran on (%smid), in the row's last slot (not a time).
__device__ __forceinline__ void trace_sm(unsigned long long* table, int row) {
    unsigned int v;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
    if (row >= 0 && row < kTraceRows) table[row * kTraceSlots + kTraceSlots - 1] = v;
}

}  // namespace smd

// Host: copy a table out (n stamps) or zero it.
#define SMD_TRACE_COPY_FN(fn, name)                                                            \
    int fn(uint64_t* host, int n, bool clear) {                                                \
        if (clear) {                                                                           \
            static unsigned long long zeros[smd::kTraceRows * smd::kTraceSlots];               \
            return cudaMemcpyToSymbol(name, zeros, sizeof(zeros)) == cudaSuccess ? SMD_OK      \
                                                                                 : SMD_ERR_LAUNCH; \
        }                                                                                      \
        return cudaMemcpyFromSymbol(host, name, sizeof(unsigned long long) * n) == cudaSuccess \
                   ? SMD_OK                                                                    \
                   : SMD_ERR_LAUNCH;                                                           \
    }

#else

#define SMD_TRACE_TABLE(name)
// (The row expression is named, not evaluated: no code, no unused warnings.)
#define SMD_STAMP(name, row, slot) ((void)sizeof(row))
#define SMD_TRACE_SM(name, row) ((void)sizeof(row))
#define SMD_TRACE_COPY_FN(fn, name) \
    int fn(uint64_t*, int, bool) { return SMD_ERR_PLAN; }

#endif
