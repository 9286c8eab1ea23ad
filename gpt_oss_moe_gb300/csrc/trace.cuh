// Per-CTA phase timestamps of the layer's kernels, compiled in only by the
// "trace" build variant (-DMOE_TRACE): each kernel records %globaltimer (ns)
// at fixed points of each of its first kTraceCtas CTAs into a file-scope
// device array, which moe_trace_read copies to the host.  Every call
// overwrites the same slots, so a read describes the last call.
#pragma once

#include <cstddef>

namespace moe {

constexpr int kTraceCtas = 512;
constexpr int kTracePoints = 8;   // every kernel: 8 slots per CTA

#ifdef MOE_TRACE
#define MOE_TRACE_ARRAY(name, kernels) \
    static __device__ unsigned long long name[kernels][kTraceCtas][kTracePoints]
#define MOE_TRACE_POINT(name, k, cta, pt)                                  \
    do {                                                                   \
        const int _c = (cta);                                              \
        if (_c >= 0 && _c < kTraceCtas) {                                  \
            unsigned long long _t;                                         \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(_t));         \
            name[k][_c][pt] = _t;                                          \
        }                                                                  \
    } while (0)
#define MOE_TRACE_COPY(name, dst, cap)                                              \
    do {                                                                            \
        const size_t _n = sizeof(name) / sizeof(unsigned long long);                \
        if ((cap) < _n) return 0;                                                   \
        if (cudaMemcpyFromSymbol((dst), name, sizeof(name)) != cudaSuccess) return 0; \
        return _n;                                                                  \
    } while (0)
#else
#define MOE_TRACE_ARRAY(name, kernels) static_assert(true, "")
#define MOE_TRACE_POINT(name, k, cta, pt) ((void)0)
#define MOE_TRACE_COPY(name, dst, cap) \
    do {                               \
        (void)(dst);                   \
        (void)(cap);                   \
        return 0;                      \
    } while (0)
#endif

// Copy one file's trace array to dst (cap elements); returns the element
// count, 0 when tracing is not compiled in or cap is too small.
size_t trace_copy_router(unsigned long long* dst, size_t cap);
size_t trace_copy_permute(unsigned long long* dst, size_t cap);
size_t trace_copy_gemm(unsigned long long* dst, size_t cap);
size_t trace_copy_attn(unsigned long long* dst, size_t cap);

}  // namespace moe
