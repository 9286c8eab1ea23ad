// Stage checks of the layer's intermediate results, for finding the first
// stage that goes wrong (xserv docs/19-gpt-oss-moe.md, "Phase 19:
// gpt-oss-20b", §3 and §4: the page's two bugs were located by NaN and
// magnitude checks after each stage behind an environment switch).  Off by
// default; moe_api.cu launches one check after each stage when
// MOE_CHECK_STAGES=1.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float value_of(const void* buf, size_t i, int dtype) {
    if (dtype == 1) return static_cast<const float*>(buf)[i];
    if (dtype == 3) return __half2float(static_cast<const __half*>(buf)[i]);
    if (dtype == 2) {
        __nv_fp8_e4m3 c;
        c.__x = static_cast<const uint8_t*>(buf)[i];
        return static_cast<float>(c);
    }
    return __bfloat162float(static_cast<const __nv_bfloat16*>(buf)[i]);
}

__global__ void __launch_bounds__(kThreads)
    stage_check_kernel(const void* buf, size_t n, int dtype, int stage, int32_t* status) {
    pdl_wait();
    int bad = 0;
    float mx = 0.f;
    for (size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * kThreads) {
        const float v = value_of(buf, i, dtype);
        if (isfinite(v))
            mx = fmaxf(mx, fabsf(v));
        else
            ++bad;
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        bad += __shfl_xor_sync(0xffffffffu, bad, d);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    }
    if ((threadIdx.x & 31) == 0) {
        int32_t* w = status + kStageStatsWord + 2 * stage;
        if (bad) {
            atomicAdd(w, bad);
            atomicOr(status + kStatusWord, MOE_DEV_NONFINITE);
        }
        // non-negative floats order like their bit patterns
        atomicMax(w + 1, __float_as_int(mx));
    }
}

}  // namespace

cudaError_t launch_stage_check(const void* buf, size_t n, int dtype, int stage, int32_t* status,
                               cudaStream_t s) {
    if (stage < 0 || stage >= kNumStages) return cudaErrorInvalidValue;
    size_t blocks = (n + kThreads - 1) / kThreads;
    if (blocks > 1024) blocks = 1024;
    if (blocks == 0) blocks = 1;
    stage_check_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(buf, n, dtype, stage,
                                                                           status);
    return cudaGetLastError();
}

}  // namespace moe
