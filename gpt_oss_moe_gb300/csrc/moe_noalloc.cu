// moe_forward_noalloc: the layer forward for callers that cannot allocate
// device memory.
//
// Some hosts hand a plugin only its input and output buffers and plan every
// other byte of device memory themselves (a serving runtime with a fixed
// memory budget, an embedded engine that forbids cudaMalloc after start-up,
// or a thread where cudaMalloc's implicit synchronisation would stall other
// work).  Such a caller cannot provide the workspace moe_forward asks for.
// This entry point runs the same kernels as moe_forward but keeps their
// scratch in one fixed-size array that lives in the library's own device
// memory, so the call allocates nothing.
//
// The array is a file-scope `static __device__` object: every GPU that loads
// the library holds its kNoallocScratchBytes until the process exits.  In
// host code its name is only a host-side stand-in, never a device address, so
// the first call on each device looks the real address up with
// cudaGetSymbolAddress (with that device current) and caches it.
#include <atomic>
#include <mutex>

#include "moe_internal.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

constexpr size_t kNoallocScratchBytes = static_cast<size_t>(MOE_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxNoallocDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxNoallocDevices] = {};
// Test switch ("noalloc_poison" of moe_set_tuning): the next call first fills
// the array's status word and counters with non-zero bytes, as a call that
// gave up on the device could have left them.
std::atomic<int> g_noalloc_poison{0};

// Device address of the scratch array on the current device (set-up on the
// first call per device).
moe_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoallocDevices)
        return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return MOE_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

}  // namespace

void set_noalloc_poison(int on) { g_noalloc_poison.store(on ? 1 : 0); }

}  // namespace moe

extern "C" moe_status moe_forward_noalloc(const moe_shape* shape, const void* hidden,
                                          const void* router_w, const void* router_b,
                                          moe_weight gate_up, moe_weight down, void* out,
                                          int out_is_fp32, int32_t* topk_ids_out,
                                          float* topk_w_out, int32_t* device_status_out,
                                          cudaStream_t stream) {
    if (!shape) return MOE_ERR_ARG;
    const size_t need = moe_workspace_bytes(shape);
    if (need == 0)
        return shape->wfmt == MOE_W_BF16 || shape->wfmt == MOE_W_MXFP4 ||
                       shape->wfmt == MOE_W_FP8 || shape->wfmt == MOE_W_MXFP4_MXFP8
                   ? MOE_ERR_SHAPE
                   : MOE_ERR_ARG;
    if (shape->T == 0) return MOE_OK;
    if (need > moe::kNoallocScratchBytes) return MOE_ERR_WORKSPACE;
    if (device_status_out && (reinterpret_cast<uintptr_t>(device_status_out) & 3u))
        return MOE_ERR_ALIGN;
    void* scratch = nullptr;
    moe_status st = moe::noalloc_scratch(&scratch);
    if (st != MOE_OK) return st;
    // The array keeps the previous call's contents.  The status word and the
    // block of completion counters after it (router tickets, expert totals,
    // GEMM K-split tickets) must start from zero: a call completes only if
    // every counter it uses starts at zero, and a call that gave up on the
    // device (a wait timeout, a bad tile) leaves some of them set.  A caller
    // of this entry point cannot reach the array to clear it, so every call
    // clears them itself (256 + 134,528 bytes).  Every other region is fully
    // rewritten by the kernels before it is read.
    const size_t clear_bytes = 256 + moe::kCounterBytes;
    if (moe::g_noalloc_poison.exchange(0) &&
        cudaMemsetAsync(scratch, 0x5A, clear_bytes, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemsetAsync(scratch, 0, clear_bytes, stream) != cudaSuccess) return MOE_ERR_CUDA;
    st = moe_forward(shape, hidden, router_w, router_b, gate_up, down, out, out_is_fp32,
                     topk_ids_out, topk_w_out, scratch, moe::kNoallocScratchBytes, stream);
    if (st != MOE_OK) return st;
    if (device_status_out &&
        cudaMemcpyAsync(device_status_out, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
