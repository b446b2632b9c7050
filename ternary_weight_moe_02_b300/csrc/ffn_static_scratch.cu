// maple_moe_ffn_static_scratch: the expert FFN for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain a workspace: a plugin loaded into a host
// process whose device memory is owned by that host's own allocator, code that runs
// while a stream is being captured into a CUDA graph (where cudaMalloc is not
// allowed), or a real-time loop that must never enter the allocator.  This entry
// point takes no workspace: its scratch is one file-scope device array of fixed
// size, which every GPU that loads this library keeps until the process exits.
//
// In host code the array's name is only a host-side stand-in, not a device address,
// so the device address is looked up with cudaGetSymbolAddress, once per device,
// with that device current, on the first call made on that device; that first call
// should therefore come before any stream capture.  After the look-up every call runs
// maple_moe_ffn's checks and kernels with the array as its workspace, always on the
// CUDA-core path: the grouped tensor-core path needs per-tile operand blocks far
// larger than the array.  Nothing in the array
// needs to start at zero: every kernel writes what it later reads, so the contents
// left by the previous call are simply overwritten.  All calls share the one array,
// so calls that overlap on the GPU (other streams, other host threads) race on it
// and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "maple.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;  // 2 MiB per device

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" MAPLE_API int maple_moe_ffn_static_scratch(const maple_experts* ex, const uint16_t* x,
                                                      const int32_t* idx, const float* w,
                                                      int32_t T, int32_t k, float* y,
                                                      void* stream) {
    // Argument checks are maple_moe_ffn's own; a call it rejects (or an empty one,
    // T == 0) is forwarded without scratch, so it reports exactly as it would.
    if (!ex || T <= 0 || k < 1 || ex->E < 1 || ex->I < 1)
        return maple::moe_ffn_entry(ex, x, idx, w, T, k, y, nullptr, 0, stream, MAPLE_FFN_CORES);
    const size_t need = maple::moe_ffn_workspace_bytes(T, k, ex, MAPLE_FFN_CORES);
    if (need > kStaticScratchBytes)
        return maple::report_error(MAPLE_ERR_WORKSPACE,
                                   "moe_ffn_static_scratch: T=%d k=%d I=%d needs %zu bytes of "
                                   "scratch; the static array holds %zu",
                                   T, k, ex->I, need, kStaticScratchBytes);
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return maple::report_error(MAPLE_ERR_CUDA, "moe_ffn_static_scratch: cudaGetDevice: %s",
                                   cudaGetErrorString(err));
    if (dev < 0 || dev >= kMaxDevices)
        return maple::report_error(MAPLE_ERR_UNSUPPORTED_SHAPE,
                                   "moe_ffn_static_scratch: device %d >= %d", dev, kMaxDevices);
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (g_scratch_addr[dev] == nullptr) {
            void* p = nullptr;
            err = cudaGetSymbolAddress(&p, g_static_scratch);
            if (err != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return maple::report_error(MAPLE_ERR_CUDA,
                                           "moe_ffn_static_scratch: cudaGetSymbolAddress: %s",
                                           cudaGetErrorString(err));
            }
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    return maple::moe_ffn_entry(ex, x, idx, w, T, k, y, scratch, kStaticScratchBytes, stream, MAPLE_FFN_CORES);
}
