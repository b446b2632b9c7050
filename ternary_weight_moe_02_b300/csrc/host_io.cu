// Device-side copies between pinned (mapped) host memory and device memory, for the
// entry points whose activations live in host memory.  A copy kernel, unlike a memcpy
// node, takes part in programmatic dependent launch: the copy-in overlaps the tail of
// the previous kernel and the next kernel's start overlaps the copy's tail, so a step
// fed from host memory keeps the launch chain of a device-resident one.
#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

constexpr int kIoThreads = 256;

__global__ void __launch_bounds__(kIoThreads) io_copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                              int64_t n16) {
    pdl_wait();  // the destination may still be read by the previous kernel
    pdl_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * kIoThreads + threadIdx.x; i < n16; i += (int64_t)gridDim.x * kIoThreads)
        dst[i] = src[i];
}

__global__ void __launch_bounds__(kIoThreads) io_copy1_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                             int64_t n) {
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * kIoThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kIoThreads)
        dst[i] = src[i];
}

}  // namespace

// The device address of host memory the device can reach (pinned with mapping, which
// unified addressing gives every pinned allocation), or nullptr.
void* mapped_host_pointer(const void* host) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
        cudaGetLastError();  // a plain pageable pointer: clear the error
        return nullptr;
    }
    return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}

cudaError_t launch_io_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream, const DeviceInfo& dev) {
    if (bytes == 0) return cudaSuccess;
    const bool wide = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | bytes) & 15u) == 0;
    const int64_t n = wide ? (int64_t)(bytes / 16) : (int64_t)bytes;
    int64_t blocks = (n + kIoThreads - 1) / kIoThreads;
    const int64_t cap = (int64_t)dev.sm_count * 4;
    blocks = blocks < cap ? blocks : cap;
    if (wide)
        return launch_pdl(io_copy16_kernel, dim3((unsigned)blocks), dim3(kIoThreads), 0, stream,
                          reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n);
    return launch_pdl(io_copy1_kernel, dim3((unsigned)blocks), dim3(kIoThreads), 0, stream,
                      reinterpret_cast<const uint8_t*>(src), reinterpret_cast<uint8_t*>(dst), n);
}

}  // namespace maple
