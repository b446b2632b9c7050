// Device helpers shared by the CUDA kernels of libmaple (internal header).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace maple {

constexpr unsigned kFullMask = 0xffffffffu;

// Programmatic dependent launch: wait until the preceding grid on the stream has
// finished and its writes are visible.  Every kernel calls this before it reads
// anything a previous kernel wrote (and before it writes anything a previous
// kernel may still read), in every thread that does so.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next grid on the stream start its prologue early.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// bf16 -> fp32 is a 16-bit left shift of the bit pattern (exact).
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xffff0000u); }

// Butterfly sum over the warp: every lane ends with the same, order-fixed value.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ldg_nc_u8(const uint8_t* p) {
    uint16_t r;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// Shared-memory table of one packed byte: for each of its five trits, the top byte
// of the fp32 value +0.5 (0x3f), -0.5 (0xbf) or 0 (0x00).  Trits 0..3 live in .x,
// trit 4 in byte 0 of .y.  A single byte-permute turns one of them into the fp32
// multiplier {+0.5, -0.5, 0}; the factor 2 is folded into the row scale.
struct TritLut {
    uint2 entry[243];
};

__device__ __forceinline__ void build_trit_lut(TritLut& lut, int tid, int nthreads) {
    for (int c = tid; c < 243; c += nthreads) {
        int code = c;
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            int digit = code % 3;
            code /= 3;
            uint32_t top = digit == 2 ? 0x3fu : (digit == 0 ? 0xbfu : 0x00u);
            if (i < 4)
                lo |= top << (8 * i);
            else
                hi = top;
        }
        lut.entry[c] = make_uint2(lo, hi);
    }
}

// fp32 multiplier (+-0.5 or 0) of trit i (0..4) of a table entry.
template <int I>
__device__ __forceinline__ float trit_half(uint2 e) {
    if constexpr (I < 4)
        return __uint_as_float(__byte_perm(e.x, 0u, 0x0444u | (I << 12)));
    else
        return __uint_as_float(__byte_perm(e.y, 0u, 0x0444u));
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Launch with the programmatic-stream-serialization attribute (PDL).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace maple
