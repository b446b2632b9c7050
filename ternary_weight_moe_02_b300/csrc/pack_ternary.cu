// Packing of weight rows that are already ternary.
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// section "The claim, verified from the bytes": the released checkpoint stores every
// expert weight as a bf16 value -s, 0 or +s of its row.  Absmean ternarization of such
// a row keeps the trits but rescales the row by (1 - z), z its share of zeros; this
// packing keeps the checkpoint's own scale instead: s = max_j |w_j| and q_j = sign(w_j)
// (+0 and -0 give 0), five trits per byte as in the absmean packing ("The 5.31 GB claim
// reconciles").  A row with two different nonzero magnitudes is not ternary: it is
// counted, and still gets those trits and that scale.
//
// Shapes the staged absmean pack kernel takes (W 16-byte aligned, K a multiple of 8 up
// to 49152) run through its already-ternary form (pack.cu); the kernel here serves the
// rest.  One warp per row, one pass: lane l packs bytes b = l, l + 32, ... (its five weights
// 5b .. 5b + 4 are 10 contiguous bytes, so a warp's loads cover 320 contiguous bytes)
// and keeps the largest and the smallest nonzero magnitude it met; the row is ternary
// when the two agree after a warp reduction.  Magnitudes are compared as bf16 bit
// patterns, which order finite non-negative values exactly.
#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

constexpr int kPtWarps = 8;

__global__ void __launch_bounds__(kPtWarps * 32)
    pack_ternary_kernel(const uint16_t* __restrict__ W, int64_t rows, int64_t K, uint8_t* __restrict__ packed,
                        float* __restrict__ scales, int32_t* __restrict__ bad_rows) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nb = (K + 4) / 5;
    for (int64_t r = (int64_t)blockIdx.x * kPtWarps + (threadIdx.x >> 5); r < rows;
         r += (int64_t)gridDim.x * kPtWarps) {
        const uint16_t* wr = W + r * K;
        uint8_t* pr = packed + r * nb;
        uint32_t mx = 0u, mn = 0x7fffu;  // largest / smallest nonzero magnitude (bf16 bits)
#pragma unroll 2
        for (int64_t b = lane; b < nb; b += 32) {
            uint32_t bits[5];
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                const int64_t j = 5 * b + i;
                bits[i] = j < K ? (uint32_t)__ldg(wr + j) : 0u;
            }
            uint32_t code = 0u, place = 1u;
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                const uint32_t mag = bits[i] & 0x7fffu;
                const uint32_t digit = mag == 0u ? 1u : ((bits[i] & 0x8000u) ? 0u : 2u);  // q + 1
                code += digit * place;
                place *= 3u;
                if (mag != 0u) {
                    mx = max(mx, mag);
                    mn = min(mn, mag);
                }
            }
            pr[b] = (uint8_t)code;
        }
        mx = __reduce_max_sync(kFullMask, mx);
        mn = __reduce_min_sync(kFullMask, mn);
        if (lane == 0) {
            scales[r] = __uint_as_float(mx << 16);
            if (bad_rows != nullptr && mx != 0u && mn != mx) atomicAdd(bad_rows, 1);
        }
    }
}

}  // namespace

cudaError_t launch_pack_ternary(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed, float* scales,
                                int32_t* bad_rows, cudaStream_t stream, const DeviceInfo& dev) {
    // shapes the staged pack kernel takes run there (threshold 0, max scale)
    bool taken = false;
    const cudaError_t err = launch_pack_exact_staged(W, rows, K, packed, scales, bad_rows, stream, dev, &taken);
    if (taken) return err;
    const int64_t want = (rows + kPtWarps - 1) / kPtWarps;
    const int64_t cap = (int64_t)dev.sm_count * 8;
    const int grid = (int)(want < cap ? want : cap);
    return launch_pdl(pack_ternary_kernel, dim3(grid), dim3(kPtWarps * 32), 0, stream, W, rows, K, packed, scales,
                      bad_rows);
}

}  // namespace maple
