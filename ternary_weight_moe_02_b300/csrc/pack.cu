// Absmean ternarization + five-trits-per-byte packing, and the inverse (unpack).
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// section "The claim, verified from the bytes": every row is -s, 0, +s with one s per
// output row (absmean, BitNet b1.58 shape); section "The 5.31 GB claim reconciles":
// five trits per byte (3^5 = 243 <= 256) plus per-row scales.
//
// ternarize_pack is HBM-bound: it reads 2 B and writes 0.2 B per weight.  One warp
// owns one row at a time (grid-stride over rows); the row is read twice, the second
// time from L1, so DRAM sees it once.
#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

// Sum of |w| over one bf16 row, as every lane of the warp sees it.  Per lane: the
// eight values of a 16-byte chunk are added pairwise, chunk sums are accumulated
// with Kahan compensation, then the lanes are combined by a butterfly.  The
// relative error stays below ~10 fp32 ulps for any K.
__device__ __forceinline__ float row_abs_sum(const uint16_t* __restrict__ wr, int64_t K,
                                             bool vec, int lane) {
    float sum = 0.f, comp = 0.f;
    auto kahan_add = [&](float a) {
        float y = a - comp;
        float t = sum + y;
        comp = (t - sum) - y;
        sum = t;
    };
    if (vec) {
        const uint4* w4 = reinterpret_cast<const uint4*>(wr);
        const int64_t n4 = K >> 3;
        for (int64_t c0 = lane; c0 < n4; c0 += 32 * 4) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                int64_t c = c0 + 32 * u;
                v[u] = c < n4 ? ldg_nc_v4(w4 + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float a0 = fabsf(bf16_lo(v[u].x)) + fabsf(bf16_hi(v[u].x));
                float a1 = fabsf(bf16_lo(v[u].y)) + fabsf(bf16_hi(v[u].y));
                float a2 = fabsf(bf16_lo(v[u].z)) + fabsf(bf16_hi(v[u].z));
                float a3 = fabsf(bf16_lo(v[u].w)) + fabsf(bf16_hi(v[u].w));
                kahan_add((a0 + a1) + (a2 + a3));
            }
        }
    } else {
        for (int64_t j = lane; j < K; j += 32) kahan_add(fabsf(bf16_bits_to_float(wr[j])));
    }
    return warp_sum(sum - comp);
}

__global__ void __launch_bounds__(256)
    ternarize_pack_kernel(const uint16_t* __restrict__ W, int64_t rows, int64_t K,
                          uint8_t* __restrict__ packed, float* __restrict__ scales, int vec) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t nb = (K + 4) / 5;
    for (int64_t r = gw; r < rows; r += nw) {
        const uint16_t* wr = W + r * K;
        const float total = row_abs_sum(wr, K, vec != 0, lane);
        const float s = __fdiv_rn(total, (float)K);
        const float thr = 0.5f * s;  // exact: |w| > s/2  <=>  round(|w|/s) >= 1
        uint8_t* pr = packed + r * nb;
        for (int64_t b = lane; b < nb; b += 32) {
            int code = 0, place = 1;
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                const int64_t j = 5 * b + i;
                int digit = 1;
                if (j < K) {
                    const float v = bf16_bits_to_float(wr[j]);
                    digit = fabsf(v) > thr ? (v > 0.f ? 2 : 0) : 1;
                }
                code += digit * place;
                place *= 3;
            }
            pr[b] = (uint8_t)code;
        }
        if (lane == 0) scales[r] = s;
    }
}

__global__ void __launch_bounds__(256)
    unpack_kernel(const uint8_t* __restrict__ packed, const float* __restrict__ scales,
                  int64_t rows, int64_t K, float* __restrict__ out, int32_t* bad_codes) {
    pdl_wait();
    const int64_t nb = (K + 4) / 5;
    const int64_t total = rows * nb;
    int bad = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / nb, b = i - r * nb;
        int code = packed[i];
        if (code >= 243) {
            ++bad;
            code = 121;
        }
        const float s = scales[r];
#pragma unroll
        for (int d = 0; d < 5; ++d) {
            const int digit = code % 3;
            code /= 3;
            const int64_t j = 5 * b + d;
            if (j < K) out[r * K + j] = (float)(digit - 1) * s;
        }
    }
    if (bad_codes != nullptr && bad != 0) atomicAdd(bad_codes, bad);
}

}  // namespace

cudaError_t launch_ternarize_pack(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed,
                                  float* scales, cudaStream_t stream, const DeviceInfo& dev) {
    const int vec = (K % 8 == 0) && (reinterpret_cast<uintptr_t>(W) % 16 == 0);
    const int64_t want = (rows + 7) / 8;
    const int64_t cap = (int64_t)dev.sm_count * 8;
    const int grid = (int)(want < cap ? want : cap);
    return launch_pdl(ternarize_pack_kernel, dim3(grid), dim3(256), 0, stream, W, rows, K, packed,
                      scales, vec);
}

cudaError_t launch_unpack(const uint8_t* packed, const float* scales, int64_t rows, int64_t K,
                          float* W_out, int32_t* bad_codes, cudaStream_t stream,
                          const DeviceInfo& dev) {
    const int64_t total = rows * ((K + 4) / 5);
    const int64_t want = (total + 255) / 256;
    const int64_t cap = (int64_t)dev.sm_count * 16;
    const int grid = (int)(want < cap ? want : cap);
    return launch_pdl(unpack_kernel, dim3(grid), dim3(256), 0, stream, packed, scales, rows, K,
                      W_out, bad_codes);
}

}  // namespace maple
