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

// Bulk-copy path (K % 8 == 0, 16-byte aligned W, K <= kPkMaxK).  Each warp streams
// its rows (grid-stride) through two shared-memory row buffers: lane 0 bulk-copies the
// next row while the warp works on the current one, so every row is read from DRAM
// once.  The row sum reads 16-byte chunks; each output byte b (lane-strided) is built
// from its five weights as 121 + P - N, where P / N add 3^i for weight i above +s/2 /
// below -s/2 (the base-3 code with digit q + 1, written out).
constexpr int kPkWarps = 8;
constexpr int kPkMaxK = 8192;

__global__ void __launch_bounds__(kPkWarps * 32)
    ternarize_pack_tma_kernel(const uint16_t* __restrict__ W, int64_t rows, int K,
                              uint8_t* __restrict__ packed, float* __restrict__ scales, int* status) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[kPkWarps][2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rowbytes = 2 * K;  // a multiple of 16
    uint16_t* const buf0 = reinterpret_cast<uint16_t*>(smem + (size_t)warp * 2 * rowbytes);
    const int64_t gw = (int64_t)blockIdx.x * kPkWarps + warp;
    const int64_t nw = (int64_t)gridDim.x * kPkWarps;
    const int nb = (K + 4) / 5;
    if (lane == 0) {
        mbar_init(&bars[warp][0], 1);
        mbar_init(&bars[warp][1], 1);
    }
    __syncwarp();
    pdl_wait();
    if (gw < rows && lane == 0) {
        mbar_arrive_expect_tx(&bars[warp][0], rowbytes);
        bulk_copy_g2s(buf0, W + gw * K, rowbytes, &bars[warp][0]);
    }
    uint32_t phase0 = 0, phase1 = 0;
    int slot = 0;
    bool ok = true;
    for (int64_t r = gw; r < rows; r += nw) {
        const int64_t rn = r + nw;
        if (rn < rows && lane == 0) {
            // the other buffer was last read (generic proxy) before the previous __syncwarp
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&bars[warp][slot ^ 1], rowbytes);
            bulk_copy_g2s(buf0 + (slot ^ 1) * K, W + rn * K, rowbytes, &bars[warp][slot ^ 1]);
        }
        const uint32_t ph = slot ? phase1 : phase0;
        if (!mbar_wait_bounded(&bars[warp][slot], ph, status)) ok = false;
        if (slot)
            phase1 ^= 1u;
        else
            phase0 ^= 1u;
        if (!__all_sync(kFullMask, ok)) break;
        const uint16_t* row = buf0 + slot * K;

        // row sum of |w|: pairwise inside 16-byte chunks, Kahan across them, butterfly
        float sum = 0.f, comp = 0.f;
        const uint4* r4 = reinterpret_cast<const uint4*>(row);
        for (int c = lane; c < (K >> 3); c += 32) {
            const uint4 v = r4[c];
            const float a0 = fabsf(bf16_lo(v.x)) + fabsf(bf16_hi(v.x));
            const float a1 = fabsf(bf16_lo(v.y)) + fabsf(bf16_hi(v.y));
            const float a2 = fabsf(bf16_lo(v.z)) + fabsf(bf16_hi(v.z));
            const float a3 = fabsf(bf16_lo(v.w)) + fabsf(bf16_hi(v.w));
            const float y = ((a0 + a1) + (a2 + a3)) - comp;
            const float t = sum + y;
            comp = (t - sum) - y;
            sum = t;
        }
        const float total = warp_sum(sum - comp);
        const float s = __fdiv_rn(total, (float)K);
        const float thr = 0.5f * s;  // exact: |w| > s/2  <=>  round(|w|/s) >= 1

        const uint32_t* row32 = reinterpret_cast<const uint32_t*>(row);
        uint8_t* out = packed + r * nb;
        for (int b = lane; b < nb; b += 32) {
            const int e0 = 5 * b;             // first weight of the byte
            const int wi = e0 >> 1;           // its 32-bit word
            const uint32_t sh = (e0 & 1) * 16;
            const uint32_t w0 = row32[wi], w1 = row32[wi + 1], w2 = row32[wi + 2];
            const uint32_t v0 = __funnelshift_r(w0, w1, sh);  // weights e0, e0+1
            const uint32_t v1 = __funnelshift_r(w1, w2, sh);  // e0+2, e0+3
            const uint32_t v2 = __funnelshift_r(w2, w2, sh);  // e0+4 (low half)
            const float f0 = __uint_as_float(v0 << 16), f1 = __uint_as_float(v0 & 0xffff0000u);
            const float f2 = __uint_as_float(v1 << 16), f3 = __uint_as_float(v1 & 0xffff0000u);
            const float f4 = __uint_as_float(v2 << 16);
            int P = 0, N = 0;
            if (e0 + 4 < K) {  // all five weights exist (every byte but a K-tail one)
                P += (f0 > thr) ? 1 : 0;
                N += (f0 < -thr) ? 1 : 0;
                P += (f1 > thr) ? 3 : 0;
                N += (f1 < -thr) ? 3 : 0;
                P += (f2 > thr) ? 9 : 0;
                N += (f2 < -thr) ? 9 : 0;
                P += (f3 > thr) ? 27 : 0;
                N += (f3 < -thr) ? 27 : 0;
                P += (f4 > thr) ? 81 : 0;
                N += (f4 < -thr) ? 81 : 0;
            } else {
                const float f[5] = {f0, f1, f2, f3, f4};
                int place = 1;
                for (int i = 0; i < 5 && e0 + i < K; ++i) {
                    if (f[i] > thr) P += place;
                    if (f[i] < -thr) N += place;
                    place *= 3;
                }
            }
            out[b] = (uint8_t)(121 + P - N);
        }
        if (lane == 0) scales[r] = s;
        __syncwarp();  // every lane is done with this buffer before it is refilled
        slot ^= 1;
    }
    // a row prefetched but not consumed (only after a failed wait) must land first
    if (!ok && lane == 0) {
        mbar_wait_bounded(&bars[warp][0], phase0, nullptr);
        mbar_wait_bounded(&bars[warp][1], phase1, nullptr);
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
    if (vec && K <= kPkMaxK) {
        // two row buffers per warp, plus 16 bytes: the last byte's third 32-bit load may
        // run past the end of the row (those weights are masked)
        const size_t smem = (size_t)kPkWarps * 2 * 2 * K + 16;
        cudaError_t err = ensure_dynamic_smem(ternarize_pack_tma_kernel, smem);
        if (err != cudaSuccess) return err;
        const int per_sm = smem <= 56 * 1024 ? 4 : (smem <= 110 * 1024 ? 2 : 1);
        const int64_t want = (rows + kPkWarps - 1) / kPkWarps;
        const int64_t cap = (int64_t)dev.sm_count * per_sm;
        const int grid = (int)(want < cap ? want : cap);
        return launch_pdl(ternarize_pack_tma_kernel, dim3(grid), dim3(kPkWarps * 32), smem, stream, W,
                          rows, (int)K, packed, scales, dev.status);
    }
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
