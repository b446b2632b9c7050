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

// Bulk-copy path (K % 8 == 0, 16-byte aligned W, two stages of R row slots per warp
// fit in shared memory).  Each warp streams blocks of R consecutive rows (R a power of
// two, chosen so that a block is about 4 KB) through two stages: lane 0 issues the next
// block's row copies while the warp packs the current one, so every row is read from
// DRAM once.  A row slot is 2K bytes followed by kPkPad zero bytes, which the last,
// ragged unit of a row reads as +0 weights (digit 1, the zero trit).  Within a stage,
// G = 32 / R lanes own each row: they sum it, reduce among themselves, and pack it.
//
// Per row: the sum of |w| reads 16-byte chunks (Kahan across pairs of chunks).  The
// packing then works on units of ten weights (five 32-bit words, two output bytes) with
// integer arithmetic only:
//   * |w| > thr, for a bf16 w and an fp32 thr >= 0, is the same test as |w| > t where
//     t is thr truncated to bf16 (the largest bf16 <= thr); on the 15-bit magnitudes of
//     both halves of a word at once it is bit 15 of (|w| + 0x7fff - t), which never
//     carries out of its half;
//   * the base-3 digit q + 1 of a weight is 2p + z, p = (|w| > thr and w > 0), z = not
//     (|w| > thr); trit_field puts p at bit 15 and z at bit 14 of each half, so each half
//     holds (q + 1) * 2^14;
//   * mul.hi by c_lo * 2^18 + c_hi * 4 gives c_lo (q_lo + 1) + c_hi (q_hi + 1) in the
//     low 16 bits (the higher bits get a harmless c_lo * 2^16 term), so three products
//     summed give a byte's code, the sum over five weights of 3^i (q_i + 1).
constexpr int kPkMaxWarps = 8;
constexpr int kPkStageBytes = 4096;
constexpr int kPkMaxK = 49152;
constexpr int kPkPad = 32;

template <uint32_t kLut>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(kLut));
    return d;
}

__device__ __forceinline__ uint32_t trit_field(uint32_t x, uint32_t c2) {
    const uint32_t y = (x & 0x7fff7fffu) + c2;             // bit 15 of a half: |w| > threshold
    const uint32_t p = lop3<0x20>(y, x, 0x80008000u);      // y & ~x & mask: above, positive
    return lop3<0xF2>(p, y >> 1, 0x40004000u);             // p | (~(y >> 1) & mask): not above
}

// multipliers c_lo * 2^18 + c_hi * 4 for the words of a ten-weight unit: byte A takes
// weights 0..4 (3^0..3^4), byte B weights 5..9; word 2 holds weight 4 and weight 5
__host__ __device__ constexpr uint32_t pk_mul(uint32_t c_lo, uint32_t c_hi) {
    return (c_lo << 18) | (c_hi << 2);
}

__device__ __forceinline__ uint32_t pack_unit(const uint32_t* w, uint32_t c2) {
    const uint32_t f0 = trit_field(w[0], c2), f1 = trit_field(w[1], c2), f2 = trit_field(w[2], c2);
    const uint32_t f3 = trit_field(w[3], c2), f4 = trit_field(w[4], c2);
    const uint32_t a = __umulhi(f0, pk_mul(1, 3)) + __umulhi(f1, pk_mul(9, 27)) + __umulhi(f2, pk_mul(81, 0));
    const uint32_t b = __umulhi(f2, pk_mul(0, 1)) + __umulhi(f3, pk_mul(3, 9)) + __umulhi(f4, pk_mul(27, 81));
    return __byte_perm(a, b, 0x0040);  // byte 0: code A, byte 1: code B
}

__device__ __forceinline__ float chunk_abs_sum(uint4 v) {
    const float a0 = fabsf(bf16_lo(v.x)) + __uint_as_float(v.x & 0x7fff0000u);
    const float a1 = fabsf(bf16_lo(v.y)) + __uint_as_float(v.y & 0x7fff0000u);
    const float a2 = fabsf(bf16_lo(v.z)) + __uint_as_float(v.z & 0x7fff0000u);
    const float a3 = fabsf(bf16_lo(v.w)) + __uint_as_float(v.w & 0x7fff0000u);
    return (a0 + a1) + (a2 + a3);
}

// Sum of |w| over a row slot, as every lane of the row's G-lane group sees it (j: the
// lane's index in the group).
template <int G>
__device__ __forceinline__ float group_row_abs_sum(const uint4* r4, int n4, int j) {
    float sum = 0.f, comp = 0.f;
    for (int c = j; c < n4; c += 2 * G) {
        const uint4 v0 = r4[c];
        const uint4 v1 = c + G < n4 ? r4[c + G] : make_uint4(0u, 0u, 0u, 0u);
        const float y = (chunk_abs_sum(v0) + chunk_abs_sum(v1)) - comp;
        const float t = sum + y;
        comp = (t - sum) - y;
        sum = t;
    }
    float v = sum - comp;
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
    return v;
}

// Per-half unsigned max / min of two packed 16-bit pairs.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Folds one word (two bf16) into the running packed maxima of the magnitudes and minima
// of (magnitude - 1) mod 2^16, which sends a zero magnitude to 0xffff, above every
// other.  Setting bit 15 of each half first keeps the subtraction from borrowing across
// halves: (|w| | 0x8000) - 1 lies in [0x7fff, 0xfffe], and the xor with 0x8000 maps it
// to |w| - 1 for |w| >= 1 and to 0xffff for |w| = 0.
__device__ __forceinline__ void fold_mag_word(uint32_t w, uint32_t& hi2, uint32_t& lo2) {
    hi2 = max_u16x2(hi2, w & 0x7fff7fffu);
    lo2 = min_u16x2(lo2, ((w | 0x80008000u) - 0x00010001u) ^ 0x80008000u);
}

// Largest and smallest nonzero magnitude (bf16 bits; 0x7fff when there is none) over
// a row slot, as every lane of the row's G-lane group sees them (j: the lane's index
// in the group).  Non-negative finite bf16 values order like their bit patterns, so
// both halves of every word are compared at once as unsigned 16-bit values.
template <int G>
__device__ __forceinline__ void group_row_mag_range(const uint4* r4, int n4, int j, uint32_t& mx, uint32_t& mn) {
    uint32_t hi2 = 0u, lo2 = 0xffffffffu;
    for (int c = j; c < n4; c += 2 * G) {
        const uint4 v0 = r4[c];
        const uint4 v1 = c + G < n4 ? r4[c + G] : make_uint4(0u, 0u, 0u, 0u);
        fold_mag_word(v0.x, hi2, lo2);
        fold_mag_word(v0.y, hi2, lo2);
        fold_mag_word(v0.z, hi2, lo2);
        fold_mag_word(v0.w, hi2, lo2);
        fold_mag_word(v1.x, hi2, lo2);
        fold_mag_word(v1.y, hi2, lo2);
        fold_mag_word(v1.z, hi2, lo2);
        fold_mag_word(v1.w, hi2, lo2);
    }
    uint32_t hi = max(hi2 & 0xffffu, hi2 >> 16);
    uint32_t lo = min(lo2 & 0xffffu, lo2 >> 16);  // (smallest nonzero magnitude - 1), or 0xffff
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) {
        hi = max(hi, __shfl_xor_sync(kFullMask, hi, o));
        lo = min(lo, __shfl_xor_sync(kFullMask, lo, o));
    }
    mx = hi;
    mn = lo == 0xffffu ? 0x7fffu : lo + 1u;
}

// Packs the units j, j + G, ... of one row slot (two per loop trip).
template <int G, bool kPairStores>
__device__ __forceinline__ void group_pack_row(const uint32_t* row32, int units, int nb, int j,
                                               uint32_t c2, uint8_t* __restrict__ out) {
    auto store = [&](int u, uint32_t ab) {
        if (kPairStores) {
            reinterpret_cast<uint16_t*>(out)[u] = (uint16_t)ab;  // nb even: every unit has A and B
        } else {
            out[2 * u] = (uint8_t)ab;
            if (2 * u + 1 < nb) out[2 * u + 1] = (uint8_t)(ab >> 8);
        }
    };
    int u = j;
    for (; u + G < units; u += 2 * G) {
        const uint32_t ab0 = pack_unit(row32 + 5 * u, c2);
        const uint32_t ab1 = pack_unit(row32 + 5 * (u + G), c2);
        store(u, ab0);
        store(u + G, ab1);
    }
    if (u < units) store(u, pack_unit(row32 + 5 * u, c2));
}

// kExact: the rows are already ternary (-s, 0, +s each): s = the largest magnitude,
// trits = signs (the packing threshold is 0), and rows with two different nonzero
// magnitudes are counted in *bad_rows (may be null).  Otherwise absmean.
template <int G, bool kPairStores, bool kExact>
__global__ void __launch_bounds__(kPkMaxWarps * 32)
    ternarize_pack_tma_kernel(const uint16_t* __restrict__ W, int64_t rows, int K,
                              uint8_t* __restrict__ packed, float* __restrict__ scales, int* status,
                              int32_t* __restrict__ bad_rows) {
    constexpr int R = 32 / G;  // rows per block
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) uint64_t bars[kPkMaxWarps][2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int rowbytes = 2 * K;              // a multiple of 16
    const int slot = rowbytes + kPkPad;      // row slot stride
    const int stagebytes = R * slot;
    unsigned char* const stage0 = smem + (size_t)warp * 2 * stagebytes;
    const int64_t nblk = (rows + R - 1) / R;
    const int64_t gw = (int64_t)blockIdx.x * nwarps + warp;
    const int64_t nw = (int64_t)gridDim.x * nwarps;
    const int nb = (K + 4) / 5;
    const int units = (nb + 1) >> 1;         // the last one holds only byte A when nb is odd
    const int q = lane / G, j = lane % G;    // this lane's row in a block, index in its group
    // zero the pads after the 2R row slots; copies never write them
    for (int i = lane; i < 2 * R * (kPkPad / 16); i += 32) {
        const int sl = i / (kPkPad / 16), part = i % (kPkPad / 16);
        *reinterpret_cast<uint4*>(stage0 + sl * slot + rowbytes + 16 * part) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (lane == 0) {
        mbar_init(&bars[warp][0], 1);
        mbar_init(&bars[warp][1], 1);
    }
    __syncwarp();
    pdl_wait();
    auto issue = [&](int64_t blk, int st) {
        const int64_t r0 = blk * R;
        const int64_t left = rows - r0;
        const int n = (int)(left < R ? left : R);
        mbar_arrive_expect_tx(&bars[warp][st], (uint32_t)(n * rowbytes));
        for (int i = 0; i < n; ++i)
            bulk_copy_g2s(stage0 + st * stagebytes + i * slot, W + (r0 + i) * K, (uint32_t)rowbytes,
                          &bars[warp][st]);
    };
    if (gw < nblk && lane == 0) issue(gw, 0);
    uint32_t phase0 = 0, phase1 = 0;
    int st = 0;
    bool ok = true;
    for (int64_t blk = gw; blk < nblk; blk += nw) {
        if (blk + nw < nblk && lane == 0) {
            // the other stage was last read (generic proxy) before the previous __syncwarp
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(blk + nw, st ^ 1);
        }
        const uint32_t ph = st ? phase1 : phase0;
        if (!mbar_wait_bounded(&bars[warp][st], ph, status)) ok = false;
        if (st)
            phase1 ^= 1u;
        else
            phase0 ^= 1u;
        if (!__all_sync(kFullMask, ok)) break;
        const int64_t r = blk * R + q;
        // a group whose row is past the end (last block) sums its stale slot harmlessly
        // and stores nothing
        const unsigned char* rowp = stage0 + st * stagebytes + q * slot;
        if constexpr (kExact) {
            uint32_t mx, mn;
            group_row_mag_range<G>(reinterpret_cast<const uint4*>(rowp), K >> 3, j, mx, mn);
            if (r < rows) {
                // threshold 0: every nonzero magnitude gives the sign trit
                group_pack_row<G, kPairStores>(reinterpret_cast<const uint32_t*>(rowp), units, nb, j,
                                               0x7fffu * 0x10001u, packed + r * nb);
                if (j == 0) {
                    scales[r] = __uint_as_float(mx << 16);
                    if (bad_rows != nullptr && mx != 0u && mn != mx) atomicAdd(bad_rows, 1);
                }
            }
        } else {
            const float total = group_row_abs_sum<G>(reinterpret_cast<const uint4*>(rowp), K >> 3, j);
            if (r < rows) {
                const float s = __fdiv_rn(total, (float)K);
                const uint32_t t16 = (__float_as_uint(0.5f * s) >> 16) & 0x7fffu;
                const uint32_t c2 = (0x7fffu - t16) * 0x10001u;
                group_pack_row<G, kPairStores>(reinterpret_cast<const uint32_t*>(rowp), units, nb, j, c2,
                                               packed + r * nb);
                if (j == 0) scales[r] = s;
            }
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
        st ^= 1;
    }
    // a block prefetched but not consumed (only after a failed wait) must land first
    if (!ok && lane == 0) {
        mbar_wait_bounded(&bars[warp][0], phase0, nullptr);
        mbar_wait_bounded(&bars[warp][1], phase1, nullptr);
    }
}

template <int G, bool kPairStores, bool kExact>
cudaError_t launch_pack_tma(const uint16_t* W, int64_t rows, int K, uint8_t* packed, float* scales,
                            int32_t* bad_rows, int warps, cudaStream_t stream, const DeviceInfo& dev) {
    constexpr int R = 32 / G;
    auto kernel = ternarize_pack_tma_kernel<G, kPairStores, kExact>;
    const size_t smem = (size_t)warps * 2 * R * (2 * (size_t)K + kPkPad);
    cudaError_t err = ensure_dynamic_smem(kernel, smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, warps * 32, smem);
    if (err != cudaSuccess) return err;
    per_sm = per_sm < 1 ? 1 : per_sm;
    const int64_t nblk = (rows + R - 1) / R;
    const int64_t want = (nblk + warps - 1) / warps;
    const int64_t cap = (int64_t)dev.sm_count * per_sm;
    const int grid = (int)(want < cap ? want : cap);
    return launch_pdl(kernel, dim3(grid), dim3(warps * 32), smem, stream, W, rows, K, packed, scales,
                      dev.status, bad_rows);
}

template <int G, bool kExact>
cudaError_t launch_pack_tma_g(const uint16_t* W, int64_t rows, int K, uint8_t* packed, float* scales,
                              int32_t* bad_rows, int warps, cudaStream_t stream, const DeviceInfo& dev) {
    const int nb = (K + 4) / 5;
    if (nb % 2 == 0 && reinterpret_cast<uintptr_t>(packed) % 2 == 0)
        return launch_pack_tma<G, true, kExact>(W, rows, K, packed, scales, bad_rows, warps, stream, dev);
    return launch_pack_tma<G, false, kExact>(W, rows, K, packed, scales, bad_rows, warps, stream, dev);
}

// The staged path (bulk copies of row blocks into shared memory) for W 16-byte aligned
// and K a multiple of 8 up to kPkMaxK: rows per block R, the largest power of two <= 32
// whose block is at most ~4 KB, and warps per CTA.  False when the shape does not take it.
bool pack_staged_plan(const uint16_t* W, int64_t K, const DeviceInfo& dev, int& R, int& warps) {
    const bool vec = (K % 8 == 0) && (reinterpret_cast<uintptr_t>(W) % 16 == 0);
    if (!vec || K > kPkMaxK) return false;
    const int rowbytes = 2 * (int)K;
    R = 1;
    while (R < 32 && 2 * R * rowbytes <= kPkStageBytes) R *= 2;
    const size_t per_warp = (size_t)2 * R * (rowbytes + kPkPad);  // two stages
    warps = (int)((dev.smem_optin - 1024) / per_warp);
    warps = warps > kPkMaxWarps ? kPkMaxWarps : warps;
    return warps >= 1;
}

template <bool kExact>
cudaError_t launch_pack_staged(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed, float* scales,
                               int32_t* bad_rows, int R, int warps, cudaStream_t stream, const DeviceInfo& dev) {
    switch (R) {
        case 1: return launch_pack_tma_g<32, kExact>(W, rows, (int)K, packed, scales, bad_rows, warps, stream, dev);
        case 2: return launch_pack_tma_g<16, kExact>(W, rows, (int)K, packed, scales, bad_rows, warps, stream, dev);
        case 4: return launch_pack_tma_g<8, kExact>(W, rows, (int)K, packed, scales, bad_rows, warps, stream, dev);
        case 8: return launch_pack_tma_g<4, kExact>(W, rows, (int)K, packed, scales, bad_rows, warps, stream, dev);
        case 16: return launch_pack_tma_g<2, kExact>(W, rows, (int)K, packed, scales, bad_rows, warps, stream, dev);
        default: return launch_pack_tma_g<1, kExact>(W, rows, (int)K, packed, scales, bad_rows, warps, stream, dev);
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
    int R = 0, warps = 0;
    if (pack_staged_plan(W, K, dev, R, warps))
        return launch_pack_staged<false>(W, rows, K, packed, scales, nullptr, R, warps, stream, dev);
    const int64_t want = (rows + 7) / 8;
    const int64_t cap = (int64_t)dev.sm_count * 8;
    const int grid = (int)(want < cap ? want : cap);
    return launch_pdl(ternarize_pack_kernel, dim3(grid), dim3(256), 0, stream, W, rows, K, packed,
                      scales, vec);
}

cudaError_t launch_pack_exact_staged(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed,
                                     float* scales, int32_t* bad_rows, cudaStream_t stream, const DeviceInfo& dev,
                                     bool* taken) {
    int R = 0, warps = 0;
    *taken = pack_staged_plan(W, K, dev, R, warps);
    if (!*taken) return cudaSuccess;
    return launch_pack_staged<true>(W, rows, K, packed, scales, bad_rows, R, warps, stream, dev);
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
