// Expert FFN of the ternary MoE layer on CUDA cores (decode path).
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// section "The shipped code does no quantization": the expert body is
// down(act(clamp(gate x, max=7)) * clamp(up x, -7, 7)); "IA de 20B Rodando a 120 tok/s
// no iPhone", section "Pesos ternarios": weight 0 skips, +1 adds, -1 subtracts.
//
// Two implementations of each stage.  The TMA path (Maple-like shapes) stages a CTA's
// packed rows, and the token's activations, in shared memory with one 1-D bulk copy
// per row group, all issued at once, and prefetches the expert's down rows into L2
// while gate/up runs.  The generic path reads bytes straight from global memory and
// takes any shape.
//
// gate/up (generic): one CTA = 16 rows of gate and the same 16 rows of up of one expert,
// for every token routed to that expert.  A warp owns 4 row pairs; lane L always owns
// the packed bytes L, L+32, ... of a row, so the activations it needs (5 per byte)
// stay in registers across rows.  Each byte is decoded through a shared-memory table
// (code -> top bytes of +-0.5/0 for its five trits); one byte-permute per trit gives
// the fp32 multiplier, one FMA accumulates it (the product is exact: +-x/2 or 0).
// The row scale (times 2) is applied once to the warp's sum, then SiLU, the clamps
// and the gate*up product give h, stored fp32 per routing slot.
//
// down (generic): one CTA = 16 output rows of one token; it walks the token's k slots in
// order i = 0..k-1, so the weighted combine is fused and deterministic (no atomics).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;

template <int MB>
__device__ __forceinline__ float ternary_dot(const uint8_t* __restrict__ row, int nbytes,
                                             const TritLut& lut, const float (&v)[MB][5],
                                             int lane) {
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        const int b = lane + 32 * m;
        if (b < nbytes) {
            const uint2 t = lut.entry[ldg_nc_u8(row + b)];
            acc = fmaf(trit_half<0>(t), v[m][0], acc);
            acc = fmaf(trit_half<1>(t), v[m][1], acc);
            acc = fmaf(trit_half<2>(t), v[m][2], acc);
            acc = fmaf(trit_half<3>(t), v[m][3], acc);
            acc = fmaf(trit_half<4>(t), v[m][4], acc);
        }
    }
    return acc;
}

template <int MB>
__global__ void __launch_bounds__(kWarps * 32)
    ffn_gateup_generic_kernel(FfnArgs a, int slot_mode) {
    __shared__ TritLut lut;
    extern __shared__ float xs[];  // [H] activations of the current token, fp32
    build_trit_lut(lut, threadIdx.x, blockDim.x);
    pdl_wait();
    pdl_launch_dependents();
    __syncthreads();

    const int S = a.T * a.k;
    int e, n, off = 0;
    if (slot_mode) {
        if ((int)blockIdx.y >= S) return;
        e = a.idx[blockIdx.y];
        n = 1;
    } else {
        if ((int)blockIdx.y >= *a.n_active) return;
        e = a.active[blockIdx.y];
        off = a.offsets[e];
        n = a.counts[e];
    }
    if (e < 0 || e >= a.E) return;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = a.H, I = a.I;
    const int Bh = (H + 4) / 5;
    const int r_base = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
    const uint8_t* gate_e = a.gate + (int64_t)e * I * Bh;
    const uint8_t* up_e = a.up + (int64_t)e * I * Bh;

    for (int j = 0; j < n; ++j) {
        const int s = slot_mode ? (int)blockIdx.y : a.perm[off + j];
        const int t = s / a.k;
        __syncthreads();
        for (int c = threadIdx.x; c < H; c += blockDim.x)
            xs[c] = bf16_bits_to_float(a.x[(int64_t)t * H + c]);
        __syncthreads();
        float xr[MB][5];
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int b = lane + 32 * m;
#pragma unroll
            for (int d = 0; d < 5; ++d) {
                const int col = 5 * b + d;
                xr[m][d] = (b < Bh && col < H) ? xs[col] : 0.f;
            }
        }
        for (int q = 0; q < kRowsPerWarp; ++q) {
            const int r = r_base + q;
            if (r >= I) break;
            const float ag = warp_sum(ternary_dot<MB>(gate_e + (int64_t)r * Bh, Bh, lut, xr, lane));
            const float au = warp_sum(ternary_dot<MB>(up_e + (int64_t)r * Bh, Bh, lut, xr, lane));
            if (lane == 0) {
                const float g = (2.f * ag) * a.s_gate[(int64_t)e * I + r];
                const float u = (2.f * au) * a.s_up[(int64_t)e * I + r];
                const float gc = fminf(g, a.clamp);
                const float uc = fminf(fmaxf(u, -a.clamp), a.clamp);
                a.h[(int64_t)s * I + r] = silu_f(gc) * uc;
            }
        }
    }
}

template <int MB>
__global__ void __launch_bounds__(kWarps * 32) ffn_down_generic_kernel(FfnArgs a) {
    __shared__ TritLut lut;
    build_trit_lut(lut, threadIdx.x, blockDim.x);
    pdl_wait();
    pdl_launch_dependents();
    __syncthreads();

    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = a.H, I = a.I;
    const int Bi = (I + 4) / 5;
    const int c_base = blockIdx.y * kRowsPerCta + warp * kRowsPerWarp;
    float yacc[kRowsPerWarp];
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) yacc[q] = 0.f;

    for (int i = 0; i < a.k; ++i) {
        const int s = t * a.k + i;
        const int e = a.idx[s];
        if (e < 0 || e >= a.E) continue;
        const float wt = a.w[s];
        const float* hs = a.h + (int64_t)s * I;
        float hr[MB][5];
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int b = lane + 32 * m;
#pragma unroll
            for (int d = 0; d < 5; ++d) {
                const int col = 5 * b + d;
                hr[m][d] = (b < Bi && col < I) ? hs[col] : 0.f;
            }
        }
        const uint8_t* down_e = a.down + (int64_t)e * H * Bi;
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; ++q) {
            const int c = c_base + q;
            if (c < H) {
                const float acc = warp_sum(ternary_dot<MB>(down_e + (int64_t)c * Bi, Bi, lut, hr, lane));
                yacc[q] += wt * (a.s_down[(int64_t)e * H + c] * (2.f * acc));
            }
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; ++q) {
            const int c = c_base + q;
            if (c < H) a.y[(int64_t)t * H + c] = yacc[q];
        }
    }
}

// ------------------------------------------------------------------ TMA path

constexpr int kGuWarps = 4;
constexpr int kGuRowsPerWarp = 2;
constexpr int kGuRows = kGuWarps * kGuRowsPerWarp;  // row pairs (gate + up) per CTA
constexpr int kDnWarps = 16;
constexpr int kDnRows = 16;  // output rows per CTA
constexpr int kDnMaxK = 12;
constexpr int kLut16Bytes = (int)sizeof(TritLut16);  // 31,104 B, a multiple of 16

// Activations of the columns a lane owns: byte b = lane + 32m covers columns 5b..5b+4,
// kept as (x0,x1), (x2,x3) pairs and x4 for packed fp32 FMAs.
template <int MB>
struct LaneCols {
    float2 x01[MB];
    float2 x23[MB];
    float x4[MB];
};

// gate/up: one CTA = kGuRows rows of gate and the same rows of up of one expert (one
// routing slot at T = 1, one active expert otherwise).  Thread 0 issues three bulk
// copies (gate rows, up rows, the first token's activations); another thread
// prefetches this CTA's share of the expert's down rows into L2 for the down kernel.
// Warp w computes row pairs 2w and 2w+1 for each token of the expert.
// Requires: I % kGuRows == 0, ceil(H/5) even, H % 8 == 0, 16-byte aligned bases.
template <int MB>
__global__ void __launch_bounds__(kGuWarps * 32, 3) ffn_gateup_tma_kernel(FfnArgs a, int slot_mode) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    TritLut16& lut = *reinterpret_cast<TritLut16*>(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, I = a.I, Bh = (H + 4) / 5;
    const int wbytes = kGuRows * Bh;  // a multiple of 16
    uint8_t* gbuf = smem + kLut16Bytes;
    uint8_t* ubuf = gbuf + wbytes;
    float* sgbuf = reinterpret_cast<float*>(ubuf + wbytes);  // kGuRows gate scales
    float* subuf = sgbuf + kGuRows;                            // kGuRows up scales
    uint16_t* xb = reinterpret_cast<uint16_t*>(subuf + kGuRows);
    // x as fp32 in lane-column order xcol[m][d][lane] = x[5 (lane + 32 m) + d]: each
    // lane then loads its columns with conflict-free 32-bit reads
    float* xcol = reinterpret_cast<float*>(xb + ((H + 7) / 8) * 8);
    if (tid == 0) {
        // the decode table needs nothing from earlier kernels: start its copy now
        mbar_init(&bar, 1);
        mbar_expect_tx(&bar, (uint32_t)kLut16Bytes);  // no arrival: phase 0 stays open
        bulk_copy_g2s(&lut, &g_lut16_image, kLut16Bytes, &bar);
    }
    pdl_wait();
    pdl_launch_dependents();

    const int S = a.T * a.k;
    int e, n, off = 0;
    if (slot_mode) {
        e = (int)blockIdx.y < S ? a.idx[blockIdx.y] : -1;
        n = 1;
    } else {
        const bool has = (int)blockIdx.y < *a.n_active;
        e = has ? a.active[blockIdx.y] : -1;
        off = has ? a.offsets[e] : 0;
        n = has ? a.counts[e] : 0;
    }
    if (e < 0 || e >= a.E) {
        // nothing to do, but the table copy issued above must land before exiting
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar, 0);
            mbar_wait_bounded(&bar, 0, a.status);
        }
        return;
    }
    const int r0 = blockIdx.x * kGuRows;
    const int s0 = slot_mode ? (int)blockIdx.y : a.perm[off];
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar, 2u * wbytes + 8u * kGuRows + 2u * H);  // the one arrival
        bulk_copy_g2s(gbuf, a.gate + ((int64_t)e * I + r0) * Bh, wbytes, &bar);
        bulk_copy_g2s(ubuf, a.up + ((int64_t)e * I + r0) * Bh, wbytes, &bar);
        bulk_copy_g2s(sgbuf, a.s_gate + (int64_t)e * I + r0, 4u * kGuRows, &bar);
        bulk_copy_g2s(subuf, a.s_up + (int64_t)e * I + r0, 4u * kGuRows, &bar);
        bulk_copy_g2s(xb, a.x + (int64_t)(s0 / a.k) * H, 2u * H, &bar);
    } else if (tid == 32 && a.prefetch_down) {
        // This CTA's share of the expert's down rows (and, for part 0, its scales).
        // prefetch_down guarantees that H * ceil(I/5) and 4 * H are multiples of 16, so
        // every start offset and length below is too.
        const int Bi = (I + 4) / 5;
        const int64_t total = (int64_t)H * Bi;
        const int parts = gridDim.x;
        const int64_t part = ((total + parts - 1) / parts + 15) / 16 * 16;
        const int64_t start = (int64_t)blockIdx.x * part;
        if (start < total) {
            const int64_t len = min(part, total - start);
            bulk_prefetch_l2(a.down + (int64_t)e * total + start, (uint32_t)len);
        }
        if (blockIdx.x == 0) bulk_prefetch_l2(a.s_down + (int64_t)e * H, 4u * H);
    }
    __syncthreads();  // the mbarrier is initialised before anyone waits on it
    {
        const bool ok = mbar_wait_bounded(&bar, 0, a.status);
        if (__syncthreads_or(!ok)) {
            if (!ok) mbar_wait_bounded(&bar, 0, nullptr);  // let copies in flight land first
            return;
        }
    }

    for (int j = 0; j < n; ++j) {
        const int s = slot_mode ? (int)blockIdx.y : a.perm[off + j];
        if (j > 0) {
            __syncthreads();  // every warp is done with the previous token
            const uint4* src = reinterpret_cast<const uint4*>(a.x + (int64_t)(s / a.k) * H);
            uint4* dst = reinterpret_cast<uint4*>(xb);
            for (int c = tid; c < H / 8; c += blockDim.x) dst[c] = src[c];
            __syncthreads();
        }
        // bf16 -> fp32 once per CTA, scattered into lane-column order
        for (int i = tid; i < 32 * MB * 5; i += blockDim.x) {
            const int l = i & 31, md = i >> 5, m = md / 5, d = md - 5 * m;
            const int col = 5 * (l + 32 * m) + d;
            xcol[i] = col < H ? bf16_bits_to_float(xb[col]) : 0.f;
        }
        __syncthreads();
        LaneCols<MB> cols;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const float* xm = xcol + (m * 5) * 32 + lane;
            cols.x01[m] = make_float2(xm[0], xm[32]);
            cols.x23[m] = make_float2(xm[64], xm[96]);
            cols.x4[m] = xm[128];
        }
        float gsum[kGuRowsPerWarp], usum[kGuRowsPerWarp];
#pragma unroll
        for (int q = 0; q < kGuRowsPerWarp; ++q) {
            const int r = warp * kGuRowsPerWarp + q;
            gsum[q] = warp_sum(lane_row_dot<MB>(gbuf + r * Bh, Bh, lut, cols.x01, cols.x23, cols.x4, lane));
            usum[q] = warp_sum(lane_row_dot<MB>(ubuf + r * Bh, Bh, lut, cols.x01, cols.x23, cols.x4, lane));
        }
        if (lane < kGuRowsPerWarp) {  // lane q finishes row pair q
            float ag = gsum[0], au = usum[0];
#pragma unroll
            for (int q = 1; q < kGuRowsPerWarp; ++q)
                if (lane == q) {
                    ag = gsum[q];
                    au = usum[q];
                }
            const int r = warp * kGuRowsPerWarp + lane;
            const float g = (2.f * ag) * sgbuf[r];
            const float u = (2.f * au) * subuf[r];
            const float gc = fminf(g, a.clamp);
            const float uc = fminf(fmaxf(u, -a.clamp), a.clamp);
            a.h[(int64_t)s * I + r0 + r] = silu_f(gc) * uc;
        }
    }
}

// down + combine: one CTA = kDnRows (16) output rows of one token.  Thread 0 arms the
// barrier with the bytes of all copies; then one thread per copy issues, for each of
// the token's k slots, the expert's 16-row group, the slot's h and the 16 row scales.
// The partial sums come from down_group_partials (two warps per slot, lanes owning
// columns); one thread per row then adds the slots in order i = 0..k-1.
// Requires: H % kDnRows == 0, I % 4 == 0, k <= kDnMaxK, 16-byte aligned bases.
template <int MB>
__global__ void __launch_bounds__(kDnWarps * 32) ffn_down_tma_kernel(FfnArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_e[kDnMaxK];
    __shared__ float s_w[kDnMaxK];
    __shared__ float s_part[kDnMaxK][kDnRows];
    TritLut16& lut = *reinterpret_cast<TritLut16*>(smem);
    const int tid = threadIdx.x;
    const int H = a.H, I = a.I, Bi = (I + 4) / 5, k = a.k;
    const int dbytes = kDnRows * Bi;  // a multiple of 16
    uint8_t* dbuf = smem + kLut16Bytes;
    float* hbuf = reinterpret_cast<float*>(dbuf + k * dbytes);
    float* sdbuf = hbuf + k * I;  // [k][kDnRows] row scales
    if (tid == 0) {
        // the decode table needs nothing from earlier kernels: start its copy now
        mbar_init(&bar, 1);
        mbar_expect_tx(&bar, (uint32_t)kLut16Bytes);  // no arrival: phase 0 stays open
        bulk_copy_g2s(&lut, &g_lut16_image, kLut16Bytes, &bar);
    }
    pdl_wait();
    pdl_launch_dependents();

    const int t = blockIdx.x;
    const int c0 = blockIdx.y * kDnRows;
    if (tid < k) {
        const int e = a.idx[t * k + tid];
        s_e[tid] = (e >= 0 && e < a.E) ? e : -1;
        s_w[tid] = a.w[t * k + tid];
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t total = 0;
        for (int i = 0; i < k; ++i)
            if (s_e[i] >= 0) total += dbytes + 4u * I + 4u * kDnRows;
        mbar_arrive_expect_tx(&bar, total);  // the one arrival of phase 0
    }
    __syncthreads();  // armed before any copy can complete
    if (tid < 3 * k) {
        const int i = tid / 3, part = tid - 3 * i, e = s_e[i];
        if (e >= 0) {
            if (part == 0)
                bulk_copy_g2s(dbuf + i * dbytes, a.down + ((int64_t)e * H + c0) * Bi, dbytes, &bar);
            else if (part == 1)
                bulk_copy_g2s(hbuf + i * I, a.h + (int64_t)(t * k + i) * I, 4u * I, &bar);
            else
                bulk_copy_g2s(sdbuf + i * kDnRows, a.s_down + (int64_t)e * H + c0, 4u * kDnRows, &bar);
        }
    }
    {
        const bool ok = mbar_wait_bounded(&bar, 0, a.status);
        if (__syncthreads_or(!ok)) {
            if (!ok) mbar_wait_bounded(&bar, 0, nullptr);  // let copies in flight land first
            return;
        }
    }
    down_group_partials<MB, false>(
        k, I, Bi, lut, [&](int i) { return dbuf + i * dbytes; }, [&](int i) { return hbuf + i * I; },
        [&](int i) { return s_e[i] >= 0; }, s_part, kDnWarps);
    __syncthreads();
    if (tid < kDnRows) {
        float y = 0.f;
        for (int i = 0; i < k; ++i)
            if (s_e[i] >= 0) y += s_w[i] * (sdbuf[i * kDnRows + tid] * (2.f * s_part[i][tid]));
        a.y[(int64_t)t * H + c0 + tid] = y;
    }
}

bool gateup_tma_ok(const FfnArgs& a) {
    const int Bh = (a.H + 4) / 5;
    return a.I % kGuRows == 0 && Bh % 2 == 0 && a.H % 8 == 0 && (Bh + 31) / 32 <= 13;
}

bool down_tma_ok(const FfnArgs& a) {
    const int Bi = (a.I + 4) / 5;
    return a.H % kDnRows == 0 && a.I % 4 == 0 && a.k <= kDnMaxK && (Bi + 31) / 32 <= 13;
}

template <int MB>
cudaError_t launch_gateup_tma_mb(const FfnArgs& a, int slot_mode, cudaStream_t stream) {
    const int S = a.T * a.k;
    const int ny = slot_mode ? S : (a.E < S ? a.E : S);
    const int Bh = (a.H + 4) / 5;
    const size_t smem = kLut16Bytes + 2 * (size_t)kGuRows * Bh + 8 * (size_t)kGuRows +
                        2 * (size_t)((a.H + 7) / 8 * 8) + 4 * (size_t)(32 * MB * 5);
    cudaError_t err = ensure_dynamic_smem(ffn_gateup_tma_kernel<MB>, smem);
    if (err != cudaSuccess) return err;
    dim3 grid(a.I / kGuRows, ny);
    return launch_pdl(ffn_gateup_tma_kernel<MB>, grid, dim3(kGuWarps * 32), smem, stream, a, slot_mode);
}

template <int MB>
cudaError_t launch_down_tma_mb(const FfnArgs& a, cudaStream_t stream) {
    const int Bi = (a.I + 4) / 5;
    const size_t smem = kLut16Bytes + (size_t)a.k * ((size_t)kDnRows * Bi + 4 * (size_t)a.I + 4 * kDnRows);
    cudaError_t err = ensure_dynamic_smem(ffn_down_tma_kernel<MB>, smem);
    if (err != cudaSuccess) return err;
    dim3 grid(a.T, a.H / kDnRows);
    return launch_pdl(ffn_down_tma_kernel<MB>, grid, dim3(kDnWarps * 32), smem, stream, a);
}

template <int MB>
cudaError_t launch_gateup_mb(const FfnArgs& a, int slot_mode, cudaStream_t stream) {
    const int S = a.T * a.k;
    const int ny = slot_mode ? S : (a.E < S ? a.E : S);
    dim3 grid((a.I + kRowsPerCta - 1) / kRowsPerCta, ny);
    return launch_pdl(ffn_gateup_generic_kernel<MB>, grid, dim3(kWarps * 32), sizeof(float) * a.H, stream,
                      a, slot_mode);
}

template <int MB>
cudaError_t launch_down_mb(const FfnArgs& a, cudaStream_t stream) {
    dim3 grid(a.T, (a.H + kRowsPerCta - 1) / kRowsPerCta);
    return launch_pdl(ffn_down_generic_kernel<MB>, grid, dim3(kWarps * 32), 0, stream, a);
}

#define MAPLE_MB_SWITCH(MBV, CALL)                \
    switch (MBV) {                                \
        case 1: return CALL(1);                   \
        case 2: return CALL(2);                   \
        case 3: return CALL(3);                   \
        case 4: return CALL(4);                   \
        case 5: return CALL(5);                   \
        case 6: return CALL(6);                   \
        case 7: return CALL(7);                   \
        case 8: return CALL(8);                   \
        case 9: return CALL(9);                   \
        case 10: return CALL(10);                 \
        case 11: return CALL(11);                 \
        case 12: return CALL(12);                 \
        case 13: return CALL(13);                 \
        default: return cudaErrorInvalidValue;    \
    }

cudaError_t launch_gateup(const FfnArgs& a, int slot_mode, cudaStream_t stream) {
    const int mb = ((a.H + 4) / 5 + 31) / 32;
    if (gateup_tma_ok(a)) {
#define MAPLE_CALL_GUT(M) launch_gateup_tma_mb<M>(a, slot_mode, stream)
        MAPLE_MB_SWITCH(mb, MAPLE_CALL_GUT)
#undef MAPLE_CALL_GUT
    }
#define MAPLE_CALL_GU(M) launch_gateup_mb<M>(a, slot_mode, stream)
    MAPLE_MB_SWITCH(mb, MAPLE_CALL_GU)
#undef MAPLE_CALL_GU
}

cudaError_t launch_down(const FfnArgs& a, cudaStream_t stream) {
    const int mb = ((a.I + 4) / 5 + 31) / 32;
    if (down_tma_ok(a)) {
#define MAPLE_CALL_DNT(M) launch_down_tma_mb<M>(a, stream)
        MAPLE_MB_SWITCH(mb, MAPLE_CALL_DNT)
#undef MAPLE_CALL_DNT
    }
#define MAPLE_CALL_DN(M) launch_down_mb<M>(a, stream)
    MAPLE_MB_SWITCH(mb, MAPLE_CALL_DN)
#undef MAPLE_CALL_DN
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

FfnWorkspaceLayout ffn_workspace_layout(int T, int k, int E, int H, int I, bool tensor) {
    const size_t S = (size_t)T * (size_t)k;
    FfnWorkspaceLayout L{};
    size_t o = 0;
    L.counts = o;
    o = align_up(o + 4 * (size_t)E, 256);
    L.offsets = o;
    o = align_up(o + 4 * ((size_t)E + 1), 256);
    L.perm = o;
    o = align_up(o + 4 * S, 256);
    L.active = o;
    o = align_up(o + 4 * (size_t)E, 256);
    L.n_active = o;
    o = align_up(o + 4, 256);
    L.h = o;
    o = align_up(o + 4 * S * (size_t)I, 256);
    L.tensor = tensor;
    L.tile_off = L.chunks = L.xs = L.hs = L.xscale = L.hscale = L.ys = o;
    if (L.tensor) {
        o = align_up(o + 4 * (((size_t)E + 1 + 3) & ~(size_t)3) + 16 * (size_t)ffn_tensor_max_tiles((int)S, E), 256);
        L.chunks = o;
        o = align_up(o + group_chunked_bytes((int)S, E), 256);
        L.xs = o;
        o = align_up(o + ffn_tensor_x_bytes((int)S, E, H), 256);
        L.hs = o;
        o = align_up(o + ffn_tensor_h_bytes((int)S, E, I), 256);
        L.xscale = o;
        o = align_up(o + ffn_tensor_scale_bytes((int)S, E), 256);
        L.hscale = o;
        o = align_up(o + ffn_tensor_scale_bytes((int)S, E), 256);
        L.ys = o;
        o = align_up(o + 4 * S * (size_t)H, 256);
    }
    L.total = o;
    return L;
}

cudaError_t launch_moe_ffn(const FfnArgs& args, cudaStream_t stream, const DeviceInfo& dev) {
    FfnArgs a = args;
    const int64_t down_bytes = (int64_t)a.H * ((a.I + 4) / 5);
    a.prefetch_down = (down_bytes % 16 == 0 && a.H % 4 == 0) ? 1 : 0;
    if (a.tensor) return launch_moe_ffn_tensor(a, stream, dev);
    const int S = a.T * a.k;
    const int slot_mode = a.T == 1 ? 1 : 0;
    if (!slot_mode) {
        cudaError_t err = launch_group_tokens(a.idx, S, a.k, a.E, a.counts, a.offsets, a.perm,
                                              a.active, a.n_active, stream, dev);
        if (err != cudaSuccess) return err;
    }
    cudaError_t err = launch_gateup(a, slot_mode, stream);
    if (err != cudaSuccess) return err;
    return launch_down(a, stream);
}

}  // namespace maple
