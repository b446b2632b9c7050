// Expert FFN of the ternary MoE layer on CUDA cores (decode path).
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// section "The shipped code does no quantization": the expert body is
// down(act(clamp(gate x, max=7)) * clamp(up x, -7, 7)); "IA de 20B Rodando a 120 tok/s
// no iPhone", section "Pesos ternarios": weight 0 skips, +1 adds, -1 subtracts.
//
// gate/up kernel: one CTA = 16 rows of gate and the same 16 rows of up of one expert,
// for every token routed to that expert.  A warp owns 4 row pairs; lane L always owns
// the packed bytes L, L+32, ... of a row, so the activations it needs (5 per byte)
// stay in registers across rows.  Each byte is decoded through a shared-memory table
// (code -> top bytes of +-0.5/0 for its five trits); one byte-permute per trit gives
// the fp32 multiplier, one FMA accumulates it (the product is exact: +-x/2 or 0).
// The row scale (times 2) is applied once to the warp's sum, then SiLU, the clamps
// and the gate*up product give h, stored fp32 per routing slot.
//
// down kernel: one CTA = 16 output rows of one token; it walks the token's k slots in
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
    ffn_gateup_kernel(FfnArgs a, int slot_mode) {
    __shared__ TritLut lut;
    extern __shared__ float xs[];  // [H] activations of the current token, fp32
    build_trit_lut(lut, threadIdx.x, blockDim.x);
    pdl_wait();
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
__global__ void __launch_bounds__(kWarps * 32) ffn_down_kernel(FfnArgs a) {
    __shared__ TritLut lut;
    build_trit_lut(lut, threadIdx.x, blockDim.x);
    pdl_wait();
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

template <int MB>
cudaError_t launch_gateup_mb(const FfnArgs& a, int slot_mode, cudaStream_t stream) {
    const int S = a.T * a.k;
    const int ny = slot_mode ? S : (a.E < S ? a.E : S);
    dim3 grid((a.I + kRowsPerCta - 1) / kRowsPerCta, ny);
    return launch_pdl(ffn_gateup_kernel<MB>, grid, dim3(kWarps * 32), sizeof(float) * a.H, stream,
                      a, slot_mode);
}

template <int MB>
cudaError_t launch_down_mb(const FfnArgs& a, cudaStream_t stream) {
    dim3 grid(a.T, (a.H + kRowsPerCta - 1) / kRowsPerCta);
    return launch_pdl(ffn_down_kernel<MB>, grid, dim3(kWarps * 32), 0, stream, a);
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
#define MAPLE_CALL_GU(M) launch_gateup_mb<M>(a, slot_mode, stream)
    MAPLE_MB_SWITCH(mb, MAPLE_CALL_GU)
#undef MAPLE_CALL_GU
}

cudaError_t launch_down(const FfnArgs& a, cudaStream_t stream) {
    const int mb = ((a.I + 4) / 5 + 31) / 32;
#define MAPLE_CALL_DN(M) launch_down_mb<M>(a, stream)
    MAPLE_MB_SWITCH(mb, MAPLE_CALL_DN)
#undef MAPLE_CALL_DN
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

FfnWorkspaceLayout ffn_workspace_layout(int T, int k, int E, int I) {
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
    L.total = o;
    return L;
}

cudaError_t launch_moe_ffn(const FfnArgs& a, cudaStream_t stream, const DeviceInfo& dev) {
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
