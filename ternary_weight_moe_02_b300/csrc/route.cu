// Full-precision MoE router: bf16 GEMV/GEMM to fp32 logits, top-k, softmax over
// the k selected.
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// section "The claim, verified from the bytes": the router stays in full precision
// and picks 8 of 256 experts from the margin between logits.
//
// Kernels 1 and 1' (logits, H a multiple of 8): bf16 x bf16 products are exact in fp32;
// lane L accumulates, with FMA, the products of the 16-byte chunks L, L + 32, ... in
// column order, then a butterfly combines the lanes (depth H/32 + 5 additions).
// Kernel 1 (up to 256 tokens) stages the token rows in shared memory and keeps one
// router row per warp in registers; kernel 1' (more tokens) is register-tiled, a warp
// computing 4 tokens x 8 experts so that each chunk of x or Wr it loads serves 8 or 4
// outputs.  Both run every logit's FMA chain in the same order and the same butterfly,
// so they give identical logits (the fused batch-1 layer kernel too).
// Kernel 1'' (H not a multiple of 8): one warp per expert row, lane L taking the
// elements L, L + 32, ... .
// Kernel 2 (select): one warp per token; k rounds of warp arg-max (ties to the lower
// expert id), then softmax of the k winners in fp32.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

constexpr int kRouteWarps = 2;   // expert rows per CTA
constexpr int kRouteTokens = 8;  // tokens per CTA

__global__ void __launch_bounds__(kRouteWarps * 32)
    route_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ Wr,
                        const float* __restrict__ bias, int T, int H, int E,
                        float* __restrict__ logits) {
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouteWarps + warp;
    const int t0 = blockIdx.y * kRouteTokens;
    if (e >= E) return;
    const int nt = min(kRouteTokens, T - t0);
    float acc[kRouteTokens];
#pragma unroll
    for (int t = 0; t < kRouteTokens; ++t) acc[t] = 0.f;
    const uint16_t* wr = Wr + (int64_t)e * H;
    for (int j = lane; j < H; j += 32) {
        const float wf = bf16_bits_to_float(wr[j]);
#pragma unroll
        for (int t = 0; t < kRouteTokens; ++t)
            if (t < nt) acc[t] = fmaf(wf, bf16_bits_to_float(x[(int64_t)(t0 + t) * H + j]), acc[t]);
    }
    const float b = bias != nullptr ? bias[e] : 0.f;
#pragma unroll
    for (int t = 0; t < kRouteTokens; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0 && t < nt) logits[(int64_t)(t0 + t) * E + e] = v + b;
    }
}

constexpr int kTileTok = 4;    // tokens per warp
constexpr int kTileExp = 8;    // experts per warp
constexpr int kTileWarpsT = 2; // warps along tokens in a CTA
constexpr int kTileWarpsE = 4; // warps along experts in a CTA

__global__ void __launch_bounds__(kTileWarpsT * kTileWarpsE * 32)
    route_logits_tiled_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ Wr,
                              const float* __restrict__ bias, int T, int H, int E,
                              float* __restrict__ logits) {
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = (blockIdx.y * kTileWarpsT + (warp % kTileWarpsT)) * kTileTok;
    const int e0 = (blockIdx.x * kTileWarpsE + (warp / kTileWarpsT)) * kTileExp;
    if (t0 >= T || e0 >= E) return;
    float acc[kTileTok][kTileExp];
#pragma unroll
    for (int t = 0; t < kTileTok; ++t)
#pragma unroll
        for (int e = 0; e < kTileExp; ++e) acc[t][e] = 0.f;
    const int n8 = H >> 3;
    for (int c = lane; c < n8; c += 32) {
        uint4 wv[kTileExp], xv[kTileTok];
#pragma unroll
        for (int e = 0; e < kTileExp; ++e)
            wv[e] = e0 + e < E ? ldg_nc_v4(reinterpret_cast<const uint4*>(Wr + (int64_t)(e0 + e) * H) + c)
                               : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int t = 0; t < kTileTok; ++t)
            xv[t] = t0 + t < T ? ldg_nc_v4(reinterpret_cast<const uint4*>(x + (int64_t)(t0 + t) * H) + c)
                               : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float wf[kTileExp], xf[kTileTok];
#pragma unroll
            for (int e = 0; e < kTileExp; ++e) {
                const uint32_t word = j < 2 ? wv[e].x : (j < 4 ? wv[e].y : (j < 6 ? wv[e].z : wv[e].w));
                wf[e] = (j & 1) ? bf16_hi(word) : bf16_lo(word);
            }
#pragma unroll
            for (int t = 0; t < kTileTok; ++t) {
                const uint32_t word = j < 2 ? xv[t].x : (j < 4 ? xv[t].y : (j < 6 ? xv[t].z : xv[t].w));
                xf[t] = (j & 1) ? bf16_hi(word) : bf16_lo(word);
            }
#pragma unroll
            for (int t = 0; t < kTileTok; ++t)
#pragma unroll
                for (int e = 0; e < kTileExp; ++e) acc[t][e] = fmaf(wf[e], xf[t], acc[t][e]);
        }
    }
#pragma unroll
    for (int t = 0; t < kTileTok; ++t)
#pragma unroll
        for (int e = 0; e < kTileExp; ++e) {
            const float v = warp_sum(acc[t][e]);
            if (lane == 0 && t0 + t < T && e0 + e < E)
                logits[(int64_t)(t0 + t) * E + e0 + e] = v + (bias != nullptr ? bias[e0 + e] : 0.f);
        }
}

// Kernel 1 (logits, up to kStagedMaxT tokens, H a multiple of 8).  A CTA takes
// kStExp experts (one per warp) and kStTok tokens: each warp
// holds its router row in registers (16-byte chunks lane + 32 u, loaded before the
// dependency wait: the router weights are a static input), one bulk copy brings the
// CTA's token rows (contiguous in x) into shared memory, and the warp runs every
// token's FMA chain from there, then the butterfly.
constexpr int kStExp = 4;
constexpr int kStTok = 16;
constexpr int kStagedMaxT = 256;

template <int MC>  // chunks per lane: H <= 256 MC
__global__ void __launch_bounds__(kStExp * 32)
    route_logits_staged_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ Wr,
                               const float* __restrict__ bias, int T, int H, int E, float* __restrict__ logits,
                               int* status) {
    extern __shared__ __align__(16) uint4 xs[];  // [nt][H / 8]
    __shared__ uint64_t bar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kStExp + warp;
    const int t0 = blockIdx.y * kStTok;
    const int nt = min(kStTok, T - t0);
    const int n8 = H >> 3;
    uint4 wv[MC];
#pragma unroll
    for (int u = 0; u < MC; ++u) {
        const int c = lane + 32 * u;
        wv[u] = (e < E && c < n8) ? ldg_nc_v4(reinterpret_cast<const uint4*>(Wr + (int64_t)e * H) + c)
                                  : make_uint4(0, 0, 0, 0);
    }
    if (threadIdx.x == 0) mbar_init(&bar, 1);
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    const float b = (bias != nullptr && e < E) ? bias[e] : 0.f;
    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)nt * (uint32_t)H * 2u;
        mbar_arrive_expect_tx(&bar, bytes);
        bulk_copy_g2s(xs, x + (int64_t)t0 * H, bytes, &bar);
    }
    // every thread waits: the copy lands before anyone reads it or the CTA exits
    const bool ok = mbar_wait_bounded(&bar, 0, status);
    if (!ok || e >= E) return;
    for (int t = 0; t < nt; ++t) {
        const uint4* xr = xs + (size_t)t * n8;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < MC; ++u) {
            const int c = lane + 32 * u;
            const uint4 xv = c < n8 ? xr[c] : make_uint4(0, 0, 0, 0);
            const float wf[8] = {bf16_lo(wv[u].x), bf16_hi(wv[u].x), bf16_lo(wv[u].y), bf16_hi(wv[u].y),
                                 bf16_lo(wv[u].z), bf16_hi(wv[u].z), bf16_lo(wv[u].w), bf16_hi(wv[u].w)};
            const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                                 bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
            for (int j = 0; j < 8; ++j) acc = fmaf(wf[j], xf[j], acc);
        }
        const float v = warp_sum(acc);
        if (lane == 0) logits[(int64_t)(t0 + t) * E + e] = v + b;
    }
}

// JE = logits held per lane (E <= 32 * JE).
template <int JE>
__global__ void __launch_bounds__(256)
    route_select_kernel(const float* __restrict__ logits, int T, int E, int k,
                        int32_t* __restrict__ idx, float* __restrict__ w) {
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    int my_idx;
    float my_w;
    const float* lt = logits + (int64_t)t * E;
    warp_topk_softmax<JE>([&](int e) { return lt[e]; }, E, k, lane, my_idx, my_w);
    if (lane < k) {
        idx[(int64_t)t * k + lane] = my_idx;
        w[(int64_t)t * k + lane] = my_w;
    }
}

}  // namespace

namespace {

// One launch of each route kernel for at most kRouteChunk tokens.
cudaError_t launch_route_chunk(const uint16_t* x, const uint16_t* Wr, const float* bias, int T, int H, int E,
                               int k, float* logits, int32_t* idx, float* w, cudaStream_t stream, int* status) {
    const int vec = (H % 8 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                    (reinterpret_cast<uintptr_t>(Wr) % 16 == 0);
    cudaError_t err;
    if (vec && T <= kStagedMaxT && H <= 256 * 16) {
        const dim3 gs((E + kStExp - 1) / kStExp, (T + kStTok - 1) / kStTok);
        const size_t smem = (size_t)(T < kStTok ? T : kStTok) * H * 2;
        if (H <= 256 * 8) {
            err = ensure_dynamic_smem(route_logits_staged_kernel<8>, smem);
            if (err == cudaSuccess)
                err = launch_pdl(route_logits_staged_kernel<8>, gs, dim3(kStExp * 32), smem, stream, x, Wr, bias, T,
                                 H, E, logits, status);
        } else {
            err = ensure_dynamic_smem(route_logits_staged_kernel<16>, smem);
            if (err == cudaSuccess)
                err = launch_pdl(route_logits_staged_kernel<16>, gs, dim3(kStExp * 32), smem, stream, x, Wr, bias,
                                 T, H, E, logits, status);
        }
    } else if (vec && route_tc_shape_ok(x, Wr, H) &&
               (err = launch_route_logits_tc(x, Wr, bias, T, H, E, logits, stream, status)) != cudaErrorNotSupported) {
        // tensor cores (more than kStagedMaxT tokens)
    } else if (vec) {
        dim3 gt((E + kTileWarpsE * kTileExp - 1) / (kTileWarpsE * kTileExp),
                (T + kTileWarpsT * kTileTok - 1) / (kTileWarpsT * kTileTok));
        err = launch_pdl(route_logits_tiled_kernel, gt, dim3(kTileWarpsT * kTileWarpsE * 32), 0, stream, x, Wr,
                         bias, T, H, E, logits);
    } else {
        dim3 g1((E + kRouteWarps - 1) / kRouteWarps, (T + kRouteTokens - 1) / kRouteTokens);
        err = launch_pdl(route_logits_kernel, g1, dim3(kRouteWarps * 32), 0, stream, x, Wr, bias, T, H, E,
                         logits);
    }
    if (err != cudaSuccess) return err;
    dim3 g2((T + 7) / 8);
    const float* cl = logits;
    if (E <= 32) return launch_pdl(route_select_kernel<1>, g2, dim3(256), 0, stream, cl, T, E, k, idx, w);
    if (E <= 64) return launch_pdl(route_select_kernel<2>, g2, dim3(256), 0, stream, cl, T, E, k, idx, w);
    if (E <= 128) return launch_pdl(route_select_kernel<4>, g2, dim3(256), 0, stream, cl, T, E, k, idx, w);
    if (E <= 256) return launch_pdl(route_select_kernel<8>, g2, dim3(256), 0, stream, cl, T, E, k, idx, w);
    if (E <= 512) return launch_pdl(route_select_kernel<16>, g2, dim3(256), 0, stream, cl, T, E, k, idx, w);
    return launch_pdl(route_select_kernel<32>, g2, dim3(256), 0, stream, cl, T, E, k, idx, w);
}

}  // namespace

// The logits kernels put T / 8 token groups in gridDim.y (at most 65535): larger calls
// run in chunks of kRouteChunk tokens (each token's logits are the same either way).
cudaError_t launch_route_topk(const uint16_t* x, const uint16_t* Wr, const float* bias, int T,
                              int H, int E, int k, float* logits, int32_t* idx, float* w,
                              cudaStream_t stream, const DeviceInfo& dev) {
    constexpr int kRouteChunk = 65535 * 8;
    int t0 = 0;
    do {
        const int n = T - t0 < kRouteChunk ? T - t0 : kRouteChunk;
        const cudaError_t err = launch_route_chunk(x + (int64_t)t0 * H, Wr, bias, n, H, E, k, logits + (int64_t)t0 * E,
                                                   idx + (int64_t)t0 * k, w + (int64_t)t0 * k, stream, dev.status);
        if (err != cudaSuccess) return err;
        t0 += n;
    } while (t0 < T);
    return cudaSuccess;
}

}  // namespace maple
