// One whole MoE layer step for a single decode token in one launch: route, gate/up and
// down + combine, separated by two grid-wide barriers instead of kernel boundaries.
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// sections "The claim, verified from the bytes" (full-precision router, 8 of 256
// experts) and "The shipped code does no quantization" (the expert body with its
// clamps); "IA de 20B Rodando a 120 tok/s no iPhone", section "Pesos ternarios"
// (skip / add / subtract).
//
// At batch 1 a layer moves ~5 MB but is a chain of dependent steps (logits -> top-k ->
// expert rows -> h -> down rows).  Separate kernels pay a launch, a completion flush
// and a dependent re-read of their inputs at every boundary; here one persistent,
// cooperative grid (one CTA per SM) keeps its state in shared memory and synchronises
// with two bounded grid barriers.
//
// Phase 0 (before the programmatic-dependent-launch wait): each CTA starts bulk copies
//   of the decode table and of its share of the router rows (static weights).
// Phase 1: each CTA computes the logits of its router rows (same accumulation order as
//   route_logits_kernel) into the caller's logits buffer; x is converted to fp32 in
//   lane-column order for phase 2.                                   -- grid barrier --
// Phase 2: every CTA reads all E logits and runs the same top-k + softmax (CTA 0 stores
//   idx and w).  It then issues, at once, bulk copies of its gate/up items (8 row pairs
//   of one expert each) and of its 16-row down group for all k experts, computes h for
//   its items and stores it.                                         -- grid barrier --
// Phase 3: each CTA with a down group copies the k slots' h, computes its 16 output
//   rows (two warps per slot, lanes owning columns) and adds the slots in order
//   i = 0..k-1.
// Every wait is bounded; a wait that gives up records MAPLE_ERR_TIMEOUT in the device
// status word and the CTA skips the remaining work but still takes part in the
// barriers and the exit count.  The last CTA to exit resets the barrier counters.
#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

constexpr int kLdWarps = 16;
constexpr int kLdThreads = kLdWarps * 32;
constexpr int kLdItemRows = 8;    // row pairs per gate/up item
constexpr int kLdDownRows = 16;   // output rows per down group
constexpr int kLdMaxItems = 8;
constexpr int kLdMaxRouterRows = 8;
constexpr int kLdMaxK = 12;
constexpr int kLdMaxDownLaneBytes = 4;  // ceil(ceil(I/5)/32) <= 4, i.e. I <= 640
constexpr int kLdBarrierCounters = 8;   // arrival counters (CTA c adds to c % 8)
constexpr int kLdLutBytes = (int)sizeof(TritLut16);
constexpr uint32_t kBarrierPolls = 1u << 22;

struct LayerArgs {
    const uint16_t* x;
    const uint16_t* Wr;
    const float* bias;
    const uint8_t* gate;
    const uint8_t* up;
    const uint8_t* down;
    const float* s_gate;
    const float* s_up;
    const float* s_down;
    int E, H, I, k;
    int nr;      // router rows per CTA (upper bound)
    int nitems;  // gate/up items per CTA (upper bound)
    float clamp;
    float* logits;
    int32_t* idx;
    float* w;
    float* y;
    float* h;         // [k][I]
    unsigned* sync;   // [0..7] barrier arrivals, [8] exits: zero on entry, zero on exit
    int* status;
};

struct LayerSmem {
    int wr, xb, xcol, gu, item_bytes, dn, dn_bytes, hb, lg, total;
};

__host__ __device__ inline LayerSmem layer_smem(int H, int I, int E, int k, int nr, int nitems, int MB) {
    const int Bh = (H + 4) / 5, Bi = (I + 4) / 5;
    LayerSmem L;
    int o = kLdLutBytes;
    L.wr = o;
    o += nr * 2 * H;
    L.xb = o;
    o += 2 * H;
    L.xcol = o;
    o += 4 * 32 * MB * 5;
    L.gu = o;
    L.item_bytes = 2 * kLdItemRows * Bh + 8 * kLdItemRows;  // gate rows, up rows, 2 x scales
    o += nitems * L.item_bytes;
    L.dn = o;
    L.dn_bytes = kLdDownRows * Bi + 4 * kLdDownRows;  // rows + scales, per slot
    o += k * L.dn_bytes;
    L.hb = o;
    o += k * 4 * I;
    L.lg = o;
    o += 4 * ((E + 3) / 4 * 4);
    L.total = o;
    return L;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Grid-wide barrier over co-resident CTAs.  Thread 0 publishes this CTA's writes
// (fence + release add) on one of kLdBarrierCounters counters; lanes 0..7 of warp 0
// poll one counter each with acquire loads until the counters sum to `target`, a
// bounded number of times.  Spreading the arrivals keeps the atomics on one counter
// few.  Returns false (and records MAPLE_ERR_TIMEOUT) if the wait gave up.
__device__ bool grid_barrier(unsigned* ctr, unsigned target, int* status, int* s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add(ctr + blockIdx.x % kLdBarrierCounters, 1u);
    }
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int ok = 1;
        uint32_t polls = 0;
        while (true) {
            const unsigned v = lane < kLdBarrierCounters ? ld_acquire(ctr + lane) : 0u;
            if (__reduce_add_sync(kFullMask, v) >= target) break;
            if (++polls > kBarrierPolls) {
                ok = 0;
                if (lane == 0) atomicExch(status, kStatusTimeout);
                break;
            }
        }
        if (lane == 0) *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

template <int MB>
__global__ void __launch_bounds__(kLdThreads, 1) moe_layer_b1_kernel(LayerArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar_in;
    __shared__ __align__(8) uint64_t bar_x;
    __shared__ __align__(8) uint64_t bar_gu[kLdMaxItems];
    __shared__ __align__(8) uint64_t bar_dn;
    __shared__ __align__(8) uint64_t bar_h;
    __shared__ int s_idx[32];
    __shared__ float s_val[32];
    __shared__ float s_w[32];
    __shared__ float s_part[kLdMaxK][kLdDownRows];
    __shared__ int s_ok, s_fail;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int H = a.H, I = a.I, E = a.E, k = a.k;
    const int Bh = (H + 4) / 5, Bi = (I + 4) / 5;
    const int ngroups = I / kLdItemRows;
    const LayerSmem L = layer_smem(H, I, E, k, a.nr, a.nitems, MB);
    unsigned* exits = a.sync + kLdBarrierCounters;
    TritLut16& lut = *reinterpret_cast<TritLut16*>(smem);
    uint16_t* wr = reinterpret_cast<uint16_t*>(smem + L.wr);
    uint16_t* xb = reinterpret_cast<uint16_t*>(smem + L.xb);
    float* xcol = reinterpret_cast<float*>(smem + L.xcol);
    uint8_t* gu = smem + L.gu;
    uint8_t* dn = smem + L.dn;
    float* hb = reinterpret_cast<float*>(smem + L.hb);
    float* lg = reinterpret_cast<float*>(smem + L.lg);

    int nr_mine = 0;
    for (int j = 0; j < a.nr; ++j)
        if (c + j * G < E) ++nr_mine;
    int n_items = 0;
    for (int n = 0; n < a.nitems; ++n)
        if (c + n * G < k * ngroups) ++n_items;
    const bool has_dn = c < H / kLdDownRows;

    // ---- phase 0: static inputs, before the dependency wait
    if (tid == 0) {
        s_fail = 0;
        mbar_init(&bar_in, 1);
        mbar_init(&bar_x, 1);
        for (int n = 0; n < kLdMaxItems; ++n) mbar_init(&bar_gu[n], 1);
        mbar_init(&bar_dn, 1);
        mbar_init(&bar_h, 1);
        mbar_arrive_expect_tx(&bar_in, (uint32_t)(kLdLutBytes + nr_mine * 2 * H));
        bulk_copy_g2s(&lut, &g_lut16_image, kLdLutBytes, &bar_in);
        for (int j = 0; j < nr_mine; ++j)
            bulk_copy_g2s(wr + j * H, a.Wr + (int64_t)(c + j * G) * H, 2u * H, &bar_in);
    }
    pdl_wait();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_x, 2u * H);
        bulk_copy_g2s(xb, a.x, 2u * H, &bar_x);
    }
    __syncthreads();  // barriers initialised before anyone waits on them
    if (!mbar_wait_bounded(&bar_in, 0, a.status) || !mbar_wait_bounded(&bar_x, 0, a.status))
        s_fail = 1;
    __syncthreads();

    // ---- phase 1: logits of this CTA's router rows; x in lane-column order
    if (!s_fail) {
        if (warp < nr_mine) {
            const int e = c + warp * G;
            const uint4* w4 = reinterpret_cast<const uint4*>(wr + warp * H);
            const uint4* x4 = reinterpret_cast<const uint4*>(xb);
            const int n8 = H >> 3;
            float acc = 0.f;
            for (int base = 0; base < n8; base += 32 * 8) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int cc = base + lane + 32 * u;
                    if (cc < n8) {
                        const uint4 wv = w4[cc], xv = x4[cc];
                        acc = fmaf(bf16_lo(wv.x), bf16_lo(xv.x), acc);
                        acc = fmaf(bf16_hi(wv.x), bf16_hi(xv.x), acc);
                        acc = fmaf(bf16_lo(wv.y), bf16_lo(xv.y), acc);
                        acc = fmaf(bf16_hi(wv.y), bf16_hi(xv.y), acc);
                        acc = fmaf(bf16_lo(wv.z), bf16_lo(xv.z), acc);
                        acc = fmaf(bf16_hi(wv.z), bf16_hi(xv.z), acc);
                        acc = fmaf(bf16_lo(wv.w), bf16_lo(xv.w), acc);
                        acc = fmaf(bf16_hi(wv.w), bf16_hi(xv.w), acc);
                    }
                }
            }
            const float v = warp_sum(acc);
            if (lane == 0) a.logits[e] = v + (a.bias != nullptr ? a.bias[e] : 0.f);
        }
        for (int i = tid; i < 32 * MB * 5; i += blockDim.x) {
            const int l = i & 31, md = i >> 5, m = md / 5, d = md - 5 * m;
            const int col = 5 * (l + 32 * m) + d;
            xcol[i] = col < H ? bf16_bits_to_float(xb[col]) : 0.f;
        }
    }
    if (!grid_barrier(a.sync, (unsigned)G, a.status, &s_ok)) s_fail = 1;

    // ---- phase 2: selection, gate/up
    bool issued_gu = false, issued_dn = false;
    if (!s_fail) {
        for (int e = tid; e < E; e += blockDim.x) {
            const float v = __ldcg(a.logits + e);
            lg[e] = (v != v) ? -INFINITY : v;  // NaN ranks last
        }
        __syncthreads();
        if (warp == 0) {
            int my_idx;
            float my_val, my_w;
            warp_topk_softmax_smem(lg, E, k, lane, my_idx, my_val, my_w);
            if (lane < k) {
                s_idx[lane] = my_idx;
                s_val[lane] = my_val;
                s_w[lane] = my_w;
                if (c == 0) {
                    a.idx[lane] = my_idx;
                    a.w[lane] = my_w;
                }
            }
        }
        __syncthreads();
        if (tid == 0) {  // arm every barrier before any copy can complete
            for (int n = 0; n < n_items; ++n)
                mbar_arrive_expect_tx(&bar_gu[n], (uint32_t)(2 * kLdItemRows * Bh + 8 * kLdItemRows));
            if (has_dn) mbar_arrive_expect_tx(&bar_dn, (uint32_t)(k * L.dn_bytes));
        }
        __syncthreads();
        // one thread per copy: 4 per gate/up item, 2 per slot for the down group
        if (tid < 4 * n_items) {
            const int n = tid >> 2, part = tid & 3;
            const int j = c + n * G, i = j / ngroups, g = j - i * ngroups, e = s_idx[i];
            const int r0 = g * kLdItemRows;
            uint8_t* it = gu + n * L.item_bytes;
            const uint32_t rows = kLdItemRows * Bh;
            if (part == 0)
                bulk_copy_g2s(it, a.gate + ((int64_t)e * I + r0) * Bh, rows, &bar_gu[n]);
            else if (part == 1)
                bulk_copy_g2s(it + rows, a.up + ((int64_t)e * I + r0) * Bh, rows, &bar_gu[n]);
            else if (part == 2)
                bulk_copy_g2s(it + 2 * rows, a.s_gate + (int64_t)e * I + r0, 4u * kLdItemRows, &bar_gu[n]);
            else
                bulk_copy_g2s(it + 2 * rows + 4 * kLdItemRows, a.s_up + (int64_t)e * I + r0,
                              4u * kLdItemRows, &bar_gu[n]);
        } else if (has_dn && tid >= 32 && tid < 32 + 2 * k) {
            const int i = (tid - 32) >> 1, part = (tid - 32) & 1, c0 = c * kLdDownRows;
            uint8_t* d = dn + i * L.dn_bytes;
            if (part == 0)
                bulk_copy_g2s(d, a.down + ((int64_t)s_idx[i] * H + c0) * Bi, kLdDownRows * Bi, &bar_dn);
            else
                bulk_copy_g2s(d + kLdDownRows * Bi, a.s_down + (int64_t)s_idx[i] * H + c0,
                              4u * kLdDownRows, &bar_dn);
        }
        issued_gu = true;
        issued_dn = has_dn;
        // lane columns of x (the same for every item)
        float2 x01[MB], x23[MB];
        float x4[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const float* xm = xcol + (m * 5) * 32 + lane;
            x01[m] = make_float2(xm[0], xm[32]);
            x23[m] = make_float2(xm[64], xm[96]);
            x4[m] = xm[128];
        }
        const int q = warp & 7;
        for (int p = 0; 2 * p < n_items; ++p) {
            const int n = 2 * p + (warp >> 3);
            if (n >= n_items) continue;
            if (!mbar_wait_bounded(&bar_gu[n], 0, a.status)) {
                s_fail = 1;
                continue;
            }
            const uint8_t* it = gu + n * L.item_bytes;
            const int rows = kLdItemRows * Bh;
            const float* sg = reinterpret_cast<const float*>(it + 2 * rows);
            const float* su = sg + kLdItemRows;
            const float ag = warp_sum(lane_row_dot<MB>(it + q * Bh, Bh, lut, x01, x23, x4, lane));
            const float au = warp_sum(lane_row_dot<MB>(it + rows + q * Bh, Bh, lut, x01, x23, x4, lane));
            if (lane == 0) {
                const int j = c + n * G, i = j / ngroups, g = j - i * ngroups;
                const int r = g * kLdItemRows + q;
                const float gv = (2.f * ag) * sg[q];
                const float uv = (2.f * au) * su[q];
                const float gc = fminf(gv, a.clamp);
                const float uc = fminf(fmaxf(uv, -a.clamp), a.clamp);
                a.h[(int64_t)i * I + r] = silu_f(gc) * uc;
                fence_proxy_async_global();  // h is read by bulk copies in phase 3
            }
        }
    }
    if (!grid_barrier(a.sync, 2u * (unsigned)G, a.status, &s_ok)) s_fail = 1;

    // ---- phase 3: down + combine for this CTA's 16 output rows
    bool issued_h = false;
    if (!s_fail && has_dn) {
        if (tid == 0) mbar_arrive_expect_tx(&bar_h, (uint32_t)(k * 4 * I));
        __syncthreads();
        if (tid < k) {
            fence_proxy_async_global();  // h was written by other CTAs' generic stores
            bulk_copy_g2s(hb + tid * I, a.h + (int64_t)tid * I, 4u * I, &bar_h);
        }
        issued_h = true;
        if (!mbar_wait_bounded(&bar_dn, 0, a.status) || !mbar_wait_bounded(&bar_h, 0, a.status)) s_fail = 1;
        __syncthreads();
        if (!s_fail) {
            down_group_partials<kLdMaxDownLaneBytes, true>(
                k, I, Bi, lut, [&](int i) { return dn + i * L.dn_bytes; }, [&](int i) { return hb + i * I; },
                [&](int) { return true; }, s_part, kLdWarps);
            __syncthreads();
            if (tid < kLdDownRows) {
                const int c0 = c * kLdDownRows;
                float yv = 0.f;
                for (int i = 0; i < k; ++i) {
                    const float* sd = reinterpret_cast<const float*>(dn + i * L.dn_bytes + kLdDownRows * Bi);
                    yv += s_w[i] * (sd[tid] * (2.f * s_part[i][tid]));
                }
                a.y[c0 + tid] = yv;
            }
        }
    }

    // ---- exit: copies this CTA issued must have landed; the last CTA out resets sync
    __syncthreads();
    if (tid == 0) {
        mbar_wait_bounded(&bar_in, 0, nullptr);
        mbar_wait_bounded(&bar_x, 0, nullptr);
        if (issued_gu)
            for (int n = 0; n < n_items; ++n) mbar_wait_bounded(&bar_gu[n], 0, nullptr);
        if (issued_dn) mbar_wait_bounded(&bar_dn, 0, nullptr);
        if (issued_h) mbar_wait_bounded(&bar_h, 0, nullptr);
        __threadfence();
        const unsigned done = atomicAdd(exits, 1u);
        if (done == (unsigned)G - 1) {
            for (int j = 0; j < kLdBarrierCounters; ++j) atomicExch(a.sync + j, 0u);
            atomicExch(exits, 0u);
        }
    }
}

#define MAPLE_LD_SWITCH(MBV, CALL)             \
    switch (MBV) {                             \
        case 1: return CALL(1);                \
        case 2: return CALL(2);                \
        case 3: return CALL(3);                \
        case 4: return CALL(4);                \
        case 5: return CALL(5);                \
        case 6: return CALL(6);                \
        case 7: return CALL(7);                \
        case 8: return CALL(8);                \
        case 9: return CALL(9);                \
        case 10: return CALL(10);              \
        case 11: return CALL(11);              \
        case 12: return CALL(12);              \
        case 13: return CALL(13);              \
        default: return cudaErrorInvalidValue; \
    }

template <int MB>
cudaError_t launch_layer_mb(const LayerArgs& a, int G, size_t smem, cudaStream_t stream) {
    cudaError_t err = ensure_dynamic_smem(moe_layer_b1_kernel<MB>, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kLdThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, moe_layer_b1_kernel<MB>, a);
}

}  // namespace

bool layer_b1_supported(int H, int I, int E, int k, const DeviceInfo& dev) {
    const int G = dev.sm_count;
    const int Bh = (H + 4) / 5, Bi = (I + 4) / 5;
    if (H % kLdDownRows != 0 || H / kLdDownRows > G) return false;
    if (I % kLdItemRows != 0 || I % 4 != 0 || Bh % 2 != 0 || (Bh + 31) / 32 > 13) return false;
    if ((Bi + 31) / 32 > kLdMaxDownLaneBytes) return false;
    if (k > kLdMaxK || k > 32 || E > 1024) return false;
    if ((E + G - 1) / G > kLdMaxRouterRows || (E + G - 1) / G > kLdWarps) return false;
    if ((k * (I / kLdItemRows) + G - 1) / G > kLdMaxItems) return false;
    const int MB = (Bh + 31) / 32;
    const LayerSmem L = layer_smem(H, I, E, k, (E + G - 1) / G, (k * (I / kLdItemRows) + G - 1) / G, MB);
    return (size_t)L.total <= dev.smem_optin - 1024 && Bi >= 1;
}

cudaError_t launch_moe_layer_b1(const LayerLaunch& p, cudaStream_t stream, const DeviceInfo& dev) {
    const int G = dev.sm_count;
    LayerArgs a;
    a.x = p.x;
    a.Wr = p.Wr;
    a.bias = p.bias;
    a.gate = p.gate;
    a.up = p.up;
    a.down = p.down;
    a.s_gate = p.s_gate;
    a.s_up = p.s_up;
    a.s_down = p.s_down;
    a.E = p.E;
    a.H = p.H;
    a.I = p.I;
    a.k = p.k;
    a.nr = (p.E + G - 1) / G;
    a.nitems = (p.k * (p.I / kLdItemRows) + G - 1) / G;
    a.clamp = p.clamp;
    a.logits = p.logits;
    a.idx = p.idx;
    a.w = p.w;
    a.y = p.y;
    a.h = p.h;
    a.sync = p.sync;
    a.status = dev.status;
    const int MB = ((p.H + 4) / 5 + 31) / 32;
    const size_t smem = (size_t)layer_smem(p.H, p.I, p.E, p.k, a.nr, a.nitems, MB).total;
#define MAPLE_CALL_LD(M) launch_layer_mb<M>(a, G, smem, stream)
    MAPLE_LD_SWITCH(MB, MAPLE_CALL_LD)
#undef MAPLE_CALL_LD
}

}  // namespace maple
