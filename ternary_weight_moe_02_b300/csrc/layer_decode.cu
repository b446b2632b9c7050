// One whole MoE layer step for a single decode token in one launch: route, gate/up,
// down and the weighted combine, with no grid-wide barrier.
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// sections "The claim, verified from the bytes" (full-precision router, 8 of 256
// experts) and "The shipped code does no quantization" (the expert body with its
// clamps); "IA de 20B Rodando a 120 tok/s no iPhone", section "Pesos ternarios"
// (skip / add / subtract).
//
// At batch 1 a layer moves ~5 MB through a chain of dependent steps (logits -> top-k ->
// expert rows -> h -> down rows -> combine).  A grid-wide barrier between the steps
// costs an L2 round trip for every CTA plus the poll, so this kernel has none.  The grid
// is C thread-block clusters of kCS = 16 CTAs, one CTA per SM (512 threads), C the
// number of such clusters the GPU runs at once (7 on a B300) or k if smaller.
// Everything that needs all CTAs of a step is exchanged inside a cluster through
// distributed shared memory:
//
// Phase 0 (before the programmatic-dependent-launch wait, static inputs only): the
//   decode table is bulk-copied into shared memory and each warp loads one of this
//   CTA's router rows (E / 16, one per warp) into registers.
// Phase 1: x is read into shared memory (plain loads through L2); each CTA computes
//   the logits of its router rows (the accumulation order of route_logits_kernel, so
//   the logits are the same bits) and stores them into the logit array of every CTA of
//   its cluster; cluster barrier.
//   Every CTA now holds all E logits and selects the same top-k, so the clusters agree
//   without talking to each other.
// Phase 2: cluster c takes slot c < C whole: CTA rank r bulk-copies its I / 16 gate/up
//   row pairs and its H / 16 down rows (and lays x out by lane columns while they are
//   in flight).  Each slot s >= C (when k > C) is split over the
//   clusters by ranges of the intermediate dimension: cluster c computes h only for
//   its range of slot s, and the down product only over those columns, since
//   down(h) is the sum of the down products over any split of h's columns.  Each CTA
//   computes h for its rows and stores it into the h arrays of every CTA of the
//   cluster; cluster barrier.
// Phase 3: each CTA computes its H / 16 down rows for its slot (and its column range of
//   each split slot), scales them by the slot's weight and stores them in part[g],
//   g = c for the whole slot, C + (s - C) C + c for a split slot.  The C CTAs owning the
//   same rows (one per cluster) count themselves on a global counter; the one that
//   arrives last adds part[0 .. C(1 + k - C)) of those rows in that order (slot order,
//   and column-range order within a split slot) into y and zeroes the counter.
//   Nobody waits on anybody.
//
// Waits on bulk copies are bounded; a wait that gives up records MAPLE_ERR_TIMEOUT in
// the device status word, the CTA skips its arithmetic (its part rows are NaN) but
// still takes part in the cluster barriers and in the combine count, so the counters
// are zero again when the grid ends.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

constexpr int kCS = 16;                 // CTAs per cluster
constexpr int kLcWarps = 16;
constexpr int kLcThreads = kLcWarps * 32;
constexpr int kLcChunks = 4;            // gate/up copy chunks of the whole slot (one mbarrier each)
constexpr int kLcMaxE = 256;            // experts: one router row per warp per CTA
constexpr int kLcMaxK = 16;             // routed slots
constexpr int kLcMaxSplit = 2;          // slots beyond the clusters, split over them
constexpr int kLcMaxDownLaneBytes = 4;  // ceil(ceil(I/5)/32) <= 4, i.e. I <= 640
constexpr int kLcUnit = 40;             // split granule: 8 gate/up rows = 8 down-row bytes
constexpr int kLcMaxUnits = 4;          // units per cluster per split slot (32 down-row bytes)
constexpr int kLcSplitCopyRows = 24;    // gate/up rows a CTA copies per split slot
constexpr int kLcLutBytes = (int)sizeof(TritLut16);
constexpr int kLcRouterChunks = 9;      // 16-byte router-row chunks per lane: H <= 2304
static_assert(kLcThreads >= 2 * kLcMaxE && kLcThreads >= 4 * (kLcMaxE / 32) * kLcMaxK, "top-k thread plan");

__host__ __device__ constexpr int align16(int v) { return (v + 15) / 16 * 16; }

struct LcArgs {
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
    int C;             // clusters (slots taken whole); slots C..k-1 are split over them
    float clamp;
    float* logits;
    int32_t* idx;
    float* w;
    float* y;
    float* y_mirror;   // null, or a second copy of y (e.g. mapped host memory)
    float* part;       // [C (1 + k - C)][H] per-slot (and per column range) contributions
    unsigned* counts;  // [kCS] combine counters: zero on entry, zero on exit
    int* status;
    uint32_t wait_polls;  // poll limit of every bounded wait
    int stall;            // test hook: 1 = CTA 0 arms one barrier for 16 bytes no copy delivers
};

// Columns [col0, col1) of the intermediate dimension that cluster c handles for a split
// slot: units of kLcUnit columns spread evenly over the C clusters.
__host__ __device__ inline void split_range(int I, int C, int c, int& col0, int& col1) {
    const int nu = (I + kLcUnit - 1) / kLcUnit;
    const int u0 = c * nu / C, u1 = (c + 1) * nu / C;
    col0 = u0 * kLcUnit;
    col1 = u1 * kLcUnit < I ? u1 * kLcUnit : I;
}

// The split-slot gate/up pairs CTA rank r computes, as offsets [p0, p1) within its
// cluster's column range of n columns, and the first row g0 (a multiple of 8) of the
// 8-row groups it copies to hold them.
__host__ __device__ inline void split_pairs(int n, int r, int& p0, int& p1, int& g0) {
    const int per = (n + kCS - 1) / kCS;
    p0 = r * per < n ? r * per : n;
    p1 = p0 + per < n ? p0 + per : n;
    g0 = p0 / 8 * 8;
}

// Shared-memory plan (byte offsets).  The expert rows go to the last region.
struct LcSmem {
    int xb, xcol, hcol, hsp, lg, sh, un;
    int chunk_rows, chunk_bytes, dn, dn_bytes, sp, sp_gu_bytes, sp_bytes, total;
};

__host__ __device__ inline LcSmem lc_smem(int H, int I, int E, int MB) {
    const int Bh = (H + 4) / 5, Bi = (I + 4) / 5;
    const int rg = I / kCS, rd = H / kCS;
    LcSmem L;
    int o = kLcLutBytes;
    L.xb = o;
    o += align16(2 * H);
    L.xcol = o;
    o += 4 * 32 * MB * 5;
    L.hcol = o;
    o += 4 * 32 * kLcMaxDownLaneBytes * 5;
    L.hsp = o;
    o += 4 * kLcMaxSplit * align16(I);
    L.lg = o;
    o += 4 * kLcMaxE;
    L.sh = o;
    o += 4 * (rg + kLcMaxSplit * kCS);
    L.un = o = align16(o);
    L.chunk_rows = rg / kLcChunks;
    L.chunk_bytes = 2 * L.chunk_rows * Bh + 8 * L.chunk_rows;  // gate rows, up rows, their scales
    L.dn = kLcChunks * L.chunk_bytes;
    L.dn_bytes = rd * Bi + 4 * rd;                              // down rows, their scales
    L.sp = L.dn + L.dn_bytes;
    L.sp_gu_bytes = 2 * kLcSplitCopyRows * Bh + 8 * kLcSplitCopyRows;
    L.sp_bytes = L.sp_gu_bytes + L.dn_bytes;  // per split slot: gate/up groups, then down rows
    o += L.sp + kLcMaxSplit * L.sp_bytes;
    L.total = o;
    return L;
}

__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Every thread of every CTA of the cluster arrives (release) and waits (acquire):
// shared-memory stores into other CTAs before it are visible to them after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bounded wait with a run-time poll limit (see mbar_wait_bounded).
__device__ __forceinline__ bool lc_wait(uint64_t* bar, uint32_t parity, int* status, uint32_t polls) {
    for (uint32_t i = 0; i < polls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    if (status != nullptr) atomicExch(status, kStatusTimeout);
    return false;
}

// Selection key of logit v of expert e: larger keys come first (larger logit, then
// lower id); +0 and -0 get the same key.  v must not be NaN.
__device__ __forceinline__ uint64_t sel_key(float v, int e) {
    return ((uint64_t)float_order_key(v + 0.0f) << 32) | (uint64_t)(0xffffffffu - (uint32_t)e);
}

// Ranks each of the ncand candidate keys among all of them, kTpc threads per candidate
// (kLcThreads / kTpc candidates at most), and stores the k best in s_sel in order.
template <int kTpc>
__device__ __forceinline__ void rank_candidates(const uint64_t* s_cand, uint64_t* s_sel, int ncand, int k, int tid) {
    constexpr int kNj = kLcThreads / kTpc / kTpc;  // candidates a thread compares with
    const int cand = tid / kTpc, sub = tid % kTpc;
    const uint64_t K = cand < ncand ? s_cand[cand] : 0;
    int rank = 0;
#pragma unroll
    for (int j = 0; j < kNj; ++j) {
        const int jj = sub + kTpc * j;
        if (jj < ncand) rank += s_cand[jj] > K ? 1 : 0;
    }
#pragma unroll
    for (int o = kTpc / 2; o > 0; o >>= 1) rank += __shfl_xor_sync(kFullMask, rank, o);
    if (cand < ncand && sub == 0 && rank < k) s_sel[rank] = K;
}

template <int MB>
__global__ void __launch_bounds__(kLcThreads, 1) moe_layer_b1_kernel(LcArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar_in;                // decode table + router rows
    __shared__ __align__(8) uint64_t bar_gu[kLcChunks];     // gate/up chunk q of the whole slot
    __shared__ __align__(8) uint64_t bar_dn;                // its down rows + scales
    __shared__ __align__(8) uint64_t bar_sg[kLcMaxSplit];   // split slot: gate/up groups
    __shared__ __align__(8) uint64_t bar_sd[kLcMaxSplit];   // split slot: down rows + scales
    __shared__ __align__(16) uint64_t s_key[kLcMaxE];       // selection keys of the logits
    __shared__ __align__(16) uint64_t s_cand[kLcMaxE / 32 * kLcMaxK];
    __shared__ uint64_t s_sel[kLcMaxK];
    __shared__ float s_w[kLcMaxK];
    __shared__ int s_fail, s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x / kCS, r = blockIdx.x % kCS;  // cluster and rank
    const int H = a.H, I = a.I, E = a.E, k = a.k, C = a.C, nsplit = a.k - a.C;
    const int Bh = (H + 4) / 5, Bi = (I + 4) / 5;
    const int nr = (E + kCS - 1) / kCS, rg = I / kCS, rd = H / kCS;
    const LcSmem L = lc_smem(H, I, E, MB);
    TritLut16& lut = *reinterpret_cast<TritLut16*>(smem);
    uint16_t* xb = reinterpret_cast<uint16_t*>(smem + L.xb);
    float* xcol = reinterpret_cast<float*>(smem + L.xcol);
    float* hcol = reinterpret_cast<float*>(smem + L.hcol);
    float* hsp = reinterpret_cast<float*>(smem + L.hsp);  // [kLcMaxSplit][align16(I)]
    float* lg = reinterpret_cast<float*>(smem + L.lg);
    float* sh = reinterpret_cast<float*>(smem + L.sh);    // this CTA's h values
    unsigned char* un = smem + L.un;
    const int e_lo = r * nr;
    const int nr_mine = E - e_lo < nr ? (E - e_lo > 0 ? E - e_lo : 0) : nr;
    const int hsp_stride = align16(I);
    int col0 = 0, col1 = 0, sp0 = 0, sp1 = 0, sg0 = 0;  // split range and this CTA's pairs
    split_range(I, C, c, col0, col1);
    split_pairs(col1 - col0, r, sp0, sp1, sg0);

    // ---- phase 0: static inputs, before the dependency wait
    if (tid == 0) {
        s_fail = 0;
        mbar_init_nofence(&bar_in, 1);
        for (int q = 0; q < kLcChunks; ++q) mbar_init_nofence(&bar_gu[q], 1);
        mbar_init_nofence(&bar_dn, 1);
        for (int s = 0; s < kLcMaxSplit; ++s) {
            mbar_init_nofence(&bar_sg[s], 1);
            mbar_init_nofence(&bar_sd[s], 1);
        }
        mbar_init_fence();
        mbar_arrive_expect_tx(&bar_in, (uint32_t)kLcLutBytes);
        bulk_copy_g2s(&lut, &g_lut16_image, kLcLutBytes, &bar_in);
    }
    // warp w's router row in registers, 16-byte chunk lane + 32 u in wv[u] (weights: no
    // dependence on the previous kernel)
    const int n8 = H >> 3;
    uint4 wv[kLcRouterChunks];
#pragma unroll
    for (int u = 0; u < kLcRouterChunks; ++u) {
        const int cc = lane + 32 * u;
        wv[u] = warp < nr_mine && cc < n8 ? __ldg(reinterpret_cast<const uint4*>(a.Wr + (int64_t)(e_lo + warp) * H) + cc)
                                         : make_uint4(0u, 0u, 0u, 0u);
    }
    pdl_wait();
    pdl_launch_dependents();
    // the token (written by the previous kernel), 8 bytes per thread through L2
    for (int i = tid; i < H / 4; i += kLcThreads)
        reinterpret_cast<uint2*>(xb)[i] = __ldcg(reinterpret_cast<const uint2*>(a.x) + i);
    __syncthreads();  // barriers initialised before anyone waits on them; x in place
    if (!lc_wait(&bar_in, 0, a.status, a.wait_polls)) s_fail = 1;
    __syncthreads();

    // ---- phase 1: this CTA's logits, into every CTA of the cluster
    if (!s_fail) {
        const uint32_t lg_s = smem_addr(lg);
        if (warp < nr_mine) {  // warp w: router row w (the per-row order of route_logits_kernel)
            const int e = e_lo + warp;
            const uint4* x4 = reinterpret_cast<const uint4*>(xb);
            float acc = 0.f;
            {
#pragma unroll
                for (int u = 0; u < kLcRouterChunks; ++u) {
                    const int cc = lane + 32 * u;
                    if (cc < n8) {
                        const uint4 xv = x4[cc];
                        acc = fmaf(bf16_lo(wv[u].x), bf16_lo(xv.x), acc);
                        acc = fmaf(bf16_hi(wv[u].x), bf16_hi(xv.x), acc);
                        acc = fmaf(bf16_lo(wv[u].y), bf16_lo(xv.y), acc);
                        acc = fmaf(bf16_hi(wv[u].y), bf16_hi(xv.y), acc);
                        acc = fmaf(bf16_lo(wv[u].z), bf16_lo(xv.z), acc);
                        acc = fmaf(bf16_hi(wv[u].z), bf16_hi(xv.z), acc);
                        acc = fmaf(bf16_lo(wv[u].w), bf16_lo(xv.w), acc);
                        acc = fmaf(bf16_hi(wv[u].w), bf16_hi(xv.w), acc);
                    }
                }
            }
            const float v = warp_sum(acc) + (a.bias != nullptr ? a.bias[e] : 0.f);
            if (c == 0 && lane == 0) a.logits[e] = v;
            // lane q stores the logit into CTA q's array (NaN ranks last)
            if (lane < kCS) st_cluster_f32(mapa_shared(lg_s + 4u * e, (uint32_t)lane), (v != v) ? -INFINITY : v);
        }
        // entries past E rank last (in this CTA's own array only)
        for (int e = E + tid; e < kLcMaxE; e += kLcThreads) lg[e] = -INFINITY;
    }
    cluster_sync();

    // ---- phase 2: selection (the same in every CTA), this CTA's expert rows, h
    bool issued = false;
    if (!s_fail) {
        // top-k by rank counting on selection keys: each group of 32 logits keeps its k
        // best as candidates (every global top-k entry is in its group's top k), then
        // each candidate is ranked among the candidates.
        if (tid < kLcMaxE) s_key[tid] = sel_key(lg[tid], tid);
        __syncthreads();
        {  // two threads per logit, each against half of its group of 32
            const int i = tid >> 1, half = tid & 1;
            const uint64_t K = s_key[i];
            const uint64_t* grp = s_key + (i & ~31) + 16 * half;
            int rank = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) rank += grp[j] > K ? 1 : 0;
            rank += __shfl_xor_sync(kFullMask, rank, 1);
            if (half == 0 && rank < k) s_cand[(i >> 5) * k + rank] = K;
        }
        __syncthreads();
        if ((kLcMaxE / 32) * k <= 64)
            rank_candidates<8>(s_cand, s_sel, (kLcMaxE / 32) * k, k, tid);
        else
            rank_candidates<4>(s_cand, s_sel, (kLcMaxE / 32) * k, k, tid);
        __syncthreads();
        // the copies need only the selected ids (from the keys); the softmax weights are
        // first read after the h exchange, so the last warp forms them off the critical
        // path while the copies are issued
        auto sel_id = [&](int i) { return (int)(0xffffffffu - (uint32_t)s_sel[i]); };
        if (warp == kLcWarps - 1) {  // softmax over the k selected: exp(l_i - l_0) / sum_j exp(l_j - l_0)
            const int my_idx = lane < k ? (int)(0xffffffffu - (uint32_t)s_sel[lane]) : 0;
            const float my_val = lane < k ? lg[my_idx] : -INFINITY;
            const float top = lg[(int)(0xffffffffu - (uint32_t)s_sel[0])];
            const float ex = lane < k ? expf(my_val - top) : 0.f;
            const float denom = warp_sum(ex);
            if (lane < k) {
                s_w[lane] = ex / denom;
                if (blockIdx.x == 0) {
                    a.idx[lane] = my_idx;
                    a.w[lane] = ex / denom;
                }
            }
        }
        // bulk copies, one issuing thread per group of barriers (lane 0 of warps 0..2+2S)
        if (lane == 0 && warp < 3 + 2 * nsplit) {
            if (warp < 2) {  // whole slot: gate/up chunks 2w, 2w + 1
                const int e = sel_id(c), cr = L.chunk_rows;
                const uint32_t rows = (uint32_t)(cr * Bh);
                for (int q = 2 * warp; q < 2 * warp + 2; ++q) {
                    unsigned char* ch = un + q * L.chunk_bytes;
                    const int64_t r0 = (int64_t)e * I + r * rg + q * cr;
                    const uint32_t extra = (a.stall && blockIdx.x == 0 && q == 0) ? 16u : 0u;
                    mbar_arrive_expect_tx(&bar_gu[q], 2u * rows + 8u * cr + extra);
                    bulk_copy_g2s(ch, a.gate + r0 * Bh, rows, &bar_gu[q]);
                    bulk_copy_g2s(ch + rows, a.up + r0 * Bh, rows, &bar_gu[q]);
                    bulk_copy_g2s(ch + 2 * rows, a.s_gate + r0, 4u * cr, &bar_gu[q]);
                    bulk_copy_g2s(ch + 2 * rows + 4 * cr, a.s_up + r0, 4u * cr, &bar_gu[q]);
                }
            } else if (warp == 2) {  // whole slot: down rows + scales
                const int64_t d0 = (int64_t)sel_id(c) * H + r * rd;
                mbar_arrive_expect_tx(&bar_dn, (uint32_t)L.dn_bytes);
                bulk_copy_g2s(un + L.dn, a.down + d0 * Bi, (uint32_t)(rd * Bi), &bar_dn);
                bulk_copy_g2s(un + L.dn + rd * Bi, a.s_down + d0, 4u * rd, &bar_dn);
            } else {
                const int s = (warp - 3) >> 1, e = sel_id(C + s);
                unsigned char* sp = un + L.sp + s * L.sp_bytes;
                if (((warp - 3) & 1) == 0) {  // split slot s: the 8-row groups holding this CTA's pairs
                    const int64_t r0 = (int64_t)e * I + col0 + sg0;
                    const int room = I - col0 - sg0;
                    const int nrows = sp1 > sp0 ? (room < kLcSplitCopyRows ? room : kLcSplitCopyRows) : 0;
                    const uint32_t rows = (uint32_t)(nrows * Bh);
                    mbar_arrive_expect_tx(&bar_sg[s], 2u * rows + 8u * nrows);
                    if (nrows > 0) {
                        bulk_copy_g2s(sp, a.gate + r0 * Bh, rows, &bar_sg[s]);
                        bulk_copy_g2s(sp + kLcSplitCopyRows * Bh, a.up + r0 * Bh, rows, &bar_sg[s]);
                        bulk_copy_g2s(sp + 2 * kLcSplitCopyRows * Bh, a.s_gate + r0, 4u * nrows, &bar_sg[s]);
                        bulk_copy_g2s(sp + 2 * kLcSplitCopyRows * Bh + 4 * kLcSplitCopyRows, a.s_up + r0,
                                      4u * nrows, &bar_sg[s]);
                    }
                } else {  // split slot s: down rows + scales (whole rows; only the range is used)
                    const int64_t d0 = (int64_t)e * H + r * rd;
                    mbar_arrive_expect_tx(&bar_sd[s], (uint32_t)L.dn_bytes);
                    bulk_copy_g2s(sp + L.sp_gu_bytes, a.down + d0 * Bi, (uint32_t)(rd * Bi), &bar_sd[s]);
                    bulk_copy_g2s(sp + L.sp_gu_bytes + rd * Bi, a.s_down + d0, 4u * rd, &bar_sd[s]);
                }
            }
        }
        issued = true;
        // x in lane-column order for the dot products (xcol[(5 m + d) 32 + l] = x[5 (l +
        // 32 m) + d]), formed while the expert rows are in flight
        for (int i = tid; i < 32 * MB * 5; i += kLcThreads) {
            const int l = i & 31, md = i >> 5, m = md / 5, d = md - 5 * m;
            const int col = 5 * (l + 32 * m) + d;
            xcol[i] = col < H ? bf16_bits_to_float(xb[col]) : 0.f;
        }
        __syncthreads();
        // lane columns of x
        float2 x01[MB], x23[MB];
        float x4[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const float* xm = xcol + (m * 5) * 32 + lane;
            x01[m] = make_float2(xm[0], xm[32]);
            x23[m] = make_float2(xm[64], xm[96]);
            x4[m] = xm[128];
        }
        // whole slot: warp w takes row pairs [w per, (w + 1) per), all in chunk w / 4;
        // lane partials of gate and up rows, then one transposed reduction: lane l ends
        // with row l >> 2 (pair l >> 3, up if bit 2)
        {
            const int q = warp / (kLcWarps / kLcChunks), per = rg / kLcWarps, cr = L.chunk_rows;
            if (!lc_wait(&bar_gu[q], 0, a.status, a.wait_polls)) {
                s_fail = 1;
            } else {
                const unsigned char* ch = un + q * L.chunk_bytes;
                const float* sg = reinterpret_cast<const float*>(ch + 2 * cr * Bh);
                const float* su = sg + cr;
                float part[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) part[i] = 0.f;
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if (p < per) {
                        const int jj = warp * per + p - q * cr;  // row within the chunk
                        part[2 * p] = lane_row_dot<MB>(ch + jj * Bh, Bh, lut, x01, x23, x4, lane);
                        part[2 * p + 1] = lane_row_dot<MB>(ch + (cr + jj) * Bh, Bh, lut, x01, x23, x4, lane);
                    }
                }
                const float mine = warp_transpose_sum<8>(part, lane);
                const float au = __shfl_down_sync(kFullMask, mine, 4);
                const int p = lane >> 3;
                if ((lane & 7) == 0 && p < per) {
                    const int j = warp * per + p, jj = j - q * cr;
                    const float gv = (2.f * mine) * sg[jj];
                    const float uv = (2.f * au) * su[jj];
                    const float gc = fminf(gv, a.clamp);
                    const float uc = fminf(fmaxf(uv, -a.clamp), a.clamp);
                    sh[j] = silu_f(gc) * uc;
                }
            }
        }
        // split slots: warp w takes this CTA's pair sp0 + w of the cluster's column range
        for (int s = 0; s < nsplit; ++s) {
            if (warp < sp1 - sp0) {
                if (!lc_wait(&bar_sg[s], 0, a.status, a.wait_polls)) {
                    s_fail = 1;
                } else {
                    const unsigned char* sp = un + L.sp + s * L.sp_bytes;
                    const int jj = sp0 + warp - sg0;  // row within the copied groups
                    float part[2];
                    part[0] = lane_row_dot<MB>(sp + jj * Bh, Bh, lut, x01, x23, x4, lane);
                    part[1] = lane_row_dot<MB>(sp + (kLcSplitCopyRows + jj) * Bh, Bh, lut, x01, x23, x4, lane);
                    const float mine = warp_transpose_sum<2>(part, lane);  // lane l: row l >> 4
                    const float au = __shfl_down_sync(kFullMask, mine, 16);
                    if (lane == 0) {
                        const float* sg = reinterpret_cast<const float*>(sp + 2 * kLcSplitCopyRows * Bh);
                        const float gv = (2.f * mine) * sg[jj];
                        const float uv = (2.f * au) * sg[kLcSplitCopyRows + jj];
                        const float gc = fminf(gv, a.clamp);
                        const float uc = fminf(fmaxf(uv, -a.clamp), a.clamp);
                        sh[rg + s * kCS + warp] = silu_f(gc) * uc;
                    }
                }
            }
        }
    }
    __syncthreads();
    // this CTA's h values into every CTA of the cluster: the whole slot's in lane-column
    // order, the split slots' by column
    if (!s_fail) {
        const uint32_t hcol_s = smem_addr(hcol), hsp_s = smem_addr(hsp);
        const int nsp = sp1 - sp0, per_dst = rg + nsplit * nsp;
        for (int i = tid; i < kCS * per_dst; i += kLcThreads) {
            const int dst = i / per_dst, j = i - dst * per_dst;
            uint32_t addr;
            float v;
            if (j < rg) {
                const int col = r * rg + j, b = col / 5, dd = col - 5 * b;
                addr = hcol_s + 4u * (uint32_t)(((b >> 5) * 5 + dd) * 32 + (b & 31));
                v = sh[j];
            } else {
                const int s = (j - rg) / nsp, jj = (j - rg) - s * nsp;
                addr = hsp_s + 4u * (uint32_t)(s * hsp_stride + col0 + sp0 + jj);
                v = sh[rg + s * kCS + jj];
            }
            st_cluster_f32(mapa_shared(addr, (uint32_t)dst), v);
        }
    }
    cluster_sync();

    // ---- phase 3: this CTA's down rows: the whole slot, then each split slot's range
    const int per = rd / kLcWarps;  // rows per warp (<= 8)
    if (!s_fail && !lc_wait(&bar_dn, 0, a.status, a.wait_polls)) s_fail = 1;
    for (int s = 0; s < nsplit; ++s)
        if (!s_fail && !lc_wait(&bar_sd[s], 0, a.status, a.wait_polls)) s_fail = 1;
    __syncthreads();
    {
        float mine = __int_as_float(0x7fc00000);  // NaN marks rows of a CTA that gave up
        if (!s_fail) {
            float2 h01[kLcMaxDownLaneBytes], h23[kLcMaxDownLaneBytes];
            float h4[kLcMaxDownLaneBytes];
#pragma unroll
            for (int m = 0; m < kLcMaxDownLaneBytes; ++m) {
                const int b = lane + 32 * m;
                float v[5];
#pragma unroll
                for (int d = 0; d < 5; ++d) {
                    const int col = 5 * b + d;
                    v[d] = (b < Bi && col < I) ? hcol[(m * 5 + d) * 32 + lane] : 0.f;
                }
                h01[m] = make_float2(v[0], v[1]);
                h23[m] = make_float2(v[2], v[3]);
                h4[m] = v[4];
            }
            const unsigned char* dn = un + L.dn;
            float part[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
                part[t] = t < per ? lane_row_dot<kLcMaxDownLaneBytes, true>(dn + (warp * per + t) * Bi, Bi, lut,
                                                                          h01, h23, h4, lane)
                                  : 0.f;
            mine = warp_transpose_sum<8>(part, lane);  // lane l: row l >> 2
            const int t = lane >> 2;
            if (t < per) {
                const float* sd = reinterpret_cast<const float*>(dn + rd * Bi);
                mine = s_w[c] * (sd[warp * per + t] * (2.f * mine));
            }
        }
        if ((lane & 3) == 0 && (lane >> 2) < per)
            a.part[(int64_t)c * H + r * rd + warp * per + (lane >> 2)] = mine;
    }
    for (int s = 0; s < nsplit; ++s) {
        // lane owns byte b0 + lane of the cluster's range of each row (<= 32 bytes)
        float mine = __int_as_float(0x7fc00000);
        if (!s_fail) {
            const unsigned char* sp = un + L.sp + s * L.sp_bytes + L.sp_gu_bytes;
            const int b0 = col0 / 5, b1 = (col1 + 4) / 5, b = b0 + lane;
            float hv[5];
#pragma unroll
            for (int d = 0; d < 5; ++d) {
                const int col = 5 * b + d;
                hv[d] = (b < b1 && col >= col0 && col < col1) ? hsp[s * hsp_stride + col] : 0.f;
            }
            const int sub = lane & 15;
            float part[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                float acc = 0.f;
                if (t < per && b < b1) {
                    const uint2 ent = lut.entry[(uint32_t)sp[(warp * per + t) * Bi + b] * 16 + sub];
                    acc = fmaf(trit_half<0>(ent), hv[0], acc);
                    acc = fmaf(trit_half<1>(ent), hv[1], acc);
                    acc = fmaf(trit_half<2>(ent), hv[2], acc);
                    acc = fmaf(trit_half<3>(ent), hv[3], acc);
                    acc = fmaf(trit_half<4>(ent), hv[4], acc);
                }
                part[t] = acc;
            }
            mine = warp_transpose_sum<8>(part, lane);  // lane l: row l >> 2
            const int t = lane >> 2;
            if (t < per) {
                const float* sd = reinterpret_cast<const float*>(sp + rd * Bi);
                mine = s_w[C + s] * (sd[warp * per + t] * (2.f * mine));
            }
        }
        if ((lane & 3) == 0 && (lane >> 2) < per)
            a.part[(int64_t)(C + s * C + c) * H + r * rd + warp * per + (lane >> 2)] = mine;
    }
    // combine: the last of the C CTAs owning these rows adds every part in order
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned before = atomicAdd(a.counts + r, 1u);
        s_last = before == (unsigned)C - 1;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        const int G = C * (1 + nsplit);  // at most kLcMaxK (1 + kLcMaxSplit)
        for (int t = tid; t < rd; t += kLcThreads) {
            float v[kLcMaxK * (1 + kLcMaxSplit)];
#pragma unroll
            for (int g = 0; g < kLcMaxK * (1 + kLcMaxSplit); ++g)
                v[g] = g < G ? __ldcg(a.part + (int64_t)g * H + r * rd + t) : 0.f;
            float yv = 0.f;
#pragma unroll
            for (int g = 0; g < kLcMaxK * (1 + kLcMaxSplit); ++g)
                if (g < G) yv += v[g];
            a.y[r * rd + t] = yv;
            if (a.y_mirror != nullptr) a.y_mirror[r * rd + t] = yv;
        }
        if (tid == 0) atomicExch(a.counts + r, 0u);
    }

    // ---- exit: the copies this CTA issued have landed
    if (tid == 0) {
        lc_wait(&bar_in, 0, nullptr, a.wait_polls);
        if (issued) {
            for (int q = 0; q < kLcChunks; ++q) lc_wait(&bar_gu[q], 0, nullptr, a.wait_polls);
            lc_wait(&bar_dn, 0, nullptr, a.wait_polls);
            for (int s = 0; s < nsplit; ++s) {
                lc_wait(&bar_sg[s], 0, nullptr, a.wait_polls);
                lc_wait(&bar_sd[s], 0, nullptr, a.wait_polls);
            }
        }
    }
}

#define MAPLE_LC_SWITCH(MBV, CALL)             \
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

// Per-device one-time attributes of an instance: 16-CTA clusters (beyond the portable
// 8) and the dynamic shared memory.
template <int MB>
cudaError_t lc_prepare(size_t smem) {
    static_assert(kCS == 16, "16-CTA clusters need the non-portable size attribute");
    cudaError_t err = ensure_dynamic_smem(moe_layer_b1_kernel<MB>, smem);
    if (err != cudaSuccess) return err;
    static std::atomic<bool> done[128];
    int dev = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (done[dev].load()) return cudaSuccess;
    err = cudaFuncSetAttribute(moe_layer_b1_kernel<MB>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    done[dev].store(true);
    return cudaSuccess;
}

template <int MB>
cudaError_t launch_lc_mb(const LcArgs& a, size_t smem, cudaStream_t stream) {
    cudaError_t err = lc_prepare<MB>(smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.C * kCS);
    cfg.blockDim = dim3(kLcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, moe_layer_b1_kernel<MB>, a);
}

template <int MB>
cudaError_t lc_max_clusters(size_t smem, int* n) {
    cudaError_t err = lc_prepare<MB>(smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kLcMaxK * kCS);
    cfg.blockDim = dim3(kLcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, moe_layer_b1_kernel<MB>, &cfg);
}

// One-shot test hooks (see maple_test_inject): consumed by the next fused launch.
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_inject_polls{0};

}  // namespace

// How many 16-CTA clusters of the instance for (H, I, E) the current device runs at
// once (cached per device and instance; 0 if the query fails).
int layer_b1_clusters(int H, int I, int E) {
    const int MB = ((H + 4) / 5 + 31) / 32;
    static std::atomic<int> cached[128][14];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128 || MB < 1 || MB > 13) return 0;
    int n = cached[dev][MB].load();
    if (n > 0) return n;
    if (layer_b1_max_clusters(H, I, E, &n) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return 0;
    }
    cached[dev][MB].store(n);
    return n;
}

void layer_b1_inject_stall(int polls) {
    if (polls < 1) {  // cancel
        g_inject_stall.store(0);
        return;
    }
    g_inject_polls.store(polls);
    g_inject_stall.store(1);
}

// An upper bound of the per-slot output rows over every cluster count C <= k:
// C (1 + k - C) groups of H fp32 values.
size_t layer_b1_part_bytes(int k, int H) {
    int g = 0;
    for (int C = 1; C <= k; ++C) g = C * (1 + k - C) > g ? C * (1 + k - C) : g;
    return 4 * (size_t)g * (size_t)H;
}

bool layer_b1_supported(int H, int I, int E, int k, const DeviceInfo& dev) {
    const int Bh = (H + 4) / 5, Bi = (I + 4) / 5;
    // down: H / 16 rows per CTA, at most 8 per warp; a router row in a warp's registers
    if (H % 8 != 0 || H % (kCS * kLcWarps) != 0 || H / kCS / kLcWarps > 8) return false;
    if ((H / 8 + 31) / 32 > kLcRouterChunks) return false;
    const int rd = H / kCS;
    if ((rd * Bi) % 16 != 0 || ((int64_t)H * Bi) % 16 != 0 || (Bi + 31) / 32 > kLcMaxDownLaneBytes) return false;
    // gate/up: I / 16 row pairs per CTA in four chunks of 16-byte-aligned row groups, at
    // most four pairs per warp
    if (I % 8 != 0 || I % (kCS * kLcWarps) != 0 || I / kCS / kLcWarps > 4) return false;
    const int cr = I / kCS / kLcChunks;
    if ((cr * Bh) % 16 != 0 || ((int64_t)I * Bh) % 16 != 0 || (8 * Bh) % 16 != 0 || (Bh + 31) / 32 > 13) return false;
    if (k < 1 || k > kLcMaxK || k > E || E > kLcMaxE || (E + kCS - 1) / kCS > kLcWarps) return false;
    const int cmax = layer_b1_clusters(H, I, E);
    if (cmax < 1) return false;
    const int C = k < cmax ? k : cmax, nsplit = k - C;
    if (nsplit > kLcMaxSplit) return false;
    if (nsplit > 0) {
        // a cluster's range: at most kLcMaxUnits units (32 down-row bytes, one per lane);
        // a CTA's pairs fit the copied row groups and the warps
        const int nu = (I + kLcUnit - 1) / kLcUnit;
        if ((nu + C - 1) / C > kLcMaxUnits) return false;
        for (int cc = 0; cc < C; ++cc) {
            int c0, c1;
            split_range(I, C, cc, c0, c1);
            const int per = (c1 - c0 + kCS - 1) / kCS;
            if (per > kLcWarps || per + 7 > kLcSplitCopyRows) return false;
        }
    }
    const LcSmem L = lc_smem(H, I, E, (Bh + 31) / 32);
    return (size_t)L.total + 1024 <= dev.smem_optin;
}

cudaError_t launch_moe_layer_b1(const LayerLaunch& p, cudaStream_t stream, const DeviceInfo& dev) {
    LcArgs a;
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
    const int cmax = layer_b1_clusters(p.H, p.I, p.E);
    a.C = p.k < cmax ? p.k : cmax;
    a.clamp = p.clamp;
    a.logits = p.logits;
    a.idx = p.idx;
    a.w = p.w;
    a.y = p.y;
    a.y_mirror = p.y_mirror;
    a.part = p.part;
    a.counts = p.sync;
    a.status = dev.status;
    a.wait_polls = kWaitPolls;
    a.stall = 0;
    if (g_inject_stall.exchange(0) != 0) {
        a.stall = 1;
        const int polls = g_inject_polls.load();
        a.wait_polls = polls > 0 ? (uint32_t)polls : 1u;
    }
    const int MB = ((p.H + 4) / 5 + 31) / 32;
    const size_t smem = (size_t)lc_smem(p.H, p.I, p.E, MB).total;
#define MAPLE_CALL_LC(M) launch_lc_mb<M>(a, smem, stream)
    MAPLE_LC_SWITCH(MB, MAPLE_CALL_LC)
#undef MAPLE_CALL_LC
}

cudaError_t layer_b1_max_clusters(int H, int I, int E, int* n) {
    const int MB = ((H + 4) / 5 + 31) / 32;
    const size_t smem = (size_t)lc_smem(H, I, E, MB).total;
#define MAPLE_CALL_LCQ(M) lc_max_clusters<M>(smem, n)
    MAPLE_LC_SWITCH(MB, MAPLE_CALL_LCQ)
#undef MAPLE_CALL_LCQ
}

}  // namespace maple
