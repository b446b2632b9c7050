// Device helpers shared by the CUDA kernels of libmaple (internal header).
#pragma once

#include <mutex>
#include <cuda_runtime.h>
#include <math.h>
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
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ldg_nc_u8(const uint8_t* p) {
    uint16_t r;
    asm("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
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

// The same table replicated 16 times, indexed [code][lane % 16]: a warp's 64-bit
// lookups are served as two half-warp wavefronts, and within a half-warp every lane
// reads its own bank pair, so random codes never conflict.  243 x 16 x 8 B = 31 KB.
// The image is computed at compile time and lives in device global memory; kernels
// bulk-copy it into shared memory (it depends on no earlier kernel, so the copy may
// start before the programmatic-dependent-launch wait).
struct TritLut16 {
    uint2 entry[243 * 16];
};

struct Lut16Word {
    uint32_t lo, hi;
};
struct Lut16Image {
    Lut16Word entry[243 * 16];
};

constexpr Lut16Image make_lut16_image() {
    Lut16Image t{};
    for (int i = 0; i < 243 * 16; ++i) {
        int code = i / 16;
        uint32_t lo = 0, hi = 0;
        for (int d = 0; d < 5; ++d) {
            const int digit = code % 3;
            code /= 3;
            const uint32_t top = digit == 2 ? 0x3fu : (digit == 0 ? 0xbfu : 0x00u);
            if (d < 4)
                lo |= top << (8 * d);
            else
                hi = top;
        }
        t.entry[i] = Lut16Word{lo, hi};
    }
    return t;
}

static __device__ __align__(16) const Lut16Image g_lut16_image = make_lut16_image();
static_assert(sizeof(Lut16Image) == sizeof(TritLut16), "table image layout");
static_assert(sizeof(Lut16Image) % 16 == 0, "bulk-copy size");

// fp32 multiplier (+-0.5 or 0) of trit i (0..4) of a table entry.
template <int I>
__device__ __forceinline__ float trit_half(uint2 e) {
    if constexpr (I < 4)
        return __uint_as_float(__byte_perm(e.x, 0u, 0x0444u | (I << 12)));
    else
        return __uint_as_float(__byte_perm(e.y, 0u, 0x0444u));
}

// ---------------------------------------------------------------- TMA bulk copies
// 1-D bulk copies global -> shared memory completed on an mbarrier (transaction
// count), and bulk L2 prefetches.  Addresses must be 16-byte aligned and sizes a
// multiple of 16.

constexpr int kStatusTimeout = -5;  // MAPLE_ERR_TIMEOUT

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// mbarrier.init without the fences: initialise several barriers this way, then make
// them visible (to the async proxy and the cluster) with one mbar_init_fence().
__device__ __forceinline__ void mbar_init_nofence(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Sums v[0..R) of every lane over the warp's 32 lanes, R a power of two <= 16, with
// R - 1 + 5 - log2(R) shuffles instead of R full butterflies: at each of the first
// log2(R) levels a lane keeps half of its values (the half its lane bit selects) and
// adds its partner's copy of that half; the last levels are a plain butterfly.  Lane l
// ends with the total of value (l >> (5 - log2 R)); v[0] holds it.
template <int R>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[R], int lane) {
    static_assert(R == 1 || R == 2 || R == 4 || R == 8 || R == 16, "R");
#pragma unroll
    for (int half = R / 2, o = 16; half >= 1; half /= 2, o /= 2) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float keep = upper ? v[i + half] : v[i];
            const float send = upper ? v[i] : v[i + half];
            v[i] = keep + __shfl_xor_sync(kFullMask, send, o);
        }
    }
    constexpr int kDone = R == 1 ? 0 : (R == 2 ? 1 : (R == 4 ? 2 : (R == 8 ? 3 : 4)));
#pragma unroll
    for (int o = 16 >> kDone; o > 0; o >>= 1) v[0] += __shfl_xor_sync(kFullMask, v[0], o);
    return v[0];
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Add `bytes` to the transaction count the current phase waits for, without arriving:
// the phase completes only after the (single) arrival and every expected byte.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// try_wait with a suspend-time hint: a thread whose phase is not yet complete sleeps
// until the phase completes or the hint (ns) runs out, instead of spinning.
constexpr uint32_t kWaitSuspendNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kWaitSuspendNs)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after kWaitPolls suspended polls
// (at most kWaitPolls x kWaitSuspendNs = about 2 s).  On give-up the device status word
// records MAPLE_ERR_TIMEOUT and false is returned: the caller skips its work and
// returns.
constexpr uint32_t kWaitPolls = 2000;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status) {
    for (uint32_t i = 0; i < kWaitPolls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    if (status != nullptr) atomicExch(status, kStatusTimeout);
    return false;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Top-k of one token's E logits by one warp, then softmax over the k winners.
// Lane j < k receives the j-th largest logit's expert (ties: lower id) and its weight
// exp(l_j - l_0) / sum_i exp(l_i - l_0).  `logit(e)` returns the logit of expert e;
// NaN ranks last.  JE = logits held per lane (E <= 32 * JE); k <= 32.
template <int JE, typename LogitFn>
__device__ __forceinline__ void warp_topk_softmax(LogitFn logit, int E, int k, int lane, int& out_idx,
                                                  float& out_w) {
    float v[JE];
#pragma unroll
    for (int j = 0; j < JE; ++j) {
        const int e = lane + 32 * j;
        const float l = e < E ? logit(e) : -INFINITY;
        v[j] = (l != l) ? -INFINITY : l;
    }
    uint32_t taken = 0;
    float my_val = -INFINITY;
    int my_idx = 0;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < JE; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < be))) {
                bv = v[j];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(kFullMask, bv, o);
            const int oe = __shfl_xor_sync(kFullMask, be, o);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == r) {
            my_val = bv;
            my_idx = be;
        }
    }
    const float top = __shfl_sync(kFullMask, my_val, 0);
    const float ex = lane < k ? expf(my_val - top) : 0.f;
    const float denom = warp_sum(ex);
    out_idx = my_idx;
    out_w = ex / denom;
}

// Order-preserving 32-bit key of a float (NaN must already be replaced by -inf and
// -0 by +0, so that equal values get equal keys).
__device__ __forceinline__ uint32_t float_order_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_from_order_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of E (<= 1024) logits held in shared memory, by one warp, then softmax over
// the k winners.  Each round every lane scans its entries (lane, lane + 32, ...) for
// its best untaken one; a warp max of the keys and a warp min of the ids among the
// lanes holding that key pick the winner (larger value first, ties to the lower id).
// Lane j < k ends with winner j, its logit and exp(l_j - l_0) / sum_i exp(l_i - l_0)
// (the same softmax as warp_topk_softmax).  Entries must be NaN-free (see above).
__device__ __forceinline__ void warp_topk_softmax_smem(const float* lg, int E, int k, int lane,
                                                       int& out_idx, float& out_val, float& out_w) {
    // keys of entries lane + 32 j, j < 8, in registers; entries beyond 256 (if any) are
    // re-read from shared memory each round
    constexpr int kRegJ = 8;
    uint32_t keys[kRegJ];
#pragma unroll
    for (int j = 0; j < kRegJ; ++j) {
        const int e = lane + 32 * j;
        keys[j] = e < E ? float_order_key(lg[e] + 0.0f) : 0u;
    }
    uint32_t taken = 0;  // bit j: entry lane + 32 j already selected
    int my_idx = 0;
    float my_val = -INFINITY;
    const int nj = (E + 31) >> 5;
    for (int r = 0; r < k; ++r) {
        uint32_t best_key = 0;
        int best_e = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kRegJ; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u) && (best_e == 0x7fffffff || keys[j] > best_key)) {
                best_key = keys[j];
                best_e = e;
            }
        }
        for (int j = kRegJ; j < nj; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u)) {
                const uint32_t key = float_order_key(lg[e] + 0.0f);
                if (best_e == 0x7fffffff || key > best_key) {
                    best_key = key;
                    best_e = e;
                }
            }
        }
        const uint32_t top_key = __reduce_max_sync(kFullMask, best_key);
        const uint32_t cand = (best_e != 0x7fffffff && best_key == top_key) ? (uint32_t)best_e : 0xffffffffu;
        const int win = (int)__reduce_min_sync(kFullMask, cand);
        if ((win & 31) == lane) taken |= 1u << (win >> 5);
        if (lane == r) {
            my_idx = win;
            my_val = float_from_order_key(top_key);
        }
    }
    const float top = __shfl_sync(kFullMask, my_val, 0);
    const float ex = lane < k ? expf(my_val - top) : 0.f;
    const float denom = warp_sum(ex);
    out_idx = my_idx;
    out_val = my_val;
    out_w = ex / denom;
}

// Dot product of one packed row held in shared memory with the activations of the
// columns this lane owns: byte b = lane + 32 m covers columns 5b..5b+4, whose values
// sit in x01[m] = (x0, x1), x23[m] = (x2, x3) and x4[m].  Each byte costs one table
// lookup, five byte permutes (the +-1/2 multipliers) and two packed + one scalar FMA;
// the result is half the row's sum of +-x (the factor 2 goes with the row scale).
// CHECK_ALL: test b < nbytes at every m (MB may then exceed ceil(nbytes / 32));
// otherwise MB must equal ceil(nbytes / 32) and only the last m is tested.
template <int MB, bool CHECK_ALL = false>
__device__ __forceinline__ float lane_row_dot(const uint8_t* row, int nbytes, const TritLut16& lut,
                                              const float2* x01, const float2* x23, const float* x4,
                                              int lane) {
    // Stage the loads: all of the lane's codes, then all table entries, then the FMAs,
    // so a row costs two shared-memory latencies rather than two per byte.
    const int sub = lane & 15;
    uint32_t code[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        const int b = lane + 32 * m;
        code[m] = ((!CHECK_ALL && m + 1 < MB) || b < nbytes) ? row[b] : 121u;  // 121: five zeros
    }
    uint2 ent[MB];
#pragma unroll
    for (int m = 0; m < MB; ++m) ent[m] = lut.entry[code[m] * 16 + sub];
    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
    float a4 = 0.f;
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        a01 = __ffma2_rn(make_float2(trit_half<0>(ent[m]), trit_half<1>(ent[m])), x01[m], a01);
        a23 = __ffma2_rn(make_float2(trit_half<2>(ent[m]), trit_half<3>(ent[m])), x23[m], a23);
        a4 = fmaf(trit_half<4>(ent[m]), x4[m], a4);
    }
    return ((a01.x + a01.y) + (a23.x + a23.y)) + a4;
}

// Activations of the columns a lane owns (see lane_row_dot); `load(col)` reads column
// col < ncols, the others are 0.
template <int MB, typename Load>
__device__ __forceinline__ void load_lane_cols(float2* x01, float2* x23, float* x4, int lane,
                                               int nbytes, int ncols, Load load) {
#pragma unroll
    for (int m = 0; m < MB; ++m) {
        const int b = lane + 32 * m;
        float v[5];
#pragma unroll
        for (int d = 0; d < 5; ++d) {
            const int col = 5 * b + d;
            v[d] = (b < nbytes && col < ncols) ? load(col) : 0.f;
        }
        x01[m] = make_float2(v[0], v[1]);
        x23[m] = make_float2(v[2], v[3]);
        x4[m] = v[4];
    }
}

// Partial sums of one 16-row down group for k slots, from shared memory.  Warp w takes
// slots w/2, w/2 + nwarps/2, ... and rows (w & 1) * 8 .. + 8 of the group; lanes own
// columns (lane_row_dot), with the slot's h in plain layout h[5b + d] (conflict-free
// reads: 5 is odd).  s_part[i][row] = lane-summed partial (without the factor 2), or 0
// for a slot with live(i) false.
//   rows(i): slot i's 16 x Bi packed bytes;  hplain(i): slot i's h, I floats.
template <int MBD, bool CHECK_ALL, typename RowsFn, typename HFn, typename LiveFn>
__device__ __forceinline__ void down_group_partials(int k, int I, int Bi, const TritLut16& lut, RowsFn rows,
                                                    HFn hplain, LiveFn live, float (*s_part)[16],
                                                    int nwarps) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row0 = (warp & 1) * 8;
    for (int i = warp >> 1; i < k; i += nwarps >> 1) {
        float mine = 0.f;
        if (live(i)) {
            const float* hs = hplain(i);
            float2 x01[MBD], x23[MBD];
            float x4[MBD];
            load_lane_cols<MBD>(x01, x23, x4, lane, Bi, I, [&](int col) { return hs[col]; });
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float p = warp_sum(
                    lane_row_dot<MBD, CHECK_ALL>(rows(i) + (row0 + r) * Bi, Bi, lut, x01, x23, x4, lane));
                if (lane == r) mine = p;
            }
        }
        if (lane < 8) s_part[i][row0 + lane] = mine;
    }
}

// Raises a kernel's dynamic shared-memory limit to `bytes`.  The attribute is per
// device; the last size set per (kernel, device) is remembered, keyed by the kernel's
// address (template instances share a function type), so that steady-state launches
// make no extra driver call.
template <typename Kernel>
cudaError_t ensure_dynamic_smem(Kernel* kernel, size_t bytes) {
    // static and dynamic shared memory together may exceed the 48 KB default even when
    // the dynamic part alone does not: opt in for any dynamic size
    if (bytes == 0) return cudaSuccess;
    struct Entry {
        const void* fn;
        int dev;
        size_t bytes;
    };
    constexpr int kEntries = 128;
    static Entry cache[kEntries] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const void* fn = reinterpret_cast<const void*>(kernel);
    int slot = -1;
    for (int i = 0; i < kEntries; ++i) {
        if (cache[i].fn == fn && cache[i].dev == dev) {
            if (cache[i].bytes >= bytes) return cudaSuccess;
            slot = i;
            break;
        }
        if (cache[i].fn == nullptr) {
            slot = i;
            break;
        }
    }
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err == cudaSuccess && slot >= 0) cache[slot] = Entry{fn, dev, bytes};
    return err;
}

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
