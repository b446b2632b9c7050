// Host-resident experts streamed into an HBM cache on demand.
//
// "Maple Preview 接入 Mference：M4 MacBook 上 500MB 内存跑 20B MoE" (opening paragraph,
// and section "接入 Mference 后的实测结果"): the Mference port keeps the MoE experts
// outside the accelerator's memory and reads a token's experts when its routing asks
// for them.  Here the experts of a layer live in pinned host memory (a "pool", any
// layout maple_experts describes, as device-accessible host pointers) and a cache of C
// expert slots lives in HBM.  Per step, entirely on the device (no host round trip, so
// a step can be captured in a CUDA graph):
//
//   cache_plan_kernel (one CTA): marks the experts the step's idx routes to; a routed
//     expert already in a slot is a hit; every miss takes the least recently used slot
//     no routed expert holds (ties to the lower slot; empty slots first), in increasing
//     expert order, so the plan is deterministic.  Writes idx_slot (each slot of idx
//     renamed to its cache slot, -1 for ids outside [0, E)) and the list of copies.
//   cache_copy_kernel: each listed expert's six arrays (gate and up rows, down rows,
//     their scales) are read from the pool with 16-byte loads across the host link and
//     written into its slot; kCopyParts CTAs per expert.
//
// The FFN then runs unchanged on the cache, as a layer of C experts, with idx_slot.
#include "common.cuh"
#include "kernels.h"
#include "maple.h"

namespace maple {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCopyParts = 16;   // CTAs per fetched expert
constexpr int kCopyThreads = 256;

struct CacheArgs {
    maple_experts pool;   // E experts, host memory the device can read
    maple_experts slots;  // C experts in HBM (slots.E = C)
    int32_t* slot_of;     // [E]: slot holding expert e, or -1
    int32_t* expert_of;   // [C]: expert in slot s, or -1
    uint32_t* last_use;   // [C]: step stamp of the slot's last use (0: never)
    uint32_t* stats;      // [4]: steps, hits, misses, experts copied
    const int32_t* idx;   // [S] routed expert ids
    int S;
    int32_t* idx_slot;    // [S] written
    int32_t* jobs;        // workspace: [0] number of copies, then (slot, expert) pairs
    int* status;
};

__global__ void __launch_bounds__(kPlanThreads) cache_plan_kernel(CacheArgs a) {
    __shared__ unsigned char need[1024];    // routed this step
    __shared__ unsigned char in_use[1024];  // slot holds an expert routed this step
    __shared__ int miss_rank[1024];         // rank of expert e among this step's misses
    __shared__ int s_nmiss, s_nfree;
    __shared__ uint32_t s_stamp;
    __shared__ int victim_of_rank[1024];
    const int tid = threadIdx.x;
    const int E = a.pool.E, C = a.slots.E;
    pdl_wait();
    pdl_launch_dependents();
    for (int e = tid; e < 1024; e += kPlanThreads) need[e] = 0;
    for (int s = tid; s < 1024; s += kPlanThreads) in_use[s] = 0;
    if (tid == 0) {
        s_stamp = a.stats[0] + 1u;
        a.stats[0] = s_stamp;
    }
    __syncthreads();
    for (int s = tid; s < a.S; s += kPlanThreads) {
        const int e = a.idx[s];
        if (e >= 0 && e < E) need[e] = 1;
    }
    __syncthreads();
    // hits mark their slot; misses are ranked in increasing expert order
    const bool miss = tid < E && need[tid] && a.slot_of[tid] < 0;
    if (tid < E && need[tid] && !miss) {
        const int s = a.slot_of[tid];
        in_use[s] = 1;
        a.last_use[s] = s_stamp;
    }
    {
        // block-wide exclusive scan of the miss flags
        __shared__ int warp_sums[kPlanThreads / 32];
        const int lane = tid & 31, warp = tid >> 5;
        const unsigned m = __ballot_sync(kFullMask, miss);
        const int before = __popc(m & ((1u << lane) - 1u));
        if (lane == 0) warp_sums[warp] = __popc(m);
        __syncthreads();
        if (warp == 0) {
            int v = warp_sums[lane], incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(kFullMask, incl, o);
                if (lane >= o) incl += n;
            }
            warp_sums[lane] = incl - v;
            if (lane == 31) s_nmiss = incl;
        }
        __syncthreads();
        if (tid < 1024) miss_rank[tid] = miss ? warp_sums[warp] + before : -1;
    }
    __syncthreads();
    // victims: the slots no routed expert holds, ranked by (last use, slot)
    if (tid == 0) s_nfree = 0;
    __syncthreads();
    if (tid < C && !in_use[tid]) {
        const uint32_t mine = a.last_use[tid];
        int rank = 0;
        for (int u = 0; u < C; ++u) {
            if (in_use[u]) continue;
            const uint32_t lu = a.last_use[u];
            rank += (lu < mine || (lu == mine && u < tid)) ? 1 : 0;
        }
        if (rank < 1024) victim_of_rank[rank] = tid;
        atomicAdd(&s_nfree, 1);
    }
    __syncthreads();
    const int nmiss = s_nmiss;
    if (nmiss > s_nfree) {  // more routed experts than slots: nothing is fetched
        if (tid == 0) {
            atomicExch(a.status, -7);  // MAPLE_ERR_WORKSPACE: the cache is too small
            a.jobs[0] = 0;
        }
        for (int s = tid; s < a.S; s += kPlanThreads) a.idx_slot[s] = -1;
        return;
    }
    // evict the victims' old experts first, then assign
    if (tid < E && miss_rank[tid] >= 0) {
        const int v = victim_of_rank[miss_rank[tid]];
        const int old = a.expert_of[v];
        if (old >= 0) a.slot_of[old] = -1;
    }
    __syncthreads();
    if (tid < E && miss_rank[tid] >= 0) {
        const int r = miss_rank[tid], v = victim_of_rank[r];
        a.expert_of[v] = tid;
        a.slot_of[tid] = v;
        a.last_use[v] = s_stamp;
        a.jobs[1 + 2 * r] = v;
        a.jobs[2 + 2 * r] = tid;
    }
    const int nneed = __syncthreads_count(tid < E && need[tid]);
    if (tid == 0) {
        a.jobs[0] = nmiss;
        a.stats[1] += (uint32_t)(nneed - nmiss);
        a.stats[2] += (uint32_t)nmiss;
        a.stats[3] += (uint32_t)nmiss;
    }
    __threadfence_block();
    __syncthreads();
    for (int s = tid; s < a.S; s += kPlanThreads) {
        const int e = a.idx[s];
        a.idx_slot[s] = (e >= 0 && e < E) ? a.slot_of[e] : -1;
    }
}

// Copies [begin, end) 16-byte chunks of one array from the pool to a slot.
__device__ __forceinline__ void copy_chunks(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n,
                                            int part, int tid) {
    const int64_t begin = n * part / kCopyParts, end = n * (part + 1) / kCopyParts;
    int64_t i = begin + tid;
    for (; i + 3 * kCopyThreads < end; i += 4 * kCopyThreads) {
        const uint4 v0 = src[i], v1 = src[i + kCopyThreads], v2 = src[i + 2 * kCopyThreads],
                    v3 = src[i + 3 * kCopyThreads];
        dst[i] = v0;
        dst[i + kCopyThreads] = v1;
        dst[i + 2 * kCopyThreads] = v2;
        dst[i + 3 * kCopyThreads] = v3;
    }
    for (; i < end; i += kCopyThreads) dst[i] = src[i];
}

__global__ void __launch_bounds__(kCopyThreads) cache_copy_kernel(CacheArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int job = blockIdx.x / kCopyParts, part = blockIdx.x % kCopyParts;
    if (job >= a.jobs[0]) return;
    const int v = a.jobs[1 + 2 * job], e = a.jobs[2 + 2 * job];
    const int H = a.slots.H, I = a.slots.I;
    const int64_t gu = (int64_t)I * ((H + 4) / 5), dn = (int64_t)H * ((I + 4) / 5);
    const int tid = threadIdx.x;
    copy_chunks(reinterpret_cast<const uint4*>(a.pool.gate + e * gu), reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.slots.gate) + v * gu), gu / 16, part, tid);
    copy_chunks(reinterpret_cast<const uint4*>(a.pool.up + e * gu), reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.slots.up) + v * gu), gu / 16, part, tid);
    copy_chunks(reinterpret_cast<const uint4*>(a.pool.down + e * dn), reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.slots.down) + v * dn), dn / 16, part, tid);
    copy_chunks(reinterpret_cast<const uint4*>(a.pool.s_gate + (int64_t)e * I), reinterpret_cast<uint4*>(const_cast<float*>(a.slots.s_gate) + (int64_t)v * I), I / 4, part, tid);
    copy_chunks(reinterpret_cast<const uint4*>(a.pool.s_up + (int64_t)e * I), reinterpret_cast<uint4*>(const_cast<float*>(a.slots.s_up) + (int64_t)v * I), I / 4, part, tid);
    copy_chunks(reinterpret_cast<const uint4*>(a.pool.s_down + (int64_t)e * H), reinterpret_cast<uint4*>(const_cast<float*>(a.slots.s_down) + (int64_t)v * H), H / 4, part, tid);
}

}  // namespace

// The arrays of one expert must be whole 16-byte chunks at 16-byte aligned offsets.
bool cache_shape_ok(int H, int I) {
    const int64_t gu = (int64_t)I * ((H + 4) / 5), dn = (int64_t)H * ((I + 4) / 5);
    return gu % 16 == 0 && dn % 16 == 0 && I % 4 == 0 && H % 4 == 0;
}

cudaError_t launch_cache_fetch(const maple_experts& pool, const maple_experts& slots, int32_t* slot_of,
                               int32_t* expert_of, uint32_t* last_use, uint32_t* stats, const int32_t* idx,
                               int S, int32_t* idx_slot, int32_t* jobs, cudaStream_t stream,
                               const DeviceInfo& dev) {
    CacheArgs a;
    a.pool = pool;
    a.slots = slots;
    a.slot_of = slot_of;
    a.expert_of = expert_of;
    a.last_use = last_use;
    a.stats = stats;
    a.idx = idx;
    a.S = S;
    a.idx_slot = idx_slot;
    a.jobs = jobs;
    a.status = dev.status;
    cudaError_t err = launch_pdl(cache_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, a);
    if (err != cudaSuccess) return err;
    // at most min(S, C, E) experts are copied
    int maxjobs = S < slots.E ? S : slots.E;
    maxjobs = maxjobs < pool.E ? maxjobs : pool.E;
    return launch_pdl(cache_copy_kernel, dim3(maxjobs * kCopyParts), dim3(kCopyThreads), 0, stream, a);
}

}  // namespace maple
