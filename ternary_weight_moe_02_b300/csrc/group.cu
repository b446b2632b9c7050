// Token-to-expert grouping: histogram, exclusive scan and a stable placement of the
// T*k routing slots by expert (a counting sort), in one CTA of 1024 threads.
//
// The grouping is not on the pages; it follows from batching tokens that share an
// expert so that each expert's packed rows are read once per step.  Stable order
// (slots of one expert in increasing slot number) makes the result unique.
//
// Placement walks the slots in chunks of 1024 in order.  Inside a warp, lanes with
// the same expert find each other with match.any and rank themselves by lane; the
// per-warp counts of each expert (shared memory) give the offset of a warp inside
// the chunk; a running cursor per expert carries the chunks.
#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

constexpr int kGroupThreads = 1024;
constexpr int kGroupWarps = kGroupThreads / 32;

__global__ void __launch_bounds__(kGroupThreads)
    group_tokens_kernel(const int32_t* __restrict__ idx, int S, int E,
                        int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ perm, int32_t* __restrict__ active,
                        int32_t* __restrict__ n_active) {
    extern __shared__ int32_t smem[];
    int32_t* hist = smem;                 // [E]
    int32_t* cursor = hist + E;           // [E]
    int32_t* warp_cnt = cursor + E;       // [kGroupWarps][E]
    __shared__ int32_t scan_part[kGroupWarps];
    __shared__ int32_t scan_flag[kGroupWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kGroupThreads) hist[e] = 0;
    for (int i = tid; i < kGroupWarps * E; i += kGroupThreads) warp_cnt[i] = 0;
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    for (int s = tid; s < S; s += kGroupThreads) {
        const int e = idx[s];
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();

    // Exclusive scan of counts (and of the "non-empty" flags) over E <= 1024 entries:
    // thread e holds entry e.
    {
        const int c = tid < E ? hist[tid] : 0;
        const int f = c > 0 ? 1 : 0;
        int ci = c, fi = f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int cn = __shfl_up_sync(kFullMask, ci, o);
            const int fn = __shfl_up_sync(kFullMask, fi, o);
            if (lane >= o) {
                ci += cn;
                fi += fn;
            }
        }
        if (lane == 31) {
            scan_part[warp] = ci;
            scan_flag[warp] = fi;
        }
        __syncthreads();
        if (warp == 0) {
            int p = scan_part[lane], q = scan_flag[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int pn = __shfl_up_sync(kFullMask, p, o);
                const int qn = __shfl_up_sync(kFullMask, q, o);
                if (lane >= o) {
                    p += pn;
                    q += qn;
                }
            }
            scan_part[lane] = p;
            scan_flag[lane] = q;
        }
        __syncthreads();
        const int base_c = warp > 0 ? scan_part[warp - 1] : 0;
        const int base_f = warp > 0 ? scan_flag[warp - 1] : 0;
        const int excl_c = base_c + ci - c;
        const int excl_f = base_f + fi - f;
        if (tid < E) {
            counts[tid] = c;
            offsets[tid] = excl_c;
            cursor[tid] = excl_c;
            if (active != nullptr && f) active[excl_f] = tid;
        }
        if (tid == E - 1) {
            offsets[E] = excl_c + c;
            if (n_active != nullptr) *n_active = excl_f + f;
        }
    }
    __syncthreads();

    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < S; base += kGroupThreads) {
        const int s = base + tid;
        int e = s < S ? idx[s] : -1;
        const bool valid = e >= 0 && e < E;
        if (!valid) e = -1;
        const unsigned peers = __match_any_sync(kFullMask, e);
        const int rank = __popc(peers & lt_mask);
        if (valid && rank == 0) warp_cnt[warp * E + e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int pre = 0;
            for (int w2 = 0; w2 < warp; ++w2) pre += warp_cnt[w2 * E + e];
            perm[cursor[e] + pre + rank] = s;
        }
        __syncthreads();
        for (int ee = tid; ee < E; ee += kGroupThreads) {
            int tot = 0;
            for (int w2 = 0; w2 < kGroupWarps; ++w2) {
                tot += warp_cnt[w2 * E + ee];
                warp_cnt[w2 * E + ee] = 0;
            }
            cursor[ee] += tot;
        }
        __syncthreads();
    }
}

}  // namespace

size_t group_tokens_smem_bytes(int E) { return sizeof(int32_t) * (size_t)E * (2 + kGroupWarps); }

cudaError_t launch_group_tokens(const int32_t* idx, int S, int k, int E, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* active,
                                int32_t* n_active, cudaStream_t stream, const DeviceInfo& dev) {
    (void)k;
    const size_t smem = group_tokens_smem_bytes(E);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(group_tokens_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    (void)dev;
    return launch_pdl(group_tokens_kernel, dim3(1), dim3(kGroupThreads), smem, stream, idx, S, E,
                      counts, offsets, perm, active, n_active);
}

}  // namespace maple
