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
                        int32_t* __restrict__ n_active, int nt, int32_t* __restrict__ tile_off,
                        int4* __restrict__ tile_info) {
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
        // the grouped tensor-core path's tile table (nt > 0): tile_off[e] = sum over
        // e' < e of ceil(counts[e'] / nt), and per tile (expert, first token, tokens,
        // grouped position of its first token)
        if (nt > 0) {
            const int v = (c + nt - 1) / nt;
            int vi = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int vn = __shfl_up_sync(kFullMask, vi, o);
                if (lane >= o) vi += vn;
            }
            __syncthreads();  // every thread has read the counts scan's partials
            if (lane == 31) scan_part[warp] = vi;
            __syncthreads();
            if (warp == 0) {
                int p = scan_part[lane];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int pn = __shfl_up_sync(kFullMask, p, o);
                    if (lane >= o) p += pn;
                }
                scan_part[lane] = p;
            }
            __syncthreads();
            const int excl_v = (warp > 0 ? scan_part[warp - 1] : 0) + vi - v;
            if (tid < E) tile_off[tid] = excl_v;
            if (tid == E - 1) tile_off[E] = excl_v + v;
            for (int t = 0; t < v; ++t) {
                const int n0 = t * nt, left = c - n0;
                tile_info[excl_v + t] = make_int4(tid, n0, left < nt ? left : nt, excl_c + n0);
            }
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

// Multi-CTA grouping for many slots (same result as group_tokens_kernel): chunks of
// kChunk slots; (1) a histogram per chunk, (2) one CTA turns them into counts,
// offsets, the active list and each chunk's base position per expert, (3) each chunk
// places its slots stably (match.any ranks inside a warp, per-warp counts across the
// chunk's warps).
constexpr int kChunk = 1024;

__global__ void __launch_bounds__(kChunk) group_hist_kernel(const int32_t* __restrict__ idx, int S, int E,
                                                            int32_t* __restrict__ chunk_counts) {
    extern __shared__ int32_t hist[];  // [E]
    for (int e = threadIdx.x; e < E; e += kChunk) hist[e] = 0;
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    const int s = blockIdx.x * kChunk + threadIdx.x;
    if (s < S) {
        const int e = idx[s];
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kChunk) chunk_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// One CTA of 1024 threads, thread e < E owns expert e.  chunk_counts is turned into the
// chunks' base positions in place.
__global__ void __launch_bounds__(kGroupThreads)
    group_scan_kernel(int32_t* __restrict__ chunk_counts, int C, int E, int32_t* __restrict__ counts,
                      int32_t* __restrict__ offsets, int32_t* __restrict__ active, int32_t* __restrict__ n_active) {
    __shared__ int32_t scan_part[kGroupWarps];
    __shared__ int32_t scan_flag[kGroupWarps];
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int c_tot = 0;
    if (tid < E)
        for (int c = 0; c < C; ++c) c_tot += chunk_counts[(int64_t)c * E + tid];
    const int f = c_tot > 0 ? 1 : 0;
    int ci = c_tot, fi = f;
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
    const int excl_c = (warp > 0 ? scan_part[warp - 1] : 0) + ci - c_tot;
    const int excl_f = (warp > 0 ? scan_flag[warp - 1] : 0) + fi - f;
    if (tid < E) {
        counts[tid] = c_tot;
        offsets[tid] = excl_c;
        if (active != nullptr && f) active[excl_f] = tid;
        int base = excl_c;
        for (int c = 0; c < C; ++c) {
            const int n = chunk_counts[(int64_t)c * E + tid];
            chunk_counts[(int64_t)c * E + tid] = base;
            base += n;
        }
    }
    if (tid == E - 1) {
        offsets[E] = excl_c + c_tot;
        if (n_active != nullptr) *n_active = excl_f + f;
    }
}

__global__ void __launch_bounds__(kChunk) group_place_kernel(const int32_t* __restrict__ idx, int S, int E,
                                                             const int32_t* __restrict__ chunk_base,
                                                             int32_t* __restrict__ perm) {
    extern __shared__ int32_t warp_cnt[];  // [kChunk / 32][E]
    constexpr int kW = kChunk / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kW * E; i += kChunk) warp_cnt[i] = 0;
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    const int s = blockIdx.x * kChunk + tid;
    int e = s < S ? idx[s] : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1;
    const unsigned peers = __match_any_sync(kFullMask, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) warp_cnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (valid) {
        int pre = 0;
        for (int w2 = 0; w2 < warp; ++w2) pre += warp_cnt[w2 * E + e];
        perm[chunk_base[(int64_t)blockIdx.x * E + e] + pre + rank] = s;
    }
}

}  // namespace

size_t group_chunked_bytes(int S, int E) { return sizeof(int32_t) * (size_t)((S + kChunk - 1) / kChunk) * E; }

cudaError_t launch_group_tokens_chunked(const int32_t* idx, int S, int E, int32_t* counts, int32_t* offsets,
                                        int32_t* perm, int32_t* active, int32_t* n_active, int32_t* chunk_scratch,
                                        cudaStream_t stream) {
    const int C = (S + kChunk - 1) / kChunk;
    cudaError_t err = launch_pdl(group_hist_kernel, dim3(C), dim3(kChunk), sizeof(int32_t) * (size_t)E, stream, idx,
                                 S, E, chunk_scratch);
    if (err != cudaSuccess) return err;
    err = launch_pdl(group_scan_kernel, dim3(1), dim3(kGroupThreads), 0, stream, chunk_scratch, C, E, counts, offsets,
                     active, n_active);
    if (err != cudaSuccess) return err;
    const size_t smem = sizeof(int32_t) * (size_t)(kChunk / 32) * E;
    err = ensure_dynamic_smem(group_place_kernel, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(group_place_kernel, dim3(C), dim3(kChunk), smem, stream, idx, S, E,
                      (const int32_t*)chunk_scratch, perm);
}

size_t group_tokens_smem_bytes(int E) { return sizeof(int32_t) * (size_t)E * (2 + kGroupWarps); }

cudaError_t launch_group_tokens(const int32_t* idx, int S, int k, int E, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* active,
                                int32_t* n_active, cudaStream_t stream, const DeviceInfo& dev, int nt,
                                int32_t* tile_off, int4* tile_info) {
    (void)k;
    const size_t smem = group_tokens_smem_bytes(E);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(group_tokens_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
    }
    (void)dev;
    return launch_pdl(group_tokens_kernel, dim3(1), dim3(kGroupThreads), smem, stream, idx, S, E,
                      counts, offsets, perm, active, n_active, nt, tile_off, tile_info);
}

}  // namespace maple
