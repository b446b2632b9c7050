// Expert FFN on the tcgen05 tensor cores (grouped path: tokens batched per expert).
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// sections "The claim, verified from the bytes" (one scale per output row, trits
// -1/0/+1) and "The shipped code does no quantization" (the expert body
// down(act(clamp(gate x, max=7)) * clamp(up x, -7, 7))).  The pages give no kernel for
// many tokens per expert; a trit is exact in bf16, so the sums can run on the tensor
// cores with fp32 accumulation.
//
// Per expert e with n_e routed tokens (slots grouped by expert, tiles of NT tokens;
// NT = 128 for prefill-sized calls, 16 for decode batches):
//   gate/up CTA: D[128 x NT] = A . X^T, A = 64 gate rows and the same 64 up rows of e,
//     X = the tokens' bf16 activations (gathered once per call into expert order,
//     loaded by TMA); fp32 accumulation in tensor memory.  Epilogue:
//     h = silu(min(s_g g, clamp)) * clamp(s_u u, -clamp, clamp), rounded to bf16, stored
//     per slot in expert order.
//   down CTA: D[128 x NT] = A_down . H^T over I; epilogue w_slot * s_d * D stored per
//     slot (fp32); a combine kernel adds each token's k slots in order 0..k-1.
//
// A is decoded from the packed bytes straight into tensor memory: thread r of lane
// quarter r / 32 owns weight row r (TMEM lane r) and writes its K values as bf16 +-0.5
// or 0 (half the trit, exact; the epilogues scale by 2 s), two per 32-bit column, with
// tcgen05.st; the MMA reads A from tensor memory.  B (tokens) sits in shared memory
// K-major without swizzle: element (n, k) of a stage at (k / 8) * (NT * 16) + n * 16 +
// (k % 8) * 2.  The gather kernel (for x) and the gate/up epilogue (for h) store each
// tile's rows in global memory in that same order (chunk-major, [tile][K/8][NT][8]),
// so a stage is one contiguous block loaded by one 1-D bulk copy.  K tiles hold 80
// values (16 packed bytes per row).
// Eight producer warps fill a ring of four stages; one thread issues five tcgen05.mma
// (K = 16 each) per stage and commits them to the stage's "empty" mbarrier, which the
// producers wait for before refilling the stage.  All waits are bounded.
#include <cuda_bf16.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"

namespace maple {

namespace {

constexpr int kRows = 128;                 // MMA M: weight rows per CTA
constexpr int kKTile = 80;                 // K values per stage (16 packed bytes)
constexpr int kChunks = kKTile / 8;        // 16-byte core-matrix columns per B stage
constexpr int kMaxStages = 4;
constexpr int kAStride = 48;               // TMEM column stride between A stages (40 used)
constexpr int kLutReps = 4;                // copies of the decode table, by lane & 3
constexpr int kLutBytes = 256 * kLutReps * 8;  // 8 KB
constexpr int kProducerWarps = 8;          // decode A, load B; warp 8 issues the MMAs
constexpr int kThreads = (kProducerWarps + 1) * 32;

template <int NT>
struct TileCfg {
    static constexpr int kStages = 4;                                    // ring depth
    static constexpr int kStageB = kChunks * NT * 16;                    // bytes of a B stage
    static constexpr int kABase = NT < 32 ? 32 : NT;                     // first A column
    static constexpr int kUsedCols = kABase + kStages * kAStride;
    static constexpr int kTmemCols = kUsedCols <= 256 ? 256 : 512;       // power of two
    // instruction descriptor: D fp32, A and B bf16, both K-major, N = NT, M = 128
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) |
                                       ((uint32_t)(kRows >> 4) << 24);
};

// ----------------------------------------------------------------- tcgen05 helpers

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    // start address, leading (K-direction) and stride (row-group) byte offsets, >> 4;
    // bits 46-47: descriptor version 1; swizzle field (bits 61-63) 0: none
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
           ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[tmem] . B[smem descriptor]
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// 16 and 4 consecutive 32-bit columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* w) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]),
        "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* w) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3])
                 : "memory");
}

// 8 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// ----------------------------------------------------------------- decode table

// For each code, the high bytes of the five bf16 values +-0.5 / 0 of its trits (0xBF
// for -1, 0x00 for 0, 0x3F for +1; the low byte of those bf16 values is zero), bytes
// 5-7 zero; the invalid codes 243..255 give five zeros.  kLutReps copies interleaved by
// entry ([code][copy]) so that the 8-byte loads of a half-warp spread over more banks.
__device__ __forceinline__ void build_half_lut(uint2* lut, int tid, int nthreads) {
    for (int i = tid; i < 256 * kLutReps; i += nthreads) {
        const int c = i / kLutReps;
        uint32_t b[5] = {0u, 0u, 0u, 0u, 0u};
        if (c < 243) {
            int code = c;
#pragma unroll
            for (int t = 0; t < 5; ++t) {
                const int d = code % 3;
                code /= 3;
                b[t] = d == 0 ? 0xBFu : (d == 2 ? 0x3Fu : 0u);
            }
        }
        lut[i] = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4]);
    }
}

// Decodes packed bytes [16 kt + 8 h, +8) of one row (bytes at or past rb read as the
// all-zero code 121) into 20 words of two bf16 each (K order).  Two bytes (ten values)
// become five words by byte permutes of their two table entries.
__device__ __forceinline__ void decode_half_tile(const uint8_t* row, int rb, int kt, int h, const uint2* lut,
                                                 int rep, uint32_t* words) {
    const int b0 = 16 * kt + 8 * h;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int ba = b0 + 2 * p, bb = ba + 1;
        const int ca = ba < rb ? row[ba] : 121;
        const int cb = bb < rb ? row[bb] : 121;
        const uint2 ea = lut[ca * kLutReps + rep];
        const uint2 eb = lut[cb * kLutReps + rep];
        words[5 * p + 0] = __byte_perm(ea.x, ea.y, 0x1505);  // 0, a0, 0, a1
        words[5 * p + 1] = __byte_perm(ea.x, ea.y, 0x3525);  // 0, a2, 0, a3
        words[5 * p + 2] = __byte_perm(ea.y, eb.x, 0x4101);  // 0, a4, 0, b0
        words[5 * p + 3] = __byte_perm(eb.x, eb.y, 0x2515);  // 0, b1, 0, b2
        words[5 * p + 4] = __byte_perm(eb.x, eb.y, 0x4535);  // 0, b3, 0, b4
    }
}

struct TcArgs {
    const uint8_t* gate;
    const uint8_t* up;
    const uint8_t* down;
    const float* s_gate;
    const float* s_up;
    const float* s_down;
    int E, H, I, k;
    float clamp;
    const uint16_t* x;
    const float* w;
    const int32_t* idx;
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* perm;
    const int32_t* tile_off;  // [E + 1] prefix of ceil(counts / NT)
    uint16_t* xs;             // [tile][H / 8][NT][8] bf16: each tile's token rows
    uint16_t* hs;             // [tile][I / 8][NT][8] bf16: each tile's h rows
    float* ys;                // [T k][H] fp32, per original slot
    float* y;                 // [T][H]
    int T;
    int* status;
};

// Shared-memory plan of a grouped CTA: the decode table, the CTA's packed rows, the B
// stages.  The epilogue reuses the packed rows and the stages.
__host__ __device__ constexpr size_t tc_packed_offset() { return (size_t)kLutBytes; }
__host__ __device__ constexpr size_t tc_stage_offset(int row_bytes) {
    return (tc_packed_offset() + (size_t)kRows * row_bytes + 127) / 128 * 128;
}
template <int NT>
__host__ __device__ constexpr size_t tc_smem_bytes(int row_bytes) {
    return tc_stage_offset(row_bytes) + (size_t)TileCfg<NT>::kStages * TileCfg<NT>::kStageB;
}

// Finds the expert and token range of grid row `tile`; false when past the last tile.
// The tile table, counts and offsets come from kernels that completed before the
// previous one started, so they are read (through L2) before this grid's PDL wait.
template <int NT>
__device__ __forceinline__ bool tc_tile(const TcArgs& a, int tile, int& e, int& n0, int& nv, int& pos0) {
    if (tile >= __ldcg(a.tile_off + a.E)) return false;
    int lo = 0, hi = a.E - 1;  // largest e with tile_off[e] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldcg(a.tile_off + mid) <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    e = lo;
    n0 = (tile - __ldcg(a.tile_off + e)) * NT;
    const int left = __ldcg(a.counts + e) - n0;
    nv = left < NT ? left : NT;
    pos0 = __ldcg(a.offsets + e) + n0;
    return nv > 0;
}

// Barriers of a grouped CTA: full[s] (one arrival per producer thread once its A words
// are in tensor memory), bfull[s] (the B tile's TMA bytes), empty[s] (MMA commit),
// done (commit after the last MMA), packed (bulk copy of the CTA's packed rows).
struct TcBars {
    uint64_t full[kMaxStages];
    uint64_t bfull[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t done;
    uint64_t packed;
};

// Warp-specialised main loop.  Warp w < 8 produces: its thread owns row 32 (w & 3) +
// lane (the warp's TMEM lane quarter) and decodes half w >> 2 of that row's 16 bytes of
// each K tile into A stage s (tensor memory), then arrives on full[s]; thread 0 also
// copies the stage's B block (this K tile's chunks of the tile's operand block bsrc,
// fewer at the K tail) with one bulk copy onto bfull[s].
// Warp 8 lane 0 waits for both, issues the stage's five MMAs and commits empty[s]; its
// last commit goes to done.  Returns false if a bounded wait gave up.
template <int NT>
__device__ bool tc_mainloop(unsigned char* smem, const uint8_t* packed, int rb, int Kdim, const uint16_t* bsrc,
                            uint32_t tmem, TcBars& bars, int* status) {
    using Cfg = TileCfg<NT>;
    constexpr int S = Cfg::kStages;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint2* lut = reinterpret_cast<const uint2*>(smem);
    unsigned char* stages = smem + tc_stage_offset(rb);
    const int KT = (Kdim + kKTile - 1) / kKTile;
    bool ok = true;
    int issued = 0;  // B tiles thread 0 has loaded
    if (warp < kProducerWarps) {
        const int q = warp & 3, h = warp >> 2, r = 32 * q + lane;
        const uint8_t* my_row = packed + r * rb;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        // tile j + 1 is decoded while tile j's tensor-memory stores complete
        uint32_t cur[20], nxt[20];
        decode_half_tile(my_row, rb, 0, h, lut, lane & (kLutReps - 1), cur);
        for (int j = 0; j < KT && ok; ++j) {
            const int s = j % S;
            if (j >= S && !mbar_wait_bounded(&bars.empty[s], (uint32_t)(((j - S) / S) & 1), status)) {
                ok = false;
                break;
            }
            if (tid == 0) {
                const int left = Kdim / 8 - j * kChunks;
                const uint32_t bytes = (uint32_t)((left < kChunks ? left : kChunks) * NT * 16);
                mbar_arrive_expect_tx(&bars.bfull[s], bytes);
                bulk_copy_g2s(stages + s * Cfg::kStageB, bsrc + (size_t)j * kChunks * NT * 8, bytes, &bars.bfull[s]);
                issued = j + 1;
            }
            const uint32_t col = (uint32_t)(Cfg::kABase + s * kAStride + 20 * h);
            tmem_st16(lane_base + col, cur);
            tmem_st4(lane_base + col + 16, cur + 16);
            if (j + 1 < KT) decode_half_tile(my_row, rb, j + 1, h, lut, lane & (kLutReps - 1), nxt);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(&bars.full[s]);
#pragma unroll
            for (int i = 0; i < 20; ++i) cur[i] = nxt[i];
        }
    } else if (tid == kProducerWarps * 32) {
        for (int j = 0; j < KT; ++j) {
            const int s = j % S;
            const uint32_t par = (uint32_t)((j / S) & 1);
            if (!mbar_wait_bounded(&bars.full[s], par, status) || !mbar_wait_bounded(&bars.bfull[s], par, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = tmem + (uint32_t)(Cfg::kABase + s * kAStride);
            const uint32_t b0 = smem_addr(stages + s * Cfg::kStageB);
#pragma unroll
            for (int qk = 0; qk < kKTile / 16; ++qk) {
                const uint64_t bd = smem_desc(b0 + qk * 2 * (NT * 16), NT * 16, 128);
                mma_tmem_a(tmem, a0 + 8 * qk, bd, Cfg::kIdesc, (j | qk) != 0 ? 1u : 0u);
            }
            mma_commit(j == KT - 1 ? &bars.done : &bars.empty[s]);
        }
    }
    __syncwarp();
    // every thread waits for the last MMA (the epilogue reads TMEM and reuses shared memory)
    if (ok && !mbar_wait_bounded(&bars.done, 0, status)) ok = false;
    if (!ok && tid == 0) {
        // the last B load of each stage may still be in flight: let it land first
        for (int t = issued - S > 0 ? issued - S : 0; t < issued; ++t)
            mbar_wait_bounded(&bars.bfull[t % S], (uint32_t)((t / S) & 1), nullptr);
    }
    tc_fence_after();
    return !__syncthreads_or(!ok);
}

// CTA prologue shared by both stages: decode table, zeroed B stages, barriers, TMEM
// (warp 8), and the bulk copy of the CTA's packed rows (nrows_copy rows of rb bytes
// from src0 and, when src1 is set, as many from src1).
__device__ bool tc_prologue(unsigned char* smem, TcBars& bars, uint32_t* tmem_slot, uint32_t tmem_cols,
                            const uint8_t* src0, const uint8_t* src1, int nrows_copy, int rb, size_t stage_bytes,
                            int* status) {
    const int tid = threadIdx.x;
    build_half_lut(reinterpret_cast<uint2*>(smem), tid, blockDim.x);
    // zero the B stages: the K tail's chunks are never copied, and the MMA multiplies
    // them by zero A values, which must not meet NaN bit patterns
    uint4* st4 = reinterpret_cast<uint4*>(smem + tc_stage_offset(rb));
    for (size_t i = tid; i < stage_bytes / 16; i += blockDim.x) st4[i] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (tid == 0) {
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&bars.full[i], kProducerWarps * 32);
            mbar_init(&bars.bfull[i], 1);
            mbar_init(&bars.empty[i], 1);
        }
        mbar_init(&bars.done, 1);
        mbar_init(&bars.packed, 1);
        const uint32_t bytes = (uint32_t)(nrows_copy * rb);
        mbar_arrive_expect_tx(&bars.packed, src1 ? 2 * bytes : bytes);
        bulk_copy_g2s(smem + tc_packed_offset(), src0, bytes, &bars.packed);
        if (src1) bulk_copy_g2s(smem + tc_packed_offset() + bytes, src1, bytes, &bars.packed);
    }
    if ((tid >> 5) == kProducerWarps) tmem_alloc(tmem_slot, tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool ok = mbar_wait_bounded(&bars.packed, 0, status);
    return !__syncthreads_or(!ok);
}

__device__ __forceinline__ void tc_release(uint32_t tmem, uint32_t tmem_cols) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == kProducerWarps) tmem_dealloc(tmem, tmem_cols);
}

// gate/up: grid (I / 64, max tiles); rows 0..63 of the CTA are gate rows m0..m0+63 of
// the expert, rows 64..127 the same up rows.
template <int NT>
__global__ void __launch_bounds__(kThreads, 1) tc_gateup_kernel(TcArgs a) {
    using Cfg = TileCfg<NT>;
    constexpr int CW = NT / 2;  // columns per epilogue warp (two warps per lane quarter)
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ TcBars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ float s_scale[kRows];  // 2 s of rows 0..127 (gate rows, then up rows)
    int e, n0, nv, pos0;
    if (!tc_tile<NT>(a, blockIdx.y, e, n0, nv, pos0)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, I = a.I, Bh = (H + 4) / 5;
    const int m0 = blockIdx.x * (kRows / 2);
    const int tile = blockIdx.y;
    if (tid < kRows)
        s_scale[tid] = 2.f * (tid < kRows / 2 ? a.s_gate[(int64_t)e * I + m0 + tid]
                                             : a.s_up[(int64_t)e * I + m0 + tid - kRows / 2]);
    const uint8_t* gsrc = a.gate + ((int64_t)e * I + m0) * Bh;
    const uint8_t* usrc = a.up + ((int64_t)e * I + m0) * Bh;
    // everything up to here reads data no kernel of this call writes
    bool ok = tc_prologue(smem, bars, &tmem_slot, Cfg::kTmemCols, gsrc, usrc, kRows / 2, Bh,
                          (size_t)Cfg::kStages * Cfg::kStageB, a.status);
    const uint32_t tmem = tmem_slot;
    pdl_wait();  // the gathered x of the previous kernel
    pdl_launch_dependents();
    if (ok) ok = tc_mainloop<NT>(smem, smem + tc_packed_offset(), Bh, H, a.xs + (size_t)tile * H * NT, tmem, bars, a.status);
    if (ok) {
        // epilogue: warps 0-7 read rows 32 (w & 3) + lane and columns CW (w >> 2) .. +CW,
        // store min(2 s_g g, clamp) (gate rows) or clamp(2 s_u u) (up rows); then every
        // thread forms h = silu(g) u for its share of the tile and rounds it to bf16
        unsigned char* epi = smem + tc_packed_offset();
        float* G = reinterpret_cast<float*>(epi);                             // [NT][64]
        float* U = G + NT * 64;                                               // [NT][64]
        uint16_t* Hs = reinterpret_cast<uint16_t*>(U + NT * 64);              // [NT][64]
        if (warp < kProducerWarps) {
            const int q = warp & 3, c0 = CW * (warp >> 2), r = 32 * q + lane;
            const uint32_t addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
            const float sc = s_scale[r];
            float v[CW];
#pragma unroll
            for (int i = 0; i < CW; i += 8) tmem_ld8(addr + i, v + i);
            if (q < 2) {
#pragma unroll
                for (int i = 0; i < CW; ++i) G[(c0 + i) * 64 + r] = fminf(sc * v[i], a.clamp);
            } else {
#pragma unroll
                for (int i = 0; i < CW; ++i) U[(c0 + i) * 64 + r - 64] = fminf(fmaxf(sc * v[i], -a.clamp), a.clamp);
            }
        }
        __syncthreads();
        for (int i = tid; i < nv * 64; i += kThreads)
            Hs[i] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_f(G[i]) * U[i]));
        __syncthreads();
        // the tile's h rows, chunk-major: chunk m0 / 8 + part, row nn
        uint16_t* hblk = a.hs + (size_t)tile * I * NT;
        for (int i = tid; i < nv * 8; i += kThreads) {
            const int part = i / nv, nn = i - part * nv;
            *reinterpret_cast<uint4*>(hblk + ((size_t)(m0 / 8 + part) * NT + nn) * 8) =
                *reinterpret_cast<const uint4*>(Hs + nn * 64 + 8 * part);
        }
    }
    tc_release(tmem, Cfg::kTmemCols);
}

// down: grid (H / 128, max tiles); the CTA's 128 rows are down rows m0..m0+127.
template <int NT>
__global__ void __launch_bounds__(kThreads, 1) tc_down_kernel(TcArgs a) {
    using Cfg = TileCfg<NT>;
    constexpr int CW = NT / 2;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ TcBars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_slot[NT];
    __shared__ float s_w[NT];
    __shared__ float s_scale[kRows];
    int e, n0, nv, pos0;
    if (!tc_tile<NT>(a, blockIdx.y, e, n0, nv, pos0)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, I = a.I, Bi = (I + 4) / 5;
    const int m0 = blockIdx.x * kRows;
    if (tid < NT) {
        const int slot = tid < nv ? __ldcg(a.perm + pos0 + tid) : 0;
        s_slot[tid] = slot;
        s_w[tid] = tid < nv ? __ldcg(a.w + slot) : 0.f;
    }
    if (tid < kRows) s_scale[tid] = 2.f * a.s_down[(int64_t)e * H + m0 + tid];
    const uint8_t* dsrc = a.down + ((int64_t)e * H + m0) * Bi;
    // everything up to here reads data no kernel of this call writes after the grouping
    bool ok = tc_prologue(smem, bars, &tmem_slot, Cfg::kTmemCols, dsrc, nullptr, kRows, Bi,
                          (size_t)Cfg::kStages * Cfg::kStageB, a.status);
    const uint32_t tmem = tmem_slot;
    pdl_wait();  // h of the gate/up kernel
    pdl_launch_dependents();
    if (ok)
        ok = tc_mainloop<NT>(smem, smem + tc_packed_offset(), Bi, I, a.hs + (size_t)blockIdx.y * I * NT, tmem, bars,
                             a.status);
    if (ok) {
        float* Ys = reinterpret_cast<float*>(smem + tc_packed_offset());  // [NT][kRows]
        if (warp < kProducerWarps) {
            const int q = warp & 3, c0 = CW * (warp >> 2), r = 32 * q + lane;
            const uint32_t addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
            const float sd = s_scale[r];
            float v[CW];
#pragma unroll
            for (int i = 0; i < CW; i += 8) tmem_ld8(addr + i, v + i);
#pragma unroll
            for (int i = 0; i < CW; ++i) Ys[(c0 + i) * kRows + r] = s_w[c0 + i] * (sd * v[i]);
        }
        __syncthreads();
        for (int i = tid; i < nv * (kRows / 4); i += kThreads) {
            const int nn = i / (kRows / 4), part = i % (kRows / 4);
            *reinterpret_cast<float4*>(a.ys + (int64_t)s_slot[nn] * H + m0 + 4 * part) =
                *reinterpret_cast<const float4*>(Ys + nn * kRows + 4 * part);
        }
    }
    tc_release(tmem, Cfg::kTmemCols);
}

// One CTA per tile: the tile's token rows of x, chunk-major ([H / 8][NT][8]).  Rows
// past the tile's tokens are left as they are: they only reach output columns that
// the epilogues never store.
template <int NT>
__global__ void __launch_bounds__(256) tc_gather_kernel(TcArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    int e, n0, nv, pos0;
    if (!tc_tile<NT>(a, blockIdx.x, e, n0, nv, pos0)) return;
    const int H8 = a.H / 8;
    uint4* blk = reinterpret_cast<uint4*>(a.xs + (size_t)blockIdx.x * a.H * NT);
    for (int i = threadIdx.x; i < H8 * nv; i += blockDim.x) {
        const int c = i / nv, r = i - c * nv;
        blk[c * NT + r] = reinterpret_cast<const uint4*>(a.x + (int64_t)(a.perm[pos0 + r] / a.k) * a.H)[c];
    }
}

// y[t] = sum over i = 0..k-1 of the slot outputs of token t (slots of invalid experts
// add nothing), four columns per thread.
__global__ void __launch_bounds__(256) tc_combine_kernel(TcArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int H4 = a.H / 4;
    const int64_t total = (int64_t)a.T * H4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / H4), c4 = (int)(i - (int64_t)t * H4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < a.k; ++j) {
            const int s = t * a.k + j;
            const int e = a.idx[s];
            if (e < 0 || e >= a.E) continue;
            const float4 v = reinterpret_cast<const float4*>(a.ys + (int64_t)s * a.H)[c4];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        reinterpret_cast<float4*>(a.y + (int64_t)t * a.H)[c4] = acc;
    }
}

// tile_off[e] = sum over e' < e of ceil(counts[e'] / nt); one CTA, E <= 1024.
__global__ void __launch_bounds__(1024) tc_tile_prefix_kernel(const int32_t* __restrict__ counts, int E, int nt,
                                                              int32_t* __restrict__ tile_off) {
    __shared__ int32_t part[32];
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v = tid < E ? (counts[tid] + nt - 1) / nt : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) part[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int p = part[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFullMask, p, o);
            if (lane >= o) p += n;
        }
        part[lane] = p;
    }
    __syncthreads();
    const int excl = (warp > 0 ? part[warp - 1] : 0) + incl - v;
    if (tid < E) tile_off[tid] = excl;
    if (tid == E - 1) tile_off[E] = excl + v;
}

}  // namespace

// Token-tile width of a call: 128 when the slots average at least 64 per expert
// (prefill), 16 otherwise (decode batches: fewer padded MMA columns and a smaller
// TMEM allocation, so that two CTAs share an SM).
int ffn_tensor_tile_tokens(int S, int E) { return (int64_t)S >= 64 * (int64_t)E ? 128 : 16; }

// An upper bound of the number of tiles, sum over experts of ceil(n_e / NT).
int ffn_tensor_max_tiles(int S, int E) {
    const int nt = ffn_tensor_tile_tokens(S, E);
    return (S + nt - 1) / nt + (E < S ? E : S);
}

// MAPLE_FFN_PATH=tensor or =cores forces a path (for parity tests of both on the same
// inputs); otherwise the tensor path runs once there are at least half as many slots
// as experts (on the Maple layer, 16 tokens and up: measured faster than the CUDA-core
// kernels from there on, slower below).
bool ffn_use_tensor(int T, int k, int E, int H, int I) {
    if (!ffn_tensor_shape_ok(H, I) || T < 1) return false;
    const char* env = getenv("MAPLE_FFN_PATH");
    if (env != nullptr && strcmp(env, "tensor") == 0) return true;
    if (env != nullptr && strcmp(env, "cores") == 0) return false;
    return 2 * (int64_t)T * k >= (int64_t)E;
}

// H a multiple of the 128 down rows of a CTA, I of the 64 gate (and up) rows; both at
// least 128 so that a B box (10 chunks of 8 values) fits inside a row.
bool ffn_tensor_shape_ok(int H, int I) {
    return H % kRows == 0 && I % (kRows / 2) == 0 && H >= 128 && I >= 128 && H <= 2080 && I <= 2080;
}

size_t ffn_tensor_x_bytes(int S, int E, int H) {
    const int nt = ffn_tensor_tile_tokens(S, E);
    return (size_t)ffn_tensor_max_tiles(S, E) * H * nt * 2;
}

size_t ffn_tensor_h_bytes(int S, int E, int I) {
    const int nt = ffn_tensor_tile_tokens(S, E);
    return (size_t)ffn_tensor_max_tiles(S, E) * I * nt * 2;
}

namespace {

template <int NT>
cudaError_t launch_tc_ffn(const TcArgs& a, int S, cudaStream_t stream) {
    const int tiles = ffn_tensor_max_tiles(S, a.E);
    const int Bh = (a.H + 4) / 5, Bi = (a.I + 4) / 5;
    const size_t smem_gu = tc_smem_bytes<NT>(Bh), smem_dn = tc_smem_bytes<NT>(Bi);
    auto gu = tc_gateup_kernel<NT>;
    auto dn = tc_down_kernel<NT>;
    cudaError_t err = ensure_dynamic_smem(gu, smem_gu);
    if (err != cudaSuccess) return err;
    err = ensure_dynamic_smem(dn, smem_dn);
    if (err != cudaSuccess) return err;
    err = launch_pdl(tc_gather_kernel<NT>, dim3(tiles), dim3(256), 0, stream, a);
    if (err != cudaSuccess) return err;
    err = launch_pdl(gu, dim3(a.I / (kRows / 2), tiles), dim3(kThreads), smem_gu, stream, a);
    if (err != cudaSuccess) return err;
    return launch_pdl(dn, dim3(a.H / kRows, tiles), dim3(kThreads), smem_dn, stream, a);
}

}  // namespace

cudaError_t launch_moe_ffn_tensor(const FfnArgs& f, cudaStream_t stream, const DeviceInfo& dev) {
    const int S = f.T * f.k;
    const int nt = ffn_tensor_tile_tokens(S, f.E);
    // one CTA groups a few thousand slots fastest; beyond that, chunks in parallel
    cudaError_t err = S > 4096 ? launch_group_tokens_chunked(f.idx, S, f.E, f.counts, f.offsets, f.perm, f.active,
                                                             f.n_active, f.chunks, stream)
                               : launch_group_tokens(f.idx, S, f.k, f.E, f.counts, f.offsets, f.perm, f.active,
                                                     f.n_active, stream, dev);
    if (err != cudaSuccess) return err;
    err = launch_pdl(tc_tile_prefix_kernel, dim3(1), dim3(1024), 0, stream, (const int32_t*)f.counts, f.E, nt,
                     f.tile_off);
    if (err != cudaSuccess) return err;
    TcArgs a;
    a.gate = f.gate;
    a.up = f.up;
    a.down = f.down;
    a.s_gate = f.s_gate;
    a.s_up = f.s_up;
    a.s_down = f.s_down;
    a.E = f.E;
    a.H = f.H;
    a.I = f.I;
    a.k = f.k;
    a.clamp = f.clamp;
    a.x = f.x;
    a.w = f.w;
    a.idx = f.idx;
    a.counts = f.counts;
    a.offsets = f.offsets;
    a.perm = f.perm;
    a.tile_off = f.tile_off;
    a.xs = f.xs;
    a.hs = f.hs;
    a.ys = f.ys;
    a.y = f.y;
    a.T = f.T;
    a.status = f.status;
    err = nt == 128 ? launch_tc_ffn<128>(a, S, stream) : launch_tc_ffn<16>(a, S, stream);
    if (err != cudaSuccess) return err;
    const int64_t work = (int64_t)f.T * (f.H / 4);
    const int64_t want = (work + 255) / 256;
    const int64_t cap = (int64_t)dev.sm_count * 8;
    return launch_pdl(tc_combine_kernel, dim3((unsigned)(want < cap ? want : cap)), dim3(256), 0, stream, a);
}

}  // namespace maple
