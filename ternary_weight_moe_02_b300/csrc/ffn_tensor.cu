// Expert FFN on the tcgen05 tensor cores (grouped path: tokens batched per expert).
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// sections "The claim, verified from the bytes" (one scale per output row, trits
// -1/0/+1) and "The shipped code does no quantization" (the expert body
// down(act(clamp(gate x, max=7)) * clamp(up x, -7, 7))).  The pages give no kernel for
// many tokens per expert.  Here the sums run on the tensor cores as fp8 (e4m3) MMAs
// with fp32 accumulation, without rounding the operands:
//   * a trit -1 / 0 / +1 is exact in e4m3;
//   * a bf16 row (of x, or of h) whose largest magnitude lies in [2^e, 2^(e+1)) gets the
//     power-of-two scale s = 2^(e - 7); each value v is split into two e4m3 values with
//     v = s (hi + lo): hi is v / s rounded to e4m3 (four significant bits) and lo the
//     rest, also an e4m3 value.  Both are exact whenever |v / s| >= 2^-2 (bf16 carries
//     eight significant bits); smaller values keep their bits down to s 2^-9;
//   * the MMA multiplies the trits by the hi and by the lo rows as separate columns of
//     one product, and the epilogue adds the two accumulators and applies s.
//
// Per expert e with n_e routed tokens (slots grouped by expert, tiles of NT tokens;
// NT = 64 for prefill-sized calls, 16 for decode batches):
//   split x: each tile's token rows of x into hi/lo rows and scales;
//   gate/up item: D[128 x 2NT] = A . B^T, A = 64 gate rows and the same 64 up rows of e
//     (interleaved), B = the tile's hi rows then its lo rows; epilogue
//     h = silu(min(s_g g, clamp)) * clamp(s_u u, -clamp, clamp), rounded to bf16 and
//     stored by grouped position;
//   split h: each tile's h rows into hi/lo rows and scales, as for x;
//   down item: D[128 x 2NT] = A_down . B^T over I; epilogue w_slot * s_d * s_h * D per
//     slot (fp32); a combine kernel adds each token's k slots in order 0..k-1.
//
// A is decoded from the packed bytes straight into tensor memory: the thread of TMEM
// lane r decodes that lane's weight row and writes its K values as e4m3, four per
// 32-bit column (K order from the low byte), with tcgen05.st; the MMA reads A from
// tensor memory.  B sits in shared memory K-major without swizzle: byte (n, k) of a
// stage at (k / 16) * (2NT * 16) + n * 16 + k % 16.  The split kernels store each
// tile's rows in global memory in that order ([K / 16][2NT][16] bytes), so a stage of B
// is one contiguous block loaded by one 1-D bulk copy.  The gate/up and down items run
// in the persistent streaming kernels below.  All waits are bounded.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace maple {

namespace {

constexpr int kRows = 128;                 // MMA M: weight rows of an item
constexpr int kKTile = 160;                // K values of 32 packed bytes
constexpr int kLutReps = 16;               // copies of the decode table, by lane & 15
constexpr int kLutBytes = 256 * kLutReps * 8;  // 32 KB

// ----------------------------------------------------------------- tcgen05 helpers
// (allocation, fences, descriptors, commits and loads: tcgen05.cuh)

// D[tmem] (+)= A[tmem] . B[smem descriptor], e4m3 x e4m3 -> fp32
__device__ __forceinline__ void mma_f8_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
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



// ----------------------------------------------------------------- e4m3 split

// Two floats to two e4m3, rounded to nearest even with saturation; byte 0 from a.
__device__ __forceinline__ uint32_t e4m3x2_from(float a, float b) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(b), "f"(a));
    return d;
}

// The two e4m3 values in bytes 0 and 1 of p, exactly, as floats.
__device__ __forceinline__ void e4m3x2_to(uint32_t p, float& a, float& b) {
    asm("{\n.reg .b32 h2;\n.reg .b16 lo, hi;\n"
        "cvt.rn.f16x2.e4m3x2 h2, %2;\n"
        "mov.b32 {lo, hi}, h2;\n"
        "cvt.f32.f16 %0, lo;\n"
        "cvt.f32.f16 %1, hi;\n}\n"
        : "=f"(a), "=f"(b)
        : "h"((uint16_t)p));
}

// The split scale 2^(e - 7) of a row whose largest magnitude m lies in [2^e, 2^(e+1))
// (1 for an all-zero row; e held to [-100, 127] so that 1 / s stays finite).
__device__ __forceinline__ float split_scale(float m) {
    if (!(m > 0.f)) return 1.f;
    int e = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;
    e = e < -100 ? -100 : (e > 127 ? 127 : e);
    return ldexpf(1.f, e - 7);
}

// Eight values (already divided by the row's scale) into eight hi and eight lo bytes.
__device__ __forceinline__ void split8(const float* v, uint2& hi, uint2& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        h[p] = e4m3x2_from(v[2 * p], v[2 * p + 1]);
        float b0, b1;
        e4m3x2_to(h[p], b0, b1);
        l[p] = e4m3x2_from(v[2 * p] - b0, v[2 * p + 1] - b1);
    }
    hi = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    lo = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}

// ----------------------------------------------------------------- decode table

// For each code, the e4m3 values of its five trits (0xB8 = -1, 0x00 = 0, 0x38 = +1) in
// bytes 0-4, bytes 5-7 zero; the invalid codes 243..255 give five zeros.  kLutReps
// copies interleaved by entry ([code][copy], 8 bytes): copy lane & 15 of a warp's 32
// loads falls in bank pair 2 (lane & 15), so a load takes the minimum two wavefronts.
// Built at compile time; every CTA bulk-copies it into shared memory.
struct F8LutImage {
    uint32_t word[256 * kLutReps * 2];
};

constexpr F8LutImage make_f8_lut_image() {
    F8LutImage t{};
    for (int c = 0; c < 256; ++c) {
        uint32_t b[5] = {0u, 0u, 0u, 0u, 0u};
        if (c < 243) {
            int code = c;
            for (int i = 0; i < 5; ++i) {
                const int d = code % 3;
                code /= 3;
                b[i] = d == 0 ? 0xB8u : (d == 2 ? 0x38u : 0u);
            }
        }
        for (int r = 0; r < kLutReps; ++r) {
            t.word[2 * (c * kLutReps + r)] = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
            t.word[2 * (c * kLutReps + r) + 1] = b[4];
        }
    }
    return t;
}

__device__ __align__(16) const F8LutImage g_f8_lut_image = make_f8_lut_image();
static_assert(sizeof(F8LutImage) == kLutBytes, "table image size");

// Shared-memory loads at 32-bit shared addresses (the decode's operands always live
// in shared memory; the explicit form keeps them off the generic path).
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

// Bytes [A, A + 16) of the packed rows (shared address base_s, 16-byte aligned) as four
// words, from five aligned word loads and funnel shifts.  Reads up to 3 bytes past
// A + 16.
__device__ __forceinline__ void load_bytes16(uint32_t base_s, uint32_t A, uint32_t* a) {
    const uint32_t w = base_s + (A & ~3u);
    const uint32_t sh = (A & 3u) * 8;
    uint32_t t[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) t[i] = lds32(w + 4 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = __funnelshift_r(t[i], t[i + 1], sh);
}

// Decodes bytes [b0, b0 + 16) of the row at byte offset row_off of the packed rows
// (shared address packed_s; bytes at or past rb read as the all-zero code 121) into 20
// words of four e4m3 each, in K order: every four codes (twenty values) become five
// words by byte permutes of their table entries (lut_s: this lane's copy of entry 0).
template <bool kTail>
__device__ __forceinline__ void decode_half_tile_impl(uint32_t packed_s, uint32_t row_off, int rb, int b0,
                                                      uint32_t lut_s, uint32_t* words) {
    uint32_t a[4];
    load_bytes16(packed_s, row_off + (uint32_t)b0, a);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint2 en[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t c = (a[g] >> (8 * i)) & 0xFFu;
            if (kTail && b0 + 4 * g + i >= rb) c = 121u;
            en[i] = lds64(lut_s + c * (kLutReps * 8));
        }
        words[5 * g + 0] = en[0].x;                                // values 0-3 of code 0
        words[5 * g + 1] = __byte_perm(en[0].y, en[1].x, 0x6540);  // 0.4, 1.0, 1.1, 1.2
        words[5 * g + 2] = __byte_perm(__byte_perm(en[1].x, en[1].y, 0x0043), en[2].x, 0x5410);  // 1.3, 1.4, 2.0, 2.1
        words[5 * g + 3] = __byte_perm(__byte_perm(en[2].x, en[2].y, 0x0432), en[3].x, 0x4210);  // 2.2-2.4, 3.0
        words[5 * g + 4] = __byte_perm(en[3].x, en[3].y, 0x4321);  // 3.1-3.4
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
    const int4* tile_info;    // [tiles] expert, first token, tokens, first grouped position
    uint8_t* xs;              // [tile][H / 16][2NT][16] e4m3: each tile's x rows, hi then lo
    uint8_t* hs;              // [tile][I / 16][2NT][16] e4m3: each tile's h rows, hi then lo
    float* xscale;            // [tile][NT] split scales of the x rows
    float* hscale;            // [tile][NT] split scales of the h rows
    uint16_t* hrow;           // [T k][I] bf16 h by grouped position
    float* ys;                // [T k][H] fp32, per original slot
    float* y;                 // [T][H]
    int T;
    int* status;
};

// Finds the expert and token range of grid row `tile`; false when past the last tile.
// The tile table comes from a kernel that completed before the previous one started,
// so it is read (through L2) before this grid's PDL wait; both loads are in flight at
// once.
template <int NT>
__device__ __forceinline__ bool tc_tile(const TcArgs& a, int tile, int& e, int& n0, int& nv, int& pos0) {
    const int total = __ldcg(a.tile_off + a.E);
    const int4 info = __ldcg(a.tile_info + tile);
    if (tile >= total) return false;
    e = info.x;
    n0 = info.y;
    nv = info.z;
    pos0 = info.w;
    return nv > 0;
}

// Columns [c0, c0 + CB) of this thread's lane plus columns [NT + c0, NT + c0 + CB):
// the hi and lo accumulators of CB tokens, summed (all loads issued, then one wait).
template <int NT, int CB>
__device__ __forceinline__ void tmem_ld_sum(uint32_t lane_addr, int c0, float* v) {
    static_assert(CB % 16 == 0, "blocks of 16 columns");
    uint32_t hi[CB], lo[CB];
#pragma unroll
    for (int i = 0; i < CB; i += 16) {
        tmem_ld16(lane_addr + (uint32_t)(c0 + i), hi + i);
        tmem_ld16(lane_addr + (uint32_t)(NT + c0 + i), lo + i);
    }
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < CB; ++i) v[i] = __uint_as_float(hi[i]) + __uint_as_float(lo[i]);
}

// ----------------------------------------------------------------- streaming kernels
//
// Grouped tiles of NT = 16 (decode batches) or 64 (prefill) tokens, through one
// persistent CTA per SM per stage, with the work of consecutive items overlapped
// instead of a CTA per item run start to finish.  An item is one 128-row block of one
// tile: for gate/up the 64 gate and the same 64 up rows of block b of the tile's
// expert, for down 128 down rows.  CTA c takes items c, c + grid, c + 2 grid, ... .
// The K dimension moves through a ring of stages of kSuper K tiles each (A in tensor
// memory, B in shared memory), one "full" barrier per stage for both operands, so that
// the MMA thread waits once and issues 5 kSuper MMAs per stage.  Roles (warps):
//   0-15  producers: decode A into the ring, stage after stage across item boundaries:
//         thread (w, lane) owns TMEM lane 32 (w & 3) + lane and packed bytes
//         [16 (w >> 2), +16) of each 64-byte stage of that lane's row;
//   16    lane 0 issues the MMAs into one of kAccs accumulators (item it into
//         it % kAccs), commits each stage back to its producers and each item to the
//         epilogue; the warp owns the tensor memory;
//   17    lane 0 copies the items' packed rows into npk buffers, as far ahead as the
//         producers free them (weights: issued before the PDL wait);
//   18    lane 0 copies the tiles' B operands (split x or h) into the ring;
//   19-   epilogue (4 warps, or 8 on 64-token tiles): drain the item's accumulator (TMEM
//         lane quarter warp % 4) 16 tokens at a time, free it, and finish the item as
//         the per-item kernels do.
// Gate/up items interleave their rows in tensor memory: lane 2j holds gate row j and
// lane 2j + 1 the same up row, so that the two values h needs meet in one warp (a
// shuffle) instead of in shared memory.
// One MMA of M = 128, K = 32 occupies the tensor pipe about as long at N = 32 as at
// N = 128 (about 100 cycles, measured), so 64-token tiles (N = 128) cost about as much
// per MMA as 16-token ones and do four times the work.
// Every wait is bounded; a wait that gives up records MAPLE_ERR_TIMEOUT and raises a
// CTA-wide abort flag that ends the other roles' waits, after which copies and MMAs
// still in flight are waited for before the CTA frees its tensor memory and exits.
constexpr int kPsProducers = 16;             // producer warps
constexpr int kPsMmaWarp = 16, kPsPackWarp = 17, kPsBWarp = 18, kPsEpiWarp0 = 19;
constexpr int kPsMaxPacked = 4;              // packed-row buffers (at least 2)
constexpr int kPsMaxStages = 4;
constexpr int kPsMaxAccs = 4;
constexpr int kPsTmemCols = 512;
constexpr int kPsAccCol = 256;               // accumulators in [256, 512), A stages below:
                                             // A operands above column 256 measured slower

template <int NT>
struct PsCfg {
    static constexpr int kN = 2 * NT;                         // MMA N: hi and lo rows
    static constexpr int kSuper = 2;                          // K tiles per ring stage
    static constexpr int kKS = kSuper * kKTile;               // K values per stage
    static constexpr int kRowBytesS = kKS / 5;                // packed bytes of a row per stage
    static constexpr int kChunksS = kKS / 16;                 // B chunks per stage
    static constexpr int kStageB = kChunksS * kN * 16;        // bytes of a B stage
    static constexpr int kStageCols = kKS / 4;                // A columns per stage
    static constexpr int kStages = NT <= 16 ? 3 : 2;          // ring depth (shared memory)
    static constexpr int kAccs = 256 / kN < kPsMaxAccs ? 256 / kN : kPsMaxAccs;
    // epilogue warps: one per tensor-memory lane quarter, two (taking alternate groups
    // of 16 tokens) when a tile has several groups
    static constexpr int kEpiWarps = NT >= 32 ? 8 : 4;
    static constexpr int kEpiThreads = 32 * kEpiWarps;
    static constexpr int kThreads = 32 * kPsEpiWarp0 + kEpiThreads;
    // instruction descriptor as in TileCfg: D fp32, A and B e4m3, both K-major, N, M = 128
    static constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
    static_assert(kRowBytesS == 4 * 16, "four producer parts of 16 bytes per stage row");
    static_assert(kStages * kStageCols <= kPsAccCol && kAccs * kN <= kPsTmemCols - kPsAccCol, "tensor memory");
    static_assert(kStages <= kPsMaxStages && kAccs >= 2 && NT % 16 == 0 && NT <= 64, "plan");
};

struct PsBars {
    uint64_t pk_full[kPsMaxPacked], pk_empty[kPsMaxPacked];
    uint64_t full[kPsMaxStages], empty[kPsMaxStages];
    uint64_t acc_full[kPsMaxAccs], acc_empty[kPsMaxAccs];
    uint64_t lut, fin;
    int abort;
};

// Shared-memory plan: decode table, npk packed-row buffers of pk_stride bytes, the B ring.
__host__ __device__ constexpr size_t ps_pk_stride(int row_bytes) { return ((size_t)kRows * row_bytes + 127) / 128 * 128; }
__host__ __device__ constexpr size_t ps_b_offset(int row_bytes, int npk) {
    return (size_t)kLutBytes + (size_t)npk * ps_pk_stride(row_bytes);
}
template <int NT>
__host__ __device__ constexpr size_t ps_smem_bytes(int row_bytes, int npk) {
    return ps_b_offset(row_bytes, npk) + (size_t)PsCfg<NT>::kStages * PsCfg<NT>::kStageB;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded waits that also end when another role has raised the abort flag.  The spin
// form (single-thread roles whose waits are short) polls without suspending, up to
// about 4e9 cycles; the other tests once, then suspends between polls.
__device__ __noinline__ bool ps_give_up(int* status, volatile int* abort) {
    *abort = 1;
    if (status != nullptr) atomicExch(status, kStatusTimeout);
    return false;
}
__device__ __forceinline__ bool ps_wait_spin(uint64_t* bar, uint32_t parity, int* status, volatile int* abort) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (clock64() - t0 < 4000000000ll) {
        if (mbar_test_wait(bar, parity)) return true;
        if (*abort) return false;
    }
    return ps_give_up(status, abort);
}
__device__ __forceinline__ bool ps_wait(uint64_t* bar, uint32_t parity, int* status, volatile int* abort) {
    if (mbar_test_wait(bar, parity)) return true;
    for (uint32_t i = 0; i < kWaitPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
    }
    return ps_give_up(status, abort);
}

// Whether any of the kThreads epilogue threads (named barrier 1) passes pred = true;
// all of them must call it.
template <int kThreads>
__device__ __forceinline__ bool bar_any_epi(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\n"
        "setp.ne.u32 q, %1, 0;\n"
        "bar.red.or.pred p, 1, %2, q;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(kThreads)
        : "memory");
    return r != 0;
}

// Bytes [b0, b0 + 16) of a row (zeros at and past rb) as 20 words of e4m3.
__device__ __forceinline__ void ps_decode16(uint32_t packed_s, uint32_t row_off, int rb, int b0, uint32_t lut_s,
                                            uint32_t* words) {
    if (b0 + 16 <= rb)
        decode_half_tile_impl<false>(packed_s, row_off, rb, b0, lut_s, words);
    else
        decode_half_tile_impl<true>(packed_s, row_off, rb, b0, lut_s, words);
}

template <int NT, bool kDown>
__global__ void __launch_bounds__(PsCfg<NT>::kThreads, 1) tc_stream_kernel(TcArgs a, int npk) {
    using Cfg = PsCfg<NT>;
    constexpr int S = Cfg::kStages, NACC = Cfg::kAccs;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ PsBars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ float2 s_tok[NACC][NT];  // per-token epilogue values of the items in flight
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, I = a.I;
    const int Kdim = kDown ? I : H;
    const int rb = (Kdim + 4) / 5;                     // packed bytes per row
    const int nblk = kDown ? H / kRows : I / (kRows / 2);
    const int NS = (Kdim + Cfg::kKS - 1) / Cfg::kKS;   // ring stages per item
    // the tile table is complete before this grid starts (see tc_tile)
    const int n_items = __ldcg(a.tile_off + a.E) * nblk;
    if ((int)blockIdx.x >= n_items) return;
    const int stride = gridDim.x;
    const size_t pk_stride = ps_pk_stride(rb);
    unsigned char* pk0 = smem + kLutBytes;
    unsigned char* bring = smem + ps_b_offset(rb, npk);
    volatile int* abort = &bars.abort;
    if (warp == kPsMmaWarp) {
        if (lane == 0) {
            for (int i = 0; i < kPsMaxPacked; ++i) {
                mbar_init(&bars.pk_full[i], 1);
                mbar_init(&bars.pk_empty[i], kPsProducers * 32);
            }
            for (int i = 0; i < S; ++i) {
                mbar_init(&bars.full[i], kPsProducers * 32 + 1);  // producers + the B copy
                mbar_init(&bars.empty[i], 1);
            }
            for (int i = 0; i < NACC; ++i) {
                mbar_init(&bars.acc_full[i], 1);
                mbar_init(&bars.acc_empty[i], Cfg::kEpiThreads);
            }
            mbar_init(&bars.lut, 1);
            mbar_init(&bars.fin, 1);
            bars.abort = 0;
        }
        __syncwarp();
        tmem_alloc(&tmem_slot, kPsTmemCols);
    }
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp < kPsProducers) {
        // ---- producers.  Waits are taken by every lane and voted on, so that the warp
        // stays converged for the .sync.aligned tensor-memory stores.
        const int q = warp & 3, part = warp >> 2, r = 32 * q + lane;
        // packed row of TMEM lane r: gate/up rows interleaved (gate j at 2j, up j at 2j + 1)
        const int prow = kDown ? r : ((r & 1) ? kRows / 2 + (r >> 1) : (r >> 1));
        const uint32_t row_off = (uint32_t)(prow * rb);
        const uint32_t lut_s = smem_addr(smem) + 8u * (uint32_t)(lane & (kLutReps - 1));
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(kFullMask, ps_wait(bar, parity, a.status, abort));
        };
        bool ok = wait_all(&bars.lut, 0) && wait_all(&bars.pk_full[0], 0);
        // ring stage s of fill round `round` (its empty barrier is waited for from the
        // second round on, parity (round - 1) & 1); packed-row buffer pk of the item and
        // the parity of its full barrier; the decoded words alternate between wa and wb
        int it = 0, st = 0, s = 0, round = 0, pk = 0;
        uint32_t pk_ph = 0;
        const uint32_t pk_base = smem_addr(pk0);
        uint32_t pk_addr = pk_base;
        uint32_t wa[20], wb[20];
        if (ok) ps_decode16(pk_addr, row_off, rb, 16 * part, lut_s, wa);
        // stores `cur` into stage s, decodes the next stage into `nxt`; false when this
        // CTA has no further stage (or a wait gave up)
        auto step = [&](const uint32_t* cur, uint32_t* nxt) {
            if (round > 0 && !wait_all(&bars.empty[s], (uint32_t)((round - 1) & 1))) {
                ok = false;
                return false;
            }
            const uint32_t col = (uint32_t)(s * Cfg::kStageCols + 20 * part);
            tmem_st16(lane_base + col, cur);
            tmem_st4(lane_base + col + 16, cur + 16);
            bool more = true;
            if (st + 1 < NS) {
                ++st;
                ps_decode16(pk_addr, row_off, rb, Cfg::kRowBytesS * st + 16 * part, lut_s, nxt);
            } else {
                mbar_arrive(&bars.pk_empty[pk]);  // this item's packed rows are read
                ++it;
                st = 0;
                if (++pk == npk) {
                    pk = 0;
                    pk_ph ^= 1u;
                }
                pk_addr = pk_base + (uint32_t)((size_t)pk * pk_stride);
                more = (int)blockIdx.x + it * stride < n_items;
                if (more && !wait_all(&bars.pk_full[pk], pk_ph)) more = false;
                if (more) ps_decode16(pk_addr, row_off, rb, 16 * part, lut_s, nxt);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(&bars.full[s]);
            if (++s == S) {
                s = 0;
                ++round;
            }
            return more;
        };
        while (ok) {
            if (!step(wa, wb) || !step(wb, wa)) break;
        }
    } else if (warp == kPsMmaWarp) {
        // ---- MMA issue
        if (lane == 0) {
            // ring stage s and its phase ph; B descriptors step through the start-address
            // field (shared addresses below 256 KB: no carry out of it)
            int s = 0;
            uint32_t ph = 0;
            const uint64_t bdesc0 = smem_desc(smem_addr(bring), Cfg::kN * 16, 128);
            constexpr uint64_t kQkStep = (uint64_t)((2 * Cfg::kN * 16) >> 4);
            constexpr uint64_t kStStep = (uint64_t)(Cfg::kStageB >> 4);
            const int nq_last = (Kdim - (NS - 1) * Cfg::kKS) / 32;
            bool ok = true;
            for (int it = 0; ok && (int)blockIdx.x + it * stride < n_items; ++it) {
                const int acc = it % NACC;
                if (it >= NACC &&
                    !ps_wait_spin(&bars.acc_empty[acc], (uint32_t)((it / NACC - 1) & 1), a.status, abort))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(kPsAccCol + acc * Cfg::kN);
                for (int st = 0; st < NS; ++st) {
                    if (!ps_wait_spin(&bars.full[s], ph, a.status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = tmem + (uint32_t)(s * Cfg::kStageCols);
                    const uint64_t bd = bdesc0 + (uint64_t)s * kStStep;
                    // only the K range the stage's copy filled (Kdim is a multiple of 32):
                    // the rest of a B stage may hold another tile's rows, whose padding
                    // rows are not guaranteed finite
                    const int nq = st == NS - 1 ? nq_last : Cfg::kKS / 32;
#pragma unroll
                    for (int qk = 0; qk < Cfg::kKS / 32; ++qk)
                        if (qk < nq)
                            mma_f8_tmem_a(d, a0 + 8 * qk, bd + qk * kQkStep, Cfg::kIdesc, (st | qk) != 0 ? 1u : 0u);
                    mma_commit(&bars.empty[s]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) mma_commit(&bars.acc_full[acc]);
            }
            // every MMA issued has completed before the tensor memory is freed
            mma_commit(&bars.fin);
            mbar_wait_bounded(&bars.fin, 0, a.status);
        }
        __syncwarp();
    } else if (warp == kPsPackWarp) {
        // ---- packed rows (weights: no dependence on the previous kernel)
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars.lut, (uint32_t)kLutBytes);
            bulk_copy_g2s(smem, &g_f8_lut_image, (uint32_t)kLutBytes, &bars.lut);
            int it = 0;
            for (; (int)blockIdx.x + it * stride < n_items; ++it) {
                const int p = it % npk;
                if (it >= npk && !ps_wait_spin(&bars.pk_empty[p], (uint32_t)((it / npk - 1) & 1), a.status, abort))
                    break;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // reads done -> refill
                const int item = (int)blockIdx.x + it * stride;
                const int4 info = __ldcg(a.tile_info + item / nblk);
                const int blk = item % nblk;
                unsigned char* dst = pk0 + (size_t)p * pk_stride;
                if (kDown) {
                    const uint32_t bytes = (uint32_t)(kRows * rb);
                    mbar_arrive_expect_tx(&bars.pk_full[p], bytes);
                    bulk_copy_g2s(dst, a.down + ((int64_t)info.x * H + (int64_t)blk * kRows) * rb, bytes,
                                  &bars.pk_full[p]);
                } else {
                    const uint32_t bytes = (uint32_t)((kRows / 2) * rb);
                    const int64_t r0 = (int64_t)info.x * I + (int64_t)blk * (kRows / 2);
                    mbar_arrive_expect_tx(&bars.pk_full[p], 2 * bytes);
                    bulk_copy_g2s(dst, a.gate + r0 * rb, bytes, &bars.pk_full[p]);
                    bulk_copy_g2s(dst + bytes, a.up + r0 * rb, bytes, &bars.pk_full[p]);
                }
            }
            // copies still in flight land before the CTA leaves
            mbar_wait_bounded(&bars.lut, 0, nullptr);
            for (int j = it - npk > 0 ? it - npk : 0; j < it; ++j)
                mbar_wait_bounded(&bars.pk_full[j % npk], (uint32_t)((j / npk) & 1), nullptr);
        }
        __syncwarp();
    } else if (warp == kPsBWarp) {
        // ---- B operands (written by the previous kernel)
        pdl_wait();
        if (lane == 0) {
            const uint8_t* bbase = kDown ? a.hs : a.xs;
            uint32_t g = 0;
            bool ok = true;
            for (int it = 0; ok && (int)blockIdx.x + it * stride < n_items; ++it) {
                const int tile = ((int)blockIdx.x + it * stride) / nblk;
                const uint8_t* bsrc = bbase + (size_t)tile * Kdim * Cfg::kN;
                for (int st = 0; st < NS; ++st, ++g) {
                    const int s = (int)(g % S);
                    if (g >= (uint32_t)S && !ps_wait_spin(&bars.empty[s], ((g / S) - 1) & 1, a.status, abort)) {
                        ok = false;
                        break;
                    }
                    const int left = Kdim / 16 - st * Cfg::kChunksS;
                    const uint32_t bytes = (uint32_t)((left < Cfg::kChunksS ? left : Cfg::kChunksS) * Cfg::kN * 16);
                    mbar_arrive_expect_tx(&bars.full[s], bytes);
                    bulk_copy_g2s(bring + (size_t)s * Cfg::kStageB, bsrc + (size_t)st * Cfg::kStageB, bytes,
                                  &bars.full[s]);
                }
            }
            // the last copy into each stage lands before the CTA leaves
            for (uint32_t j = g > (uint32_t)S ? g - S : 0u; j < g; ++j)
                mbar_wait_bounded(&bars.full[j % S], (j / S) & 1, nullptr);
        }
        __syncwarp();
    } else {
        // ---- epilogue: TMEM lane quarter warp % 4, lane r of the item's 128; with eight
        // epilogue warps the two of a quarter take alternate groups of 16 tokens
        pdl_wait();
        const int q = warp & 3, r = 32 * q + lane;
        const int half = Cfg::kEpiWarps > 4 ? (warp - kPsEpiWarp0) >> 2 : 0;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16);
        const bool up_side = !kDown && (r & 1);
        // An item's per-item values are loaded one item ahead, so that their dependent
        // global loads overlap the previous item's work: each thread's row scale, and
        // the per-token values, which the first epilogue warp loads into registers and
        // publishes in shared memory once the previous item is stored (the named
        // barrier of the item orders them): the x split scale (gate/up), or the slot and
        // the routing weight times the h split scale (down).
        constexpr int TPL = (NT + 31) / 32;  // per-token values a lane of that warp loads
        auto valid = [&](int it) { return (int)blockIdx.x + it * stride < n_items; };
        auto record = [&](int it) {
            return valid(it) ? __ldcg(a.tile_info + ((int)blockIdx.x + it * stride) / nblk) : make_int4(0, 0, 0, 0);
        };
        auto load_tokens = [&](int it, int4 info, float2* tv) {
            const int tile = ((int)blockIdx.x + it * stride) / nblk, nv = valid(it) ? info.z : 0, pos0 = info.w;
#pragma unroll
            for (int u = 0; u < TPL; ++u) {
                const int t = lane + 32 * u;
                tv[u] = make_float2(0.f, 0.f);
                if (t < NT && t < nv) {
                    if (kDown) {
                        const int slot = __ldcg(a.perm + pos0 + t);
                        tv[u] = make_float2(__int_as_float(slot), __ldcg(a.w + slot) * a.hscale[(size_t)tile * NT + t]);
                    } else {
                        tv[u].x = a.xscale[(size_t)tile * NT + t];
                    }
                }
            }
        };
        auto publish = [&](int it, const float2* tv) {
#pragma unroll
            for (int u = 0; u < TPL; ++u)
                if (lane + 32 * u < NT) s_tok[it % NACC][lane + 32 * u] = tv[u];
        };
        auto load_row_scale = [&](int it, int4 info) {
            if (!valid(it)) return 0.f;
            const int blk = ((int)blockIdx.x + it * stride) % nblk, e = info.x;
            return kDown ? a.s_down[(int64_t)e * H + blk * kRows + r]
                         : (up_side ? a.s_up[(int64_t)e * I + blk * (kRows / 2) + (r >> 1)]
                                    : a.s_gate[(int64_t)e * I + blk * (kRows / 2) + (r >> 1)]);
        };
        int4 info_cur = record(0), info_nxt = record(1);
        float row_scale_cur = load_row_scale(0, info_cur);
        {
            float2 tv0[TPL];
            if (warp == kPsEpiWarp0) {
                load_tokens(0, info_cur, tv0);
                publish(0, tv0);
            }
        }
        for (int it = 0; valid(it); ++it) {
            const int item = (int)blockIdx.x + it * stride;
            const int blk = item % nblk, acc = it % NACC;
            const int nv = info_cur.z, pos0 = info_cur.w;
            const float row_scale = row_scale_cur;
            const int m = kDown ? blk * kRows : blk * (kRows / 2);
            const int j = kDown ? r : (r >> 1);  // down row, or gate/up row pair
            // the next item's values, in flight while this one is finished
            const int4 info_after = record(it + 2);
            const float row_scale_nxt = load_row_scale(it + 1, info_nxt);
            float2 tv_nxt[TPL];
            if (warp == kPsEpiWarp0) load_tokens(it + 1, info_nxt, tv_nxt);
            // one decision for all epilogue threads (they meet at a named barrier)
            const bool got = ps_wait(&bars.acc_full[acc], (uint32_t)((it / NACC) & 1), a.status, abort);
            if (bar_any_epi<Cfg::kEpiThreads>(!got)) break;
            tc_fence_after();
            const uint32_t base = lane_addr + (uint32_t)(kPsAccCol + acc * Cfg::kN);
#pragma unroll 1
            for (int b = half; b < NT / 16; b += Cfg::kEpiWarps / 4) {
                float v[16];
                tmem_ld_sum<NT, 16>(base, 16 * b, v);
                if (kDown) {
                    float* yr = a.ys + m + r;
                    // every shared-memory read before the first store: the stores go
                    // through a generic pointer, which the compiler cannot tell apart
                    // from shared memory, so interleaving them would serialise the loop
                    float2 tv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) tv[i] = s_tok[acc][16 * b + i];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (16 * b + i < nv) yr[(int64_t)__float_as_int(tv[i].x) * H] = tv[i].y * (row_scale * v[i]);
                } else {
                    // gate lane keeps tokens 16b..16b+7, the up lane 16b+8..16b+15; each
                    // hands the other half to its partner lane (r ^ 1)
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float tt = row_scale * s_tok[acc][16 * b + i].x * v[i];
                        v[i] = fminf(up_side ? fmaxf(tt, -a.clamp) : tt, a.clamp);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float got_v = __shfl_xor_sync(kFullMask, up_side ? v[i] : v[8 + i], 1);
                        const float g = up_side ? got_v : v[i];
                        const float u = up_side ? v[8 + i] : got_v;
                        const int t = 16 * b + (up_side ? 8 : 0) + i;
                        // silu with the fast exponential and division (a quotient of 0 once
                        // exp(-g) overflows): h is rounded to bf16 next
                        const __nv_bfloat16 hb = __float2bfloat16_rn(__fdividef(g, 1.f + __expf(-g)) * u);
                        if (t < nv) a.hrow[(int64_t)(pos0 + t) * I + m + j] = __bfloat16_as_ushort(hb);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bars.acc_empty[acc]);  // drained
            if (warp == kPsEpiWarp0 && valid(it + 1)) publish(it + 1, tv_nxt);
            info_cur = info_nxt;
            info_nxt = info_after;
            row_scale_cur = row_scale_nxt;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kPsMmaWarp) tmem_dealloc(tmem, kPsTmemCols);
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 p, float* v) {
    v[0] = bf16_lo(p.x);
    v[1] = bf16_hi(p.x);
    v[2] = bf16_lo(p.y);
    v[3] = bf16_hi(p.y);
    v[4] = bf16_lo(p.z);
    v[5] = bf16_hi(p.z);
    v[6] = bf16_lo(p.w);
    v[7] = bf16_hi(p.w);
}

// Largest |v| of a bf16 row of `cols` values (a multiple of 8) by one warp, as fp32 bits.
__device__ __forceinline__ uint32_t warp_row_absmax(const uint4* row, int cols, int lane) {
    uint32_t m = 0;
    for (int c = lane; c < cols / 8; c += 32) {
        const uint4 p = row[c];
        const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m = max(m, (w4[i] & 0x7fffu) << 16);
            m = max(m, w4[i] & 0x7fff0000u);
        }
    }
    return __reduce_max_sync(kFullMask, m);
}

// Splits row n of a tile (bf16, `cols` values, split scale s) into its hi row n and lo
// row NT + n of the tile's operand block ([cols / 16][2NT][16] bytes), chunk by chunk:
// thread (n, p) takes chunks p, p + P, ... of 16 values, so that a warp's lanes
// (consecutive rows of one chunk) store contiguous 16-byte rows.
template <int NT>
__device__ __forceinline__ void split_row_chunks(const uint4* row, int cols, float s, uint8_t* blk, int n, int p,
                                                 int P) {
    const float inv = 1.f / s;  // a power of two: exact
#pragma unroll 8
    for (int c = p; c < cols / 16; c += P) {
        float v[16];
        bf16x8_to_f32(row[2 * c], v);
        bf16x8_to_f32(row[2 * c + 1], v + 8);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= inv;
        uint2 h0, l0, h1, l1;
        split8(v, h0, l0);
        split8(v + 8, h1, l1);
        uint8_t* chunk = blk + (size_t)c * (2 * NT * 16);
        *reinterpret_cast<uint4*>(chunk + n * 16) = make_uint4(h0.x, h0.y, h1.x, h1.y);
        *reinterpret_cast<uint4*>(chunk + (NT + n) * 16) = make_uint4(l0.x, l0.y, l1.x, l1.y);
    }
}

// The split kernels run one CTA per 16 rows of a tile (grid: tiles x NT / 16): row
// maxima first (one warp per two rows), then the split, thread (row, chunk phase) of
// the CTA's 16 rows, so that a warp stores two 256-byte runs per step.
constexpr int kSplitRows = 16;

// One CTA per 16 rows of a tile: those tokens' x rows split into hi and lo rows, and
// their scales.  Rows past the tile's tokens are left as they are: they only reach
// accumulator columns that the epilogues never store.
template <int NT>
__global__ void __launch_bounds__(256) tc_gather_kernel(TcArgs a) {
    __shared__ float s_scale[kSplitRows];
    __shared__ const uint4* s_row[kSplitRows];
    pdl_wait();
    pdl_launch_dependents();
    int e, n0, nv, pos0;
    if (!tc_tile<NT>(a, blockIdx.x, e, n0, nv, pos0)) return;
    const int r0 = blockIdx.y * kSplitRows;
    if (r0 >= nv) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t* blk = a.xs + (size_t)blockIdx.x * a.H * (2 * NT);
    for (int n = r0 + warp; n < nv && n < r0 + kSplitRows; n += 8) {
        const uint4* xr = reinterpret_cast<const uint4*>(a.x + (int64_t)(a.perm[pos0 + n] / a.k) * a.H);
        const uint32_t m = warp_row_absmax(xr, a.H, lane);
        if (lane == 0) {
            const float sc = split_scale(__uint_as_float(m));
            s_scale[n - r0] = sc;
            s_row[n - r0] = xr;
            a.xscale[(size_t)blockIdx.x * NT + n] = sc;
        }
    }
    __syncthreads();
    const int n = r0 + tid % kSplitRows;
    if (n < nv) split_row_chunks<NT>(s_row[n - r0], a.H, s_scale[n - r0], blk, n, tid / kSplitRows, 256 / kSplitRows);
}

// One CTA per 16 rows of a tile: those h rows (bf16, by grouped position) split into hi
// and lo rows with the scale of each row's largest |h|, found first as in the x split.
template <int NT>
__global__ void __launch_bounds__(256) tc_split_h_kernel(TcArgs a) {
    __shared__ float s_scale[kSplitRows];
    pdl_wait();
    pdl_launch_dependents();
    int e, n0, nv, pos0;
    if (!tc_tile<NT>(a, blockIdx.x, e, n0, nv, pos0)) return;
    const int r0 = blockIdx.y * kSplitRows;
    if (r0 >= nv) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint8_t* blk = a.hs + (size_t)blockIdx.x * a.I * (2 * NT);
    for (int n = r0 + warp; n < nv && n < r0 + kSplitRows; n += 8) {
        const uint32_t m = warp_row_absmax(reinterpret_cast<const uint4*>(a.hrow + (int64_t)(pos0 + n) * a.I), a.I, lane);
        if (lane == 0) {
            const float sc = split_scale(__uint_as_float(m));
            s_scale[n - r0] = sc;
            a.hscale[(size_t)blockIdx.x * NT + n] = sc;
        }
    }
    __syncthreads();
    const int n = r0 + tid % kSplitRows;
    if (n < nv) {
        const uint4* hr = reinterpret_cast<const uint4*>(a.hrow + (int64_t)(pos0 + n) * a.I);
        split_row_chunks<NT>(hr, a.I, s_scale[n - r0], blk, n, tid / kSplitRows, 256 / kSplitRows);
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

// tile_off[e] = sum over e' < e of ceil(counts[e'] / nt), and for each tile t of expert
// e its record (e, first token n0 within the expert, tokens, grouped position of token
// n0); one CTA, E <= 1024.
__global__ void __launch_bounds__(1024) tc_tile_prefix_kernel(const int32_t* __restrict__ counts,
                                                              const int32_t* __restrict__ offsets, int E, int nt,
                                                              int32_t* __restrict__ tile_off,
                                                              int4* __restrict__ tile_info) {
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
    for (int t = 0; t < v; ++t) {
        const int n0 = t * nt, left = counts[tid] - n0;
        tile_info[excl + t] = make_int4(tid, n0, left < nt ? left : nt, offsets[tid] + n0);
    }
}

}  // namespace

// Token-tile width of a call: 64 when the slots average at least 64 per expert
// (prefill), 16 otherwise (decode batches: fewer padded MMA columns).
int ffn_tensor_tile_tokens(int S, int E) { return (int64_t)S >= 64 * (int64_t)E ? 64 : 16; }

// An upper bound of the number of tiles, sum over experts of ceil(n_e / NT).
int ffn_tensor_max_tiles(int S, int E) {
    const int nt = ffn_tensor_tile_tokens(S, E);
    return (S + nt - 1) / nt + (E < S ? E : S);
}

// Whether the grouped kernels can take a call: a shape they support, and at most 65535
// tiles, which bounds the operand workspace (2NT (H + I) bytes a tile: 21 GB at the
// Maple shape); beyond that, more than about 4.2 million slots, only the CUDA-core
// kernels run.
bool ffn_tensor_allowed(int T, int k, int E, int H, int I) {
    if (!ffn_tensor_shape_ok(H, I) || T < 1) return false;
    return ffn_tensor_max_tiles(T * k, E) <= 65535;
}

// The automatic choice: the tensor path from 32 slots on, and once there are at least
// an eighth as many slots as experts (on the Maple layer, 4 tokens and up: measured on
// B300 through the FFN call alone, CUDA cores / tensor cores 20.7 / 26.6 us at 2
// tokens, 34.7 / 34.4 at 4, 59.0 / 48.1 at 8, 108.6 / 63.2 at 16).  The grouped path's
// fixed kernels (tile table, x and h splits, combine) outweigh its MMAs below that.
bool ffn_use_tensor(int T, int k, int E, int H, int I) {
    const int64_t S = (int64_t)T * k;
    return ffn_tensor_allowed(T, k, E, H, I) && S >= 32 && 8 * S >= (int64_t)E;
}

// H a multiple of the 128 down rows of an item, I of the 64 gate (and up) rows; both at
// least 128, and at most 2080 so that a CTA's two packed-row buffers and its B stages
// fit in shared memory.
bool ffn_tensor_shape_ok(int H, int I) {
    return H % kRows == 0 && I % (kRows / 2) == 0 && H >= 128 && I >= 128 && H <= 2080 && I <= 2080;
}

// Operand blocks: per tile, 2NT rows (hi, lo) of H (x) or I (h) e4m3 values.
size_t ffn_tensor_x_bytes(int S, int E, int H) {
    return (size_t)ffn_tensor_max_tiles(S, E) * H * 2 * ffn_tensor_tile_tokens(S, E);
}

size_t ffn_tensor_h_bytes(int S, int E, int I) {
    return (size_t)ffn_tensor_max_tiles(S, E) * I * 2 * ffn_tensor_tile_tokens(S, E);
}

// Split scales: one fp32 per tile row.
size_t ffn_tensor_scale_bytes(int S, int E) {
    return sizeof(float) * (size_t)ffn_tensor_max_tiles(S, E) * ffn_tensor_tile_tokens(S, E);
}

namespace {

// The streaming kernels, one CTA per SM (fewer when there are fewer items), each stage
// with as many packed-row buffers (2 to 4) as shared memory holds.
template <int NT>
cudaError_t launch_tc_ffn_stream(const TcArgs& a, int S, cudaStream_t stream, int sm_count) {
    const int tiles = ffn_tensor_max_tiles(S, a.E);
    const int Bh = (a.H + 4) / 5, Bi = (a.I + 4) / 5;
    constexpr size_t kSmemLimit = 227 * 1024;
    auto npk_for = [&](int rb) {
        int n = kPsMaxPacked;
        while (n > 2 && ps_smem_bytes<NT>(rb, n) > kSmemLimit) --n;
        return n;
    };
    const int npk_gu = npk_for(Bh), npk_dn = npk_for(Bi);
    const size_t smem_gu = ps_smem_bytes<NT>(Bh, npk_gu), smem_dn = ps_smem_bytes<NT>(Bi, npk_dn);
    auto gu = tc_stream_kernel<NT, false>;
    auto dn = tc_stream_kernel<NT, true>;
    cudaError_t err = ensure_dynamic_smem(gu, smem_gu);
    if (err != cudaSuccess) return err;
    err = ensure_dynamic_smem(dn, smem_dn);
    if (err != cudaSuccess) return err;
    const int64_t items_gu = (int64_t)tiles * (a.I / (kRows / 2)), items_dn = (int64_t)tiles * (a.H / kRows);
    const int grid_gu = (int)(items_gu < sm_count ? items_gu : sm_count);
    const int grid_dn = (int)(items_dn < sm_count ? items_dn : sm_count);
    err = launch_pdl(tc_gather_kernel<NT>, dim3(tiles, NT / kSplitRows), dim3(256), 0, stream, a);
    if (err != cudaSuccess) return err;
    err = launch_pdl(gu, dim3(grid_gu), dim3(PsCfg<NT>::kThreads), smem_gu, stream, a, npk_gu);
    if (err != cudaSuccess) return err;
    err = launch_pdl(tc_split_h_kernel<NT>, dim3(tiles, NT / kSplitRows), dim3(256), 0, stream, a);
    if (err != cudaSuccess) return err;
    return launch_pdl(dn, dim3(grid_dn), dim3(PsCfg<NT>::kThreads), smem_dn, stream, a, npk_dn);
}

}  // namespace

cudaError_t launch_moe_ffn_tensor(const FfnArgs& f, cudaStream_t stream, const DeviceInfo& dev) {
    const int S = f.T * f.k;
    const int nt = ffn_tensor_tile_tokens(S, f.E);
    int4* tile_info = reinterpret_cast<int4*>(f.tile_off + ((f.E + 1 + 3) & ~3));
    // one CTA groups a few thousand slots fastest, writing the tile table as it goes;
    // beyond that, chunks in parallel, then the tile table
    cudaError_t err;
    if (S > 4096) {
        err = launch_group_tokens_chunked(f.idx, S, f.E, f.counts, f.offsets, f.perm, f.active, f.n_active, f.chunks,
                                          stream);
        if (err != cudaSuccess) return err;
        err = launch_pdl(tc_tile_prefix_kernel, dim3(1), dim3(1024), 0, stream, (const int32_t*)f.counts,
                         (const int32_t*)f.offsets, f.E, nt, f.tile_off, tile_info);
    } else {
        err = launch_group_tokens(f.idx, S, f.k, f.E, f.counts, f.offsets, f.perm, f.active, f.n_active, stream,
                                  dev, nt, f.tile_off, tile_info);
    }
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
    a.tile_info = reinterpret_cast<const int4*>(f.tile_off + ((f.E + 1 + 3) & ~3));
    a.xs = f.xs;
    a.hs = f.hs;
    a.xscale = f.xscale;
    a.hscale = f.hscale;
    a.hrow = reinterpret_cast<uint16_t*>(f.h);
    a.ys = f.ys;
    a.y = f.y;
    a.T = f.T;
    a.status = f.status;
    err = nt == 64 ? launch_tc_ffn_stream<64>(a, S, stream, dev.sm_count)
                  : launch_tc_ffn_stream<16>(a, S, stream, dev.sm_count);
    if (err != cudaSuccess) return err;
    const int64_t work = (int64_t)f.T * (f.H / 4);
    const int64_t want = (work + 255) / 256;
    const int64_t cap = (int64_t)dev.sm_count * 8;
    return launch_pdl(tc_combine_kernel, dim3((unsigned)(want < cap ? want : cap)), dim3(256), 0, stream, a);
}

}  // namespace maple
