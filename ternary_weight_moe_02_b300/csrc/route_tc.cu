// Router logits on the tensor cores, for calls with many tokens.
//
// "Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
// section "The claim, verified from the bytes": the router stays in full precision (a
// bf16 linear map of the hidden state to the 256 expert logits).  With hundreds or
// thousands of tokens that map is a plain dense contraction,
//   logits[T][E] = x[T][H] . Wr[E][H]^T (+ bias[E]),
// and runs here as bf16 x bf16 -> fp32 MMAs (tcgen05.mma kind::f16, both operands in
// shared memory).  The products are exact in fp32; the MMAs sum them in an order of
// their own, so these logits differ from the CUDA-core kernels' by rounding (within
// the fp32 summation bound of a K-deep sum).
//
// A CTA computes a block of 128 tokens x 128 experts over all of H:
//   warp 0, lane 0 (loads): per K stage of 64 values, one TMA box load of x (64 values
//     x 128 token rows, whole 128-byte lines) and one of Wr (64 values x 128 expert
//     rows), in the 128-byte swizzled K-major layout the MMA descriptors name, on the
//     stage's "full" barrier;
//   warp 1, lane 0 (MMA): four MMAs (K = 16) per stage into one 128-column fp32
//     accumulator in tensor memory, committing the stage's "empty" barrier, and the
//     "done" barrier after the last stage;
//   all four warps (epilogue): thread r of lane quarter r / 32 reads token row r's 128
//     logits from tensor memory into shared memory; then each warp stores whole rows
//     (lane l the experts l + 32 j) with the bias added.
// Token rows past T, expert rows past E and values past H read as zeros (the TMA
// out-of-bounds fill) and are not stored.  Every wait is bounded (MAPLE_ERR_TIMEOUT).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace maple {

namespace {

constexpr int kRtM = 128;                      // tokens per CTA (MMA M)
constexpr int kRtN = 128;                      // experts per CTA (MMA N)
constexpr int kRtK = 64;                       // K values per stage
constexpr int kRtStages = 4;
constexpr int kRtSwizzleBytes = 128;           // 128-byte swizzle: one 64-value row of a stage
constexpr int kRtStageA = kRtM * kRtK * 2;     // 16 KB
constexpr int kRtStageB = kRtN * kRtK * 2;     // 16 KB
constexpr int kRtSmem = kRtStages * (kRtStageA + kRtStageB) + 1024;  // + alignment of the stages
static_assert(kRtK * 2 == kRtSwizzleBytes, "a stage row is one swizzle row");
constexpr int kRtThreads = 128;
constexpr int kRtPitch = kRtN + 1;             // floats per row of the staged logits block
static_assert(kRtM * kRtPitch * 4 <= kRtSmem, "staged block fits the operand stages");
// instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9 and
// 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24
constexpr uint32_t kRtIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRtN >> 3) << 17) |
                              ((uint32_t)(kRtM >> 4) << 24);

struct RtBars {
    uint64_t full[kRtStages], empty[kRtStages], done;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// Shared-memory descriptor of a K-major operand in the 128-byte swizzled layout that TMA
// writes with CU_TENSOR_MAP_SWIZZLE_128B: rows of 128 bytes (64 bf16), the 16-byte
// pieces of row r XOR-permuted by r % 8, 8-row groups 1024 bytes apart (SBO); the
// leading offset is unused for this layout (1).  Start address >> 4 in bits 0-13,
// version 1 at bit 46, layout type 2 (128-byte swizzle) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

// D[tmem] (+)= A[smem descriptor] . B[smem descriptor]^T, bf16 x bf16 -> fp32
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kRtIdesc), "r"(accumulate)
        : "memory");
}

__global__ void __launch_bounds__(kRtThreads, 1)
    route_logits_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                           const float* __restrict__ bias, int T, int H, int E, float* __restrict__ logits,
                           int* status) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ RtBars bars;
    __shared__ uint32_t tmem_slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kRtM, e0 = blockIdx.y * kRtN;
    const int KS = (H + kRtK - 1) / kRtK;
    // the stages on a 1024-byte boundary (the 128-byte swizzle repeats every 8 rows)
    unsigned char* sa = smem + ((1024u - (smem_addr(smem) & 1023u)) & 1023u);
    unsigned char* sb = sa + kRtStages * kRtStageA;
    if (tid == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            mbar_init_nofence(&bars.full[s], 1);
            mbar_init_nofence(&bars.empty[s], 1);
        }
        mbar_init_nofence(&bars.done, 1);
        mbar_init_fence();
    }
    if (warp == 2) tmem_alloc(&tmem_slot, kRtN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    pdl_wait();  // x, the bias and the logits buffer may belong to earlier kernels
    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int ks = 0; ks < KS && ok; ++ks) {
                const int s = ks % kRtStages;
                if (ks >= kRtStages && !mbar_wait_bounded(&bars.empty[s], ((ks / kRtStages) - 1) & 1, status)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bars.full[s], (uint32_t)(kRtStageA + kRtStageB));
                tma_load_2d(sa + s * kRtStageA, &map_x, ks * kRtK, t0, &bars.full[s]);
                tma_load_2d(sb + s * kRtStageB, &map_w, ks * kRtK, e0, &bars.full[s]);
                issued = ks + 1;
            }
            // the last loads into each stage land before the CTA leaves
            for (int j = issued - kRtStages > 0 ? issued - kRtStages : 0; j < issued; ++j)
                mbar_wait_bounded(&bars.full[j % kRtStages], (j / kRtStages) & 1, nullptr);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            for (int ks = 0; ks < KS; ++ks) {
                const int s = ks % kRtStages;
                if (!mbar_wait_bounded(&bars.full[s], (ks / kRtStages) & 1, status)) break;
                tc_fence_after();
                const uint32_t a0 = smem_addr(sa + s * kRtStageA), b0 = smem_addr(sb + s * kRtStageB);
#pragma unroll
                for (int kk = 0; kk < kRtK / 16; ++kk) {
                    // K = 16 values = 32 bytes along the swizzled 128-byte rows
                    const uint64_t ad = smem_desc_sw128(a0 + kk * 32);
                    const uint64_t bd = smem_desc_sw128(b0 + kk * 32);
                    mma_bf16_ss(tmem, ad, bd, (ks | kk) != 0 ? 1u : 0u);
                }
                mma_commit(&bars.empty[s]);
            }
            mma_commit(&bars.done);  // after every MMA issued, including on a give-up
        }
        __syncwarp();
    }
    pdl_launch_dependents();
    // epilogue: the block's logits go through shared memory (the operand stages are
    // free once every MMA is done), so that each warp stores whole 512-byte runs of a
    // token's row instead of one word of 32 different rows per store
    const bool got = mbar_wait_bounded(&bars.done, 0, status);
    tc_fence_after();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // stages: TMA writes -> generic
    float* blk = reinterpret_cast<float*>(smem);                    // [kRtM][kRtPitch]
    {
        const int r = 32 * warp + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll 1
        for (int c0 = 0; c0 < kRtN; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(lane_addr + (uint32_t)c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) blk[r * kRtPitch + c0 + i] = __uint_as_float(v[i]);
        }
    }
    __syncthreads();
    if (got) {
        float b[kRtN / 32];
#pragma unroll
        for (int jj = 0; jj < kRtN / 32; ++jj) {
            const int e = e0 + lane + 32 * jj;
            b[jj] = (bias != nullptr && e < E) ? bias[e] : 0.f;
        }
        for (int row = warp; row < kRtM; row += kRtThreads / 32) {
            const int t = t0 + row;
            if (t >= T) break;
            float* out = logits + (int64_t)t * E;
#pragma unroll
            for (int jj = 0; jj < kRtN / 32; ++jj) {
                const int e = e0 + lane + 32 * jj;
                if (e < E) out[e] = blk[row * kRtPitch + lane + 32 * jj] + b[jj];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) tmem_dealloc(tmem, kRtN);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A [rows][H] bf16 row-major matrix as a TMA map with boxes of 64 values x box_rows rows,
// written to shared memory in the 128-byte swizzled layout.
bool encode_rows(CUtensorMap* map, const uint16_t* base, int rows, int H, int box_rows) {
    const auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kRtK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The shapes the tensor-core logits kernel takes: rows of 16-byte aligned bf16 values
// (H a multiple of 8, x and Wr 16-byte aligned).
bool route_tc_shape_ok(const void* x, const void* Wr, int H) {
    return H % 8 == 0 && H >= 8 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(Wr) % 16 == 0;
}

// cudaErrorNotSupported when the driver offers no tensor-map encoder (the caller then
// uses the CUDA-core kernels).
cudaError_t launch_route_logits_tc(const uint16_t* x, const uint16_t* Wr, const float* bias, int T, int H, int E,
                                   float* logits, cudaStream_t stream, int* status) {
    CUtensorMap mx, mw;
    if (!encode_rows(&mx, x, T, H, kRtM) || !encode_rows(&mw, Wr, E, H, kRtN)) return cudaErrorNotSupported;
    cudaError_t err = ensure_dynamic_smem(route_logits_tc_kernel, (size_t)kRtSmem);
    if (err != cudaSuccess) return err;
    const dim3 grid((T + kRtM - 1) / kRtM, (E + kRtN - 1) / kRtN);
    return launch_pdl(route_logits_tc_kernel, grid, dim3(kRtThreads), (size_t)kRtSmem, stream, mx, mw, bias, T, H, E,
                      logits, status);
}

}  // namespace maple
