// Internal launchers of libmaple (C++ linkage; the public C-ABI is include/maple.h).
// Each returns the cudaError_t of its launch(es); arguments are already validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

struct maple_experts;

namespace maple {

// Sets the per-thread text behind maple_last_error() and returns `status`.
int report_error(int status, const char* fmt, ...);

struct DeviceInfo {
    int device;
    int sm_count;
    size_t smem_optin;
    int* status;  // device status word (MAPLE_ERR_TIMEOUT after a bounded wait gave up)
};
cudaError_t device_info(DeviceInfo* info);

cudaError_t launch_ternarize_pack(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed,
                                  float* scales, cudaStream_t stream, const DeviceInfo& dev);

cudaError_t launch_pack_ternary(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed, float* scales,
                                int32_t* bad_rows, cudaStream_t stream, const DeviceInfo& dev);
// The staged pack kernel in its already-ternary form; *taken is false (and nothing is
// launched) when the shape does not take the staged path.
cudaError_t launch_pack_exact_staged(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed,
                                     float* scales, int32_t* bad_rows, cudaStream_t stream, const DeviceInfo& dev,
                                     bool* taken);

cudaError_t launch_unpack(const uint8_t* packed, const float* scales, int64_t rows, int64_t K,
                          float* W_out, int32_t* bad_codes, cudaStream_t stream,
                          const DeviceInfo& dev);

// Router logits on the tensor cores (route_tc.cu); cudaErrorNotSupported when the
// driver offers no tensor-map encoder.
bool route_tc_shape_ok(const void* x, const void* Wr, int H);
cudaError_t launch_route_logits_tc(const uint16_t* x, const uint16_t* Wr, const float* bias, int T, int H, int E,
                                   float* logits, cudaStream_t stream, int* status);
cudaError_t launch_route_topk(const uint16_t* x, const uint16_t* Wr, const float* bias, int T,
                              int H, int E, int k, float* logits, int32_t* idx, float* w,
                              cudaStream_t stream, const DeviceInfo& dev);

// Grouping with optional outputs used by the FFN: `active` lists the experts with a
// non-zero count in increasing id order and `n_active` receives their number.
// Host I/O (host_io.cu): the device address of mapped pinned host memory (nullptr for
// other memory), and a copy kernel chained by programmatic dependent launch.
void* mapped_host_pointer(const void* host);
cudaError_t launch_io_copy(const void* src, void* dst, size_t bytes, cudaStream_t stream, const DeviceInfo& dev);

// With nt > 0 it also writes the grouped tensor-core path's tile table (tile_off[E + 1],
// tile_info: one record per tile of nt tokens), as tc_tile_prefix_kernel does.
cudaError_t launch_group_tokens(const int32_t* idx, int S, int k, int E, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* active,
                                int32_t* n_active, cudaStream_t stream, const DeviceInfo& dev, int nt = 0,
                                int32_t* tile_off = nullptr, int4* tile_info = nullptr);
size_t group_tokens_smem_bytes(int E);
// The same grouping spread over chunks of 1024 slots (for many slots); chunk_scratch
// holds group_chunked_bytes(S, E) bytes.
size_t group_chunked_bytes(int S, int E);
cudaError_t launch_group_tokens_chunked(const int32_t* idx, int S, int E, int32_t* counts, int32_t* offsets,
                                        int32_t* perm, int32_t* active, int32_t* n_active, int32_t* chunk_scratch,
                                        cudaStream_t stream);

struct FfnArgs {
    const uint8_t* gate;
    const uint8_t* up;
    const uint8_t* down;
    const float* s_gate;
    const float* s_up;
    const float* s_down;
    int E, H, I;
    float clamp;
    const uint16_t* x;
    const int32_t* idx;
    const float* w;
    int T, k;
    float* y;
    // workspace views
    int32_t* counts;   // [E]
    int32_t* offsets;  // [E+1]
    int32_t* perm;     // [T*k]
    int32_t* active;   // [E]
    int32_t* n_active; // [1]
    float* h;          // [T*k][I] (bf16 [T*k][I] on the tensor path)
    int32_t* tile_off; // tensor path only: [E+1] tile prefix, then from the next 16-byte boundary
                       // [max tiles] int4 tile records
    int32_t* chunks;   // grouping scratch of the tensor path
    uint8_t* xs;       // tensor path only: per tile, the tokens' x rows split into e4m3 hi/lo rows
    uint8_t* hs;       // tensor path only: per tile, the tokens' h rows split likewise
    float* xscale;     // tensor path only: split scale of each tile row of xs
    float* hscale;     // tensor path only: split scale of each tile row of hs
    float* ys;         // [T*k][H] tensor path only
    int* status;       // device status word
    int prefetch_down; // 1 if the down rows may be bulk-prefetched (16-byte multiples)
    int tensor;        // 1: grouped tensor-core path (the workspace holds its regions)
};

struct FfnWorkspaceLayout {
    size_t counts, offsets, perm, active, n_active, h, tile_off, chunks, xs, hs, xscale, hscale, ys, total;
    bool tensor;
};
// `tensor`: lay out the regions of the grouped tensor-core path too.
FfnWorkspaceLayout ffn_workspace_layout(int T, int k, int E, int H, int I, bool tensor);

cudaError_t launch_moe_ffn(const FfnArgs& a, cudaStream_t stream, const DeviceInfo& dev);

// Grouped tensor-core FFN (tcgen05): shapes it takes, the path choice for a call, and
// the launch (group, tile prefix, split x, gate/up, split h, down, combine).
bool ffn_tensor_shape_ok(int H, int I);
bool ffn_tensor_allowed(int T, int k, int E, int H, int I);
bool ffn_use_tensor(int T, int k, int E, int H, int I);
int ffn_tensor_tile_tokens(int S, int E);
int ffn_tensor_max_tiles(int S, int E);
size_t ffn_tensor_x_bytes(int S, int E, int H);
size_t ffn_tensor_h_bytes(int S, int E, int I);
size_t ffn_tensor_scale_bytes(int S, int E);
cudaError_t launch_moe_ffn_tensor(const FfnArgs& a, cudaStream_t stream, const DeviceInfo& dev);

// maple_moe_ffn with the path named by the caller: MAPLE_FFN_AUTO (the choice of
// ffn_use_tensor), MAPLE_FFN_CORES or MAPLE_FFN_TENSOR (an error when the grouped
// kernels cannot take the call).  moe_ffn_workspace_bytes is the workspace such a call
// needs (0 for arguments the call would reject).
size_t moe_ffn_workspace_bytes(int T, int k, const ::maple_experts* ex, int path);
int moe_ffn_entry(const ::maple_experts* ex, const uint16_t* x, const int32_t* idx, const float* w, int T, int k,
                  float* y, void* ws, size_t ws_bytes, void* stream, int path);

// Fused single-token layer step (route + gate/up + down + combine in one launch of
// 16-CTA clusters: slot c < C on cluster c, slots past C split over the clusters).
struct LayerLaunch {
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
    float clamp;
    float* logits;
    int32_t* idx;
    float* w;
    float* y;
    float* part;     // [k][H] scratch (layer_b1_part_bytes)
    unsigned* sync;  // 16 combine counters, zero on entry and on exit
    float* y_mirror = nullptr;  // optional second copy of y (a device address of mapped host memory)
};
// How many 16-CTA clusters of the fused kernel for (H, I, E) the current device runs
// at once (0 if it cannot tell).
int layer_b1_clusters(int H, int I, int E);
bool layer_b1_supported(int H, int I, int E, int k, const DeviceInfo& dev);
size_t layer_b1_part_bytes(int k, int H);
cudaError_t launch_moe_layer_b1(const LayerLaunch& p, cudaStream_t stream, const DeviceInfo& dev);
// How many of the kernel's 16-CTA clusters can be resident at once on this device.
cudaError_t layer_b1_max_clusters(int H, int I, int E, int* n);
// Test hook: the next fused launch arms one copy barrier of its first CTA for 16 bytes
// that no copy delivers and gives every bounded wait `polls` polls.
void layer_b1_inject_stall(int polls);

// Expert cache: host-resident pool -> HBM slots (plan + copy kernels).
bool cache_shape_ok(int H, int I);
cudaError_t launch_cache_fetch(const ::maple_experts& pool, const ::maple_experts& slots, int32_t* slot_of,
                               int32_t* expert_of, uint32_t* last_use, uint32_t* stats, const int32_t* idx,
                               int S, int32_t* idx_slot, int32_t* jobs, cudaStream_t stream, const DeviceInfo& dev);

}  // namespace maple
