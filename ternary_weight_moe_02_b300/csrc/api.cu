// C-ABI entry points of libmaple.so (declared in include/maple.h): argument
// validation, status codes and per-thread error text, then the kernel launches.
#include <math.h>
#include <stdarg.h>

#include <atomic>
#include <stdio.h>
#include <string.h>

#include "maple.h"
#include "kernels.h"

namespace {

thread_local char g_last_error[512] = "";

// Device status word: a kernel whose bounded wait gave up records MAPLE_ERR_TIMEOUT
// here; maple_check_device_status reads and clears it.
__device__ int g_device_status;

int fail(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int ok() {
    g_last_error[0] = '\0';
    return MAPLE_OK;
}

int cuda_fail(cudaError_t err, const char* what) {
    cudaGetLastError();  // clear the sticky-free launch error so later calls start clean
    return fail(MAPLE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// One-shot injected launch failure (maple_test_inject): consumed by the next call that
// would launch kernels, which then reports MAPLE_ERR_CUDA and launches nothing.
std::atomic<int> g_inject_launch_error{0};

// Every entry point that launches kernels calls this once its arguments are checked.
int get_device(maple::DeviceInfo* dev, const char* what) {
    if (g_inject_launch_error.exchange(0) != 0)
        return fail(MAPLE_ERR_CUDA, "%s: injected launch failure (maple_test_inject)", what);
    cudaError_t err = maple::device_info(dev);
    if (err != cudaSuccess) return cuda_fail(err, what);
    return MAPLE_OK;
}

}  // namespace

namespace maple {

int report_error(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

cudaError_t device_info(DeviceInfo* info) {
    static int cached_sm[128];
    static size_t cached_smem[128];
    static int* cached_status[128];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (cached_sm[dev] == 0) {
        int sm = 0, smem = 0;
        err = cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (err != cudaSuccess) return err;
        void* status = nullptr;
        err = cudaGetSymbolAddress(&status, g_device_status);
        if (err != cudaSuccess) return err;
        cached_status[dev] = static_cast<int*>(status);
        cached_smem[dev] = (size_t)smem;
        cached_sm[dev] = sm;
    }
    info->device = dev;
    info->sm_count = cached_sm[dev];
    info->smem_optin = cached_smem[dev];
    info->status = cached_status[dev];
    return cudaSuccess;
}

}  // namespace maple

extern "C" {

int maple_version(void) { return 100; }

const char* maple_status_string(int status) {
    switch (status) {
        case MAPLE_OK: return "MAPLE_OK";
        case MAPLE_ERR_INVALID_ARG: return "MAPLE_ERR_INVALID_ARG";
        case MAPLE_ERR_UNSUPPORTED_SHAPE: return "MAPLE_ERR_UNSUPPORTED_SHAPE";
        case MAPLE_ERR_MISALIGNED: return "MAPLE_ERR_MISALIGNED";
        case MAPLE_ERR_CUDA: return "MAPLE_ERR_CUDA";
        case MAPLE_ERR_TIMEOUT: return "MAPLE_ERR_TIMEOUT";
        case MAPLE_ERR_BAD_CODE: return "MAPLE_ERR_BAD_CODE";
        case MAPLE_ERR_WORKSPACE: return "MAPLE_ERR_WORKSPACE";
        default: return "MAPLE_ERR_UNKNOWN";
    }
}

const char* maple_last_error(void) { return g_last_error; }

int maple_test_inject(int32_t kind, int32_t value) {
    switch (kind) {
        case MAPLE_INJECT_NONE:
            g_inject_launch_error.store(0);
            maple::layer_b1_inject_stall(-1);
            return ok();
        case MAPLE_INJECT_COPY_STALL:
            if (value < 1 || value > 100000) return fail(MAPLE_ERR_INVALID_ARG, "test_inject: polls=%d (1..100000)", value);
            maple::layer_b1_inject_stall(value);
            return ok();
        case MAPLE_INJECT_LAUNCH_ERROR:
            g_inject_launch_error.store(1);
            return ok();
        default:
            return fail(MAPLE_ERR_INVALID_ARG, "test_inject: kind=%d", kind);
    }
}

int maple_check_device_status(void* stream) {
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "check_device_status")) return st;
    cudaError_t err = cudaStreamSynchronize((cudaStream_t)stream);
    if (err != cudaSuccess) return cuda_fail(err, "check_device_status: stream synchronize");
    int value = 0;
    err = cudaMemcpy(&value, dev.status, sizeof value, cudaMemcpyDeviceToHost);
    if (err != cudaSuccess) return cuda_fail(err, "check_device_status: read");
    if (value == MAPLE_OK) return ok();
    const int zero = 0;
    err = cudaMemcpy(dev.status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (err != cudaSuccess) return cuda_fail(err, "check_device_status: clear");
    return fail(value, "check_device_status: a kernel reported %s (a bounded device wait gave up)",
                maple_status_string(value));
}

int maple_ternarize_pack(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed,
                         float* scales, void* stream) {
    if (rows < 0 || K < 1) return fail(MAPLE_ERR_INVALID_ARG, "ternarize_pack: rows=%lld K=%lld", (long long)rows, (long long)K);
    if (K > (int64_t(1) << 24)) return fail(MAPLE_ERR_UNSUPPORTED_SHAPE, "ternarize_pack: K=%lld > 2^24", (long long)K);
    if (rows == 0) return ok();
    if (!W || !packed || !scales) return fail(MAPLE_ERR_INVALID_ARG, "ternarize_pack: null pointer");
    if (!aligned(W, 2) || !aligned(scales, 4)) return fail(MAPLE_ERR_MISALIGNED, "ternarize_pack: W needs 2-byte and scales 4-byte alignment");
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "ternarize_pack")) return st;
    cudaError_t err = maple::launch_ternarize_pack(W, rows, K, packed, scales, (cudaStream_t)stream, dev);
    if (err != cudaSuccess) return cuda_fail(err, "ternarize_pack launch");
    return ok();
}

int maple_pack_ternary(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed, float* scales,
                       int32_t* bad_rows, void* stream) {
    if (rows < 0 || K < 1) return fail(MAPLE_ERR_INVALID_ARG, "pack_ternary: rows=%lld K=%lld", (long long)rows, (long long)K);
    if (K > (int64_t(1) << 24)) return fail(MAPLE_ERR_UNSUPPORTED_SHAPE, "pack_ternary: K=%lld > 2^24", (long long)K);
    if (rows == 0) return ok();
    if (!W || !packed || !scales) return fail(MAPLE_ERR_INVALID_ARG, "pack_ternary: null pointer");
    if (!aligned(W, 2) || !aligned(scales, 4) || !aligned(bad_rows, 4))
        return fail(MAPLE_ERR_MISALIGNED, "pack_ternary: W needs 2-byte, scales and bad_rows 4-byte alignment");
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "pack_ternary")) return st;
    cudaError_t err = maple::launch_pack_ternary(W, rows, K, packed, scales, bad_rows, (cudaStream_t)stream, dev);
    if (err != cudaSuccess) return cuda_fail(err, "pack_ternary launch");
    return ok();
}

int maple_unpack(const uint8_t* packed, const float* scales, int64_t rows, int64_t K,
                 float* W_out, int32_t* bad_codes, void* stream) {
    if (rows < 0 || K < 1) return fail(MAPLE_ERR_INVALID_ARG, "unpack: rows=%lld K=%lld", (long long)rows, (long long)K);
    if (rows == 0) return ok();
    if (!packed || !scales || !W_out) return fail(MAPLE_ERR_INVALID_ARG, "unpack: null pointer");
    if (!aligned(scales, 4) || !aligned(W_out, 4) || !aligned(bad_codes, 4)) return fail(MAPLE_ERR_MISALIGNED, "unpack: fp32/int32 arrays need 4-byte alignment");
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "unpack")) return st;
    cudaError_t err = maple::launch_unpack(packed, scales, rows, K, W_out, bad_codes, (cudaStream_t)stream, dev);
    if (err != cudaSuccess) return cuda_fail(err, "unpack launch");
    return ok();
}

int maple_route_topk(const uint16_t* x, const uint16_t* Wr, const float* bias, int32_t T,
                     int32_t H, int32_t E, int32_t k, float* logits, int32_t* idx, float* w,
                     void* stream) {
    if (T < 0 || H < 1 || E < 1 || k < 1 || k > E) return fail(MAPLE_ERR_INVALID_ARG, "route_topk: T=%d H=%d E=%d k=%d", T, H, E, k);
    if (H > 65536 || E > 1024 || k > 32) return fail(MAPLE_ERR_UNSUPPORTED_SHAPE, "route_topk: H=%d (<=65536) E=%d (<=1024) k=%d (<=32)", H, E, k);
    if (T == 0) return ok();
    if (!x || !Wr || !logits || !idx || !w) return fail(MAPLE_ERR_INVALID_ARG, "route_topk: null pointer");
    if (!aligned(x, 16) || !aligned(Wr, 16)) return fail(MAPLE_ERR_MISALIGNED, "route_topk: x and Wr need 16-byte alignment");
    if (!aligned(bias, 4) || !aligned(logits, 4) || !aligned(idx, 4) || !aligned(w, 4)) return fail(MAPLE_ERR_MISALIGNED, "route_topk: fp32/int32 arrays need 4-byte alignment");
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "route_topk")) return st;
    cudaError_t err = maple::launch_route_topk(x, Wr, bias, T, H, E, k, logits, idx, w, (cudaStream_t)stream, dev);
    if (err != cudaSuccess) return cuda_fail(err, "route_topk launch");
    return ok();
}

int maple_group_tokens(const int32_t* idx, int32_t T, int32_t k, int32_t E, int32_t* counts,
                       int32_t* offsets, int32_t* perm, void* stream) {
    if (T < 0 || k < 1 || E < 1) return fail(MAPLE_ERR_INVALID_ARG, "group_tokens: T=%d k=%d E=%d", T, k, E);
    if (E > 1024 || (int64_t)T * k > (int64_t(1) << 24)) return fail(MAPLE_ERR_UNSUPPORTED_SHAPE, "group_tokens: E=%d (<=1024) T*k=%lld (<=2^24)", E, (long long)T * k);
    if (!counts || !offsets) return fail(MAPLE_ERR_INVALID_ARG, "group_tokens: null pointer");
    if (T > 0 && (!idx || !perm)) return fail(MAPLE_ERR_INVALID_ARG, "group_tokens: null pointer");
    if (!aligned(idx, 4) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm, 4)) return fail(MAPLE_ERR_MISALIGNED, "group_tokens: int32 arrays need 4-byte alignment");
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "group_tokens")) return st;
    cudaError_t err = maple::launch_group_tokens(idx, T * k, k, E, counts, offsets, perm, nullptr, nullptr, (cudaStream_t)stream, dev);
    if (err != cudaSuccess) return cuda_fail(err, "group_tokens launch");
    return ok();
}

size_t maple_moe_ffn_workspace_size(int32_t T, int32_t k, const maple_experts* ex) {
    return maple::moe_ffn_workspace_bytes(T, k, ex, MAPLE_FFN_AUTO);
}

size_t maple_moe_ffn_workspace_size_ex(int32_t T, int32_t k, const maple_experts* ex, int32_t path) {
    return maple::moe_ffn_workspace_bytes(T, k, ex, path);
}

int maple_moe_ffn(const maple_experts* ex, const uint16_t* x, const int32_t* idx,
                  const float* w, int32_t T, int32_t k, float* y, void* ws, size_t ws_bytes,
                  void* stream) {
    return maple::moe_ffn_entry(ex, x, idx, w, T, k, y, ws, ws_bytes, stream, MAPLE_FFN_AUTO);
}

int maple_moe_ffn_ex(const maple_experts* ex, const uint16_t* x, const int32_t* idx, const float* w,
                     int32_t T, int32_t k, float* y, int32_t path, void* ws, size_t ws_bytes, void* stream) {
    return maple::moe_ffn_entry(ex, x, idx, w, T, k, y, ws, ws_bytes, stream, path);
}

}  // extern "C"

namespace {

// The path a call takes: *tensor is set, and false is returned when `path` is not one
// of the three values or names the tensor path for a call its kernels cannot take.
bool resolve_ffn_path(int path, int T, int k, int E, int H, int I, bool* tensor) {
    switch (path) {
        case MAPLE_FFN_AUTO: *tensor = maple::ffn_use_tensor(T, k, E, H, I); return true;
        case MAPLE_FFN_CORES: *tensor = false; return true;
        case MAPLE_FFN_TENSOR: *tensor = true; return maple::ffn_tensor_allowed(T, k, E, H, I);
        default: return false;
    }
}

}  // namespace

size_t maple::moe_ffn_workspace_bytes(int T, int k, const maple_experts* ex, int path) {
    if (!ex || T < 0 || k < 1 || ex->E < 1 || ex->H < 1 || ex->I < 1) return 0;
    bool tensor = false;
    if (!resolve_ffn_path(path, T, k, ex->E, ex->H, ex->I, &tensor)) return 0;
    return maple::ffn_workspace_layout(T, k, ex->E, ex->H, ex->I, tensor).total;
}

int maple::moe_ffn_entry(const maple_experts* ex, const uint16_t* x, const int32_t* idx, const float* w, int T,
                         int k, float* y, void* ws, size_t ws_bytes, void* stream, int path) {
    if (!ex) return fail(MAPLE_ERR_INVALID_ARG, "moe_ffn: null experts");
    const int E = ex->E, H = ex->H, I = ex->I;
    if (T < 0 || k < 1 || E < 1 || H < 1 || I < 1) return fail(MAPLE_ERR_INVALID_ARG, "moe_ffn: T=%d k=%d E=%d H=%d I=%d", T, k, E, H, I);
    if (!(ex->clamp > 0.f)) return fail(MAPLE_ERR_INVALID_ARG, "moe_ffn: clamp must be > 0 (INFINITY for none)");
    if (k > 64 || E > 1024 || H > 2080 || I > 2080 || (int64_t)T * k > (int64_t(1) << 24))
        return fail(MAPLE_ERR_UNSUPPORTED_SHAPE, "moe_ffn: k=%d (<=64) E=%d (<=1024) H=%d (<=2080) I=%d (<=2080) T*k=%lld (<=2^24)", k, E, H, I, (long long)T * k);
    if (T == 0) return ok();
    if (!ex->gate || !ex->up || !ex->down || !ex->s_gate || !ex->s_up || !ex->s_down || !x || !idx || !w || !y)
        return fail(MAPLE_ERR_INVALID_ARG, "moe_ffn: null pointer");
    if (!aligned(ex->gate, 16) || !aligned(ex->up, 16) || !aligned(ex->down, 16) || !aligned(ex->s_gate, 16) ||
        !aligned(ex->s_up, 16) || !aligned(ex->s_down, 16) || !aligned(x, 16) || !aligned(ws, 16))
        return fail(MAPLE_ERR_MISALIGNED, "moe_ffn: packed weights, scales, x and ws need 16-byte alignment");
    if (!aligned(idx, 4) || !aligned(w, 4) || !aligned(y, 4)) return fail(MAPLE_ERR_MISALIGNED, "moe_ffn: idx, w, y need 4-byte alignment");
    if (path != MAPLE_FFN_AUTO && path != MAPLE_FFN_CORES && path != MAPLE_FFN_TENSOR)
        return fail(MAPLE_ERR_INVALID_ARG, "moe_ffn: path=%d (MAPLE_FFN_AUTO, _CORES or _TENSOR)", path);
    bool tensor = false;
    if (!resolve_ffn_path(path, T, k, E, H, I, &tensor))
        return fail(MAPLE_ERR_UNSUPPORTED_SHAPE,
                    "moe_ffn: the tensor-core path takes H a multiple of 128 and I of 64, both in [128, 2080] "
                    "(H=%d I=%d), and at most 65535 token tiles", H, I);
    const maple::FfnWorkspaceLayout L = maple::ffn_workspace_layout(T, k, E, H, I, tensor);
    if (!ws || ws_bytes < L.total) return fail(MAPLE_ERR_WORKSPACE, "moe_ffn: workspace %zu bytes < %zu needed", ws_bytes, L.total);
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "moe_ffn")) return st;
    char* base = static_cast<char*>(ws);
    maple::FfnArgs a;
    a.gate = ex->gate;
    a.up = ex->up;
    a.down = ex->down;
    a.s_gate = ex->s_gate;
    a.s_up = ex->s_up;
    a.s_down = ex->s_down;
    a.E = E;
    a.H = H;
    a.I = I;
    a.clamp = ex->clamp;
    a.x = x;
    a.idx = idx;
    a.w = w;
    a.T = T;
    a.k = k;
    a.y = y;
    a.counts = reinterpret_cast<int32_t*>(base + L.counts);
    a.offsets = reinterpret_cast<int32_t*>(base + L.offsets);
    a.perm = reinterpret_cast<int32_t*>(base + L.perm);
    a.active = reinterpret_cast<int32_t*>(base + L.active);
    a.n_active = reinterpret_cast<int32_t*>(base + L.n_active);
    a.h = reinterpret_cast<float*>(base + L.h);
    a.tile_off = reinterpret_cast<int32_t*>(base + L.tile_off);
    a.chunks = reinterpret_cast<int32_t*>(base + L.chunks);
    a.xs = reinterpret_cast<uint8_t*>(base + L.xs);
    a.hs = reinterpret_cast<uint8_t*>(base + L.hs);
    a.xscale = reinterpret_cast<float*>(base + L.xscale);
    a.hscale = reinterpret_cast<float*>(base + L.hscale);
    a.ys = reinterpret_cast<float*>(base + L.ys);
    a.status = dev.status;
    a.tensor = tensor ? 1 : 0;
    cudaError_t err = maple::launch_moe_ffn(a, (cudaStream_t)stream, dev);
    if (err != cudaSuccess) return cuda_fail(err, "moe_ffn launch");
    return ok();
}

extern "C" {

// Workspace of maple_moe_layer: 256 bytes of counters, then either the FFN workspace
// (two-call path) or, at T = 1, the fused kernel's per-slot outputs [k][H] fp32.
size_t maple_moe_layer_workspace_size(int32_t T, int32_t k, const maple_experts* ex) {
    const size_t ffn = maple_moe_ffn_workspace_size(T, k, ex);
    if (ffn == 0) return 0;
    const size_t part = T == 1 ? (maple::layer_b1_part_bytes(k, ex->H) + 255) / 256 * 256 : 0;
    return 256 + (ffn > part ? ffn : part);
}

}  // extern "C"

namespace {

// Argument checks of maple_moe_layer (MAPLE_OK, or the status it reports).
int check_layer_args(const uint16_t* x, const uint16_t* Wr, const float* bias, const maple_experts* ex, int32_t T,
                     int32_t k, float* logits, int32_t* idx, float* w, float* y, void* ws, size_t ws_bytes) {
    if (!ex) return fail(MAPLE_ERR_INVALID_ARG, "moe_layer: null experts");
    const int E = ex->E, H = ex->H, I = ex->I;
    if (T < 0 || H < 1 || E < 1 || I < 1 || k < 1 || k > E) return fail(MAPLE_ERR_INVALID_ARG, "moe_layer: T=%d H=%d E=%d I=%d k=%d", T, H, E, I, k);
    if (!(ex->clamp > 0.f)) return fail(MAPLE_ERR_INVALID_ARG, "moe_layer: clamp must be > 0 (INFINITY for none)");
    if (E > 1024 || k > 32 || H > 2080 || I > 2080 || (int64_t)T * k > (int64_t(1) << 24))
        return fail(MAPLE_ERR_UNSUPPORTED_SHAPE, "moe_layer: E=%d (<=1024) k=%d (<=32) H=%d (<=2080) I=%d (<=2080) T*k=%lld", E, k, H, I, (long long)T * k);
    if (T == 0) return MAPLE_OK;  // nothing to do: the pointers are not looked at
    if (!x || !Wr || !logits || !idx || !w || !y || !ex->gate || !ex->up || !ex->down || !ex->s_gate || !ex->s_up || !ex->s_down)
        return fail(MAPLE_ERR_INVALID_ARG, "moe_layer: null pointer");
    if (!aligned(x, 16) || !aligned(Wr, 16) || !aligned(ws, 16) || !aligned(ex->gate, 16) || !aligned(ex->up, 16) ||
        !aligned(ex->down, 16) || !aligned(ex->s_gate, 16) || !aligned(ex->s_up, 16) || !aligned(ex->s_down, 16))
        return fail(MAPLE_ERR_MISALIGNED, "moe_layer: x, Wr, ws, packed weights and scales need 16-byte alignment");
    if (!aligned(bias, 4) || !aligned(logits, 4) || !aligned(idx, 4) || !aligned(w, 4) || !aligned(y, 4))
        return fail(MAPLE_ERR_MISALIGNED, "moe_layer: fp32/int32 arrays need 4-byte alignment");
    const size_t need = maple_moe_layer_workspace_size(T, k, ex);
    if (!ws || ws_bytes < need) return fail(MAPLE_ERR_WORKSPACE, "moe_layer: workspace %zu bytes < %zu needed", ws_bytes, need);
    return MAPLE_OK;
}

// maple_moe_layer; y_mirror (may be null): where the fused single-token launch also
// writes y, *mirrored telling whether it did (the two-call path does not).
int moe_layer_impl(const uint16_t* x, const uint16_t* Wr, const float* bias, const maple_experts* ex, int32_t T,
                   int32_t k, float* logits, int32_t* idx, float* w, float* y, void* ws, size_t ws_bytes,
                   void* stream, float* y_mirror, bool* mirrored) {
    *mirrored = false;
    if (int st = check_layer_args(x, Wr, bias, ex, T, k, logits, idx, w, y, ws, ws_bytes)) return st;
    if (T == 0) return ok();
    const int E = ex->E, H = ex->H, I = ex->I;
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "moe_layer")) return st;
    char* base = static_cast<char*>(ws);
    if (T == 1 && maple::layer_b1_supported(H, I, E, k, dev)) {
        maple::LayerLaunch p;
        p.x = x;
        p.Wr = Wr;
        p.bias = bias;
        p.gate = ex->gate;
        p.up = ex->up;
        p.down = ex->down;
        p.s_gate = ex->s_gate;
        p.s_up = ex->s_up;
        p.s_down = ex->s_down;
        p.E = E;
        p.H = H;
        p.I = I;
        p.k = k;
        p.clamp = ex->clamp;
        p.logits = logits;
        p.idx = idx;
        p.w = w;
        p.y = y;
        p.part = reinterpret_cast<float*>(base + 256);
        p.sync = reinterpret_cast<unsigned*>(base);
        p.y_mirror = y_mirror;
        cudaError_t err = maple::launch_moe_layer_b1(p, (cudaStream_t)stream, dev);
        if (err != cudaSuccess) return cuda_fail(err, "moe_layer launch");
        *mirrored = y_mirror != nullptr;
        return ok();
    }
    // general sizes: the two calls in sequence
    int st = maple_route_topk(x, Wr, bias, T, H, E, k, logits, idx, w, stream);
    if (st != MAPLE_OK) return st;
    return maple_moe_ffn(ex, x, idx, w, T, k, y, base + 256, ws_bytes - 256, stream);
}

}  // namespace

extern "C" {

int maple_moe_layer(const uint16_t* x, const uint16_t* Wr, const float* bias,
                    const maple_experts* ex, int32_t T, int32_t k, float* logits, int32_t* idx,
                    float* w, float* y, void* ws, size_t ws_bytes, void* stream) {
    bool mirrored = false;
    return moe_layer_impl(x, Wr, bias, ex, T, k, logits, idx, w, y, ws, ws_bytes, stream, nullptr, &mirrored);
}

int maple_moe_layer_host(const uint16_t* x_host, uint16_t* x_dev, const uint16_t* Wr, const float* bias,
                         const maple_experts* ex, int32_t T, int32_t k, float* logits, int32_t* idx, float* w,
                         float* y, float* y_host, void* ws, size_t ws_bytes, void* stream) {
    // every check of the layer call first, so that a rejected call enqueues nothing
    if (int st = check_layer_args(x_dev, Wr, bias, ex, T, k, logits, idx, w, y, ws, ws_bytes)) return st;
    if (T == 0) return ok();
    if (!x_host || !y_host) return fail(MAPLE_ERR_INVALID_ARG, "moe_layer_host: null host buffer");
    const size_t x_bytes = (size_t)T * (size_t)ex->H * 2, y_bytes = (size_t)T * (size_t)ex->H * 4;
    cudaStream_t s = (cudaStream_t)stream;
    // pinned host buffers the device can address: copy kernels chained with the layer
    // by programmatic dependent launch; other host memory: plain async copies
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "moe_layer_host")) return st;
    void* xm = maple::mapped_host_pointer(x_host);
    void* ym = maple::mapped_host_pointer(y_host);
    cudaError_t err = xm && ym ? maple::launch_io_copy(xm, x_dev, x_bytes, s, dev)
                   : cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, s);
    if (err != cudaSuccess) return cuda_fail(err, "moe_layer_host: copy x in");
    // the fused single-token launch writes y to the mapped host buffer itself
    bool mirrored = false;
    const int st = moe_layer_impl(x_dev, Wr, bias, ex, T, k, logits, idx, w, y, ws, ws_bytes, stream,
                                  xm && ym ? static_cast<float*>(ym) : nullptr, &mirrored);
    if (st != MAPLE_OK) return st;
    if (mirrored) return ok();
    err = xm && ym ? maple::launch_io_copy(y, ym, y_bytes, s, dev)
                   : cudaMemcpyAsync(y_host, y, y_bytes, cudaMemcpyDeviceToHost, s);
    if (err != cudaSuccess) return cuda_fail(err, "moe_layer_host: copy y out");
    return ok();
}

size_t maple_cache_fetch_workspace_size(int32_t T, int32_t k) {
    if (T < 0 || k < 1) return 0;
    return 4 * (1 + 2 * (size_t)T * (size_t)k);
}

int maple_cache_fetch(const maple_experts* pool, const maple_expert_cache* cache, const int32_t* idx, int32_t T,
                      int32_t k, int32_t* idx_slot, void* ws, size_t ws_bytes, void* stream) {
    if (!pool || !cache) return fail(MAPLE_ERR_INVALID_ARG, "cache_fetch: null pool or cache");
    const maple_experts& sl = cache->slots;
    const int E = pool->E, C = sl.E, H = pool->H, I = pool->I;
    if (T < 0 || k < 1 || E < 1 || C < 1 || H < 1 || I < 1)
        return fail(MAPLE_ERR_INVALID_ARG, "cache_fetch: T=%d k=%d E=%d C=%d H=%d I=%d", T, k, E, C, H, I);
    if (sl.H != H || sl.I != I) return fail(MAPLE_ERR_INVALID_ARG, "cache_fetch: pool and slots differ in H or I");
    if (E > 1024 || C > 1024 || (int64_t)T * k > C)
        return fail(MAPLE_ERR_UNSUPPORTED_SHAPE, "cache_fetch: E=%d, C=%d (both <= 1024) and T*k=%lld <= C needed", E, C,
                    (long long)T * k);
    if (!maple::cache_shape_ok(H, I))
        return fail(MAPLE_ERR_UNSUPPORTED_SHAPE, "cache_fetch: an expert's arrays must be whole 16-byte chunks (H=%d I=%d)", H, I);
    if (T == 0) return ok();
    const maple_experts* both[2] = {pool, &sl};
    for (const maple_experts* ex : both) {
        if (!ex->gate || !ex->up || !ex->down || !ex->s_gate || !ex->s_up || !ex->s_down)
            return fail(MAPLE_ERR_INVALID_ARG, "cache_fetch: null expert array");
        if (!aligned(ex->gate, 16) || !aligned(ex->up, 16) || !aligned(ex->down, 16) || !aligned(ex->s_gate, 16) ||
            !aligned(ex->s_up, 16) || !aligned(ex->s_down, 16))
            return fail(MAPLE_ERR_MISALIGNED, "cache_fetch: expert arrays need 16-byte alignment");
    }
    if (!cache->slot_of || !cache->expert_of || !cache->last_use || !cache->stats || !idx || !idx_slot)
        return fail(MAPLE_ERR_INVALID_ARG, "cache_fetch: null pointer");
    if (!aligned(cache->slot_of, 4) || !aligned(cache->expert_of, 4) || !aligned(cache->last_use, 4) ||
        !aligned(cache->stats, 4) || !aligned(idx, 4) || !aligned(idx_slot, 4) || !aligned(ws, 4))
        return fail(MAPLE_ERR_MISALIGNED, "cache_fetch: int arrays need 4-byte alignment");
    const size_t need = maple_cache_fetch_workspace_size(T, k);
    if (!ws || ws_bytes < need) return fail(MAPLE_ERR_WORKSPACE, "cache_fetch: workspace %zu bytes < %zu needed", ws_bytes, need);
    maple::DeviceInfo dev;
    if (int st = get_device(&dev, "cache_fetch")) return st;
    cudaError_t err = maple::launch_cache_fetch(*pool, sl, cache->slot_of, cache->expert_of, cache->last_use, cache->stats,
                                                idx, T * k, idx_slot, static_cast<int32_t*>(ws), (cudaStream_t)stream, dev);
    if (err != cudaSuccess) return cuda_fail(err, "cache_fetch launch");
    return ok();
}

}  // extern "C"
