/*
 * maple.h -- C-ABI of libmaple.so: the ternary mixture-of-experts FFN step of
 * DeepGrove's Maple-Preview on one NVIDIA B300 (sm_103a).
 *
 * Conventions shared by every entry point
 *  - Every call returns an int status: MAPLE_OK (0) or a negative MAPLE_ERR_* code.
 *    On error nothing has been launched, except for MAPLE_ERR_CUDA, which reports a
 *    failed launch.  maple_last_error() gives a one-line reason (per host thread).
 *  - Array arguments are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or keeps them.  bf16 arrays are passed as uint16_t bit
 *    patterns.  Scratch memory comes from a caller-provided workspace whose size is
 *    given by the matching *_workspace_size call.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work is
 *    asynchronous and ordered on that stream; the host never synchronises.  Errors
 *    raised while kernels run surface at the caller's next synchronisation.
 *  - Kernels are launched with programmatic dependent launch: each one waits for
 *    the preceding work on the stream before it touches memory that work produced.
 *  - Sizes of zero are valid no-ops where stated.  Inputs must be finite.
 *
 * Packed ternary format (shared by every call)
 *  A weight matrix [rows x K] is stored as rows of ceil(K/5) bytes, row-major, with
 *  no padding between rows.  Byte b of row r holds the trits q of columns
 *  5b .. 5b+4 as sum_i (q_{5b+i} + 1) * 3^i (column 5b is the least significant
 *  base-3 digit); columns at or past K are trit 0.  Codes 243..255 are invalid.
 *  One fp32 scale per row: the dequantized weight is q * s.
 *  ("Maple-Preview: a 20B reasoning model where 97% of the weights are -1, 0, or +1",
 *  sections "The claim, verified from the bytes" and "The 5.31 GB claim reconciles":
 *  -s/0/+s per output row, five trits per byte since 3^5 = 243 <= 256.)
 */
#ifndef MAPLE_H
#define MAPLE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MAPLE_API __attribute__((visibility("default")))
#else
#define MAPLE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MAPLE_OK 0
#define MAPLE_ERR_INVALID_ARG (-1)       /* null pointer, negative size, k out of range */
#define MAPLE_ERR_UNSUPPORTED_SHAPE (-2) /* a size beyond the limits stated per call */
#define MAPLE_ERR_MISALIGNED (-3)        /* a pointer that breaks the stated alignment */
#define MAPLE_ERR_CUDA (-4)              /* a CUDA launch or attribute call failed */
#define MAPLE_ERR_TIMEOUT (-5)           /* a bounded device wait gave up */
#define MAPLE_ERR_BAD_CODE (-6)          /* packed byte >= 243 (reported by maple_unpack) */
#define MAPLE_ERR_WORKSPACE (-7)         /* workspace missing or smaller than required */

/* Expert weights of one MoE layer, all device pointers, 16-byte aligned.
 *   gate, up : [E][I][ceil(H/5)] packed bytes   s_gate, s_up : [E][I] fp32
 *   down     : [E][H][ceil(I/5)] packed bytes   s_down       : [E][H] fp32
 * clamp: bound of the activation clamps of the shipped forward (7.0f for Maple;
 * INFINITY gives plain SwiGLU).  Must be > 0. */
typedef struct maple_experts {
    const uint8_t* gate;
    const uint8_t* up;
    const uint8_t* down;
    const float* s_gate;
    const float* s_up;
    const float* s_down;
    int32_t E;
    int32_t H;
    int32_t I;
    float clamp;
} maple_experts;

/* Library version (major * 10000 + minor * 100 + patch). */
MAPLE_API int maple_version(void);

/* Static string naming a status code. */
MAPLE_API const char* maple_status_string(int status);

/* Reason for the last non-OK status returned on this host thread ("" if none). */
MAPLE_API const char* maple_last_error(void);

/*
 * Synchronise `stream`, then read and clear this device's status word.  Kernels
 * that wait on the completion of their own asynchronous copies do so with a bounded
 * number of polls; a wait that gives up records MAPLE_ERR_TIMEOUT in the word, skips
 * its work and returns, so the context stays usable.  Returns MAPLE_OK, the recorded
 * status, or MAPLE_ERR_CUDA if the synchronisation itself failed.
 */
MAPLE_API int maple_check_device_status(void* stream);

/*
 * Failure injection, for tests of the error paths (no GPU fault, trap or hang is ever
 * involved).  Each injection is one-shot and process-wide: the next call it applies to
 * consumes it.  The pages have no counterpart; this is test support.
 *   MAPLE_INJECT_NONE         cancel pending injections (value ignored).
 *   MAPLE_INJECT_COPY_STALL   the next single-token maple_moe_layer launch of the fused
 *                             kernel arms one bulk-copy barrier of its first CTA for 16
 *                             bytes that no copy delivers, and limits every bounded wait
 *                             of that launch to `value` polls (1..100000, each at most
 *                             ~1 ms).  The wait gives up, the device status word records
 *                             MAPLE_ERR_TIMEOUT (see maple_check_device_status), y rows
 *                             of that CTA are NaN, and the kernel still ends normally;
 *                             the next call needs no clean-up.
 *   MAPLE_INJECT_LAUNCH_ERROR the next call that would launch kernels returns
 *                             MAPLE_ERR_CUDA ("injected launch failure") and launches
 *                             nothing, as a failed launch does.
 * Returns MAPLE_OK, or MAPLE_ERR_INVALID_ARG for an unknown kind or value.
 */
#define MAPLE_INJECT_NONE 0
#define MAPLE_INJECT_COPY_STALL 1
#define MAPLE_INJECT_LAUNCH_ERROR 2
MAPLE_API int maple_test_inject(int32_t kind, int32_t value);

/*
 * Absmean ternarization + 5-trit packing of a bf16 row-major matrix W [rows x K].
 * Per row: s = (1/K) * sum_j |w_j| (fp32), q_j = clamp(round(w_j / s), -1, 1) with
 * round-half-to-even, i.e. q_j = sign(w_j) if |w_j| > s/2 else 0; s = 0 gives all 0.
 * ("Maple-Preview ...", section "The claim, verified from the bytes": rows are
 * exactly -s, 0, +s, the BitNet b1.58 absmean shape; "The 5.31 GB claim
 * reconciles": five trits per byte.)
 *   W      : [rows][K] bf16, 2-byte aligned (16-byte aligned with K % 8 == 0 takes
 *            the vector path)
 *   packed : [rows][ceil(K/5)] bytes, written
 *   scales : [rows] fp32, written
 * Limits: rows >= 0 (0 is a no-op), 1 <= K <= 2^24.
 */
MAPLE_API int maple_ternarize_pack(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed,
                         float* scales, void* stream);

/*
 * 5-trit packing of a bf16 row-major matrix W [rows x K] whose rows are already
 * ternary, such as the expert weights of the released bf16 checkpoint, where each
 * weight is -s, 0 or +s of its row.  Per row: s = max_j |w_j| (exact in fp32) and
 * q_j = sign(w_j) (0 for +0 and -0), packed as by maple_ternarize_pack.  (Absmean
 * ternarization of such a row gives the same trits but the scale (1 - z) s, z the
 * row's share of zeros.)  ("Maple-Preview ...", section "The claim, verified from the
 * bytes": exactly three values per row; "The 5.31 GB claim reconciles": five trits
 * per byte.)
 *   W        : [rows][K] bf16, finite, 2-byte aligned
 *   packed   : [rows][ceil(K/5)] bytes, written
 *   scales   : [rows] fp32, written
 *   bad_rows : optional device int32 counter; the kernel adds the number of rows with
 *              two different nonzero magnitudes (not ternary: they are still packed
 *              with sign trits and the max scale).  May be NULL.
 * Limits: rows >= 0 (0 is a no-op), 1 <= K <= 2^24.
 */
MAPLE_API int maple_pack_ternary(const uint16_t* W, int64_t rows, int64_t K, uint8_t* packed, float* scales,
                                 int32_t* bad_rows, void* stream);

/*
 * Dequantize packed rows back to fp32: W_out[r][j] = q_rj * s_r (inverse of the
 * packing above; a test and inspection helper, not on the hot path).
 *   packed : [rows][ceil(K/5)], scales : [rows], W_out : [rows][K] fp32 (written)
 *   bad_codes : optional device int32 counter; the kernel adds the number of bytes
 *               >= 243 it met (those decode as five zero trits).  May be NULL.
 * Limits: rows >= 0, K >= 1.
 */
MAPLE_API int maple_unpack(const uint8_t* packed, const float* scales, int64_t rows, int64_t K,
                 float* W_out, int32_t* bad_codes, void* stream);

/*
 * Full-precision router: logits = x Wr^T (+ bias) in fp32, top-k per token,
 * softmax over the k selected.
 * ("Maple-Preview ...", section "The claim, verified from the bytes": the router is
 * kept in full precision and picks 8 of 256 experts from the logit margin;
 * "IA de 20B Rodando a 120 tok/s no iPhone", section "256 experts, 8 ativos".)
 *   x      : [T][H] bf16, 16-byte aligned      Wr : [E][H] bf16, 16-byte aligned
 *   bias   : [E] fp32 or NULL
 *   logits : [T][E] fp32, written (also the intermediate between the two kernels)
 *   idx    : [T][k] int32, written: expert ids by descending logit, ties to the
 *            lower id
 *   w      : [T][k] fp32, written: exp(l_i - l_0) / sum_j exp(l_j - l_0)
 * Limits: T >= 0 (0 is a no-op), 1 <= H <= 65536, 1 <= E <= 1024, 1 <= k <= min(E, 32).
 */
MAPLE_API int maple_route_topk(const uint16_t* x, const uint16_t* Wr, const float* bias, int32_t T,
                     int32_t H, int32_t E, int32_t k, float* logits, int32_t* idx, float* w,
                     void* stream);

/*
 * Token-to-expert grouping of the T*k routing slots (slot s = t*k + i).
 *   idx     : [T][k] int32; ids outside [0, E) are left out of every group
 *   counts  : [E] int32, written: slots routed to each expert
 *   offsets : [E+1] int32, written: exclusive prefix sum of counts
 *   perm    : [T*k] int32, written: perm[offsets[e] .. offsets[e+1]) lists the
 *             slots of expert e in increasing slot order (stable)
 * Limits: T >= 0, 1 <= k, T*k <= 2^24, 1 <= E <= 1024.
 */
MAPLE_API int maple_group_tokens(const int32_t* idx, int32_t T, int32_t k, int32_t E, int32_t* counts,
                       int32_t* offsets, int32_t* perm, void* stream);

/* Bytes of workspace maple_moe_ffn needs for T tokens with k slots each. */
MAPLE_API size_t maple_moe_ffn_workspace_size(int32_t T, int32_t k, const maple_experts* ex);

/*
 * The expert FFN with weighted combine, for T tokens routed to k experts each:
 *   y_t = sum_{i<k} w[t][i] * down_e( silu(min(gate_e x_t, clamp)) * clamp(up_e x_t) )
 * with e = idx[t][i]; a weight 0 is skipped, +1 adds, -1 subtracts; each row's scale
 * is applied once to its sum.  The k terms are added in order i = 0..k-1 (fixed
 * order: the result is deterministic).
 * ("Maple-Preview ...", section "The shipped code does no quantization": the
 * MapleMLP forward with its clamps; "IA de 20B ...", section "Pesos ternarios":
 * skip / add / subtract.)
 * Two internal paths give results within the same bound: with at least 32 slots and an
 * eighth as many slots as experts (T*k >= 32, 8*T*k >= E) and H a multiple of 128, I of
 * 64, both in [128, 2080], the sums run on the tensor cores (fp8 MMAs on trits and on
 * exact two-part splits of the bf16 activations; h is rounded to bf16 between the two
 * projections); otherwise on CUDA cores with fp32 h.  maple_moe_ffn_ex below names the
 * path explicitly.
 *   ex  : expert weights (see maple_experts)
 *   x   : [T][H] bf16, 16-byte aligned
 *   idx : [T][k] int32 (ids outside [0, E) contribute 0)   w : [T][k] fp32
 *   y   : [T][H] fp32, written
 *   ws  : device workspace of at least maple_moe_ffn_workspace_size(T, k, ex) bytes,
 *         16-byte aligned; contents on entry are ignored
 * Limits: T >= 0 (0 is a no-op), 1 <= k <= 64, T*k <= 2^24, 1 <= E <= 1024,
 *         1 <= H <= 2080, 1 <= I <= 2080.
 */
MAPLE_API int maple_moe_ffn(const maple_experts* ex, const uint16_t* x, const int32_t* idx,
                  const float* w, int32_t T, int32_t k, float* y, void* ws, size_t ws_bytes,
                  void* stream);

/* FFN paths of maple_moe_ffn_ex (maple_moe_ffn always takes MAPLE_FFN_AUTO). */
#define MAPLE_FFN_AUTO 0   /* tensor cores when T*k >= 32, 8*T*k >= E and the shape allows it */
#define MAPLE_FFN_CORES 1  /* CUDA-core kernels, fp32 h (any shape within the limits) */
#define MAPLE_FFN_TENSOR 2 /* grouped tensor-core kernels (H % 128 == 0, I % 64 == 0,
                              both in [128, 2080]); MAPLE_ERR_UNSUPPORTED_SHAPE otherwise */

/* Bytes of workspace maple_moe_ffn_ex needs on `path` (0 when the call would be
 * rejected: invalid arguments, an unknown path, a tensor path the shape does not allow). */
MAPLE_API size_t maple_moe_ffn_workspace_size_ex(int32_t T, int32_t k, const maple_experts* ex,
                                                 int32_t path);

/*
 * maple_moe_ffn with the internal path named by the caller instead of chosen from the
 * load: the same arguments, limits and result bound, plus `path` (MAPLE_FFN_AUTO,
 * MAPLE_FFN_CORES or MAPLE_FFN_TENSOR; anything else is MAPLE_ERR_INVALID_ARG).  The
 * two paths differ only in rounding (the tensor path rounds h to bf16), so a caller
 * that needs the same bits across batch sizes can pin one of them.  The workspace
 * must hold maple_moe_ffn_workspace_size_ex(T, k, ex, path) bytes.
 * ("Maple-Preview ...", section "The shipped code does no quantization".)
 */
MAPLE_API int maple_moe_ffn_ex(const maple_experts* ex, const uint16_t* x, const int32_t* idx,
                               const float* w, int32_t T, int32_t k, float* y, int32_t path,
                               void* ws, size_t ws_bytes, void* stream);

/* Bytes of workspace maple_moe_layer needs (256 bytes of counters + the FFN's). */
MAPLE_API size_t maple_moe_layer_workspace_size(int32_t T, int32_t k, const maple_experts* ex);

/*
 * One MoE layer step: maple_route_topk followed by maple_moe_ffn, with the same
 * arguments, outputs and results (logits, idx, w and y are all written).
 * ("Maple-Preview ...", sections "The claim, verified from the bytes" and "The shipped
 * code does no quantization".)  For a single token (T = 1) at Maple-like sizes (E <=
 * 256, k <= 16, I a multiple of 256 up to 640, H a multiple of 128 up to 4096) the
 * whole step is one launch of one 16-CTA thread-block cluster per routed slot: each
 * cluster computes all E logits (a share per CTA, exchanged in distributed shared
 * memory), every CTA selects the same top-k, cluster i then computes slot i's expert
 * (h exchanged inside the cluster), and the k slots are added into y in the order
 * i = 0..k-1 by whichever CTA finishes a row block last.  No CTA waits for another
 * cluster; waits on copies are bounded (MAPLE_ERR_TIMEOUT via
 * maple_check_device_status).  The results are those of the two calls: the same
 * logits, idx and w bits, y within the FFN bound.  Other sizes run the two calls in
 * sequence.
 *   Wr : [E][H] bf16 router (E = ex->E), bias : [E] fp32 or NULL
 *   ws : device workspace of at least maple_moe_layer_workspace_size(T, k, ex) bytes,
 *        16-byte aligned; its first 256 bytes must be zero before the first call (for
 *        example cudaMemsetAsync once after allocating it).  Every call, including one
 *        whose bounded wait gave up, leaves them zero again.
 * Limits: those of maple_route_topk and maple_moe_ffn (k <= 32).
 */
MAPLE_API int maple_moe_layer(const uint16_t* x, const uint16_t* Wr, const float* bias,
                              const maple_experts* ex, int32_t T, int32_t k, float* logits,
                              int32_t* idx, float* w, float* y, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * maple_moe_layer for callers whose activations live in host memory: enqueues on
 * `stream` the copy of the T tokens x_host -> x_dev, the layer step on x_dev (exactly
 * maple_moe_layer, same arguments and results) and the copy y -> y_host, then returns.
 * y_host holds the result once the stream has synchronised.  Pinned host buffers
 * (cudaHostAlloc / cudaHostRegister, mapped: every pinned allocation is under unified
 * addressing) are copied by kernels that chain with the layer's kernels (the fused
 * single-token launch writes y_host itself, besides y); other host memory by
 * asynchronous copies.
 * ("Maple-Preview ...", sections "The claim, verified from the bytes" and "The shipped
 * code does no quantization".)
 *   x_host : [T][H] bf16, host     x_dev : [T][H] bf16 device staging, 16-byte aligned
 *   y      : [T][H] fp32 device    y_host : [T][H] fp32, host
 * Errors: those of maple_moe_layer (checked before anything is enqueued), an invalid
 * argument for a null host buffer, MAPLE_ERR_CUDA if a copy cannot be enqueued.
 */
MAPLE_API int maple_moe_layer_host(const uint16_t* x_host, uint16_t* x_dev, const uint16_t* Wr,
                                   const float* bias, const maple_experts* ex, int32_t T, int32_t k,
                                   float* logits, int32_t* idx, float* w, float* y, float* y_host,
                                   void* ws, size_t ws_bytes, void* stream);

/*
 * Expert cache: the experts of a layer kept in host memory (a "pool") and streamed into
 * C slots of device memory when a step routes to them, in the manner of the Mference
 * port that keeps MoE experts off the accelerator and reads them on demand
 * ("Maple Preview 接入 Mference：M4 MacBook 上 500MB 内存跑 20B MoE", opening paragraph
 * and section "接入 Mference 后的实测结果").
 *   slots     : a layer of C experts in device memory (slots.E = C, same H and I as the
 *               pool, 16-byte aligned arrays); its clamp is the FFN's
 *   slot_of   : [E] device int32, the slot holding expert e or -1; all -1 initially
 *   expert_of : [C] device int32, the expert in slot s or -1; all -1 initially
 *   last_use  : [C] device uint32, step of the slot's last use; all 0 initially
 *   stats     : [4] device uint32, zero initially: steps, hits, misses, experts copied
 * The tables belong to the cache; only maple_cache_fetch changes them.
 */
typedef struct maple_expert_cache {
    maple_experts slots;
    int32_t* slot_of;
    int32_t* expert_of;
    uint32_t* last_use;
    uint32_t* stats;
} maple_expert_cache;

/* Bytes of workspace maple_cache_fetch needs. */
MAPLE_API size_t maple_cache_fetch_workspace_size(int32_t T, int32_t k);

/*
 * Makes every expert that idx routes to resident in the cache and renames idx to slots:
 * a routed expert already in a slot is a hit (its last use is updated); each miss takes
 * the least recently used slot that no expert of this step holds (empty slots first,
 * ties to the lower slot), misses taken in increasing expert order, and is copied from
 * the pool (16-byte loads across the host link).  Then
 *   maple_moe_ffn(&cache->slots, x, idx_slot, w, ...)
 * computes the step's FFN exactly as on the pool's experts.  Everything runs on the
 * device, ordered on `stream` (no host synchronisation).
 *   pool     : E experts whose arrays the device can read (pinned host memory on a
 *              system with unified addressing, or device memory), 16-byte aligned
 *   idx      : [T][k] int32 device; ids outside [0, E) become -1 in idx_slot
 *   idx_slot : [T][k] int32 device, written
 *   ws       : device workspace of maple_cache_fetch_workspace_size(T, k) bytes
 * Limits: E <= 1024, C <= 1024, T*k <= C (every routed expert fits), each expert array
 * a whole number of 16-byte chunks.
 */
MAPLE_API int maple_cache_fetch(const maple_experts* pool, const maple_expert_cache* cache, const int32_t* idx,
                                int32_t T, int32_t k, int32_t* idx_slot, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * maple_moe_ffn without a workspace argument, for callers that cannot allocate device
 * memory: a plugin whose host process owns every device allocation, code running
 * while a stream is captured into a CUDA graph (cudaMalloc is not allowed there), or
 * a loop that must never enter an allocator.  The paper has no counterpart: this is
 * a packaging of maple_moe_ffn, with the same arguments (minus ws / ws_bytes), the
 * same limits and the same result.
 * Scratch lives in one static 2 MiB device array per GPU, held from the library's
 * load until process exit.  The call always takes the CUDA-core FFN kernels (the
 * grouped tensor-core path's operand blocks would not fit), whose scratch is the
 * [T*k][I] fp32 h array plus index arrays: a call needing more than 2 MiB (at
 * Maple's shapes: T > 127 with k = 8, I = 512) returns MAPLE_ERR_WORKSPACE and
 * launches nothing.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) and should come before any stream
 * capture.  The array is shared by every call and keeps the previous call's
 * contents (none of it needs clearing); calls that overlap on the GPU race on it,
 * so the caller must serialise them.  Allocates nothing.
 */
MAPLE_API int maple_moe_ffn_static_scratch(const maple_experts* ex, const uint16_t* x,
                                           const int32_t* idx, const float* w, int32_t T,
                                           int32_t k, float* y, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MAPLE_H */
