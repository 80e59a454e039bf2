/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) mixture-of-experts SwiGLU FFN
 * forward pass.
 *
 * The layer (per token t of x [T, D]):
 *   logits = x[t] . Wg (+ router_bias)                 router GEMM
 *   ids[t, 0..k-1] = the k largest logits, descending,  top-k
 *                    equal logits -> lower expert index
 *   w[t, j] = softmax over the k selected logits        gate weights
 *   slots s = t*k + j are sorted stably by expert id    permutation
 *   h = silu(x W1[e]) * (x W3[e])  per routed slot      grouped GEMM W1||W3
 *   y = h W2[e]                                         grouped GEMM W2
 *   out[t] = sum_j w[t, j] * y[t, j]  (+ shared(x[t]))  weighted combine
 * Sources: "Chinchilla scaling, MoE, and fused Triton kernels", section
 * "PyTorch MoE implementation" (router, top-k, softmax over the selected
 * logits, stable argsort, bincount, grouped GEMMs, inverse permutation,
 * weighted sum); "Triton MoE Kernels & Memory Checkpointing", Part A,
 * section 2 (SwiGLU expert W2(silu(W1 x) * W3 x), top-2 of 8 routed experts
 * plus an always-on shared expert) and section 10.3 (sort-by-expert layout,
 * per-expert counts and offsets).
 *
 * Conventions for every entry point:
 *  - Pointers named *_host are host memory; every other pointer is device
 *    memory on the current CUDA device.  The caller owns all memory and the
 *    stream; the library never allocates, frees or synchronises (except
 *    moe_device_error, which reads one word back).
 *  - Tensors are contiguous and row-major.  bf16 tensors are passed as
 *    void*.  Every device pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    only enqueued; results are ready when the stream reaches that point.
 *  - Arguments are validated on the host before anything is enqueued.  A
 *    bad argument returns MOE_ERR_INVALID_ARG, a shape outside the limits
 *    below returns MOE_ERR_UNSUPPORTED_SHAPE; nothing is launched in either
 *    case.  A failed launch returns MOE_ERR_CUDA.  There is no fallback path.
 *  - Kernels that wait on on-chip barriers give up after a bounded time and
 *    record MOE_ERR_DEVICE_TIMEOUT in a device word, read by
 *    moe_device_error().
 *
 * Shape limits: 0 <= T <= 2^24; D and F multiples of 64 in [64, 8192]
 * (the 8192 cap is the page's hard cap on d_model and d_ff);
 * 1 <= E <= 128; 1 <= k <= min(E, 16).
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,
  MOE_ERR_UNSUPPORTED_SHAPE = -2,
  MOE_ERR_CUDA = -3,
  MOE_ERR_WORKSPACE = -4,
  MOE_ERR_DEVICE_TIMEOUT = -5
} moe_status;

#define MOE_MAX_EXPERTS 128
#define MOE_MAX_TOPK 16
#define MOE_MAX_DIM 8192

/* Layer dimensions: T tokens, D = d_model, F = d_ff, E routed experts, top-k. */
typedef struct {
  int32_t T, D, F, E, k;
} moe_dims;

/* Optional per-call settings of moe_ffn_forward / moe_ffn_forward_host. */
typedef struct {
  /* cudaEvent_t handles recorded on `stream` at the stage boundaries:
   * [0] before routing, [1] after routing, [2] after the permutation,
   * [3] after W1||W3, [4] after W2, [5] after the combine.
   * moe_ffn_forward_host records [6] after the host->device copy of x (before
   * [0]) and [7] after the device->host copy of out.  moe_ffn_backward uses
   * [0..8] (see there).  NULL entries are skipped. */
  void* stage_events[12];
  /* Routing fixed from outside: ids [T, k] int32 and weights [T, k] fp32 in
   * device memory replace the router when both are non-NULL. */
  const int32_t* ids_in;
  const float* weights_in;
  /* MOE_FFN_CHAINED: run W1||W3 and W2 as one chained kernel that keeps h on
   * chip (moe_grouped_ffn_chained); needs D <= MOE_CHAINED_MAX_D.  The h
   * region of the workspace is then left untouched, and stage_events[3] is
   * recorded together with [4] after the chained kernel. */
  uint32_t flags;
} moe_ffn_options;

#define MOE_FFN_CHAINED 1u
#define MOE_CHAINED_MAX_D 256

/* Bytes of device workspace moe_ffn_forward needs for these dimensions
 * (has_shared != 0 when the shared expert is used; host_io != 0 adds the
 * device staging buffers used by moe_ffn_forward_host).  The workspace holds,
 * each 256-byte aligned: the packed router weights (moe_route_scratch_size
 * bytes), ids [T,k] i32, w [T,k] f32, block histogram
 * [ceil(T/16), E] i32 (of which the first ceil(T/TB) rows are used, TB =
 * moe_route_block_tokens(T)), counts [E] i32, offsets [E+1] i32, perm [T*k] i32,
 * inv [T*k] i32, x_sorted [T*k, D] bf16, h [T*k (+T), F] bf16,
 * y [T*k, D] bf16, (shared) ys [T, D] fp32, then (host_io) x [T, D] and
 * out [T, D] bf16. */
size_t moe_ffn_workspace_size(moe_dims d, int has_shared, int host_io);

/* Forward pass of one MoE SwiGLU FFN layer.
 *   x [T, D] bf16; Wg [D, E] bf16; router_bias [E] fp32 or NULL (added to the
 *   logits in fp32); W1, W3 [E, D, F] bf16; W2 [E, F, D] bf16;
 *   Ws1, Ws3 [D, F] and Ws2 [F, D] bf16: the shared expert, all three NULL
 *   for none; out [T, D] bf16.  Router logits and gate weights are fp32, GEMMs
 *   accumulate in fp32, h and y are stored as bf16, the combine sums in fp32
 *   and rounds once to bf16.  `workspace` holds moe_ffn_workspace_size(d,
 *   has_shared, 0) bytes; after the call it contains the routing, the
 *   permutation and the intermediates in the layout described above.
 *   opts may be NULL. */
moe_status moe_ffn_forward(const void* x, const void* Wg, const float* router_bias,
                           const void* W1, const void* W3, const void* W2,
                           const void* Ws1, const void* Ws3, const void* Ws2,
                           moe_dims d, void* out, void* workspace, size_t ws_bytes,
                           const moe_ffn_options* opts, void* stream);

/* The same forward pass with the activations in host memory: x_host [T, D]
 * bf16 is copied to the device, the layer runs, and out_host [T, D] bf16 is
 * copied back, all enqueued on `stream` (use pinned host memory for
 * asynchronous copies).  Weights stay in device memory.  `workspace` holds
 * moe_ffn_workspace_size(d, has_shared, 1) bytes. */
moe_status moe_ffn_forward_host(const void* x_host, const void* Wg, const float* router_bias,
                                const void* W1, const void* W3, const void* W2,
                                const void* Ws1, const void* Ws3, const void* Ws2,
                                moe_dims d, void* out_host, void* workspace, size_t ws_bytes,
                                const moe_ffn_options* opts, void* stream);

/* ---- Backward pass ---------------------------------------------------- */

/* Bytes of device workspace moe_ffn_backward needs.  With S_pad =
 * T*k + 64*E and R = S_pad (+T with the shared expert) it holds, each
 * 256-byte aligned: y_bar [S_pad, D], h_bar [R, F], g_bar|u_bar [R, 2F],
 * h [R, F], x_bar [R, D] (bf16, the routed rows of each expert padded to a
 * multiple of 64 rows in expert order, the shared rows from S_pad), the
 * gate-weight and selected-logit gradients [T, k] fp32, the router-
 * gradient partials ((T*k/64 + E) * (D + 1) fp32), Wg^T [E, D] bf16 and
 * the weight-gradient partial sums of groups split along their rows
 * ((kb / 80 + 2) * 2 * D * F fp32, kb = (T*k + 64 E) / 64 (+ ceil(T / 64))).
 * 0 for unsupported dimensions. */
size_t moe_ffn_backward_workspace_size(moe_dims d, int has_shared);

/* Gradients of L = sum(d_out * out) for the layer moe_ffn_forward computed
 * ("Triton MoE Kernels & Memory Checkpointing", Part A, section 8: the
 * SwiGLU expert's gradients -- h_bar split into g_bar = h_bar*u*silu'(g) and
 * u_bar = h_bar*silu(g), x_bar = g_bar W1^T + u_bar W3^T, the weight
 * gradients as outer products -- written as hand-made kernels; and the chain
 * rule through the combine, softmax and router of "Chinchilla scaling, MoE,
 * and fused Triton kernels", section "PyTorch MoE implementation").
 *   Inputs: the forward's x, Wg, W1, W3, W2, Ws1..Ws2 (as moe_ffn_forward) and
 *   d_out [T, D] bf16, plus the forward's workspace (fwd_workspace,
 *   fwd_ws_bytes >= moe_ffn_workspace_size(d, has_shared, 0)) holding the
 *   routing, permutation, x_sorted and y of that forward call; it is read
 *   only.  g and u are recomputed (the activations are not stored).
 *   Outputs: dx [T, D] bf16; dW1, dW3 [E, D, F], dW2 [E, F, D] and, with the
 *   shared expert, dWs1, dWs3 [D, F], dWs2 [F, D] in fp32 (all written, zero
 *   for an expert with no tokens); dWg [D, E] and dbias [E] fp32 (each may be
 *   NULL to skip).  Top-k is piecewise constant: unselected logits get no
 *   gradient.
 *   opts (nullable): ids_in / weights_in must repeat the fixed routing the
 *   forward was given, and then the router gets no gradient (dWg, dbias and
 *   the router term of dx are zero / skipped); stage_events [0..8] are
 *   recorded before the combine backward, after it, after h_bar, after
 *   g_bar|u_bar, after x_bar, after dW1|dW3, after dW2, after dx and after
 *   the router gradient; flags: MOE_FFN_CHAINED if the forward call ran
 *   chained (its workspace then holds no h, and the backward stores the
 *   recomputed h in its own workspace), else 0 (the W2 gradient reads the
 *   forward's h).
 *   Precision: fp32 accumulation everywhere; y_bar, h_bar, g_bar, u_bar, h
 *   and x_bar are stored as bf16 between the GEMMs; dx is summed in fp32 and
 *   rounded once.  Deterministic (no atomics).  T = 0 returns MOE_OK without
 *   touching any buffer. */
moe_status moe_ffn_backward(const void* x, const void* Wg, const void* W1, const void* W3,
                            const void* W2, const void* Ws1, const void* Ws3, const void* Ws2,
                            const void* d_out, moe_dims d, const void* fwd_workspace,
                            size_t fwd_ws_bytes, void* dx, float* dWg, float* dbias, float* dW1,
                            float* dW3, float* dW2, float* dWs1, float* dWs3, float* dWs2,
                            void* workspace, size_t ws_bytes, const moe_ffn_options* opts,
                            void* stream);

/* ---- Stage entry points (the same kernels moe_ffn_forward launches) ---- */

/* Scratch bytes moe_route needs: the router weights repacked in the MMA
 * fragment order, (D/32) * (E rounded up to 8, 16, 32, 64 or 128) * 16 bytes. */
size_t moe_route_scratch_size(moe_dims d);

/* Router GEMM + top-k + softmax ("PyTorch MoE implementation": logits, topk,
 * softmax over the selected logits).  ids [T, k] int32, weights [T, k] fp32.
 * block_hist (nullable) receives the per-block expert histogram
 * [ceil(T/TB), E] int32 over tokens [TB b, TB b + TB), TB =
 * moe_route_block_tokens(T).  scratch (device, 16-byte aligned) holds
 * moe_route_scratch_size(d) bytes. */
moe_status moe_route(const void* x, const void* Wg, const float* router_bias, moe_dims d,
                     int32_t* ids, float* weights, int32_t* block_hist, void* scratch,
                     size_t scratch_bytes, void* stream);

/* Tokens per row of the block histogram (and per block of the permutation
 * kernel) for a batch of T tokens on the current device: 64, or 32 / 16 for
 * batches too small to give each of the device's SMs two blocks; 16 when no
 * device can be queried. */
int moe_route_block_tokens(int T);

/* Scratch bytes moe_permute needs: the block histogram, sized for the most
 * rows any device uses, ceil(T/16)*E int32. */
size_t moe_permute_scratch_size(moe_dims d);

/* Stable permutation of the T*k slots by expert id (section "PyTorch MoE
 * implementation": flatten, stable argsort, bincount; "Triton MoE Kernels",
 * section 10.3, step 2: gather to expert-sorted order, counts and offsets).
 *   ids [T, k] int32 in [0, E); counts [E]; offsets [E+1] (offsets[E] = T*k);
 *   perm [T*k]: sorted position -> slot; inv [T*k]: slot -> sorted position;
 *   x [T, D] bf16 and x_sorted [T*k, D] bf16 are both NULL or both set
 *   (x_sorted[p] = x[perm[p] / k]).  Ids outside [0, E) give undefined
 *   output.  scratch holds moe_permute_scratch_size(d) bytes. */
moe_status moe_permute(const int32_t* ids, moe_dims d, int32_t* counts, int32_t* offsets,
                       int32_t* perm, int32_t* inv, const void* x, void* x_sorted,
                       void* scratch, size_t scratch_bytes, void* stream);

/* Grouped GEMM W1||W3 with the SwiGLU epilogue ("Triton MoE Kernels",
 * sections 2 and 10.2): for each expert e and sorted row p in
 * [offsets[e], offsets[e+1]): h[p] = silu(x_sorted[p] W1[e]) * (x_sorted[p] W3[e]).
 * With the shared expert (Ws1, Ws3 non-NULL, x non-NULL) rows T*k + t of h
 * receive silu(x[t] Ws1) * (x[t] Ws3).  h holds T*k (+T) rows of F bf16. */
moe_status moe_grouped_swiglu(const void* x_sorted, const void* x, const void* W1, const void* W3,
                              const void* Ws1, const void* Ws3, const int32_t* offsets,
                              moe_dims d, void* h, void* stream);

/* Grouped GEMM W2: y[p] = h[p] W2[e] for the routed rows, y [T*k, D] bf16;
 * with the shared expert (Ws2 non-NULL) also ys[t] = h[T*k + t] Ws2, ys
 * [T, D] fp32 (required then, ignored otherwise).  The shared expert's output
 * is added to the layer's output with weight 1, so it keeps its fp32
 * accumulation instead of being rounded to bf16 first. */
moe_status moe_grouped_down(const void* h, const void* W2, const void* Ws2, const int32_t* offsets,
                            moe_dims d, void* y, float* ys, void* stream);

/* W1||W3 + SiLU*mul and W2 chained in one kernel, h never written to memory
 * ("Chinchilla scaling, MoE, and fused Triton kernels", sections "Fused Triton
 * kernel mechanism" and "Triton fused kernel implementation").  Same inputs as
 * moe_grouped_swiglu and moe_grouped_down together, same outputs y [T*k, D]
 * bf16 and (shared) ys [T, D] fp32: per 256-row tile the kernel streams F in
 * 64-column chunks, rounds each h chunk to bf16 in shared memory and
 * accumulates y in fp32 over the chunks in the order of the two separate
 * GEMMs, so y and ys equal their result.
 * MOE_ERR_UNSUPPORTED_SHAPE when D > MOE_CHAINED_MAX_D: a tile's y
 * accumulator (D fp32 columns per row) and two g|u buffers (128 columns each)
 * must fit in the 512 TMEM columns of an SM. */
moe_status moe_grouped_ffn_chained(const void* x_sorted, const void* x, const void* W1,
                                   const void* W3, const void* W2, const void* Ws1,
                                   const void* Ws3, const void* Ws2, const int32_t* offsets,
                                   moe_dims d, void* y, float* ys, void* stream);

/* Weighted combine ("PyTorch MoE implementation": inverse permutation and
 * weighted sum): out[t] = sum_j weights[t, j] * y[inv[t*k + j]] (+ ys[t] when
 * ys, the shared expert's rows [T, D] fp32, is non-NULL), summed in fp32 in
 * order j = 0..k-1 and then the shared term, rounded once to bf16. */
moe_status moe_combine(const void* y, const float* ys, const float* weights, const int32_t* inv, moe_dims d,
                       void* out, void* stream);

/* ---- Allocation-free variant ---- */

/* moe_permute without a caller-provided scratch buffer, for callers that
 * cannot allocate device memory (for example a plugin inside a host framework
 * that owns all device memory, or a path that must never call cudaMalloc).
 * The pages have no counterpart of this entry point; it exists for such
 * callers only.  Arguments and results are those of moe_permute.  The block
 * histogram lives in a fixed 65,536-entry int32 array (256 KB) in the
 * library's own device memory, held on every GPU that loads the library until
 * the process exits; calls with ceil(T/TB) * E > 65,536 (TB =
 * moe_route_block_tokens(T)) return
 * MOE_ERR_UNSUPPORTED_SHAPE.  Every call shares that array: calls whose work
 * overlaps on the GPU race and must be serialised by the caller.  The first
 * call on each device looks up the array's device address (with that device
 * current); make it before any stream capture.  It calls no cudaMalloc or
 * cudaFree. */
moe_status moe_permute_noalloc(const int32_t* ids, moe_dims d, int32_t* counts, int32_t* offsets,
                               int32_t* perm, int32_t* inv, const void* x, void* x_sorted,
                               void* stream);

/* ---- Diagnostics ---- */

/* Reads and clears the device error word of the current device (a
 * synchronous copy).  Returns MOE_OK or MOE_ERR_DEVICE_TIMEOUT. */
moe_status moe_device_error(void);

/* Failure-detection self-test: launches one CTA whose bounded mbarrier wait
 * (the wait every pipelined kernel of the library uses) can never complete;
 * it gives up after timeout_us (1 .. 10^6 microseconds), writes 1 to
 * *gave_up (device int32) and records the timeout, so that a following
 * moe_device_error() returns MOE_ERR_DEVICE_TIMEOUT.  The GPU context stays
 * usable: nothing faults and nothing is left running. */
moe_status moe_selftest_wait_timeout(int timeout_us, int32_t* gave_up, void* stream);

/* Number of kernels this library has launched since it was loaded. */
uint64_t moe_launch_count(void);

/* Static text for a status code. */
const char* moe_status_str(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
