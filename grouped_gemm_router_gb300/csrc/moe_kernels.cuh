// Host-side launchers shared between the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe_ffn.h"

namespace moe {

// Counts kernel launches (moe_launch_count).
void note_launch();

// Host-side checks shared by every entry point (moe_api.cu): the shape
// limits of the header, and a CUDA error mapped to MOE_ERR_CUDA.
moe_status check_dims(const moe_dims& d);
moe_status cuda_status(cudaError_t e);

// Launches `kernel` on `s`; with `pdl` it may start while the previous kernel
// of the stream finishes (it calls griddep_wait before reading that kernel's
// results).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---- routing / permutation (route_permute.cu) ----
int current_device_sms();       // SM count of the current device (0: none)
int route_block_tokens(int T);  // tokens per permutation block / histogram row (16, 32 or 64)
int route_blocks(int T);        // ceil(T / route_block_tokens(T)) on the current device
int route_blocks_max(int T);    // ceil(T / 16): the most histogram rows on any device
size_t route_packed_bytes(int D, int E);  // router weights in MMA fragment order
// Packs Wg into wpack_buf (route_packed_bytes bytes), then routes.
cudaError_t launch_route(const uint16_t* x, const uint16_t* Wg, const float* bias, const moe_dims& d,
                         void* wpack_buf, int32_t* ids, float* w, int32_t* hist, cudaStream_t s,
                         bool pdl = false);
cudaError_t launch_hist(const int32_t* ids, const moe_dims& d, int32_t* hist, cudaStream_t s,
                        bool pdl = false);
cudaError_t launch_scatter(const int32_t* ids, const int32_t* hist, const moe_dims& d, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, const uint16_t* x,
                           uint16_t* x_sorted, cudaStream_t s, bool pdl = false);

// ---- combine (combine.cu) ----
// ys: the shared expert's rows [T, D] fp32, or nullptr without it.
cudaError_t launch_combine(const uint16_t* y, const float* ys, const float* w, const int32_t* inv,
                           const moe_dims& d, uint16_t* out, cudaStream_t s, bool pdl = false);

// ---- grouped GEMMs (grouped_gemm.cu) ----
// W1||W3 with SwiGLU epilogue: A = x_sorted [S, D] (+ x [T, D] for the shared
// group), B = W1/W3 [E, D, F] (+ Ws1/Ws3 [D, F]), C = h [S (+T), F].
cudaError_t launch_grouped_swiglu(const uint16_t* x_sorted, const uint16_t* x, const uint16_t* W1,
                                  const uint16_t* W3, const uint16_t* Ws1, const uint16_t* Ws3,
                                  const int32_t* offsets, const moe_dims& d, uint16_t* h,
                                  cudaStream_t s, bool pdl = false);
// W2: A = h [S (+T), F], B = W2 [E, F, D] (+ Ws2 [F, D]), C = y [S, D] bf16
// and (with Ws2) ys [T, D] fp32.
cudaError_t launch_grouped_down(const uint16_t* h, const uint16_t* W2, const uint16_t* Ws2,
                                const int32_t* offsets, const moe_dims& d, uint16_t* y, float* ys,
                                cudaStream_t s, bool pdl = false);

// W1||W3 + SiLU*mul and W2 chained in one kernel (chained_ffn.cu): same
// inputs as the two grouped GEMMs, y [S, D] bf16 and (shared) ys [T, D] fp32
// out, h never stored.
// Requires D <= kChainedMaxD.
constexpr int kChainedMaxD = 256;
cudaError_t launch_chained_ffn(const uint16_t* x_sorted, const uint16_t* x, const uint16_t* W1,
                               const uint16_t* W3, const uint16_t* W2, const uint16_t* Ws1,
                               const uint16_t* Ws3, const uint16_t* Ws2, const int32_t* offsets,
                               const moe_dims& d, uint16_t* y, float* ys, cudaStream_t s, bool pdl = false);

// ---- backward (grouped_gemm_bwd.cu, backward.cu) ----
// Padded sorted layout of the gradient buffers: group e at rows
// [prow0_e, prow0_e + round_up(n_e, 64)), the shared group at rows
// [S_pad, S_pad + T).
struct BwdLayout {
  moe_dims d;
  bool shared;
  int S_pad;  // bwd_padded_rows(d)
};
int bwd_padded_rows(const moe_dims& d);
// h_bar = y_bar W2^T per group (shared: d_out Ws2^T).
cudaError_t launch_bwd_dgrad_w2(const BwdLayout& L, const int32_t* offsets, const uint16_t* ybar,
                                const uint16_t* d_out, const uint16_t* W2, const uint16_t* Ws2,
                                uint16_t* hbar, cudaStream_t s, bool pdl);
// Recomputes g, u and writes g_bar | u_bar [rows, 2F] and h [rows, F].
cudaError_t launch_bwd_act(const BwdLayout& L, const int32_t* offsets, const uint16_t* x_sorted,
                           const uint16_t* x, const uint16_t* W1, const uint16_t* W3,
                           const uint16_t* Ws1, const uint16_t* Ws3, const uint16_t* hbar,
                           uint16_t* gu, uint16_t* h, cudaStream_t s, bool pdl);
// x_bar = g_bar W1^T + u_bar W3^T per group.
cudaError_t launch_bwd_dgrad_x(const BwdLayout& L, const int32_t* offsets, const uint16_t* gu,
                               const uint16_t* W1, const uint16_t* W3, const uint16_t* Ws1,
                               const uint16_t* Ws3, uint16_t* xbar, cudaStream_t s, bool pdl);
// C[e] = A[rows_e]^T B[rows_e] in fp32, columns [0, n_split) to w_a, the rest
// to w_b.  Long groups are split along the rows; their partials go to `part`
// (bwd_wgrad_part_floats floats) and a second launch adds them in order.
size_t bwd_wgrad_part_floats(const moe_dims& d, bool shared);
cudaError_t launch_bwd_wgrad(const BwdLayout& L, const int32_t* offsets, const uint16_t* A,
                             int a_padded, int M, const uint16_t* A_sh, const uint16_t* B, int N,
                             const uint16_t* B_sh, int n_split, float* w_a, float* w_b, float* ws_a,
                             float* ws_b, float* part, cudaStream_t s, bool pdl);
// Combine backward: y_bar (padded layout, padding rows zeroed), the gradient of
// the gate weights and of the selected logits (zero when routed_in).
// Also writes Wg^T [E, D] into wgt (unless routed_in).
cudaError_t launch_combine_bwd(const BwdLayout& L, const uint16_t* d_out, const uint16_t* y,
                               const float* w, const int32_t* ids, const int32_t* inv,
                               const int32_t* offsets, int routed_in, uint16_t* ybar, float* wbar,
                               float* lbar, const uint16_t* Wg, uint16_t* wgt, cudaStream_t s, bool pdl);
// dx[t] = sum_j x_bar[slot j] (+ x_bar[shared row]) + sum_j lbar[t,j] Wg^T[ids[t,j], :].
cudaError_t launch_dx_gather(const BwdLayout& L, const uint16_t* xbar, const int32_t* ids,
                             const int32_t* inv, const int32_t* offsets, const float* lbar,
                             const uint16_t* wgt, uint16_t* dx, cudaStream_t s, bool pdl);
// dWg[:, e] = sum over expert e's sorted rows of l_bar[perm[p]] x_sorted[p] and
// dbias[e] = sum of those l_bar, via group-aligned chunk partials summed in
// order (deterministic); `part` holds bwd_router_part_floats(d) floats.
size_t bwd_router_part_floats(const moe_dims& d);
cudaError_t launch_router_bwd(const BwdLayout& L, const uint16_t* x_sorted, const int32_t* perm,
                              const int32_t* offsets, const float* lbar, float* part, float* dWg,
                              float* dbias, cudaStream_t s, bool pdl);

// 2-D bf16 TMA descriptor of a row-major [rows, cols] matrix with a
// {box_cols, box_rows} box: 128-byte swizzle (64-byte for 32-column boxes),
// zero fill outside the tensor (grouped_gemm.cu).
cudaError_t tensor_map_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                          uint32_t box_rows, uint32_t box_cols);
// 3-D bf16 TMA descriptor of a row-major [rows, cols] matrix (cols % 64 == 0)
// viewed as {64 columns, rows, cols / 64 column blocks}: a box {64, box_rows,
// nblk} lands nblk consecutive 64-column blocks of box_rows rows (128 bytes a
// row, 128-byte swizzle) in one TMA operation; blocks past the last column
// read zeros (grouped_gemm.cu).
cudaError_t tensor_map_blocks(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t nblk,
                              uint32_t box_rows = 64);
// 3-D fp32 TMA descriptor of a packed [d2][d1][d0] array with a {box0, box1, 1}
// box: 64-byte swizzle for 16-float boxes (128-byte for 32), none otherwise.
cudaError_t tensor_map_f32_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint32_t box0, uint32_t box1);

// Device address of the error word that moe_device_error reads, on the
// current device.
cudaError_t device_error_address(unsigned int** p);

// One-CTA kernel whose bounded mbarrier wait must time out (*gave_up = 1).
cudaError_t launch_wait_timeout_selftest(uint64_t timeout_ns, int* gave_up, cudaStream_t s);
// Reads and clears the device error word (synchronous).
cudaError_t read_clear_device_error(unsigned int* value);

}  // namespace moe
