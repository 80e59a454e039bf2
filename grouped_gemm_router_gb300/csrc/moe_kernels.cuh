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
int route_block_tokens(int T);  // tokens per router / permutation block (16, 32 or 64)
int route_blocks(int T);        // ceil(T / route_block_tokens(T))
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
cudaError_t launch_combine(const uint16_t* y, const float* w, const int32_t* inv, const moe_dims& d,
                           int has_shared, uint16_t* out, cudaStream_t s, bool pdl = false);

// ---- grouped GEMMs (grouped_gemm.cu) ----
// W1||W3 with SwiGLU epilogue: A = x_sorted [S, D] (+ x [T, D] for the shared
// group), B = W1/W3 [E, D, F] (+ Ws1/Ws3 [D, F]), C = h [S (+T), F].
cudaError_t launch_grouped_swiglu(const uint16_t* x_sorted, const uint16_t* x, const uint16_t* W1,
                                  const uint16_t* W3, const uint16_t* Ws1, const uint16_t* Ws3,
                                  const int32_t* offsets, const moe_dims& d, uint16_t* h,
                                  cudaStream_t s, bool pdl = false);
// W2: A = h [S (+T), F], B = W2 [E, F, D] (+ Ws2 [F, D]), C = y [S (+T), D].
cudaError_t launch_grouped_down(const uint16_t* h, const uint16_t* W2, const uint16_t* Ws2,
                                const int32_t* offsets, const moe_dims& d, uint16_t* y,
                                cudaStream_t s, bool pdl = false);

// W1||W3 + SiLU*mul and W2 chained in one kernel (chained_ffn.cu): same
// inputs as the two grouped GEMMs, y [S (+T), D] out, h never stored.
// Requires D <= kChainedMaxD.
constexpr int kChainedMaxD = 256;
cudaError_t launch_chained_ffn(const uint16_t* x_sorted, const uint16_t* x, const uint16_t* W1,
                               const uint16_t* W3, const uint16_t* W2, const uint16_t* Ws1,
                               const uint16_t* Ws3, const uint16_t* Ws2, const int32_t* offsets,
                               const moe_dims& d, uint16_t* y, cudaStream_t s, bool pdl = false);

// 2-D bf16 TMA descriptor of a row-major [rows, cols] matrix with a
// {box_cols, box_rows} box: 128-byte swizzle (64-byte for 32-column boxes),
// zero fill outside the tensor (grouped_gemm.cu).
cudaError_t tensor_map_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                          uint32_t box_rows, uint32_t box_cols);

// Device address of the error word that moe_device_error reads, on the
// current device.
cudaError_t device_error_address(unsigned int** p);

// One-CTA kernel whose bounded mbarrier wait must time out (*gave_up = 1).
cudaError_t launch_wait_timeout_selftest(uint64_t timeout_ns, int* gave_up, cudaStream_t s);
// Reads and clears the device error word (synchronous).
cudaError_t read_clear_device_error(unsigned int* value);

}  // namespace moe
