// Weighted un-permute and combine.
//
// Source: "Chinchilla scaling, MoE, and fused Triton kernels", section
// "PyTorch MoE implementation": the inverse permutation brings each token's k
// expert outputs back to token order and they are summed with the gate
// weights.  The shared expert of "Triton MoE Kernels & Memory Checkpointing",
// Part A, section 2 is added with weight 1.
//
// A gather (one warp per token, 16-byte vectors) instead of a scatter with
// atomics: every output row is written exactly once and the summation order
// is fixed (j = 0..k-1, then the shared term), so the result is
// deterministic.  The routed rows of y are bf16; the shared expert's rows ys
// are fp32 (its term enters with weight 1, so its own rounding is kept out of
// the sum).
#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;

MOE_DEV void fma_bf16x8(float (&acc)[8], float w, const uint4& v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = fmaf(w, bf16_lo(u[q]), acc[2 * q]);
    acc[2 * q + 1] = fmaf(w, bf16_hi(u[q]), acc[2 * q + 1]);
  }
}

// One warp per token.  KMAX >= k is a compile-time bound so the k row
// pointers and weights stay in registers; each lane loads all k (+1) rows of
// U 16-byte column chunks before doing any arithmetic.  Every y row is read
// once and every out row written once, so both go through L2 with the
// evict-first (streaming) policy: the L2 is full of the grouped GEMM's dirty
// y lines when this kernel starts, and the streamed lines should be the
// first to leave.
template <int KMAX, int U>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const uint4* __restrict__ y, const float4* __restrict__ ys, const float* __restrict__ w,
    const int32_t* __restrict__ inv, int T, int D, int k, uint4* __restrict__ out) {
  griddep_wait();  // y comes from the previous kernel
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kCombineWarps + warp;
  if (t >= T) return;
  const int n16 = D >> 3;
  int my_row = 0;
  float my_w = 0.f;
  if (lane < k) {
    my_row = inv[static_cast<size_t>(t) * k + lane];
    my_w = w[static_cast<size_t>(t) * k + lane];
  }
  const uint4* rows[KMAX];
  float ws[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    rows[j] = y + static_cast<size_t>(__shfl_sync(0xffffffffu, my_row, j)) * n16;
    ws[j] = __shfl_sync(0xffffffffu, my_w, j);
  }
  const bool has_shared = ys != nullptr;
  const float4* ysh = has_shared ? ys + static_cast<size_t>(t) * (2 * n16) : nullptr;
  uint4* orow = out + static_cast<size_t>(t) * n16;
  for (int c0 = lane; c0 < n16; c0 += 32 * U) {
    uint4 v[U][KMAX];
    float4 vs[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 32 * u;
      const bool in = c < n16;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k && in) v[u][j] = __ldcs(rows[j] + c);
      if (has_shared && in) {
        vs[u][0] = __ldcs(ysh + 2 * c);
        vs[u][1] = __ldcs(ysh + 2 * c + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 32 * u;
      if (c >= n16) break;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) fma_bf16x8(acc, ws[j], v[u][j]);
      if (has_shared) {
        acc[0] += vs[u][0].x;
        acc[1] += vs[u][0].y;
        acc[2] += vs[u][0].z;
        acc[3] += vs[u][0].w;
        acc[4] += vs[u][1].x;
        acc[5] += vs[u][1].y;
        acc[6] += vs[u][1].z;
        acc[7] += vs[u][1].w;
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      __stcs(orow + c, o);
    }
  }
}

template <int KMAX, int U>
static cudaError_t launch_combine_k(const uint16_t* y, const float* ys, const float* w, const int32_t* inv,
                                    const moe_dims& d, uint16_t* out, cudaStream_t s, bool pdl) {
  const int grid = (d.T + kCombineWarps - 1) / kCombineWarps;
  return launch_kernel(combine_kernel<KMAX, U>, dim3(grid), dim3(kCombineThreads), 0, s, pdl,
                       reinterpret_cast<const uint4*>(y), reinterpret_cast<const float4*>(ys), w, inv, d.T, d.D,
                       d.k, reinterpret_cast<uint4*>(out));
}

cudaError_t launch_combine(const uint16_t* y, const float* ys, const float* w, const int32_t* inv,
                           const moe_dims& d, uint16_t* out, cudaStream_t s, bool pdl) {
  if (d.k <= 1) return launch_combine_k<1, 4>(y, ys, w, inv, d, out, s, pdl);
  if (d.k <= 2) return launch_combine_k<2, 3>(y, ys, w, inv, d, out, s, pdl);
  if (d.k <= 4) return launch_combine_k<4, 2>(y, ys, w, inv, d, out, s, pdl);
  if (d.k <= 8) return launch_combine_k<8, 1>(y, ys, w, inv, d, out, s, pdl);
  return launch_combine_k<16, 1>(y, ys, w, inv, d, out, s, pdl);
}

}  // namespace moe
