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
// deterministic.
#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const uint4* __restrict__ y, const float* __restrict__ w, const int32_t* __restrict__ inv, int T,
    int D, int k, int S, int has_shared, uint4* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kCombineWarps + warp;
  if (t >= T) return;
  const int n16 = D >> 3;
  // lane j < k fetches slot t*k + j; broadcast below
  int my_row = 0;
  float my_w = 0.f;
  if (lane < k) {
    my_row = inv[static_cast<size_t>(t) * k + lane];
    my_w = w[static_cast<size_t>(t) * k + lane];
  }
  int rows[MOE_MAX_TOPK];
  float ws[MOE_MAX_TOPK];
#pragma unroll
  for (int j = 0; j < MOE_MAX_TOPK; ++j) {
    rows[j] = __shfl_sync(0xffffffffu, my_row, j);
    ws[j] = __shfl_sync(0xffffffffu, my_w, j);
  }
  const uint4* ysh = y + static_cast<size_t>(S + t) * n16;
  for (int c = lane; c < n16; c += 32) {
    uint4 v[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j)
      if (j < k) v[j] = __ldg(y + static_cast<size_t>(rows[j]) * n16 + c);
    uint4 vs = make_uint4(0, 0, 0, 0);
    if (has_shared) vs = __ldg(ysh + c);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
      if (j < k) {
        const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = fmaf(ws[j], bf16_lo(u[q]), acc[2 * q]);
          acc[2 * q + 1] = fmaf(ws[j], bf16_hi(u[q]), acc[2 * q + 1]);
        }
      }
    }
    if (has_shared) {
      const uint32_t u[4] = {vs.x, vs.y, vs.z, vs.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += bf16_lo(u[q]);
        acc[2 * q + 1] += bf16_hi(u[q]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    out[static_cast<size_t>(t) * n16 + c] = o;
  }
}

cudaError_t launch_combine(const uint16_t* y, const float* w, const int32_t* inv, const moe_dims& d,
                           int has_shared, uint16_t* out, cudaStream_t s) {
  const int grid = (d.T + kCombineWarps - 1) / kCombineWarps;
  combine_kernel<<<grid, kCombineThreads, 0, s>>>(reinterpret_cast<const uint4*>(y), w, inv, d.T, d.D,
                                                  d.k, d.T * d.k, has_shared,
                                                  reinterpret_cast<uint4*>(out));
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
