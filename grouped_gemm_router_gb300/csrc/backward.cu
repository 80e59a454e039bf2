// Backward of the combine, the un-permute and the router.
//
// Forward ("Chinchilla scaling, MoE, and fused Triton kernels", section
// "PyTorch MoE implementation"): out[t] = sum_j w[t,j] y[inv[t k + j]] (+ the
// shared expert), w = softmax of the k selected router logits, logits = x Wg
// (+ bias).  The chain rule gives, for the incoming gradient d_out:
//   y_bar[slot] = w[t,j] d_out[t]            (into the padded sorted layout)
//   w_bar[t,j]  = <d_out[t], y[slot]>
//   l_bar[t,j]  = w[t,j] (w_bar[t,j] - sum_i w[t,i] w_bar[t,i])   (softmax)
//   dx[t]       = sum_j x_bar[slot j] (+ shared x_bar[t]) + sum_j l_bar[t,j] Wg[:, ids[t,j]]
//   dWg         = x^T l_bar (scattered to the selected experts),  dbias = sum_t l_bar
//                 (computed over the sorted rows: dWg[:, e] = sum over expert e's rows of
//                 l_bar x_sorted)
// All are gathers with fixed summation orders (no atomics), so the results
// are deterministic.  Top-k itself is piecewise constant: unselected logits
// get no gradient.
#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;

// prow0[e] (e <= E): exclusive prefix sum of the group sizes rounded up to 64.
MOE_DEV void padded_starts(const int32_t* offsets, int E, int* prow0) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    int loc = 0;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) loc += (offsets[e + 1] - offsets[e] + 63) & ~63;
    }
    int incl = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - loc;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < E) {
        prow0[e] = run;
        run += (offsets[e + 1] - offsets[e] + 63) & ~63;
      }
    }
    if (lane == 31) prow0[E] = incl;
  }
  __syncthreads();
}

MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// One warp per token (y_bar, w_bar, l_bar); warp i < 64 E also zeroes padding
// row i % 64 of group i / 64 when it exists.
__global__ void __launch_bounds__(kBwdThreads) combine_bwd_kernel(
    const uint4* __restrict__ d_out, const uint4* __restrict__ y, const float* __restrict__ w,
    const int32_t* __restrict__ ids, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, int E, int T, int k, int D, int routed_in,
    uint4* __restrict__ ybar, float* __restrict__ wbar, float* __restrict__ lbar,
    const uint16_t* __restrict__ Wg, uint16_t* __restrict__ wgt) {
  __shared__ int prow0[MOE_MAX_EXPERTS + 1];
  griddep_wait();
  griddep_launch_dependents();
  // Wg^T [E, D] for the router term of dx (contiguous rows per expert)
  if (!routed_in)
    for (int i = blockIdx.x * kBwdThreads + threadIdx.x; i < E * D; i += gridDim.x * kBwdThreads) {
      const int e = i / D, d = i - e * D;
      wgt[i] = Wg[static_cast<size_t>(d) * E + e];
    }
  padded_starts(offsets, E, prow0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kBwdWarps + warp;
  const int n16 = D >> 3;
  if (gw < T) {
    const int t = gw;
    int my_p = -1, my_P = -1;
    float my_w = 0.f;
    if (lane < k) {
      const size_t s = static_cast<size_t>(t) * k + lane;
      const int e = ids[s];
      my_w = w[s];
      if (e >= 0 && e < E) {
        my_p = inv[s];
        my_P = prow0[e] + my_p - offsets[e];
      }
    }
    const uint4* drow = d_out + static_cast<size_t>(t) * n16;
    float my_wbar = 0.f;
    for (int j = 0; j < k; ++j) {
      const int p = __shfl_sync(0xffffffffu, my_p, j);
      const int P = __shfl_sync(0xffffffffu, my_P, j);
      const float wj = __shfl_sync(0xffffffffu, my_w, j);
      if (p < 0) continue;
      const uint4* yrow = y + static_cast<size_t>(p) * n16;
      uint4* brow = ybar + static_cast<size_t>(P) * n16;
      float dot = 0.f;
      for (int c = lane; c < n16; c += 32) {
        const uint4 dv = __ldg(drow + c), yv = __ldg(yrow + c);
        const uint32_t du[4] = {dv.x, dv.y, dv.z, dv.w}, yu[4] = {yv.x, yv.y, yv.z, yv.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float d0 = bf16_lo(du[q]), d1 = bf16_hi(du[q]);
          dot = fmaf(d0, bf16_lo(yu[q]), dot);
          dot = fmaf(d1, bf16_hi(yu[q]), dot);
          o[q] = pack_bf16x2(wj * d0, wj * d1);
        }
        brow[c] = make_uint4(o[0], o[1], o[2], o[3]);
      }
      dot = warp_sum(dot);
      if (lane == j) my_wbar = dot;
    }
    const float s = warp_sum(lane < k ? my_w * my_wbar : 0.f);
    if (lane < k) {
      const size_t i = static_cast<size_t>(t) * k + lane;
      wbar[i] = my_wbar;
      lbar[i] = (routed_in || my_p < 0) ? 0.f : my_w * (my_wbar - s);
    }
  }
  if (gw < 64 * E) {
    const int e = gw >> 6, r = gw & 63;
    const int P = prow0[e] + (offsets[e + 1] - offsets[e]) + r;
    if (P < prow0[e + 1]) {
      uint4* brow = ybar + static_cast<size_t>(P) * n16;
      for (int c = lane; c < n16; c += 32) brow[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

// One warp per token: dx[t] = sum_j x_bar[slot j] (+ x_bar[S_pad + t])
// (+ sum_j l_bar[t,j] Wg[:, ids[t,j]]), summed in fp32 in that order.
__global__ void __launch_bounds__(kBwdThreads) dx_gather_kernel(
    const uint4* __restrict__ xbar, const int32_t* __restrict__ ids, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, const float* __restrict__ lbar,
    const uint4* __restrict__ wgt, int E, int T, int k, int D, int S_pad, int has_shared,
    uint4* __restrict__ dx) {
  __shared__ int prow0[MOE_MAX_EXPERTS + 1];
  griddep_wait();
  griddep_launch_dependents();
  padded_starts(offsets, E, prow0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kBwdWarps + warp;
  if (t >= T) return;
  const int n16 = D >> 3;
  int my_P = -1, my_e = 0;
  float my_l = 0.f;
  if (lane < k) {
    const size_t s = static_cast<size_t>(t) * k + lane;
    const int e = ids[s];
    if (e >= 0 && e < E) {
      my_P = prow0[e] + inv[s] - offsets[e];
      my_e = e;
      if (lbar != nullptr) my_l = lbar[s];
    }
  }
  for (int c = lane; c < n16; c += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int P = __shfl_sync(0xffffffffu, my_P, j);
      if (P < 0) continue;
      const uint4 v = __ldg(xbar + static_cast<size_t>(P) * n16 + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += bf16_lo(u[q]);
        acc[2 * q + 1] += bf16_hi(u[q]);
      }
    }
    if (has_shared) {
      const uint4 v = __ldg(xbar + static_cast<size_t>(S_pad + t) * n16 + c);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += bf16_lo(u[q]);
        acc[2 * q + 1] += bf16_hi(u[q]);
      }
    }
    if (lbar != nullptr) {
      for (int j = 0; j < k; ++j) {
        const float l = __shfl_sync(0xffffffffu, my_l, j);
        const int e = __shfl_sync(0xffffffffu, my_e, j);
        if (l == 0.f) continue;
        const uint4 v = __ldg(wgt + static_cast<size_t>(e) * n16 + c);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = fmaf(l, bf16_lo(u[q]), acc[2 * q]);
          acc[2 * q + 1] = fmaf(l, bf16_hi(u[q]), acc[2 * q + 1]);
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = pack_bf16x2(acc[2 * q], acc[2 * q + 1]);
    dx[static_cast<size_t>(t) * n16 + c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Router gradient over the sorted rows: dWg[:, e] = sum over the rows p of
// expert e of l_bar[perm[p]] x_sorted[p, :], dbias[e] = sum of those
// l_bar.  Rows are cut into chunks of kRouterRows that never cross a group;
// block (chunk, column slab) writes the partial sums of its chunk, and the
// reduce kernel adds each expert's chunks in order.
constexpr int kRouterRows = 64;

// Group and first row of global chunk `c` (chunks are numbered group by
// group); false past the last chunk.
MOE_DEV bool chunk_of(const int32_t* offsets, int E, int c, int* e_out, int* r0, int* r1) {
  int base = 0;
  for (int e = 0; e < E; ++e) {
    const int n = offsets[e + 1] - offsets[e];
    const int nc = (n + kRouterRows - 1) / kRouterRows;
    if (c < base + nc) {
      *e_out = e;
      *r0 = offsets[e] + (c - base) * kRouterRows;
      *r1 = min(*r0 + kRouterRows, offsets[e + 1]);
      return true;
    }
    base += nc;
  }
  return false;
}

// Block (chunk, column block): thread (h, c) adds rows h, h + 2, ... of the
// chunk for 8-column group c; the two halves are added in order h = 0, 1.
__global__ void __launch_bounds__(kBwdThreads) router_bwd_partial_kernel(
    const uint4* __restrict__ x_sorted, const int32_t* __restrict__ perm, const float* __restrict__ lbar,
    const int32_t* __restrict__ offsets, int E, int D, float* __restrict__ part,
    float* __restrict__ part_bias) {
  __shared__ float lw[kRouterRows];
  __shared__ float4 half1[kBwdThreads / 2][2];
  griddep_wait();
  griddep_launch_dependents();
  int e, r0, r1;
  if (!chunk_of(offsets, E, blockIdx.x, &e, &r0, &r1)) return;
  const int n = r1 - r0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) lw[i] = lbar[perm[r0 + i]];
  __syncthreads();
  const int n16 = D >> 3;
  const int cols = blockDim.x / 2;  // 8-column groups per block
  const int h = threadIdx.x / cols, tc = threadIdx.x % cols;
  const int c = blockIdx.y * cols + tc;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (c < n16) {
    const uint4* col = x_sorted + static_cast<size_t>(r0) * n16 + c;
#pragma unroll 8
    for (int r = h; r < n; r += 2) {
      const uint4 v = __ldg(col + static_cast<size_t>(r) * n16);
      const float l = lw[r];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = fmaf(l, bf16_lo(u[q]), acc[2 * q]);
        acc[2 * q + 1] = fmaf(l, bf16_hi(u[q]), acc[2 * q + 1]);
      }
    }
  }
  if (h == 1) {
    half1[tc][0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    half1[tc][1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  __syncthreads();
  if (h == 0 && c < n16) {
    const float4 p0 = half1[tc][0], p1 = half1[tc][1];
    float4* dst = reinterpret_cast<float4*>(part + static_cast<size_t>(blockIdx.x) * D + 8 * c);
    dst[0] = make_float4(acc[0] + p0.x, acc[1] + p0.y, acc[2] + p0.z, acc[3] + p0.w);
    dst[1] = make_float4(acc[4] + p1.x, acc[5] + p1.y, acc[6] + p1.z, acc[7] + p1.w);
  }
  if (blockIdx.y == 0 && threadIdx.x < 32) {
    float sb = 0.f;
    for (int i = threadIdx.x; i < n; i += 32) sb += lw[i];
    sb = warp_sum(sb);
    if (threadIdx.x == 0) part_bias[blockIdx.x] = sb;
  }
}

// dWg[d][e] and dbias[e]: expert e's chunk partials added in a fixed order.
// Block (column block, e): 4 x 64 threads; quarter j of the threads adds the
// chunks j, j + 4, ... of expert e for its column, the four sums are then
// added in order j = 0..3 (column block 0 also adds the bias partials).
constexpr int kRedCols = 64;
constexpr int kRedSplit = 4;

__global__ void __launch_bounds__(kRedCols * kRedSplit) router_bwd_reduce_kernel(
    const float* __restrict__ part, const float* __restrict__ part_bias, const int32_t* __restrict__ offsets,
    int D, int E, float* __restrict__ dWg, float* __restrict__ dbias) {
  __shared__ float sums[kRedSplit][kRedCols + 1];
  griddep_wait();
  griddep_launch_dependents();
  const int e = blockIdx.y;
  const int tc = threadIdx.x % kRedCols, j = threadIdx.x / kRedCols;
  const int d = blockIdx.x * kRedCols + tc;
  int base = 0;
  for (int g = 0; g < e; ++g) base += (offsets[g + 1] - offsets[g] + kRouterRows - 1) / kRouterRows;
  const int nc = (offsets[e + 1] - offsets[e] + kRouterRows - 1) / kRouterRows;
  float s = 0.f, sb = 0.f;
  if (d < D) {
#pragma unroll 8
    for (int c = j; c < nc; c += kRedSplit) s += part[static_cast<size_t>(base + c) * D + d];
  }
  if (blockIdx.x == 0 && tc == 0)
    for (int c = j; c < nc; c += kRedSplit) sb += part_bias[base + c];
  sums[j][tc] = s;
  if (blockIdx.x == 0 && tc == 0) sums[j][kRedCols] = sb;
  __syncthreads();
  if (j == 0) {
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < kRedSplit; ++q) t += sums[q][tc];
    if (d < D && dWg != nullptr) dWg[static_cast<size_t>(d) * E + e] = t;
    if (blockIdx.x == 0 && tc == 0 && dbias != nullptr) {
      float tb = 0.f;
#pragma unroll
      for (int q = 0; q < kRedSplit; ++q) tb += sums[q][kRedCols];
      dbias[e] = tb;
    }
  }
}

// Upper bound of the number of group-aligned row chunks.
int router_chunks(const moe_dims& d) { return (d.T * d.k) / kRouterRows + d.E; }

}  // namespace

cudaError_t launch_combine_bwd(const BwdLayout& L, const uint16_t* d_out, const uint16_t* y,
                               const float* w, const int32_t* ids, const int32_t* inv,
                               const int32_t* offsets, int routed_in, uint16_t* ybar, float* wbar,
                               float* lbar, const uint16_t* Wg, uint16_t* wgt, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const int warps = d.T > 64 * d.E ? d.T : 64 * d.E;
  const dim3 grid((warps + kBwdWarps - 1) / kBwdWarps);
  return launch_kernel(combine_bwd_kernel, grid, dim3(kBwdThreads), 0, s, pdl,
                       reinterpret_cast<const uint4*>(d_out), reinterpret_cast<const uint4*>(y), w, ids,
                       inv, offsets, d.E, d.T, d.k, d.D, routed_in, reinterpret_cast<uint4*>(ybar), wbar,
                       lbar, Wg, wgt);
}

cudaError_t launch_dx_gather(const BwdLayout& L, const uint16_t* xbar, const int32_t* ids,
                             const int32_t* inv, const int32_t* offsets, const float* lbar,
                             const uint16_t* wgt, uint16_t* dx, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const dim3 grid((d.T + kBwdWarps - 1) / kBwdWarps);
  return launch_kernel(dx_gather_kernel, grid, dim3(kBwdThreads), 0, s, pdl,
                       reinterpret_cast<const uint4*>(xbar), ids, inv, offsets, lbar,
                       reinterpret_cast<const uint4*>(wgt), d.E, d.T, d.k, d.D, L.S_pad,
                       L.shared ? 1 : 0, reinterpret_cast<uint4*>(dx));
}

size_t bwd_router_part_floats(const moe_dims& d) {
  return static_cast<size_t>(router_chunks(d)) * (static_cast<size_t>(d.D) + 1);
}

cudaError_t launch_router_bwd(const BwdLayout& L, const uint16_t* x_sorted, const int32_t* perm,
                              const int32_t* offsets, const float* lbar, float* part, float* dWg,
                              float* dbias, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const int nch = router_chunks(d);
  float* part_bias = part + static_cast<size_t>(nch) * d.D;
  // two threads per 8 columns (each half of the chunk's rows), up to 256 threads per block
  const int n16 = d.D / 8;
  const int cols = n16 >= kBwdThreads / 2 ? kBwdThreads / 2 : (n16 + 15) / 16 * 16;
  const int threads = 2 * cols;
  const dim3 grid(nch, (n16 + cols - 1) / cols);
  cudaError_t e = launch_kernel(router_bwd_partial_kernel, grid, dim3(threads), 0, s, pdl,
                                reinterpret_cast<const uint4*>(x_sorted), perm, lbar, offsets, d.E, d.D,
                                part, part_bias);
  if (e != cudaSuccess) return e;
  return launch_kernel(router_bwd_reduce_kernel, dim3((d.D + kRedCols - 1) / kRedCols, d.E),
                       dim3(kRedCols * kRedSplit), 0, s, pdl, static_cast<const float*>(part),
                       static_cast<const float*>(part_bias), offsets, d.D, d.E, dWg, dbias);
}

}  // namespace moe
