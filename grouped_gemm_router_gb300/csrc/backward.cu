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
// All are gathers with fixed summation orders (no atomics), so the results
// are deterministic.  Top-k itself is piecewise constant: unselected logits
// get no gradient.
#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kRouterTokens = 256;  // tokens per router-gradient partial
constexpr int kRouterCols = 64;     // x columns per router-gradient block

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
    uint4* __restrict__ ybar, float* __restrict__ wbar, float* __restrict__ lbar) {
  __shared__ int prow0[MOE_MAX_EXPERTS + 1];
  griddep_wait();
  griddep_launch_dependents();
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
    const uint16_t* __restrict__ Wg, int E, int T, int k, int D, int S_pad, int has_shared,
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
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint16_t wv = Wg[static_cast<size_t>(c * 8 + i) * E + e];
          acc[i] = fmaf(l, __uint_as_float(static_cast<uint32_t>(wv) << 16), acc[i]);
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = pack_bf16x2(acc[2 * q], acc[2 * q + 1]);
    dx[static_cast<size_t>(t) * n16 + c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Partial router gradients of one chunk of kRouterTokens tokens and
// kRouterCols columns of x: part[chunk][d][e] = sum_t x[t,d] l_bar[t,e] and
// (column block 0) part_bias[chunk][e] = sum_t l_bar[t,e].
__global__ void __launch_bounds__(kRouterCols) router_bwd_partial_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ ids, const float* __restrict__ lbar,
    int T, int D, int E, int k, float* __restrict__ part, float* __restrict__ part_bias) {
  extern __shared__ float acc[];  // [E][kRouterCols]
  __shared__ float bacc[MOE_MAX_EXPERTS];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  const int d = blockIdx.x * kRouterCols + tid;
  const int chunk = blockIdx.y;
  for (int e = 0; e < E; ++e) acc[e * kRouterCols + tid] = 0.f;
  for (int e = tid; e < E; e += kRouterCols) bacc[e] = 0.f;
  __syncthreads();
  const int t0 = chunk * kRouterTokens, t1 = min(t0 + kRouterTokens, T);
  for (int t = t0; t < t1; ++t) {
    const float xv = d < D ? __uint_as_float(static_cast<uint32_t>(x[static_cast<size_t>(t) * D + d]) << 16) : 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = ids[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= E) continue;
      const float l = lbar[static_cast<size_t>(t) * k + j];
      acc[e * kRouterCols + tid] = fmaf(xv, l, acc[e * kRouterCols + tid]);
      if (blockIdx.x == 0 && tid == 0) bacc[e] += l;
    }
  }
  __syncthreads();
  if (d < D)
    for (int e = 0; e < E; ++e) part[(static_cast<size_t>(chunk) * D + d) * E + e] = acc[e * kRouterCols + tid];
  if (blockIdx.x == 0)
    for (int e = tid; e < E; e += kRouterCols) part_bias[static_cast<size_t>(chunk) * E + e] = bacc[e];
}

// dWg[d][e] and dbias[e]: the partials summed over the chunks in order.
__global__ void router_bwd_reduce_kernel(const float* __restrict__ part, const float* __restrict__ part_bias,
                                         int nchunks, int D, int E, float* __restrict__ dWg,
                                         float* __restrict__ dbias) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int n = D * E;
  if (i < n) {
    if (dWg == nullptr) return;
    float s = 0.f;
    for (int c = 0; c < nchunks; ++c) s += part[static_cast<size_t>(c) * n + i];
    dWg[i] = s;
  } else if (i < n + E && dbias != nullptr) {
    const int e = i - n;
    float s = 0.f;
    for (int c = 0; c < nchunks; ++c) s += part_bias[static_cast<size_t>(c) * E + e];
    dbias[e] = s;
  }
}

int router_chunks(int T) { return (T + kRouterTokens - 1) / kRouterTokens; }

}  // namespace

cudaError_t launch_combine_bwd(const BwdLayout& L, const uint16_t* d_out, const uint16_t* y,
                               const float* w, const int32_t* ids, const int32_t* inv,
                               const int32_t* offsets, int routed_in, uint16_t* ybar, float* wbar,
                               float* lbar, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const int warps = d.T > 64 * d.E ? d.T : 64 * d.E;
  const dim3 grid((warps + kBwdWarps - 1) / kBwdWarps);
  return launch_kernel(combine_bwd_kernel, grid, dim3(kBwdThreads), 0, s, pdl,
                       reinterpret_cast<const uint4*>(d_out), reinterpret_cast<const uint4*>(y), w, ids,
                       inv, offsets, d.E, d.T, d.k, d.D, routed_in, reinterpret_cast<uint4*>(ybar), wbar,
                       lbar);
}

cudaError_t launch_dx_gather(const BwdLayout& L, const uint16_t* xbar, const int32_t* ids,
                             const int32_t* inv, const int32_t* offsets, const float* lbar,
                             const uint16_t* Wg, uint16_t* dx, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const dim3 grid((d.T + kBwdWarps - 1) / kBwdWarps);
  return launch_kernel(dx_gather_kernel, grid, dim3(kBwdThreads), 0, s, pdl,
                       reinterpret_cast<const uint4*>(xbar), ids, inv, offsets, lbar, Wg, d.E, d.T, d.k,
                       d.D, L.S_pad, L.shared ? 1 : 0, reinterpret_cast<uint4*>(dx));
}

size_t bwd_router_part_floats(const moe_dims& d) {
  return static_cast<size_t>(router_chunks(d.T)) * (static_cast<size_t>(d.D) * d.E + d.E);
}

cudaError_t launch_router_bwd(const BwdLayout& L, const uint16_t* x, const int32_t* ids,
                              const float* lbar, float* part, float* dWg, float* dbias,
                              cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const int nch = router_chunks(d.T);
  float* part_bias = part + static_cast<size_t>(nch) * d.D * d.E;
  const dim3 grid((d.D + kRouterCols - 1) / kRouterCols, nch);
  const size_t smem = sizeof(float) * d.E * kRouterCols;
  cudaError_t e = launch_kernel(router_bwd_partial_kernel, grid, dim3(kRouterCols), smem, s, pdl, x, ids,
                                lbar, d.T, d.D, d.E, d.k, part, part_bias);
  if (e != cudaSuccess) return e;
  const int n = d.D * d.E + d.E;
  return launch_kernel(router_bwd_reduce_kernel, dim3((n + 255) / 256), dim3(256), 0, s, pdl,
                       static_cast<const float*>(part), static_cast<const float*>(part_bias), nch, d.D,
                       d.E, dWg, dbias);
}

}  // namespace moe
