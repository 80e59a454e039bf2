// Router GEMM + top-k + softmax, and the stable expert-grouped permutation.
//
// Sources: "Chinchilla scaling, MoE, and fused Triton kernels", section
// "PyTorch MoE implementation" (logits = x . gate_w, top-k, softmax over the
// selected logits, stable argsort of the flattened ids, bincount, gather);
// "Triton MoE Kernels & Memory Checkpointing", Part A, section 10.3, steps
// 1-2 (sort-by-expert layout, counts and offsets as a cumulative sum).
//
// Both kernels read activations once from HBM with 16-byte loads; the router
// GEMM (N = E, a few experts wide) runs on warp-level bf16 MMA because it is
// far too narrow for a tcgen05 tile and the kernel is bound by reading x.
#include <math.h>

#include <mutex>

#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

constexpr int kRouteThreads = 256;  // 8 warps per router block

// SM count of the current device, cached per device; 0 when it cannot be read.
int current_device_sms() {
  static int sms[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms[dev] = 0;
  return sms[dev];
}

// Tokens per router / permutation block on the current device: 64 when that
// still gives every SM two blocks, else 32 or 16, so that small batches spread
// over the whole GPU.  16 when the device cannot be queried (the most blocks,
// which every workspace is sized for).
int route_block_tokens(int T) {
  const int sms = current_device_sms();
  if (sms <= 0) return 16;
  if (T >= 64 * 2 * sms) return 64;
  if (T >= 32 * 2 * sms) return 32;
  return 16;
}

int route_blocks(int T) {
  const int tb = route_block_tokens(T);
  return (T + tb - 1) / tb;
}

int route_blocks_max(int T) { return (T + 15) / 16; }

// Expert tiles of 8 (the MMA's N) for E experts, padded to the instantiated widths.
int route_expert_tiles(int E) {
  const int nt = (E + 7) / 8;
  return nt <= 2 ? nt : nt <= 4 ? 4 : nt <= 8 ? 8 : 16;
}

size_t route_packed_bytes(int D, int E) {
  return static_cast<size_t>(D / 32) * route_expert_tiles(E) * 32 * 16;
}

MOE_DEV void mma_m16n8k16_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The router's x loads put, for lane (g = lane / 4, c = lane % 4), columns
// d + 8c .. d + 8c + 7 of each 32-wide chunk into the MMA k-slots (2c, 2c+1,
// 2c+8, 2c+9) of two m16n8k16 MMAs; the order of terms in the sum over d is
// irrelevant.  The router weights are read in the matching fragment order:
// wpack[chunk][expert tile][lane] = 16 bytes holding
// Wg[32 chunk + 8c + j][8 tile + g], j = 0..7 (zero for padded experts).
// pack_wg_slot builds one such slot from Wg [D, E]; small packed weights are
// built by every router block in its shared memory, larger ones once per call
// by pack_router_weights_kernel.
MOE_DEV uint4 pack_wg_slot(const uint16_t* __restrict__ Wg, int E, int NT, int slot) {
  const int lane = slot & 31, n = (slot >> 5) % NT, kc = (slot >> 5) / NT;
  const int e = 8 * n + (lane >> 2), d0 = 32 * kc + 8 * (lane & 3);
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = e < E ? __ldg(Wg + static_cast<size_t>(d0 + 2 * j) * E + e) : 0u;
    const uint32_t hi = e < E ? __ldg(Wg + static_cast<size_t>(d0 + 2 * j + 1) * E + e) : 0u;
    w[j] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Packed router weights up to this size are packed by each router block
// into its own shared memory (no separate packing launch).
constexpr size_t kRouteSelfPackBytes = 16 * 1024;

__global__ void __launch_bounds__(256) pack_router_weights_kernel(const uint16_t* __restrict__ Wg, int D,
                                                                  int E, int NT, uint4* __restrict__ wpack) {
  griddep_launch_dependents();
  const int slot = blockIdx.x * blockDim.x + threadIdx.x;
  if (slot >= (D / 32) * NT * 32) return;
  wpack[slot] = pack_wg_slot(Wg, E, NT, slot);
}

// Resident blocks per SM the register budget is sized for: all blocks of a
// 32K-token batch (512 blocks) fit in one wave for E <= 8.
constexpr int route_min_blocks(int nt) { return nt <= 1 ? 4 : nt <= 2 ? 3 : nt <= 8 ? 2 : 1; }

// Top-k + softmax of the logits a quad holds for rows row0 (r = 0) and row1
// (r = 1): thread (g, c) has experts 8n + 2c + {0, 1} in acc[n][2r + {0, 1}].
// Each of the k rounds takes the largest not-yet-chosen logit across the
// quad (ties to the lower expert index; NaN counts as -inf); the softmax is
// over the k selected logits.  Writes ids / wts of rows < T and counts the
// selections in s_hist.
template <int NT, int KMAX>
MOE_DEV void select_topk(const float (&acc)[NT][4], int row0, int row1, int c, int T, int E, int k,
                         const float* __restrict__ bias, int32_t* __restrict__ ids, float* __restrict__ wts,
                         int* s_hist) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = r ? row1 : row0;
    float v[2 * NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = n * 8 + 2 * c + h;
        float l = acc[n][2 * r + h];
        if (bias != nullptr && e < E) l += bias[e];
        if (isnan(l)) l = -INFINITY;
        v[2 * n + h] = l;
      }
    }
    uint32_t taken = 0;
    float sel_v[KMAX];
    int sel_e[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      sel_v[j] = 0.f;
      sel_e[j] = 0;
      if (j < k) {
        float best = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 2 * NT; ++i) {
          const int e = (i >> 1) * 8 + 2 * c + (i & 1);
          if (e < E && !((taken >> i) & 1u) && (v[i] > best || (v[i] == best && e < be))) {
            best = v[i];
            be = e;
          }
        }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
          const float ob = __shfl_xor_sync(0xffffffffu, best, off);
          const int oe = __shfl_xor_sync(0xffffffffu, be, off);
          if (ob > best || (ob == best && oe < be)) {
            best = ob;
            be = oe;
          }
        }
#pragma unroll
        for (int i = 0; i < 2 * NT; ++i) {
          const int e = (i >> 1) * 8 + 2 * c + (i & 1);
          if (e == be) taken |= 1u << i;
        }
        sel_v[j] = best;
        sel_e[j] = be;
      }
    }
    float z[KMAX];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      z[j] = 0.f;
      if (j < k) {
        z[j] = expf(sel_v[j] - sel_v[0]);
        sum += z[j];
      }
    }
    if (row < T) {
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k && (j & 3) == c) {
          ids[static_cast<size_t>(row) * k + j] = sel_e[j];
          wts[static_cast<size_t>(row) * k + j] = z[j] / sum;
          atomicAdd(&s_hist[sel_e[j]], 1);
        }
      }
    }
  }
}

// Block = 8 warps for TB = 16 MT tokens (MT = 1, 2 or 4 tiles of 16 tokens).
// Warp w computes tile w % MT over the 32-wide D-chunks kc with
// kc % DS == w / MT (DS = 8 / MT warps share a tile), loading x and the packed
// weight fragments straight from memory in batches of KG chunks; the DS
// partial results of a tile are summed through shared memory.
//
// Selection: thread (g, c) holds the logits of experts 8n + 2c + {0,1} for
// rows g and g + 8.  Each of the k rounds (k <= KMAX) takes the largest
// not-yet-chosen logit (ties to the lower expert index) across the quad.
template <int NT, int KMAX>
__global__ void __launch_bounds__(kRouteThreads, route_min_blocks(NT)) route_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ Wg, const uint4* __restrict__ wpack,
    int self_pack, const float* __restrict__ bias, int T, int D, int E, int k, int TB,
    int32_t* __restrict__ ids, float* __restrict__ wts, int32_t* __restrict__ hist) {
  extern __shared__ float red[];  // [8 warps][NT][4][32]: partial logits, then (self_pack) the packed weights
  uint4* wps = reinterpret_cast<uint4*>(red + 8 * NT * 4 * 32);
  __shared__ int s_hist[MOE_MAX_EXPERTS];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int MT = TB >> 4, DS = 8 / MT;
  const int tile = warp % MT, split = warp / MT;
  const int t0 = blockIdx.x * TB + tile * 16;
  const int row0 = t0 + g, row1 = t0 + g + 8;
  const bool ok0 = row0 < T, ok1 = row1 < T;
  const uint4* xr0 = reinterpret_cast<const uint4*>(x + static_cast<size_t>(ok0 ? row0 : 0) * D);
  const uint4* xr1 = reinterpret_cast<const uint4*>(x + static_cast<size_t>(ok1 ? row1 : 0) * D);

  for (int i = threadIdx.x; i < E; i += blockDim.x) s_hist[i] = 0;

  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

  constexpr int KG = (NT >= 16) ? 1 : (NT >= 8) ? 2 : 4;  // chunks per load batch
  const int nkc = D >> 5;
  uint4 a0[KG], a1[KG];
  auto load_x = [&](int kc0) {  // x of one batch: 2 rows x KG chunks
#pragma unroll
    for (int j = 0; j < KG; ++j) {
      const int kc = kc0 + j * DS;
      const bool in = kc < nkc;
      const int q = (kc << 2) + c;  // 16-byte column index
      a0[j] = (ok0 && in) ? __ldg(xr0 + q) : make_uint4(0, 0, 0, 0);
      a1[j] = (ok1 && in) ? __ldg(xr1 + q) : make_uint4(0, 0, 0, 0);
    }
  };
  // x does not come from the previous kernel (the weight packing): start
  // streaming it before waiting for the packed weights (or packing them here
  // from Wg, an input of the call)
  load_x(split);
  if (self_pack) {
    const int nslots = (D / 32) * NT * 32;
    for (int i = threadIdx.x; i < nslots; i += kRouteThreads) wps[i] = pack_wg_slot(Wg, E, NT, i);
    __syncthreads();
  }
  griddep_wait();
  griddep_launch_dependents();
  const uint4* bsrc = self_pack ? wps : wpack;  // this block's copy, or the packing kernel's
  for (int kc0 = split; kc0 < nkc; kc0 += KG * DS) {
    if (kc0 != split) load_x(kc0);
    uint4 b[KG][NT];
#pragma unroll
    for (int j = 0; j < KG; ++j) {
      const int kc = kc0 + j * DS;
      const bool in = kc < nkc;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        b[j][n] = in ? bsrc[(static_cast<size_t>(kc) * NT + n) * 32 + lane] : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int j = 0; j < KG; ++j) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        mma_m16n8k16_bf16(acc[n], a0[j].x, a1[j].x, a0[j].y, a1[j].y, b[j][n].x, b[j][n].y);
        mma_m16n8k16_bf16(acc[n], a0[j].z, a1[j].z, a0[j].w, a1[j].w, b[j][n].z, b[j][n].w);
      }
    }
  }

  // ---- sum the DS partial results of each tile ----
  if (split > 0) {
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp * NT + n) * 4 + i) * 32 + lane] = acc[n][i];
  }
  __syncthreads();
  if (split > 0) return;
  for (int sp = 1; sp < DS; ++sp) {
    const int w2 = tile + sp * MT;
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[n][i] += red[((w2 * NT + n) * 4 + i) * 32 + lane];
  }

  select_topk<NT, KMAX>(acc, row0, row1, c, T, E, k, bias, ids, wts, s_hist);
  // only the MT selecting warps are left: sync them on a named barrier
  asm volatile("bar.sync 1, %0;" ::"r"(MT * 32) : "memory");
  if (hist != nullptr)
    for (int i = threadIdx.x; i < E; i += MT * 32)
      hist[static_cast<size_t>(blockIdx.x) * E + i] = s_hist[i];
}

// Per-block expert histogram of given ids (blocks of TB tokens, as route_kernel).
__global__ void __launch_bounds__(256) hist_kernel(const int32_t* __restrict__ ids, int T, int k,
                                                   int E, int TB, int32_t* __restrict__ hist) {
  __shared__ int s_hist[MOE_MAX_EXPERTS];
  griddep_wait();
  griddep_launch_dependents();
  for (int i = threadIdx.x; i < E; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int s0 = blockIdx.x * TB * k;  // T * k <= 2^28 fits in int
  const int ns = min(TB * k, T * k - s0);
  for (int i = threadIdx.x; i < ns; i += blockDim.x) {
    const int e = ids[s0 + i];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&s_hist[e], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    hist[static_cast<size_t>(blockIdx.x) * E + i] = s_hist[i];
}

// Scatter: block b owns the slots of tokens [TB b, TB b + TB).
//  1. From the whole block histogram it forms counts, offsets (exclusive
//     scan over experts) and this block's first position per expert
//     (offsets[e] + the counts of expert e in blocks before b).
//  2. Slots are ranked stably in rounds of 256 (one per thread): within a
//     warp by __match_any_sync, across warps by per-warp counts.
//  3. perm/inv are written and the x rows are copied to x_sorted by bulk
//     copies: the block's rows stream into two shared-memory buffers (one
//     1-D bulk load per chunk of rows, issued before the wait on the router,
//     since x does not come from it), and each of a row's k copies leaves
//     by one bulk store to its sorted position.
constexpr int kScatterThreads = 256;
constexpr int kScatterWarps = kScatterThreads / 32;
constexpr int kScatterBufBytes = 16384;  // one of the two row staging buffers

// 1-D bulk copy of `bytes` (a multiple of 16) from global memory into shared
// memory, counted on the transaction barrier `bar`.
MOE_DEV void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16) from shared to global memory,
// in the bulk async group of the executing thread.
MOE_DEV void bulk_store_1d(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ hist, int T, int k, int E, int TB,
    int nblk,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, const uint16_t* __restrict__ x, uint16_t* __restrict__ xs, int D,
    unsigned int* dev_err) {
  extern __shared__ __align__(128) uint8_t sc_stage[];  // 2 x kScatterBufBytes when x is copied
  __shared__ uint64_t sc_full[2];
  __shared__ int sc_abort;
  __shared__ int s_red_pre[kScatterThreads];
  __shared__ int s_red_tot[kScatterThreads];
  __shared__ int s_base[MOE_MAX_EXPERTS];
  __shared__ int s_wcnt[kScatterWarps][MOE_MAX_EXPERTS];
  __shared__ int s_pos[64 * MOE_MAX_TOPK];

  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = T * k;

  // ---- 0. start streaming this block's x rows (chunks of RB rows) ----
  const int t0 = b * TB;
  const int ntok = min(TB, T - t0);
  const uint32_t rowb = static_cast<uint32_t>(D) * 2u;
  const int RB = max(1, kScatterBufBytes / static_cast<int>(rowb));
  const int nch = (x != nullptr && xs != nullptr) ? (ntok + RB - 1) / RB : 0;
  auto load_chunk = [&](int c) {  // one thread
    const int r0 = c * RB, nr = min(RB, ntok - r0);
    const uint32_t bar = smem_u32(&sc_full[c & 1]);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr) * rowb);
    bulk_load_1d(smem_u32(sc_stage + (c & 1) * kScatterBufBytes), x + static_cast<size_t>(t0 + r0) * D,
                 static_cast<uint32_t>(nr) * rowb, bar);
  };
  if (tid == 0) {
    sc_abort = 0;
    if (nch > 0) {
      mbar_init(smem_u32(&sc_full[0]), 1);
      mbar_init(smem_u32(&sc_full[1]), 1);
      fence_mbar_init();
      fence_proxy_async_smem();
      load_chunk(0);
      if (nch > 1) load_chunk(1);
    }
  }
  griddep_wait();  // ids and the block histogram come from the previous kernel
  griddep_launch_dependents();

  // ---- 1. column sums of the block histogram ----
  {
    const int R = kScatterThreads / E;  // E <= 128 -> R >= 2
    const int e = tid % E, r = tid / E;
    int pre = 0, tot = 0;
    if (r < R) {
      // eight independent loads in flight per batch (these L2 reads are latency-bound)
      for (int bb0 = r; bb0 < nblk; bb0 += 8 * R) {
        int hv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int bb = bb0 + u * R;
          hv[u] = bb < nblk ? hist[static_cast<size_t>(bb) * E + e] : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          tot += hv[u];
          if (bb0 + u * R < b) pre += hv[u];
        }
      }
    }
    s_red_pre[tid] = pre;
    s_red_tot[tid] = tot;
    __syncthreads();
    if (warp == 0) {
      // lane handles experts [lane*per, lane*per + per)
      const int per = (E + 31) / 32;
      int tot_e[4], pre_e[4];
      int local = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        tot_e[i] = pre_e[i] = 0;
        const int ee = lane * per + i;
        if (i < per && ee < E) {
          for (int rr = 0; rr < R; ++rr) {
            tot_e[i] += s_red_tot[rr * E + ee];
            pre_e[i] += s_red_pre[rr * E + ee];
          }
          local += tot_e[i];
        }
      }
      int incl = local;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      int run = incl - local;  // exclusive prefix of this lane's first expert
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ee = lane * per + i;
        if (i < per && ee < E) {
          s_base[ee] = run + pre_e[i];
          if (b == 0) {
            counts[ee] = tot_e[i];
            offsets[ee] = run;
          }
          run += tot_e[i];
        }
      }
      if (b == 0 && lane == 0) offsets[E] = S;
    }
  }

  // ---- 2. stable ranks ----
  const int s0 = b * TB * k;
  const int ns = min(TB * k, S - s0);
  for (int base = 0; base < ns; base += kScatterThreads) {
    for (int i = tid; i < kScatterWarps * E; i += kScatterThreads) s_wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int li = base + tid;
    const bool valid = li < ns;
    int ex = valid ? ids[s0 + li] : -1;
    if (static_cast<unsigned>(ex) >= static_cast<unsigned>(E)) ex = -1;  // not placed
    const unsigned peers = __match_any_sync(0xffffffffu, ex);
    const unsigned lt = (1u << lane) - 1u;
    const int rank = __popc(peers & lt);
    if (ex >= 0 && (__ffs(peers) - 1) == lane) s_wcnt[warp][ex] = __popc(peers);
    __syncthreads();
    if (valid && ex < 0) {
      inv[s0 + li] = 0;  // an id outside [0, E): the slot gets no row of its own
      s_pos[li] = -1;
    }
    if (ex >= 0) {
      int pos = s_base[ex] + rank;
      for (int w = 0; w < warp; ++w) pos += s_wcnt[w][ex];
      perm[pos] = s0 + li;
      inv[s0 + li] = pos;
      s_pos[li] = pos;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kScatterThreads) {
      int add = 0;
      for (int w = 0; w < kScatterWarps; ++w) add += s_wcnt[w][e];
      s_base[e] += add;
    }
    __syncthreads();
  }

  // ---- 3. copy rows: chunk c sits in buffer c % 2; its k copies per row
  // are bulk stores issued one per thread, and the buffer is refilled with
  // chunk c + 2 once every store has read it ----
  if (nch == 0) return;
  int c = 0;
  for (; c < nch; ++c) {
    const int r0 = c * RB, nr = min(RB, ntok - r0);
    const bool ok = mbar_wait(smem_u32(&sc_full[c & 1]), (c >> 1) & 1, &sc_abort, dev_err);
    if (!__syncthreads_and(ok)) break;
    const uint32_t sbuf = smem_u32(sc_stage + (c & 1) * kScatterBufBytes);
    for (int i = tid; i < nr * k; i += kScatterThreads) {
      const int pos = s_pos[r0 * k + i];
      if (pos >= 0) bulk_store_1d(xs + static_cast<size_t>(pos) * D, sbuf + (i / k) * rowb, rowb);
    }
    bulk_commit_group();
    if (c + 2 < nch) {
      bulk_wait_group_read0();  // this thread's stores have read the buffer
      __syncthreads();
      if (tid == 0) load_chunk(c + 2);
    }
  }
  if (c < nch && tid == 0) {
    // A wait gave up: let the loads still in flight land before the block
    // exits (bounded as well; the error word is already set).
    volatile int local_abort = 0;
    for (int cc = c; cc < nch && cc < c + 2; ++cc)
      mbar_wait(smem_u32(&sc_full[cc & 1]), (cc >> 1) & 1, &local_abort, dev_err);
  }
  bulk_wait_group0();
}

template <int NT, int KMAX>
static cudaError_t launch_route_nt(const uint16_t* x, const uint16_t* Wg, const uint4* wpack, bool self_pack,
                                   const float* bias, const moe_dims& d, int32_t* ids, float* w, int32_t* hist,
                                   cudaStream_t s, bool pdl) {
  const int TB = route_block_tokens(d.T);
  constexpr size_t red_bytes = static_cast<size_t>(8) * NT * 4 * 32 * sizeof(float);
  const size_t smem = red_bytes + (self_pack ? route_packed_bytes(d.D, d.E) : 0);
  if (red_bytes + kRouteSelfPackBytes > 48 * 1024) {
    static bool attr_done[64] = {false};
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[dev]) {
      cudaError_t e = cudaFuncSetAttribute(route_kernel<NT, KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(red_bytes + kRouteSelfPackBytes));
      if (e != cudaSuccess) return e;
      attr_done[dev] = true;
    }
  }
  return launch_kernel(route_kernel<NT, KMAX>, dim3(route_blocks(d.T)), dim3(kRouteThreads), smem, s, pdl, x,
                       Wg, wpack, self_pack ? 1 : 0, bias, d.T, d.D, d.E, d.k, TB, ids, w, hist);
}

template <int NT>
static cudaError_t launch_route_k(const uint16_t* x, const uint16_t* Wg, const uint4* wpack, bool self_pack,
                                  const float* bias, const moe_dims& d, int32_t* ids, float* w, int32_t* hist,
                                  cudaStream_t s, bool pdl) {
  if (d.k <= 2) return launch_route_nt<NT, 2>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
  if (d.k <= 4) return launch_route_nt<NT, 4>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
  if (d.k <= 8) return launch_route_nt<NT, 8>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
  return launch_route_nt<NT, 16>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
}

cudaError_t launch_route(const uint16_t* x, const uint16_t* Wg, const float* bias, const moe_dims& d,
                         void* wpack_buf, int32_t* ids, float* w, int32_t* hist, cudaStream_t s,
                         bool pdl) {
  const int NT = route_expert_tiles(d.E);
  uint4* wpack = static_cast<uint4*>(wpack_buf);
  // Small packed weights: every router block packs its own copy (one launch).
  // Otherwise a packing kernel writes them once and the router follows it.
  const bool self_pack = route_packed_bytes(d.D, d.E) <= kRouteSelfPackBytes;
  if (!self_pack) {
    const int nslots = (d.D / 32) * NT * 32;
    cudaError_t e = launch_kernel(pack_router_weights_kernel, dim3((nslots + 255) / 256), dim3(256), 0, s, pdl,
                                  Wg, d.D, d.E, NT, wpack);
    if (e != cudaSuccess) return e;
    pdl = true;
  }
  switch (NT) {
    case 1: return launch_route_k<1>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
    case 2: return launch_route_k<2>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
    case 4: return launch_route_k<4>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
    case 8: return launch_route_k<8>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
    default: return launch_route_k<16>(x, Wg, wpack, self_pack, bias, d, ids, w, hist, s, pdl);
  }
}

cudaError_t launch_hist(const int32_t* ids, const moe_dims& d, int32_t* hist, cudaStream_t s, bool pdl) {
  return launch_kernel(hist_kernel, dim3(route_blocks(d.T)), dim3(256), 0, s, pdl, ids, d.T, d.k, d.E,
                       route_block_tokens(d.T), hist);
}

// Device error word of the current device (cached per device).
static cudaError_t scatter_error_word(unsigned int** out) {
  static unsigned int* words[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (words[dev] == nullptr && (e = device_error_address(&words[dev])) != cudaSuccess) return e;
  *out = words[dev];
  return cudaSuccess;
}

cudaError_t launch_scatter(const int32_t* ids, const int32_t* hist, const moe_dims& d, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, const uint16_t* x,
                           uint16_t* x_sorted, cudaStream_t s, bool pdl) {
  const int nblk = route_blocks(d.T);
  unsigned int* dev_err = nullptr;
  cudaError_t e = scatter_error_word(&dev_err);
  if (e != cudaSuccess) return e;
  const size_t smem = (x != nullptr && x_sorted != nullptr) ? 2 * kScatterBufBytes : 0;
  return launch_kernel(scatter_kernel, dim3(nblk), dim3(kScatterThreads), smem, s, pdl, ids, hist, d.T, d.k,
                       d.E, route_block_tokens(d.T), nblk, counts, offsets, perm, inv, x, x_sorted, d.D, dev_err);
}

}  // namespace moe
