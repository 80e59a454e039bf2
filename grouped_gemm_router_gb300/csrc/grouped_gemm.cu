// Persistent ragged grouped GEMM on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
// Two epilogues share one engine:
//  * SwiGLU (W1||W3): for every sorted row p of expert e,
//      h[p] = silu(x_sorted[p] W1[e]) * (x_sorted[p] W3[e]).
//    One MMA of width N = 2 * hw computes the gate g (columns [0, hw)) and the
//    up-projection u (columns [hw, 2hw)) of the same hw output columns, so g
//    and u never leave the chip; the epilogue reads both from TMEM, applies
//    silu(g) * u in fp32 and stores bf16 h.  This is the fused W1/W3 + SiLU
//    stage of "Triton MoE Kernels & Memory Checkpointing", Part A, sections 2,
//    6.2 and 10, re-tiled for sm_103a (128-row tiles instead of 16).
//  * Down (W2): y[p] = h[p] W2[e], bf16 out.
// The always-on shared expert is one more group whose A operand is x itself
// (SwiGLU) or the shared rows of h (down), and whose B operand is its own
// weights; its outputs go to rows S .. S + T of h / y.
//
// Ragged groups: group g owns rows [row0_g, row0_g + n_g).  Its m-tiles load
// 128 rows with TMA starting at row0_g + 128 m; rows past the group belong to
// the next group (or are zero-filled past the tensor) and are simply not
// stored: the epilogue predicates each row.  The tile schedule is derived on
// the device from the offsets (no host synchronisation): tiles are numbered
// group by group, n fastest, and CTA b takes tiles b, b + grid, ...
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0     TMA producer (one lane)
//   warp 1     TMEM allocator + MMA issuer (one lane)
//   warps 2-9  epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 and the
//              columns of half (w - 2) / 4 of the tile
// Pipelines: kStages shared-memory stages (full / empty mbarriers) and two
// TMEM accumulators of 256 columns (tmem_full / tmem_empty), so the epilogue
// of one tile overlaps the MMAs of the next.
//
// Shared-memory operand layouts (TMA, 128-byte swizzle):
//   A tile 128 rows x 64 k (K-major): row r at byte 128 r, 8-row atoms of
//     1024 bytes -> descriptor SBO = 1024; the k-th 16-wide slice starts
//     32 k bytes into the tile.
//   B tile 64 k x N (N-major, straight from the [K, N] row-major weights):
//     N is split in 64-column boxes of 64 k-rows x 128 bytes (8 KB each);
//     LBO = 8192 (next 64 columns), SBO = 1024 (next 8 k-rows); the k-th
//     16-deep slice starts 2048 k bytes into the tile.
#include <cudaTypedefs.h>

#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;                      // rows per tile (TMEM lanes)
constexpr int kBK = 64;                       // k per stage (128 bytes of bf16)
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;        // 16 KB
constexpr int kBBytesMax = 256 * kBK * 2;     // 32 KB
constexpr int kStageBytes = kABytes + kBBytesMax;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kMaxGroups = MOE_MAX_EXPERTS + 1;
constexpr uint32_t kTmemCols = 512;           // two 256-column accumulators
constexpr int kSmemBytes = kStages * kStageBytes + 1024;

__device__ unsigned int g_device_error = 0;

struct GemmArgs {
  const int32_t* offsets;  // [E + 1]
  int E;                   // routed groups
  int S;                   // routed rows
  int T_shared;            // rows of the shared group (0: none)
  int K;                   // reduction length (multiple of 64)
  int N;                   // output columns
  int tile_n;              // MMA N: SwiGLU 2*hw, down = output tile width
  int shared_a_row0;       // first A row of the shared group in its tensor map
  uint16_t* C;             // output [S + T_shared, N]
};

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int tile_prefix[kMaxGroups + 1];
  int row0[kMaxGroups];
  int nrows[kMaxGroups];
};

template <bool kSwiGLU>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapA_sh,
                        const __grid_constant__ CUtensorMap mapB0,
                        const __grid_constant__ CUtensorMap mapB1,
                        const __grid_constant__ CUtensorMap mapB0_sh,
                        const __grid_constant__ CUtensorMap mapB1_sh, const GemmArgs p) {
  extern __shared__ uint8_t gemm_smem_raw[];
  __shared__ Ctl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.E + (p.T_shared > 0 ? 1 : 0);
  const int hw = kSwiGLU ? p.tile_n / 2 : p.tile_n;  // output columns per tile
  const int ntn = p.N / hw;
  const int nkb = p.K / kBK;

  // ---- group table and tile prefix ----
  for (int g = threadIdx.x; g < G; g += kThreads) {
    if (g < p.E) {
      const int a = p.offsets[g], b = p.offsets[g + 1];
      ctl.row0[g] = a;
      ctl.nrows[g] = b - a;
    } else {
      ctl.row0[g] = p.S;
      ctl.nrows[g] = p.T_shared;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (G + 31) / 32;  // <= 5
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < G) local += ((ctl.nrows[g] + kBM - 1) / kBM) * ntn;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < G) {
        ctl.tile_prefix[g] = run;
        run += ((ctl.nrows[g] + kBM - 1) / kBM) * ntn;
      }
    }
    if (lane == 31) {
      ctl.tile_prefix[G] = incl;
      ctl.total_tiles = incl;
    }
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(smem_u32(&ctl.full[s]), 1);
        mbar_init(smem_u32(&ctl.empty[s]), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(smem_u32(&ctl.tfull[b]), 1);
        mbar_init(smem_u32(&ctl.tempty[b]), kEpiWarps);
      }
      mbar_init(smem_u32(&ctl.drain), 1);
      ctl.abort = 0;
      fence_mbar_init();
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.total_tiles;
  volatile int* abort_flag = &ctl.abort;
  unsigned int* dev_err = &g_device_error;

  if (warp == 0) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapB0);
      if (kSwiGLU) tma_prefetch_desc(&mapB1);
      const uint64_t pol_a = l2_policy_evict_normal();
      const uint64_t pol_b = l2_policy_evict_last();
      const uint32_t stage_tx = static_cast<uint32_t>(kABytes + p.tile_n * kBK * 2);
      int stage = 0;
      uint32_t phase = 0;
      int g = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        while (tile >= ctl.tile_prefix[g + 1]) ++g;
        const int local = tile - ctl.tile_prefix[g];
        const int m = local / ntn, n = local - m * ntn;
        const bool routed = g < p.E;
        const CUtensorMap* mA = routed ? &mapA : &mapA_sh;
        const CUtensorMap* mB0 = routed ? &mapB0 : &mapB0_sh;
        const CUtensorMap* mB1 = routed ? &mapB1 : &mapB1_sh;
        const int a_row = (routed ? ctl.row0[g] : p.shared_a_row0) + m * kBM;
        const int b_row0 = routed ? g * p.K : 0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&ctl.full[stage]);
          const uint32_t sa = smem_base + stage * kStageBytes;
          const uint32_t sb = sa + kABytes;
          mbar_arrive_expect_tx(full, stage_tx);
          tma_load_2d(sa, mA, full, kb * kBK, a_row, pol_a);
          const int brow = b_row0 + kb * kBK;
          if (kSwiGLU) {
            const int nch = hw / 64;
            for (int cch = 0; cch < nch; ++cch) {
              tma_load_2d(sb + cch * 8192, mB0, full, n * hw + cch * 64, brow, pol_b);
              tma_load_2d(sb + (nch + cch) * 8192, mB1, full, n * hw + cch * 64, brow, pol_b);
            }
          } else {
            const int nch = p.tile_n / 64;
            for (int cch = 0; cch < nch; ++cch)
              tma_load_2d(sb + cch * 8192, mB0, full, n * hw + cch * 64, brow, pol_b);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        int st = stage;
        uint32_t ph = phase;
        for (int i = 0; i < kStages && i < issued; ++i) {
          if (--st < 0) {
            st = kStages - 1;
            ph ^= 1u;
          }
          volatile int local_abort = 0;
          mbar_wait(smem_u32(&ctl.full[st]), ph, &local_abort, dev_err);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===================== MMA issuer =====================
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, static_cast<uint32_t>(p.tile_n), 1u);
      int stage = 0;
      uint32_t phase = 0;
      int i = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++i) {
        const int buf = i & 1;
        const uint32_t tph = (i >> 1) & 1;
        if (!mbar_wait(smem_u32(&ctl.tempty[buf]), tph ^ 1u, abort_flag, dev_err)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * 256;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_base + stage * kStageBytes;
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(sb + kk * 2048, 8192, 1024);
            umma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&ctl.empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&ctl.tfull[buf]));
      }
      // All MMAs issued by this thread are complete once `drain` flips.
      umma_commit(smem_u32(&ctl.drain));
      volatile int local_abort = 0;
      mbar_wait(smem_u32(&ctl.drain), 0, &local_abort, dev_err);
    }
    __syncwarp();
  } else {
    // ===================== epilogue =====================
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the tile's columns
    const int r_in_tile = q * 32 + lane;
    int g = 0;
    int i = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++i) {
      while (tile >= ctl.tile_prefix[g + 1]) ++g;
      const int local = tile - ctl.tile_prefix[g];
      const int m = local / ntn, n = local - m * ntn;
      const int buf = i & 1;
      const uint32_t tph = (i >> 1) & 1;
      const bool got = mbar_wait(smem_u32(&ctl.tfull[buf]), tph, abort_flag, dev_err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const int row = m * kBM + r_in_tile;
      const bool valid = row < ctl.nrows[g];
      uint16_t* crow = p.C + static_cast<size_t>(ctl.row0[g] + (valid ? row : 0)) * p.N + n * hw;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * 256;
      const int c_lo = half * (hw / 2), c_hi = c_lo + hw / 2;
      if (kSwiGLU) {
        for (int cc = c_lo; cc < c_hi; cc += 32) {
          uint32_t rg[32], ru[32];
          tmem_ld_32cols(taddr + cc, rg);
          tmem_ld_32cols(taddr + hw + cc, ru);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float g0 = __uint_as_float(rg[2 * j]), g1 = __uint_as_float(rg[2 * j + 1]);
            const float u0 = __uint_as_float(ru[2 * j]), u1 = __uint_as_float(ru[2 * j + 1]);
            // silu(g) = g / (1 + exp(-g)); the fast division returns 0 when
            // exp(-g) overflows, which is the limit of silu for g -> -inf.
            const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
            packed[j] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(crow + cc);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
          }
        }
      } else {
        for (int cc = c_lo; cc < c_hi; cc += 32) {
          uint32_t ra[32];
          tmem_ld_32cols(taddr + cc, ra);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            packed[j] = pack_bf16x2(__uint_as_float(ra[2 * j]), __uint_as_float(ra[2 * j + 1]));
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(crow + cc);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl.tempty[buf]));
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
  if (g_encode != nullptr) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

// 2-D bf16 tensor map of a row-major [rows, cols] matrix, box {box_cols, box_rows},
// 128-byte swizzle, zero fill outside the tensor.
cudaError_t make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     uint32_t box_cols) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct DeviceInfo {
  int device = -1;
  int sms = 0;
  bool attrs_set = false;
};
DeviceInfo g_dev[64];

cudaError_t device_setup(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  DeviceInfo& di = g_dev[dev];
  if (!di.attrs_set) {
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(grouped_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(grouped_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    di.attrs_set = true;
  }
  *sms = di.sms;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_grouped_swiglu(const uint16_t* x_sorted, const uint16_t* x, const uint16_t* W1,
                                  const uint16_t* W3, const uint16_t* Ws1, const uint16_t* Ws3,
                                  const int32_t* offsets, const moe_dims& d, uint16_t* h,
                                  cudaStream_t s) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  int sms = 0;
  if ((e = device_setup(&sms)) != cudaSuccess) return e;
  const int S = d.T * d.k;
  const bool shared = Ws1 != nullptr;
  const int hw = (d.F % 128 == 0) ? 128 : 64;
  CUtensorMap mA, mAs, mB0, mB1, mB0s, mB1s;
  if ((e = make_map(&mA, x_sorted, S, d.D, kBM, kBK)) != cudaSuccess) return e;
  if ((e = make_map(&mB0, W1, static_cast<uint64_t>(d.E) * d.D, d.F, kBK, 64)) != cudaSuccess) return e;
  if ((e = make_map(&mB1, W3, static_cast<uint64_t>(d.E) * d.D, d.F, kBK, 64)) != cudaSuccess) return e;
  if (shared) {
    if ((e = make_map(&mAs, x, d.T, d.D, kBM, kBK)) != cudaSuccess) return e;
    if ((e = make_map(&mB0s, Ws1, d.D, d.F, kBK, 64)) != cudaSuccess) return e;
    if ((e = make_map(&mB1s, Ws3, d.D, d.F, kBK, 64)) != cudaSuccess) return e;
  } else {
    mAs = mA;
    mB0s = mB0;
    mB1s = mB1;
  }
  GemmArgs a;
  a.offsets = offsets;
  a.E = d.E;
  a.S = S;
  a.T_shared = shared ? d.T : 0;
  a.K = d.D;
  a.N = d.F;
  a.tile_n = 2 * hw;
  a.shared_a_row0 = 0;
  a.C = h;
  grouped_gemm_kernel<true><<<sms, kThreads, kSmemBytes, s>>>(mA, mAs, mB0, mB1, mB0s, mB1s, a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_grouped_down(const uint16_t* h, const uint16_t* W2, const uint16_t* Ws2,
                                const int32_t* offsets, const moe_dims& d, uint16_t* y,
                                cudaStream_t s) {
  cudaError_t e = get_encoder();
  if (e != cudaSuccess) return e;
  int sms = 0;
  if ((e = device_setup(&sms)) != cudaSuccess) return e;
  const int S = d.T * d.k;
  const bool shared = Ws2 != nullptr;
  const int tn = (d.D % 256 == 0) ? 256 : (d.D % 128 == 0) ? 128 : 64;
  const uint64_t hrows = static_cast<uint64_t>(S) + (shared ? d.T : 0);
  CUtensorMap mA, mB0, mB0s;
  if ((e = make_map(&mA, h, hrows, d.F, kBM, kBK)) != cudaSuccess) return e;
  if ((e = make_map(&mB0, W2, static_cast<uint64_t>(d.E) * d.F, d.D, kBK, 64)) != cudaSuccess) return e;
  if (shared) {
    if ((e = make_map(&mB0s, Ws2, d.F, d.D, kBK, 64)) != cudaSuccess) return e;
  } else {
    mB0s = mB0;
  }
  GemmArgs a;
  a.offsets = offsets;
  a.E = d.E;
  a.S = S;
  a.T_shared = shared ? d.T : 0;
  a.K = d.F;
  a.N = d.D;
  a.tile_n = tn;
  a.shared_a_row0 = S;
  a.C = y;
  grouped_gemm_kernel<false><<<sms, kThreads, kSmemBytes, s>>>(mA, mA, mB0, mB0, mB0s, mB0s, a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t read_clear_device_error(unsigned int* value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

}  // namespace moe
