// Persistent ragged grouped GEMM on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in TMEM, operands staged by TMA), run by CTA
// pairs (clusters of two CTAs on two SMs, cta_group::2).
//
// Two epilogues share one engine:
//  * SwiGLU (W1||W3): for every sorted row p of expert e,
//      h[p] = silu(x_sorted[p] W1[e]) * (x_sorted[p] W3[e]).
//    One MMA of width N = 2 * hw computes the gate g (columns [0, hw)) and the
//    up-projection u (columns [hw, 2hw)) of the same hw output columns, so g
//    and u never leave the chip; the epilogue reads both from TMEM, applies
//    silu(g) * u in fp32 and stores bf16 h.  This is the fused W1/W3 + SiLU
//    stage of "Triton MoE Kernels & Memory Checkpointing", Part A, sections 2,
//    6.2 and 10, re-tiled for sm_103a (256-row pair tiles instead of 16).
//  * Down (W2): y[p] = h[p] W2[e], bf16 out.
// The always-on shared expert is one more group whose A operand is x itself
// (SwiGLU) or the shared rows of h (down), and whose B operand is its own
// weights; its h goes to rows S .. S + T of h (bf16), its down-projection to
// ys [T, D] in fp32: it enters the layer's output with weight 1, so it is
// the one intermediate that keeps its fp32 accumulation.
//
// Ragged groups: group g owns rows [row0_g, row0_g + n_g).  Its m-tiles load
// 256 rows with TMA starting at row0_g + 256 m; rows past the group belong to
// the next group (or are zero-filled past the tensor) and are simply not
// stored: the epilogue predicates each row (and each 32-column chunk past N).
// When a group's last m-tile has at most 128 rows, the peer CTA loads no A
// rows at all and its epilogue warps skip their TMEM reads: with many small
// groups (64 experts of ~128 rows) that halves the A stream, the bottleneck
// when the weights come from HBM.
// The tile schedule is derived on the device from the offsets (no host
// synchronisation): tiles are numbered group by group, n fastest, and pair c
// takes tiles c, c + pairs, ...
//
// CTA pair: CTA r holds rows [128 r, 128 r + 128) of the A tile and columns
// [r N/2, (r+1) N/2) of the B tile; the leader (r = 0) issues one
// tcgen05.mma.cta_group::2 per 16-deep k-slice, which writes each CTA's 128
// rows of D into that CTA's own TMEM.  Per SM, a 128x256 output tile then
// stages 16 KB of A and 16 KB of B per 64 k instead of 16 + 32 KB.
//
// Warp roles (64 + 32 kEpiWarps threads per CTA, one CTA per SM):
//   warp 0     TMA producer (one lane) -- both CTAs load their own halves
//   warp 1     TMEM allocator; MMA issuer (one lane, leader only)
//   warps 2-   epilogue (kEpiWarps): warp w reads TMEM lanes 32 (w % 4) .. + 31
//              and the columns of part (w - 2) / 4 of the tile
// Pipelines: a ring of shared-memory stages (full / empty mbarriers; 3 stages
// of 128 k for W1||W3, 6 of 64 k for W2, 192 KB either way) and two TMEM
// accumulators of 256 columns (tmem_full / tmem_empty), so the epilogue of
// one tile overlaps the MMAs of the next.
//
// Shared-memory operand layouts (TMA, 128-byte swizzle), per 64 k (one
// swizzle atom; a 128-deep stage holds two of each, back to back):
//   A 128 rows x 64 k (K-major): row r at byte 128 r, 8-row atoms of 1024
//     bytes -> descriptor SBO = 1024; the k-th 16-wide slice starts 32 k
//     bytes into the atom.  One 3-D TMA box {64, 128 rows, kBK / 64 atoms}
//     over the view {64, rows, K / 64} (strides K * 2 and 128 bytes) loads a
//     stage's atoms.
//   B kBK k x N/2 (N-major, straight from the [K, N] row-major weights): N/2
//     is split in 64-column blocks of kBK k-rows x 128 bytes; LBO = one block
//     (next 64 columns), SBO = 1024 (next 8 k-rows); the k-th 16-deep slice
//     starts 2048 k bytes into a block.  One 3-D TMA box {64 columns, kBK
//     rows, N/128 blocks} over the view {64, K rows, N / 64} (strides N * 2
//     and 128 bytes) lands the blocks in that order.
// A stage thus costs each CTA two TMA operations: per byte, the 128-deep
// stages of W1||W3 issue half as many as 64-deep ones would.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

namespace {

constexpr int kAtomK = 64;                     // k of one 128-byte swizzle atom (128 bytes of bf16)
#ifndef MOE_EPI_WARPS
#define MOE_EPI_WARPS 8
#endif
constexpr int kEpiWarps = MOE_EPI_WARPS;      // epilogue warps per CTA (8 or 16)
constexpr int kEpiParts = kEpiWarps / 4;      // column parts per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxGroups = MOE_MAX_EXPERTS + 1;
constexpr uint32_t kTmemCols = 512;           // two 256-column accumulators

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
  uint16_t* C;             // output [S + T_shared, N] (down: [S, N])
  float* Cs;               // down: the shared group's output [T_shared, N] in fp32
};


// ---------------------------------------------------------------------------
// Barriers: full[s] lives in the leader and counts both CTAs' TMA bytes;
// empty[s] and tfull[b] live in both CTAs and are signalled by the leader's
// multicast commit; tempty[b] lives in the leader and counts the epilogue
// warps of both CTAs.
// ---------------------------------------------------------------------------
constexpr int kPairBM = 256;                  // rows per pair tile
constexpr int kMaxPairStages = 6;
// The stage ring: 192 KB per CTA either way, three 128-deep stages (two
// swizzle atoms of A and of B, one TMA operation each) or six 64-deep ones.
// Halving the TMA operations per byte took W1||W3 from 277 to 258 us on
// gptoss_lite; W2, whose A rows come from HBM, ran 146 -> 149 us with them.
// So W1||W3 stages 128 k and W2 64 k -- W1||W3 too when D % 128 != 0, where
// the last deep stage would read the next expert's W1 / W3 rows (multiplied
// by zeros, but an inf there would still reach this expert's output).
template <bool kDeep>
struct Ring {
  static constexpr int kBK = kDeep ? 128 : 64;            // k per stage
  static constexpr int kStages = kDeep ? 3 : 6;
  static constexpr int kABytes = 128 * kBK * 2;           // this CTA's 128 rows
  static constexpr int kBBytesMax = 128 * kBK * 2;        // this CTA's half of N <= 256
  static constexpr int kStageBytes = kABytes + kBBytesMax;
};
constexpr int kOutBoxRows = 32;                 // one epilogue warp's rows
constexpr int kOutBoxCols = 32;                 // columns per TMA store box (64 bytes)
constexpr int kOutBoxBytes = kOutBoxRows * kOutBoxCols * 2;
constexpr int kOutBufs = 1;                      // staging buffers per epilogue warp
// Output columns per tile: SwiGLU hw = 128 (g and u make the MMA's N = 256),
// down <= 256.  Each epilogue warp holds its share of the accumulator
// columns in registers at once: kMaxBoxes 32-column boxes, kAccRegs values.
template <bool kSwiGLU>
struct EpiShape {
  static constexpr int kMaxBoxes = (kSwiGLU ? 128 : 256) / kEpiParts / kOutBoxCols;
  static constexpr int kAccRegs = kMaxBoxes * 32 * (kSwiGLU ? 2 : 1);
};
template <bool kDeep>
constexpr int pair_smem_bytes() {
  return Ring<kDeep>::kStages * Ring<kDeep>::kStageBytes + kEpiWarps * kOutBufs * kOutBoxBytes + 1024;
}

struct PairCtl {
  uint64_t full[kMaxPairStages];
  uint64_t empty[kMaxPairStages];
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

template <bool kSwiGLU, bool kDeep>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap mapA,
                             const __grid_constant__ CUtensorMap mapA_sh,
                             const __grid_constant__ CUtensorMap mapB0,
                             const __grid_constant__ CUtensorMap mapB1,
                             const __grid_constant__ CUtensorMap mapB0_sh,
                             const __grid_constant__ CUtensorMap mapB1_sh,
                             const __grid_constant__ CUtensorMap mapC,
                             const __grid_constant__ CUtensorMap mapCs, const GemmArgs p) {
  extern __shared__ uint8_t gemm_smem_raw[];
  __shared__ PairCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = leader, 1 = peer
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());
  const int G = p.E + (p.T_shared > 0 ? 1 : 0);
  const int hw = kSwiGLU ? p.tile_n / 2 : p.tile_n;  // output columns per tile
  const int ntn = (p.N + hw - 1) / hw;
  constexpr int kBK = Ring<kDeep>::kBK;
  constexpr int kPairStages = Ring<kDeep>::kStages;
  constexpr int kPairABytes = Ring<kDeep>::kABytes;
  constexpr int kPairStageBytes = Ring<kDeep>::kStageBytes;
  const int nkb = (p.K + kBK - 1) / kBK;  // a K of 64 mod 128 reads zeros past D (TMA fill)
  const int half_n = p.tile_n / 2;                    // B columns staged by this CTA
  constexpr int kMaxBoxes = EpiShape<kSwiGLU>::kMaxBoxes;
  constexpr int kAccRegs = EpiShape<kSwiGLU>::kAccRegs;

  // ---- setup that reads nothing produced by earlier kernels ----
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB0);
    if (kSwiGLU) tma_prefetch_desc(&mapB1);
    for (int st = 0; st < kPairStages; ++st) {
      mbar_init(smem_u32(&ctl.full[st]), 1);
      mbar_init(smem_u32(&ctl.empty[st]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl.tfull[b]), 1);
      mbar_init(smem_u32(&ctl.tempty[b]), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(&ctl.drain), 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&ctl.tmem_base), kTmemCols);
    tmem_relinquish_pair();
    tc_fence_before_sync();
  }
  griddep_launch_dependents();
  griddep_wait();  // offsets and the A operand come from earlier kernels

  // ---- group table and tile prefix (identical in both CTAs) ----
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
    const int per = (G + 31) / 32;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < G) local += ((ctl.nrows[g] + kPairBM - 1) / kPairBM) * ntn;
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
        run += ((ctl.nrows[g] + kPairBM - 1) / kPairBM) * ntn;
      }
    }
    if (lane == 31) {
      ctl.tile_prefix[G] = incl;
      ctl.total_tiles = incl;
    }
  }
  // barrier inits, the tile table and the TMEM allocation visible to both CTAs
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.total_tiles;
  volatile int* abort_flag = &ctl.abort;
  unsigned int* dev_err = &g_device_error;

  if (warp == 0) {
    // ===================== TMA producer (both CTAs) =====================
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_normal();
      const uint64_t pol_b = l2_policy_evict_last();
      const uint32_t b_tx = 2u * static_cast<uint32_t>(half_n * kBK * 2);
      int stage = 0;
      uint32_t phase = 0;
      int g = 0;
      int issued = 0;
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += npairs) {
        while (tile >= ctl.tile_prefix[g + 1]) ++g;
        const int local = tile - ctl.tile_prefix[g];
        const int m = local / ntn, n = local - m * ntn;
        const bool routed = g < p.E;
        const CUtensorMap* mA = routed ? &mapA : &mapA_sh;
        const int a_row = (routed ? ctl.row0[g] : p.shared_a_row0) + m * kPairBM + 128 * rank;
        const int b_row0 = routed ? g * p.K : 0;
        // A tile whose rows all lie past the group's end (the peer's half of
        // the last m-tile of a group of <= 128 more rows) is not loaded: those
        // rows are never stored, so the MMA may read stale shared memory.
        const bool peer_a = ctl.nrows[g] - m * kPairBM > 128;
        const bool load_a = leader || peer_a;
        const uint32_t pair_tx = b_tx + static_cast<uint32_t>(kPairABytes) * (peer_a ? 2u : 1u);
        // this CTA's B columns
        const CUtensorMap* mB;
        int bcol;
        if (kSwiGLU) {
          mB = leader ? (routed ? &mapB0 : &mapB0_sh) : (routed ? &mapB1 : &mapB1_sh);
          bcol = n * hw;
        } else {
          mB = routed ? &mapB0 : &mapB0_sh;
          bcol = n * hw + half_n * rank;
        }
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = map_to_cta(smem_u32(&ctl.full[stage]), 0);
          const uint32_t sa = smem_base + stage * kPairStageBytes;
          const uint32_t sb = sa + kPairABytes;
          if (leader) mbar_arrive_expect_tx(smem_u32(&ctl.full[stage]), pair_tx);
          if (load_a) tma_load_3d_pair(sa, mA, full_leader, 0, a_row, kb * (kBK / kAtomK), pol_a);
          const int brow = b_row0 + kb * kBK;
          tma_load_3d_pair(sb, mB, full_leader, 0, brow, bcol / 64, pol_b);
          ++issued;
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // Let the copies already in flight land before the CTA exits.
        int st = stage;
        uint32_t ph = phase;
        for (int i = 0; i < kPairStages && i < issued; ++i) {
          if (--st < 0) {
            st = kPairStages - 1;
            ph ^= 1u;
          }
          volatile int local_abort = 0;
          mbar_wait_cluster(smem_u32(&ctl.full[st]), ph, &local_abort, dev_err);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===================== MMA issuer (leader only) =====================
    if (lane == 0 && leader) {
      const uint32_t idesc = idesc_bf16_f32(kPairBM, static_cast<uint32_t>(p.tile_n), 1u);
      int stage = 0;
      uint32_t phase = 0;
      int i = 0;
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += npairs, ++i) {
        const int buf = i & 1;
        const uint32_t tph = (i >> 1) & 1;
        if (!mbar_wait_cluster(smem_u32(&ctl.tempty[buf]), tph ^ 1u, abort_flag, dev_err)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * 256;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(smem_u32(&ctl.full[stage]), phase, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_base + stage * kPairStageBytes;
          const uint32_t sb = sa + kPairABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // A: k-atom kk / 4 (128 rows x 128 bytes each), 16-wide slice kk % 4;
            // B: 64-column blocks of kBK k-rows (LBO = one block), slice kk
            const uint64_t adesc = smem_desc_sw128(sa + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(sb + kk * 2048, kBK * 128, 1024);
            umma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&ctl.empty[stage]), 0x3);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&ctl.tfull[buf]), 0x3);
      }
      // All MMAs issued by this thread are complete once `drain` flips.
      umma_commit_pair(smem_u32(&ctl.drain), 0x1);
      volatile int local_abort = 0;
      mbar_wait_cluster(smem_u32(&ctl.drain), 0, &local_abort, dev_err);
    }
    __syncwarp();
  } else {
    // ===================== epilogue (both CTAs) =====================
    // Warp w owns TMEM lanes 32 (w % 4) .. + 31 (32 output rows) and part
    // (w - 2) / 4 of the tile's columns, in boxes of 32 columns.  A box whose
    // 32 rows all belong to the group is written through a 64B-swizzled
    // staging buffer with one TMA store; a box that crosses the group's end is
    // stored row by row for its valid rows only.
    const int q = warp & 3;
    const int part = (warp - 2) >> 2;
    const int r_in_tile = 128 * static_cast<int>(rank) + q * 32 + lane;
    const uint32_t tempty_leader0 = map_to_cta(smem_u32(&ctl.tempty[0]), 0);
    const uint32_t tempty_leader1 = map_to_cta(smem_u32(&ctl.tempty[1]), 0);
    uint8_t* stage_out =
        smem + kPairStages * kPairStageBytes + (warp - 2) * kOutBufs * kOutBoxBytes;
    int obuf = 0;
    int g = 0;
    int i = 0;
    for (int tile = pair; tile < total; tile += npairs, ++i) {
      while (tile >= ctl.tile_prefix[g + 1]) ++g;
      const int local = tile - ctl.tile_prefix[g];
      const int m = local / ntn, n = local - m * ntn;
      const int buf = i & 1;
      const uint32_t tph = (i >> 1) & 1;
      const bool got = mbar_wait_cluster(smem_u32(&ctl.tfull[buf]), tph, abort_flag, dev_err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const int row = m * kPairBM + r_in_tile;
      const int nrows_g = ctl.nrows[g];
      const bool valid = row < nrows_g;
      const int warp_row0 = m * kPairBM + 128 * static_cast<int>(rank) + q * 32;
      const bool full_box = warp_row0 + kOutBoxRows <= nrows_g;
      const int col0 = n * hw;
      const bool f32_rows = !kSwiGLU && g >= p.E;  // the shared expert's down-projection: fp32
      uint16_t* crow = p.C + static_cast<size_t>(ctl.row0[g] + (valid ? row : 0)) * p.N + col0;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * 256;
      const int cols_per_part = hw / kEpiParts;
      const int c_first = part * cols_per_part;
      // a warp whose 32 rows all lie past the group's end has nothing to store
      const int nbox = warp_row0 < nrows_g ? cols_per_part / kOutBoxCols : 0;
      // All of this warp's accumulator columns are read in one burst with a
      // single wait, and the accumulator is handed back to the MMA issuer
      // before any math or store.  (A wait after every 32-column box cost
      // the MMAs ~14% of their cycles.)
      uint32_t acc[kAccRegs / 32][32];
      if (nbox > 0) {
#pragma unroll
        for (int b = 0; b < kMaxBoxes; ++b) {
          if (b < nbox) {
            if (kSwiGLU) {
              tmem_ld_32cols(taddr + c_first + b * kOutBoxCols, acc[2 * b]);
              tmem_ld_32cols(taddr + hw + c_first + b * kOutBoxCols, acc[2 * b + 1]);
            } else {
              tmem_ld_32cols(taddr + c_first + b * kOutBoxCols, acc[b]);
            }
          }
        }
        tmem_ld_wait();
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(buf ? tempty_leader1 : tempty_leader0);
#pragma unroll
      for (int b = 0; b < kMaxBoxes; ++b) {
        const int cc = c_first + b * kOutBoxCols;
        if (b >= nbox || col0 + cc >= p.N) break;  // past the group, or past the last column
        if (!kSwiGLU && f32_rows) {
          if (full_box)
            store_box_f32_tma(&mapCs, stage_out, acc[b], col0 + cc, warp_row0);
          else if (valid)
            store_row_f32(p.Cs + static_cast<size_t>(row) * p.N + col0 + cc, acc[b]);
          continue;
        }
        uint32_t packed[16];
        if (kSwiGLU) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float g0 = __uint_as_float(acc[2 * b][2 * j]), g1 = __uint_as_float(acc[2 * b][2 * j + 1]);
            const float u0 = __uint_as_float(acc[2 * b + 1][2 * j]), u1 = __uint_as_float(acc[2 * b + 1][2 * j + 1]);
            // silu(g) = g / (1 + exp(-g)); the fast division returns 0 when
            // exp(-g) overflows, which is the limit of silu for g -> -inf.
            const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
            packed[j] = pack_bf16x2(h0, h1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            packed[j] = pack_bf16x2(__uint_as_float(acc[b][2 * j]), __uint_as_float(acc[b][2 * j + 1]));
        }
        if (full_box) {
          // the store issued kOutBufs boxes ago has finished reading this buffer
          if (kOutBufs == 2)
            bulk_wait_group_read1();
          else
            bulk_wait_group_read0();
          __syncwarp();
          uint8_t* sbuf = stage_out + obuf * kOutBoxBytes;
          // 64B swizzle: 16-byte chunk c of row r lives at chunk c ^ ((r / 2) % 4)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4* dst = reinterpret_cast<uint4*>(sbuf + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4));
            *dst = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&mapC, smem_u32(sbuf), col0 + cc, ctl.row0[g] + warp_row0);
            bulk_commit_group();
          }
          obuf ^= (kOutBufs - 1);
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(crow + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  // Both CTAs done with TMEM and with each other's barriers before freeing.
  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Guards the lazily filled per-process / per-device state below.
std::mutex g_setup_mu;

cudaError_t get_encoder() {  // caller holds g_setup_mu
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
// 128-byte swizzle (64-byte for 32-column boxes), zero fill outside the tensor.
cudaError_t make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     uint32_t box_cols) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_cols * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D bf16 tensor map of the weights [rows, cols] (cols % 64 == 0) viewed as
// {64 columns, rows, cols / 64 column blocks}: a box {64, 64, nblk} holds nblk
// consecutive 64-column blocks of 64 rows, each block 8 KB in shared memory
// with the 128-byte swizzle; blocks past the last column read zeros.
cudaError_t make_weight_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t nblk,
                            uint32_t box_rows = 64) {
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, box_rows, nblk};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// An upper bound of the pair tiles of one launch, from the shape alone: each
// of the G groups adds at most one partial 256-row m-tile.  Pairs past it
// would find no tile, so the grid is capped by it (tiny layers).
int max_pair_tiles(long rows, int groups, int ntn) {
  const long mt = (rows + static_cast<long>(groups) * (kPairBM - 1)) / kPairBM;
  const long t = mt * ntn;
  return t > (1 << 30) ? (1 << 30) : static_cast<int>(t);
}

struct DeviceInfo {
  int device = -1;
  int sms = 0;
  int pair_clusters[3] = {0, 0, 0};  // co-resident CTA pairs: [down, swiglu, swiglu deep]
  bool attrs_set = false;
};
DeviceInfo g_dev[64];

template <bool kSwiGLU, bool kDeep>
cudaError_t launch_pair(int nclusters, const CUtensorMap& a, const CUtensorMap& as,
                        const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& b0s,
                        const CUtensorMap& b1s, const CUtensorMap& c, const CUtensorMap& cs,
                        const GemmArgs& args, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * nclusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes<kDeep>();
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<kSwiGLU, kDeep>, a, as, b0, b1, b0s, b1s, c, cs, args);
}

// One-time set-up of the current device (kernel attributes, co-resident
// cluster counts, the tensor-map encoder); returns a copy of its state.
cudaError_t device_setup(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if ((e = get_encoder()) != cudaSuccess) return e;
  DeviceInfo& di = g_dev[dev];
  if (!di.attrs_set) {
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // [0] W2, [1] W1||W3 with 64-deep stages, [2] W1||W3 with 128-deep stages
    for (int sw = 0; sw < 3; ++sw) {
      const void* fn = sw == 2   ? reinterpret_cast<const void*>(grouped_gemm_pair_kernel<true, true>)
                       : sw == 1 ? reinterpret_cast<const void*>(grouped_gemm_pair_kernel<true, false>)
                                 : reinterpret_cast<const void*>(grouped_gemm_pair_kernel<false, false>);
      const int smem = sw == 2 ? pair_smem_bytes<true>() : pair_smem_bytes<false>();
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (di.sms / 2), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int nclusters = 0;
      e = cudaOccupancyMaxActiveClusters(&nclusters, fn, &cfg);
      if (e != cudaSuccess) return e;
      if (nclusters < 1) return cudaErrorInvalidConfiguration;
      di.pair_clusters[sw] = nclusters;
    }
    di.attrs_set = true;
  }
  *out = di;
  return cudaSuccess;
}

}  // namespace

cudaError_t tensor_map_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                          uint32_t box_rows, uint32_t box_cols) {
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
  }
  return make_map(m, ptr, rows, cols, box_rows, box_cols);
}

cudaError_t tensor_map_blocks(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t nblk,
                              uint32_t box_rows) {
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
  }
  return make_weight_map(m, ptr, rows, cols, nblk, box_rows);
}

cudaError_t tensor_map_f32_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint32_t box0, uint32_t box1) {
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
  }
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = box0 * 4 == 64    ? CU_TENSOR_MAP_SWIZZLE_64B
                                : box0 * 4 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                  : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t device_error_address(unsigned int** p) {
  void* a = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&a, g_device_error);
  *p = static_cast<unsigned int*>(a);
  return e;
}

cudaError_t launch_grouped_swiglu(const uint16_t* x_sorted, const uint16_t* x, const uint16_t* W1,
                                  const uint16_t* W3, const uint16_t* Ws1, const uint16_t* Ws3,
                                  const int32_t* offsets, const moe_dims& d, uint16_t* h,
                                  cudaStream_t s, bool pdl) {
  DeviceInfo di;
  cudaError_t e = device_setup(&di);
  if (e != cudaSuccess) return e;
  const int S = d.T * d.k;
  const bool shared = Ws1 != nullptr;
  const int hw = 128;  // the last tile is half empty when F % 128 == 64
  CUtensorMap mA, mAs, mB0, mB1, mB0s, mB1s;
  const bool deep = d.D % 128 == 0;
  const int kBK = deep ? Ring<true>::kBK : Ring<false>::kBK;
  if ((e = make_weight_map(&mA, x_sorted, S, d.D, kBK / kAtomK, 128)) != cudaSuccess) return e;
  if ((e = make_weight_map(&mB0, W1, static_cast<uint64_t>(d.E) * d.D, d.F, hw / 64, kBK)) != cudaSuccess) return e;
  if ((e = make_weight_map(&mB1, W3, static_cast<uint64_t>(d.E) * d.D, d.F, hw / 64, kBK)) != cudaSuccess) return e;
  if (shared) {
    if ((e = make_weight_map(&mAs, x, d.T, d.D, kBK / kAtomK, 128)) != cudaSuccess) return e;
    if ((e = make_weight_map(&mB0s, Ws1, d.D, d.F, hw / 64, kBK)) != cudaSuccess) return e;
    if ((e = make_weight_map(&mB1s, Ws3, d.D, d.F, hw / 64, kBK)) != cudaSuccess) return e;
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
  a.Cs = nullptr;
  CUtensorMap mC;
  if ((e = make_map(&mC, h, static_cast<uint64_t>(S) + (shared ? d.T : 0), d.F, kOutBoxRows, kOutBoxCols)) !=
      cudaSuccess)
    return e;
  const int groups1 = d.E + (shared ? 1 : 0);
  const int pairs1 = std::min(di.pair_clusters[deep ? 2 : 1],
                              max_pair_tiles(static_cast<long>(S) + (shared ? d.T : 0), groups1, (d.F + hw - 1) / hw));
  e = deep ? launch_pair<true, true>(pairs1, mA, mAs, mB0, mB1, mB0s, mB1s, mC, mC, a, s, pdl)
           : launch_pair<true, false>(pairs1, mA, mAs, mB0, mB1, mB0s, mB1s, mC, mC, a, s, pdl);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_grouped_down(const uint16_t* h, const uint16_t* W2, const uint16_t* Ws2,
                                const int32_t* offsets, const moe_dims& d, uint16_t* y, float* ys,
                                cudaStream_t s, bool pdl) {
  DeviceInfo di;
  cudaError_t e = device_setup(&di);
  if (e != cudaSuccess) return e;
  const int S = d.T * d.k;
  const bool shared = Ws2 != nullptr;
  // D % 128 == 64: 128-wide tiles, the last one half empty
  const int tn = (d.D % 256 == 0) ? 256 : 128;
  const uint64_t hrows = static_cast<uint64_t>(S) + (shared ? d.T : 0);
  CUtensorMap mA, mB0, mB0s;
  constexpr int kBK = Ring<false>::kBK;
  if ((e = make_weight_map(&mA, h, hrows, d.F, kBK / kAtomK, 128)) != cudaSuccess) return e;
  if ((e = make_weight_map(&mB0, W2, static_cast<uint64_t>(d.E) * d.F, d.D, tn / 128, kBK)) != cudaSuccess) return e;
  if (shared) {
    if ((e = make_weight_map(&mB0s, Ws2, d.F, d.D, tn / 128, kBK)) != cudaSuccess) return e;
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
  a.Cs = ys;
  CUtensorMap mC, mCs;
  if ((e = make_map(&mC, y, S > 0 ? S : 1, d.D, kOutBoxRows, kOutBoxCols)) != cudaSuccess) return e;
  if (shared) {
    if ((e = tensor_map_f32_3d(&mCs, ys, d.D, d.T, 1, 16, kOutBoxRows)) != cudaSuccess) return e;
  } else {
    mCs = mC;
  }
  const int groups0 = d.E + (shared ? 1 : 0);
  const int pairs0 = std::min(di.pair_clusters[0],
                              max_pair_tiles(static_cast<long>(S) + (shared ? d.T : 0), groups0, (d.D + tn - 1) / tn));
  e = launch_pair<false, false>(pairs0, mA, mA, mB0, mB0, mB0s, mB0s, mC, mCs, a, s, pdl);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Self-test of the bounded waits: one CTA waits on an mbarrier that nothing
// arrives on; the wait gives up after timeout_ns and records the timeout in
// the device error word, exactly as a stalled pipeline of the GEMM would.
__global__ void wait_timeout_selftest_kernel(uint64_t timeout_ns, int* gave_up) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, &g_device_error, timeout_ns);
    *gave_up = ok ? 0 : 1;
  }
}

cudaError_t launch_wait_timeout_selftest(uint64_t timeout_ns, int* gave_up, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(timeout_ns, gave_up);
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
