// Chained expert FFN: W1||W3 + SiLU*mul and W2 in one kernel, with h kept on
// chip ("Chinchilla scaling, MoE, and fused Triton kernels", sections "Fused
// Triton kernel mechanism" and "Triton fused kernel implementation": one
// program per token tile streams F in blocks, applies the activation to each
// block of x W_up and accumulates block @ W_down, so the [t, F] activation is
// never written to HBM).
//
// GB300 mapping.  A CTA pair (cluster of 2, tcgen05 cta_group::2) owns a tile
// of 256 sorted rows of one group (CTA r: rows [128 r, 128 r + 128)) and
// walks F in chunks of 64 columns:
//   G1(c):  [g | u] = x_tile W1[:, c] | x_tile W3[:, c]   M=256, N=128, K=D
//           the leader stages the W1 block and the peer the W3 block, so
//           TMEM columns [0, 64) hold g and [64, 128) hold u
//   epi(c): h = silu(g) * u, rounded to bf16 and written by the epilogue
//           warps straight into a 128B-swizzled K-major shared-memory tile,
//           the A operand of G2 (each CTA holds its own 128 rows)
//   G2(c):  Y += h_c W2[c, :]                             M=256, N=D, K=64
// The x rows of the tile stay resident in shared memory for all chunks (D/64
// blocks of 16 KB per CTA).  TMEM (512 columns) holds two g|u buffers of 128
// columns, so the epilogue of chunk c overlaps G1(c + 1), and the D-column Y
// accumulator; this is why D <= 256.  The MMA issuer runs
// G1(0), G1(1), G2(0), G1(2), G2(1), ..., G2(last) and the producer streams
// the W1/W3 and W2 blocks through one ring in exactly that order.  After the
// last chunk the epilogue stores Y (bf16; the shared group's rows in fp32)
// with the row predication of the grouped GEMM (rows past the group's end
// are not stored).
//
// Accumulation order: g/u over k in 16-deep slices, Y over F in 16-deep
// slices, chunk by chunk -- the same order as the two separate grouped GEMMs,
// which also round h to bf16 between them.
//
// Barriers (full/empty: stage ring; the others as named):
//   a_full    leader, TMA bytes of both CTAs' resident x rows
//   a_empty   both, multicast commit after the tile's last G1
//   gu_full   both, multicast commit after G1(c)      [2 buffers]
//   gu_empty  leader, 16 epilogue-warp arrivals       [2]
//   h_full    leader, 16 epilogue-warp arrivals       [2]
//   h_empty   both, multicast commit after G2(c)      [2]
//   y_full    both, multicast commit after the tile's last G2
//   y_empty   leader, 16 epilogue-warp arrivals
// Every wait is bounded (MOE_WAIT_TIMEOUT_NS); on expiry the kernel records
// MOE_DEVERR_TIMEOUT in the error word, every role leaves its loop, and the
// CTA drains its copies and MMAs and frees TMEM before returning.
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

namespace {

constexpr int kBK = 64;                          // k per staged block (128 bytes of bf16)
constexpr int kFC = 64;                          // h columns per chunk
constexpr int kMaxD = kChainedMaxD;
constexpr int kStages = 7;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxGroups = MOE_MAX_EXPERTS + 1;
constexpr int kTileRows = 256;                   // rows per pair tile
constexpr int kABlock = 128 * kBK * 2;           // 16 KB: a 64-deep block of this CTA's rows
constexpr int kABytes = kMaxD / kBK * kABlock;   // resident x rows
constexpr int kBK1 = 128;                        // k per staged W1 / W3 block
constexpr int kBoxBytes = 64 * 64 * 2;           // one 64 x 64 weight box
constexpr int kStageBytes = 2 * kBoxBytes;       // W1 or W3: 128 k x 64 n; W2: 64 k x <= 128 n
constexpr int kHBytes = 128 * kFC * 2;           // 16 KB: one h chunk of this CTA's rows
constexpr int kOutBoxRows = 32;
constexpr int kOutBoxCols = 32;
constexpr int kOutBoxBytes = kOutBoxRows * kOutBoxCols * 2;
constexpr int kOffStages = kABytes;
constexpr int kOffH = kOffStages + kStages * kStageBytes;
constexpr int kOffOut = kOffH + 2 * kHBytes;
constexpr int kSmemBytes = kOffOut + kEpiWarps * kOutBoxBytes + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemGU = 2 * kFC;            // columns of one g|u buffer
constexpr uint32_t kTmemY = 2 * kTmemGU;         // Y at columns [256, 256 + D)
static_assert(kTmemY + kMaxD <= kTmemCols, "TMEM budget");

struct ChainArgs {
  const int32_t* offsets;  // [E + 1]
  int E;                   // routed groups
  int S;                   // routed rows
  int T_shared;            // rows of the shared group (0: none)
  int D;
  int F;
  uint16_t* Y;             // output of the routed rows [S, D]
  float* Ys;               // the shared group's output [T_shared, D], fp32
  unsigned int* dev_err;
};

struct ChainCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t a_full;
  uint64_t a_empty;
  uint64_t gu_full[2];
  uint64_t gu_empty[2];
  uint64_t h_full[2];
  uint64_t h_empty[2];
  uint64_t y_full;
  uint64_t y_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int tile_prefix[kMaxGroups + 1];
  int row0[kMaxGroups];
  int nrows[kMaxGroups];
};
// dynamic (with its 1 KB alignment slack) + static shared memory of one CTA
static_assert(kSmemBytes + sizeof(ChainCtl) <= 227 * 1024, "shared-memory budget");

__global__ void __launch_bounds__(kThreads, 1)
    chained_ffn_pair_kernel(const __grid_constant__ CUtensorMap mapA,
                            const __grid_constant__ CUtensorMap mapA_sh,
                            const __grid_constant__ CUtensorMap mapW1,
                            const __grid_constant__ CUtensorMap mapW3,
                            const __grid_constant__ CUtensorMap mapW1s,
                            const __grid_constant__ CUtensorMap mapW3s,
                            const __grid_constant__ CUtensorMap mapW2,
                            const __grid_constant__ CUtensorMap mapW2s,
                            const __grid_constant__ CUtensorMap mapY,
                            const __grid_constant__ CUtensorMap mapYs, const ChainArgs p) {
  extern __shared__ uint8_t chain_smem_raw[];
  __shared__ ChainCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(chain_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = leader, 1 = peer
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());
  const int G = p.E + (p.T_shared > 0 ? 1 : 0);
  const int nkb = p.D / kBK;       // 64-deep blocks of the resident x rows
  const int nst1 = (p.D + kBK1 - 1) / kBK1;  // W1 / W3 stages per chunk
  const int nch = p.F / kFC;       // F chunks
  const int halfD = p.D / 2;       // Y columns of W2 staged by this CTA
  const int nbox2 = (halfD + 63) / 64;

  // ---- setup that reads nothing produced by earlier kernels ----
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapW1);
    tma_prefetch_desc(&mapW3);
    tma_prefetch_desc(&mapW2);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(smem_u32(&ctl.full[st]), 1);
      mbar_init(smem_u32(&ctl.empty[st]), 1);
    }
    mbar_init(smem_u32(&ctl.a_full), 1);
    mbar_init(smem_u32(&ctl.a_empty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl.gu_full[b]), 1);
      mbar_init(smem_u32(&ctl.gu_empty[b]), 2 * kEpiWarps);
      mbar_init(smem_u32(&ctl.h_full[b]), 2 * kEpiWarps);
      mbar_init(smem_u32(&ctl.h_empty[b]), 1);
    }
    mbar_init(smem_u32(&ctl.y_full), 1);
    mbar_init(smem_u32(&ctl.y_empty), 2 * kEpiWarps);
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
  griddep_wait();  // offsets and x_sorted come from earlier kernels

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
      if (g < G) local += (ctl.nrows[g] + kTileRows - 1) / kTileRows;
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
        run += (ctl.nrows[g] + kTileRows - 1) / kTileRows;
      }
    }
    if (lane == 31) {
      ctl.tile_prefix[G] = incl;
      ctl.total_tiles = incl;
    }
  }
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.total_tiles;
  volatile int* abort_flag = &ctl.abort;
  unsigned int* dev_err = p.dev_err;

  if (warp == 0) {
    // ===================== TMA producer (lane 0 of both CTAs) =====================
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_normal();
      const uint64_t pol_b = l2_policy_evict_last();
      const uint32_t a_tx = 2u * static_cast<uint32_t>(nkb * kABlock);
      const uint32_t b1_tx = 2u * kStageBytes;
      const uint32_t b2_tx = 2u * static_cast<uint32_t>(nbox2 * kBoxBytes);
      int stage = 0;
      uint32_t phase = 0;
      int g = 0, i = 0, issued = 0;
      bool ok = true, a_pending = false;
      for (int tile = pair; tile < total && ok; tile += npairs, ++i) {
        while (tile >= ctl.tile_prefix[g + 1]) ++g;
        const int m = tile - ctl.tile_prefix[g];
        const bool routed = g < p.E;
        // resident x rows of the tile, once the previous tile's G1s are done
        if (!mbar_wait_cluster(smem_u32(&ctl.a_empty), (i & 1) ^ 1u, abort_flag, dev_err)) {
          ok = false;  // (the last x rows issued are those of tile i - 1)
          break;
        }
        const int a_row = (routed ? ctl.row0[g] : 0) + m * kTileRows + 128 * static_cast<int>(rank);
        const uint32_t a_full_leader = map_to_cta(smem_u32(&ctl.a_full), 0);
        if (leader) mbar_arrive_expect_tx(smem_u32(&ctl.a_full), a_tx);
        for (int kb = 0; kb < nkb; ++kb)
          tma_load_2d_pair(sbase + kb * kABlock, routed ? &mapA : &mapA_sh, a_full_leader, kb * kBK,
                           a_row, pol_a);
        a_pending = true;
        const int w1_row = routed ? g * p.D : 0;
        const int w2_row = routed ? g * p.F : 0;
        const CUtensorMap* mB1 =
            leader ? (routed ? &mapW1 : &mapW1s) : (routed ? &mapW3 : &mapW3s);
        const CUtensorMap* mB2 = routed ? &mapW2 : &mapW2s;
        for (int c = 0; c <= nch && ok; ++c) {
          if (c < nch) {  // W1 (leader) / W3 (peer) blocks of chunk c
            for (int s1 = 0; s1 < nst1; ++s1) {
              if (!mbar_wait_cluster(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, dev_err)) {
                ok = false;
                break;
              }
              const uint32_t full_leader = map_to_cta(smem_u32(&ctl.full[stage]), 0);
              if (leader) mbar_arrive_expect_tx(smem_u32(&ctl.full[stage]), b1_tx);
              // 128 k-rows (the last block of an odd number of 64-row blocks
              // also reads 64 rows past it, which no MMA uses)
              tma_load_2d_pair(sbase + kOffStages + stage * kStageBytes, mB1, full_leader, c * kFC,
                               w1_row + s1 * kBK1, pol_b);
              ++issued;
              if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
          }
          if (c >= 1) {  // W2 block of chunk c - 1: this CTA's half of the D columns
            if (!mbar_wait_cluster(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, dev_err)) {
              ok = false;
              break;
            }
            const uint32_t full_leader = map_to_cta(smem_u32(&ctl.full[stage]), 0);
            if (leader) mbar_arrive_expect_tx(smem_u32(&ctl.full[stage]), b2_tx);
            for (int b = 0; b < nbox2; ++b)
              tma_load_2d_pair(sbase + kOffStages + stage * kStageBytes + b * kBoxBytes, mB2,
                               full_leader, static_cast<int>(rank) * halfD + b * 64,
                               w2_row + (c - 1) * kFC, pol_b);
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok && leader) {
        // Let the copies already in flight land before the CTA exits.
        volatile int local_abort = 0;
        if (a_pending)
          mbar_wait_cluster(smem_u32(&ctl.a_full), static_cast<uint32_t>((i - 1) & 1), &local_abort,
                            dev_err);
        int st = stage;
        uint32_t ph = phase;
        for (int j = 0; j < kStages && j < issued; ++j) {
          if (--st < 0) {
            st = kStages - 1;
            ph ^= 1u;
          }
          mbar_wait_cluster(smem_u32(&ctl.full[st]), ph, &local_abort, dev_err);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ===================== MMA issuer (leader only) =====================
    if (lane == 0 && leader) {
      const uint32_t idesc1 = idesc_bf16_f32(kTileRows, 2 * kFC, 1u);
      const uint32_t idesc2 = idesc_bf16_f32(kTileRows, static_cast<uint32_t>(p.D), 1u);
      int stage = 0;
      uint32_t phase = 0;
      int n1 = 0, n2 = 0, i = 0;
      bool ok = true;
      for (int tile = pair; tile < total && ok; tile += npairs, ++i) {
        if (!mbar_wait_cluster(smem_u32(&ctl.a_full), i & 1, abort_flag, dev_err)) break;
        tc_fence_after_sync();
        for (int c = 0; c <= nch && ok; ++c) {
          if (c < nch) {  // G1(c) into g|u buffer n1 % 2
            const int b = n1 & 1;
            const uint32_t u = (n1 >> 1) & 1;
            if (!mbar_wait_cluster(smem_u32(&ctl.gu_empty[b]), u ^ 1u, abort_flag, dev_err)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + b * kTmemGU;
            for (int s1 = 0; s1 < nst1; ++s1) {
              if (!mbar_wait_cluster(smem_u32(&ctl.full[stage]), phase, abort_flag, dev_err)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              const uint32_t sb = sbase + kOffStages + stage * kStageBytes;
              const int nk16 = min(kBK1, p.D - s1 * kBK1) / 16;
              for (int kk = 0; kk < nk16; ++kk) {
                // k = 128 s1 + 16 kk: resident x block 2 s1 + kk / 4, slice kk % 4
                const uint32_t sa = sbase + (2 * s1 + (kk >> 2)) * kABlock + (kk & 3) * 32;
                const uint64_t adesc = smem_desc_sw128(sa, 16, 1024);
                const uint64_t bdesc = smem_desc_sw128(sb + kk * 2048, 8192, 1024);
                umma_bf16_pair(d_tmem, adesc, bdesc, idesc1, (s1 | kk) != 0 ? 1u : 0u);
              }
              umma_commit_pair(smem_u32(&ctl.empty[stage]), 0x3);
              if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            umma_commit_pair(smem_u32(&ctl.gu_full[b]), 0x3);
            if (c == nch - 1) umma_commit_pair(smem_u32(&ctl.a_empty), 0x3);
            ++n1;
          }
          if (c >= 1) {  // G2(c - 1): Y += h W2 with h from buffer n2 % 2
            const int b = n2 & 1;
            const uint32_t u = (n2 >> 1) & 1;
            if (!mbar_wait_cluster(smem_u32(&ctl.h_full[b]), u, abort_flag, dev_err)) {
              ok = false;
              break;
            }
            if (c == 1 && !mbar_wait_cluster(smem_u32(&ctl.y_empty), (i & 1) ^ 1u, abort_flag, dev_err)) {
              ok = false;
              break;
            }
            if (!mbar_wait_cluster(smem_u32(&ctl.full[stage]), phase, abort_flag, dev_err)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t sa = sbase + kOffH + b * kHBytes;
            const uint32_t sb = sbase + kOffStages + stage * kStageBytes;
#pragma unroll
            for (int kk = 0; kk < kFC / 16; ++kk) {
              const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bdesc = smem_desc_sw128(sb + kk * 2048, 8192, 1024);
              umma_bf16_pair(tmem_base + kTmemY, adesc, bdesc, idesc2,
                             (c > 1 || kk != 0) ? 1u : 0u);
            }
            umma_commit_pair(smem_u32(&ctl.empty[stage]), 0x3);
            umma_commit_pair(smem_u32(&ctl.h_empty[b]), 0x3);
            if (c == nch) umma_commit_pair(smem_u32(&ctl.y_full), 0x3);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
            ++n2;
          }
        }
      }
      // All MMAs issued by this thread are complete once `drain` flips.
      umma_commit_pair(smem_u32(&ctl.drain), 0x1);
      volatile int local_abort = 0;
      mbar_wait_cluster(smem_u32(&ctl.drain), 0, &local_abort, dev_err);
    }
    __syncwarp();
  } else {
    // ===================== epilogue (both CTAs) =====================
    // Warp w owns TMEM lanes 32 (w % 4) .. + 31 (rows 32 (w % 4) .. of this
    // CTA) and half (w - 2) / 4 of the columns: 32 of the chunk's 64 h
    // columns, and D / 2 of Y's columns.
    const int q = warp & 3;
    const int part = (warp - 2) >> 2;
    const int r = q * 32 + lane;  // row within this CTA's 128
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* stage_out = smem + kOffOut + (warp - 2) * kOutBoxBytes;
    int g = 0, i = 0, n = 0;
    bool ok = true;
    for (int tile = pair; tile < total && ok; tile += npairs, ++i) {
      while (tile >= ctl.tile_prefix[g + 1]) ++g;
      const int m = tile - ctl.tile_prefix[g];
      for (int c = 0; c < nch; ++c, ++n) {
        const int b = n & 1;
        const uint32_t u = (n >> 1) & 1;
        bool got = mbar_wait_cluster(smem_u32(&ctl.gu_full[b]), u, abort_flag, dev_err);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t rg[32], ru[32];
        tmem_ld_32cols(lane_base + b * kTmemGU + part * 32, rg);
        tmem_ld_32cols(lane_base + b * kTmemGU + kFC + part * 32, ru);
        tmem_ld_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&ctl.gu_empty[b]), 0));
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
        // the G2 that read this h buffer two chunks ago has completed
        got = mbar_wait_cluster(smem_u32(&ctl.h_empty[b]), u ^ 1u, abort_flag, dev_err);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        // K-major 128B-swizzled tile: row r at 128 r, 16-byte chunk j of the
        // row at chunk j ^ (r % 8); this warp fills chunks 4 part .. 4 part + 3
        uint8_t* hb = smem + kOffH + b * kHBytes + r * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int j = part * 4 + v;
          *reinterpret_cast<uint4*>(hb + ((j ^ (r & 7)) << 4)) =
              make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&ctl.h_full[b]), 0));
      }
      if (!ok) break;
      // ---- Y of the tile ----
      const bool got = mbar_wait_cluster(smem_u32(&ctl.y_full), i & 1, abort_flag, dev_err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const int nrows_g = ctl.nrows[g];
      const int row = m * kTileRows + 128 * static_cast<int>(rank) + r;
      const bool valid = row < nrows_g;
      const int warp_row0 = m * kTileRows + 128 * static_cast<int>(rank) + q * 32;
      const bool full_box = warp_row0 + kOutBoxRows <= nrows_g;
      const bool f32_rows = g >= p.E;  // the shared expert's rows keep fp32
      for (int cc = part * halfD; cc < (part + 1) * halfD; cc += kOutBoxCols) {
        uint32_t ra[32];
        tmem_ld_32cols(lane_base + kTmemY + cc, ra);
        tmem_ld_wait();
        if (f32_rows) {
          if (full_box)
            store_box_f32_tma(&mapYs, stage_out, ra, cc, warp_row0);
          else if (valid)
            store_row_f32(p.Ys + static_cast<size_t>(row) * p.D + cc, ra);
          continue;
        }
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          packed[j] = pack_bf16x2(__uint_as_float(ra[2 * j]), __uint_as_float(ra[2 * j + 1]));
        if (full_box) {
          bulk_wait_group_read0();  // the previous store has read the staging buffer
          __syncwarp();
          // 64B swizzle: 16-byte chunk v of row l lives at chunk v ^ ((l / 2) % 4)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4* dst = reinterpret_cast<uint4*>(stage_out + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4));
            *dst = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&mapY, smem_u32(stage_out), cc, ctl.row0[g] + warp_row0);
            bulk_commit_group();
          }
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(
              p.Y + static_cast<size_t>(ctl.row0[g] + row) * p.D + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_cta(smem_u32(&ctl.y_empty), 0));
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

// Per-device launch state: co-resident CTA pairs and the error word address.
struct ChainDevice {
  int pairs = 0;
  unsigned int* dev_err = nullptr;
};
ChainDevice g_chain_dev[64];
std::mutex g_chain_mu;

cudaError_t chain_setup(ChainDevice* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_chain_mu);
  ChainDevice& cd = g_chain_dev[dev];
  if (cd.pairs == 0) {
    e = cudaFuncSetAttribute(chained_ffn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclusters = 0;
    e = cudaOccupancyMaxActiveClusters(&nclusters, chained_ffn_pair_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (nclusters < 1) return cudaErrorInvalidConfiguration;
    e = device_error_address(&cd.dev_err);
    if (e != cudaSuccess) return e;
    cd.pairs = nclusters;
  }
  *out = cd;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_chained_ffn(const uint16_t* x_sorted, const uint16_t* x, const uint16_t* W1,
                               const uint16_t* W3, const uint16_t* W2, const uint16_t* Ws1,
                               const uint16_t* Ws3, const uint16_t* Ws2, const int32_t* offsets,
                               const moe_dims& d, uint16_t* y, float* ys, cudaStream_t s, bool pdl) {
  if (d.D > kMaxD || d.D % kBK != 0 || d.F % kFC != 0) return cudaErrorInvalidValue;
  ChainDevice cd;
  cudaError_t e = chain_setup(&cd);
  if (e != cudaSuccess) return e;
  const int S = d.T * d.k;
  const bool shared = Ws1 != nullptr;
  CUtensorMap mA, mAs, mW1, mW3, mW1s, mW3s, mW2, mW2s, mY, mYs;
  if ((e = tensor_map_2d(&mA, x_sorted, S, d.D, 128, kBK)) != cudaSuccess) return e;
  if ((e = tensor_map_2d(&mW1, W1, static_cast<uint64_t>(d.E) * d.D, d.F, kBK1, 64)) != cudaSuccess) return e;
  if ((e = tensor_map_2d(&mW3, W3, static_cast<uint64_t>(d.E) * d.D, d.F, kBK1, 64)) != cudaSuccess) return e;
  if ((e = tensor_map_2d(&mW2, W2, static_cast<uint64_t>(d.E) * d.F, d.D, kFC, 64)) != cudaSuccess) return e;
  if (shared) {
    if ((e = tensor_map_2d(&mAs, x, d.T, d.D, 128, kBK)) != cudaSuccess) return e;
    if ((e = tensor_map_2d(&mW1s, Ws1, d.D, d.F, kBK1, 64)) != cudaSuccess) return e;
    if ((e = tensor_map_2d(&mW3s, Ws3, d.D, d.F, kBK1, 64)) != cudaSuccess) return e;
    if ((e = tensor_map_2d(&mW2s, Ws2, d.F, d.D, kFC, 64)) != cudaSuccess) return e;
  } else {
    mAs = mA;
    mW1s = mW1;
    mW3s = mW3;
    mW2s = mW2;
  }
  if ((e = tensor_map_2d(&mY, y, S, d.D, kOutBoxRows, kOutBoxCols)) != cudaSuccess) return e;
  if (shared) {
    if ((e = tensor_map_f32_3d(&mYs, ys, d.D, d.T, 1, 16, kOutBoxRows)) != cudaSuccess) return e;
  } else {
    mYs = mY;
  }
  ChainArgs a;
  a.offsets = offsets;
  a.E = d.E;
  a.S = S;
  a.T_shared = shared ? d.T : 0;
  a.D = d.D;
  a.F = d.F;
  a.Y = y;
  a.Ys = ys;
  a.dev_err = cd.dev_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * cd.pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
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
  e = cudaLaunchKernelEx(&cfg, chained_ffn_pair_kernel, mA, mAs, mW1, mW3, mW1s, mW3s, mW2, mW2s, mY, mYs, a);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
