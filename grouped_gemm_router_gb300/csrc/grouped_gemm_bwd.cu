// Backward grouped GEMMs of the MoE SwiGLU FFN on tcgen05 CTA pairs.
//
// The backward of an expert y = (silu(x W1) * (x W3)) W2 over its rows
// ("Triton MoE Kernels & Memory Checkpointing", Part A, section 8, the
// autograd contract and its "dual kernels"): with y_bar the gradient of y,
//   h_bar = y_bar W2^T                                        (W2 dgrad)
//   g_bar = h_bar * u * silu'(g),  u_bar = h_bar * silu(g)    (activation)
//   x_bar = g_bar W1^T + u_bar W3^T                           (x dgrad)
//   W1_bar = x^T g_bar,  W3_bar = x^T u_bar,  W2_bar = h^T y_bar  (wgrad)
// One persistent CTA-pair kernel (same engine as the forward grouped GEMM:
// 256 x N pair tiles, a TMA stage ring of up to 192 KB, two TMEM accumulators,
// bounded waits)
// runs four modes:
//   kDgradW2  A = y_bar rows (K-major), B = W2[e]^T read K-major from the
//             rows of W2 [E*F, D]; bf16 h_bar out.
//   kActBwd   the W1||W3 forward recomputed (A = x_sorted, B = W1 | W3 as in
//             the forward); the epilogue reads h_bar and writes g_bar | u_bar
//             ([rows, 2F]) and the recomputed h ([rows, F]) in bf16.
//   kDgradX   A = g_bar | u_bar rows (K = 2F, K-major), B = W1[e]^T for the
//             first F and W3[e]^T for the rest, read K-major from the rows of
//             W1 / W3 [E*D, F]; bf16 x_bar out.
//   kWgrad    C[e] = A^T B over the rows of group e: A and B both M/N-major
//             (row-major [rows, M] and [rows, N] tiles), K = the group's
//             rows; fp32 out, zeros for an empty group.
//
// Row layouts.  The gradient buffers use a padded sorted layout: group e owns
// rows [prow0_e, prow0_e + pn_e), pn_e = n_e rounded up to 64, prow0 the
// exclusive prefix sum of pn; rows [n_e, pn_e) of y_bar are zero (the combine
// backward writes them), so every derived gradient is zero there too and a
// weight-gradient k-block never has to be masked.  x_sorted keeps the
// forward's unpadded layout (rows offsets[e] ..).  The shared expert is one
// more group whose operands have their own tensor maps over exactly T rows
// (zero fill past T) and whose outputs go to rows S_pad .. S_pad + T.
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_device.cuh"
#include "moe_kernels.cuh"

namespace moe {

namespace {

constexpr int kBK = 64;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxGroups = MOE_MAX_EXPERTS + 1;
constexpr uint32_t kTmemCols = 512;
constexpr int kTileM = 256;                   // rows per pair tile
constexpr int kTileN = 256;                   // MMA N
constexpr int kStages = 6;                    // largest stage ring (mbarrier arrays)
constexpr int kOutBoxRows = 32;
constexpr int kOutBoxCols = 32;
constexpr int kOutBoxBytes = kOutBoxRows * kOutBoxCols * 2;
constexpr int kWOutCols = 16;                 // fp32 weight-gradient store box: 32 rows x 64 bytes

enum : int { kDgradW2 = 0, kActBwd = 1, kDgradX = 2, kWgrad = 3 };

// Tensor maps per launch: A, A of the shared group, B0, B1, B0 / B1 of the
// shared group, and five output maps (C, C2 in the row modes; the weight
// gradient's w_a, w_b, ws_a, ws_b and partial slots).
constexpr int kMaps = 11;

// Weight-gradient tiles differ in length (a group's rows); up to kMaxLptTiles
// of them are assigned longest first to the least-loaded pair.
constexpr int kMaxLptTiles = 2048;
constexpr int kMaxMyTiles = 64;
// A weight-gradient group longer than kMaxChunkKb k-blocks is split along K
// into near-equal chunks whose fp32 partial sums a reduction kernel adds.
constexpr int kMaxChunkKb = 160;

// k per stage of each mode: 128 for the W2 dgrad (two swizzle atoms, one 3-D
// TMA box per operand and stage: 143 -> 141.5 us on gptoss_lite), 64 for the
// others, whose operands stream from HBM (the weight gradients and x dgrad
// ran slower with 128-deep stages) or whose epilogue binds (the SwiGLU
// backward: 346 -> 353 us with two such stages).
__host__ __device__ constexpr int bk_of(int mode) { return mode == kDgradW2 ? 128 : 64; }
__host__ __device__ constexpr int stage_bytes_of(int mode) { return 2 * 128 * bk_of(mode) * 2; }
// The activation mode gives each epilogue warp three output staging buffers
// (g_bar, u_bar and h boxes rotate through them) and gives up ring space for
// them.
__host__ __device__ constexpr int stages_of(int mode) {
  return mode == kActBwd ? (bk_of(mode) == 128 ? 2 : kStages - 1) : (bk_of(mode) == 128 ? 3 : kStages);
}
__host__ __device__ constexpr int out_boxes_of(int mode) { return mode == kActBwd ? 3 : 1; }
__host__ __device__ constexpr int smem_bytes_of(int mode) {
  return stages_of(mode) * stage_bytes_of(mode) + kEpiWarps * out_boxes_of(mode) * kOutBoxBytes + 1024;
}

template <int kMode>
struct Traits {
  static constexpr bool a_mn = kMode == kWgrad;                       // A M-major
  static constexpr bool b_mn = kMode == kActBwd || kMode == kWgrad;   // B N-major
  static constexpr bool row_tiles = kMode != kWgrad;                  // tiles over rows
};

struct BwdArgs {
  const int32_t* offsets;  // [E + 1] forward sorted-row offsets
  int E;
  int S;                   // routed rows T*k
  int S_pad;               // first row of the shared group in the padded buffers
  int T_shared;            // rows of the shared group (0: none)
  int K;                   // row modes: reduction length (kDgradX: 2F)
  int K1;                  // kDgradX: k at which B switches from W1 to W3 (= F)
  int N;                   // output columns
  int M;                   // kWgrad: output rows
  int b_rows;              // K-major B: rows of one expert's weight block (row modes)
  int a_padded;            // kWgrad: A rows in the padded layout (else unpadded)
  uint16_t* C;             // kDgradW2 / kDgradX: bf16 output [S_pad + T, N] (mapC's tensor)
  // kActBwd
  const uint16_t* hbar;    // [S_pad + T, N] incoming gradient of h
  uint16_t* gu;            // [S_pad + T, 2N] g_bar | u_bar
  uint16_t* h;             // [S_pad + T, N] recomputed h, or NULL: not stored
  // kWgrad: fp32 outputs; columns [0, n_split) go to *_a, [n_split, N) to *_b
  float* w_a;
  float* w_b;
  float* ws_a;
  float* ws_b;
  int n_split;
  float* part;             // kWgrad: partial sums of split groups [slot][M][N]
  unsigned int* dev_err;
};

struct BwdCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int tile_prefix[kMaxGroups + 1];  // by position in the tile order
  int gorder[kMaxGroups];           // group at each position of the tile order
  int my_count;                     // tiles of this pair in my_tiles, or -1: round robin
  int my_tiles[kMaxMyTiles];
  int row0[kMaxGroups];   // unpadded first row (forward layout)
  int prow0[kMaxGroups];  // padded first row (shared group: S_pad)
  int nrows[kMaxGroups];
  int pnrows[kMaxGroups];
  int nchunk[kMaxGroups];  // kWgrad: K chunks of the group
  int pslot[kMaxGroups];   // kWgrad: first partial slot of a split group
};

// Reads one bf16 x 32 chunk (64 bytes) into 16 packed words.
MOE_DEV void load_bf16x32(const uint16_t* src, uint32_t (&v)[16]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 q = s[i];
    v[4 * i] = q.x;
    v[4 * i + 1] = q.y;
    v[4 * i + 2] = q.z;
    v[4 * i + 3] = q.w;
  }
}

MOE_DEV void store_bf16x32(uint16_t* dst, const uint32_t (&v)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_bwd_kernel(const __grid_constant__ CUtensorMap mapA,
                            const __grid_constant__ CUtensorMap mapA_sh,
                            const __grid_constant__ CUtensorMap mapB0,
                            const __grid_constant__ CUtensorMap mapB1,
                            const __grid_constant__ CUtensorMap mapB0_sh,
                            const __grid_constant__ CUtensorMap mapB1_sh,
                            const __grid_constant__ CUtensorMap mapC,
                            const __grid_constant__ CUtensorMap mapC2,
                            const __grid_constant__ CUtensorMap mapC3,
                            const __grid_constant__ CUtensorMap mapC4,
                            const __grid_constant__ CUtensorMap mapC5, const BwdArgs p) {
  using Tr = Traits<kMode>;
  constexpr int kSt = stages_of(kMode);
  constexpr int kBKm = bk_of(kMode);             // k per stage of this mode
  constexpr int kStageBytes = stage_bytes_of(kMode);
  constexpr int kABytes = kStageBytes / 2;       // this CTA's half of A per stage
  extern __shared__ uint8_t bwd_smem_raw[];
  __shared__ BwdCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(bwd_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());
  const int G = p.E + (p.T_shared > 0 ? 1 : 0);
  // output columns per tile: kActBwd computes g and u of kTileN / 2 columns
  const int hw = kMode == kActBwd ? kTileN / 2 : kTileN;
  const int ntn = (p.N + hw - 1) / hw;
  const int nmt = (p.M + kTileM - 1) / kTileM;  // kWgrad
  const int half_n = kTileN / 2;
  const bool want_h = kMode == kActBwd && p.h != nullptr;  // kActBwd: also store the recomputed h

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB0);
    for (int st = 0; st < kSt; ++st) {
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
  // ---- group tables: unpadded / padded rows, tiles per group, tile order.
  // They read only the forward's offsets, so they run before waiting for the
  // previous kernel. ----
  if (warp == 0) {
    // padded starts: exclusive scan of the counts rounded up to 64
    const int per = (G + 31) / 32;
    int loc = 0;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < p.E) {
        const int a = p.offsets[g], b = p.offsets[g + 1];
        ctl.row0[g] = a;
        ctl.nrows[g] = b - a;
        ctl.pnrows[g] = (b - a + 63) & ~63;
        loc += ctl.pnrows[g];
      } else if (g < G) {
        ctl.row0[g] = 0;
        ctl.nrows[g] = p.T_shared;
        ctl.pnrows[g] = p.T_shared;
      }
    }
    int incl = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - loc;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < p.E) {
        ctl.prow0[g] = run;
        run += ctl.pnrows[g];
      } else if (g < G) {
        ctl.prow0[g] = p.S_pad;
      }
    }
    __syncwarp();
    // Tile order: group by group.  Weight-gradient tiles of the shared group
    // reduce over all T rows (k times longer than a routed tile's rows), so
    // they come first and the routed tiles fill in behind them.
    // weight gradients: groups by decreasing length (ties by index), so the
    // greedy assignment below sees the longest tiles first
    auto kblocks_of = [&](int g) { return (ctl.pnrows[g] + kBK - 1) / kBK; };
    auto nchunk_of = [&](int g) { return max(1, (kblocks_of(g) + kMaxChunkKb - 1) / kMaxChunkKb); };
    auto chunk_kb_of = [&](int g) { return (kblocks_of(g) + nchunk_of(g) - 1) / nchunk_of(g); };
    if (!Tr::row_tiles) {
      // partial slots of the split groups, in group order
      int nsl = 0;
      for (int i = 0; i < per; ++i) {
        const int g = lane * per + i;
        if (g < G) {
          ctl.nchunk[g] = nchunk_of(g);
          nsl += ctl.nchunk[g] > 1 ? ctl.nchunk[g] : 0;
        }
      }
      int sincl = nsl;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, sincl, off);
        if (lane >= off) sincl += v;
      }
      int srun = sincl - nsl;
      for (int i = 0; i < per; ++i) {
        const int g = lane * per + i;
        if (g < G) {
          ctl.pslot[g] = srun;
          srun += ctl.nchunk[g] > 1 ? ctl.nchunk[g] : 0;
        }
      }
      for (int i = 0; i < per; ++i) {
        const int g = lane * per + i;
        if (g < G) {
          const int c = chunk_kb_of(g);
          int rnk = 0;
          for (int h = 0; h < G; ++h) {
            const int ch = chunk_kb_of(h);
            rnk += (ch > c || (ch == c && h < g)) ? 1 : 0;
          }
          ctl.gorder[rnk] = g;
        }
      }
    } else {
      for (int i = 0; i < per; ++i) {
        const int g = lane * per + i;
        if (g < G) ctl.gorder[g] = g;
      }
    }
    __syncwarp();
    auto group_at = [&](int pos) { return ctl.gorder[pos]; };
    int tl = 0;
    for (int i = 0; i < per; ++i) {
      const int pos = lane * per + i;
      if (pos < G) {
        const int g = group_at(pos);
        tl += Tr::row_tiles ? ((ctl.pnrows[g] + kTileM - 1) / kTileM) * ntn : nchunk_of(g) * nmt * ntn;
      }
    }
    int tincl = tl;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, tincl, off);
      if (lane >= off) tincl += v;
    }
    int trun = tincl - tl;
    for (int i = 0; i < per; ++i) {
      const int pos = lane * per + i;
      if (pos < G) {
        const int g = group_at(pos);
        ctl.tile_prefix[pos] = trun;
        trun += Tr::row_tiles ? ((ctl.pnrows[g] + kTileM - 1) / kTileM) * ntn : nchunk_of(g) * nmt * ntn;
      }
    }
    if (lane == 31) {
      ctl.tile_prefix[G] = tincl;
      ctl.total_tiles = tincl;
    }
    __syncwarp();
    // Greedy assignment, longest first: each tile goes to the pair with the
    // least work so far (ties to the lower pair).  Every CTA computes the same
    // assignment and keeps its own pair's tiles; when any pair would exceed
    // kMaxMyTiles, all pairs use the round robin instead.
    int my_count = -1;
    const int total_t = __shfl_sync(0xffffffffu, tincl, 31);
    if (!Tr::row_tiles && total_t <= kMaxLptTiles && npairs <= 128) {
      uint32_t load[4] = {0u, 0u, 0u, 0u};
      int cnt[4] = {0, 0, 0, 0};
      int mine = 0;
      for (int pos = 0; pos < G; ++pos) {
        const int g = ctl.gorder[pos];
        const uint32_t cost = static_cast<uint32_t>(chunk_kb_of(g)) + 2u;  // + epilogue
        const int base = ctl.tile_prefix[pos];
        const int nt = ctl.tile_prefix[pos + 1] - base;
        for (int l = 0; l < nt; ++l) {
          uint32_t key = 0xFFFFFFFFu;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int pid = lane + 32 * q;
            if (pid < npairs) key = min(key, (load[q] << 8) | static_cast<uint32_t>(pid));
          }
          key = __reduce_min_sync(0xffffffffu, key);
          const int best = static_cast<int>(key & 0xFFu);
          if ((best & 31) == lane) {
            load[best >> 5] += cost;
            ++cnt[best >> 5];
          }
          if (best == pair) {
            if (lane == 0 && mine < kMaxMyTiles) ctl.my_tiles[mine] = base + l;
            ++mine;
          }
        }
      }
      int mx = max(max(cnt[0], cnt[1]), max(cnt[2], cnt[3]));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      my_count = mx <= kMaxMyTiles ? mine : -1;
      // The same tiles round robin over the largest multiple P of the tiles
      // per K chunk: every round then holds whole chunks, so the tiles that
      // read the same rows run together and share them in L2 (a chunk split
      // across rounds is read from DRAM twice).  Taken when its makespan is
      // within 1/32 of the greedy one.
      const int per_chunk = nmt * ntn;
      const int P = per_chunk > 0 ? (npairs / per_chunk) * per_chunk : 0;
      if (P > 0) {
        uint32_t lpt_max = max(max(load[0], load[1]), max(load[2], load[3]));
        uint32_t rr_max = 0;
        for (int q = 0; q < 4; ++q) {
          const int pid = lane + 32 * q;
          if (pid >= P) continue;
          uint32_t sum = 0;
          int ps = 0;
          for (int t = pid; t < total_t; t += P) {
            while (t >= ctl.tile_prefix[ps + 1]) ++ps;
            sum += static_cast<uint32_t>(chunk_kb_of(ctl.gorder[ps])) + 2u;
          }
          rr_max = max(rr_max, sum);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          lpt_max = max(lpt_max, __shfl_xor_sync(0xffffffffu, lpt_max, off));
          rr_max = max(rr_max, __shfl_xor_sync(0xffffffffu, rr_max, off));
        }
        if (rr_max <= lpt_max + lpt_max / 32) my_count = -2;
      }
    }
    if (lane == 0) ctl.my_count = my_count;
  }
  griddep_launch_dependents();
  griddep_wait();  // the operands come from the previous kernels
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.total_tiles;
  volatile int* abort_flag = &ctl.abort;
  unsigned int* dev_err = p.dev_err;

  // the it-th tile of this pair (-1: none left).  my_count: >= 0 tiles in
  // my_tiles (greedy), -1 round robin over all pairs, -2 round robin over the
  // largest multiple of the tiles per K chunk (whole chunks per round).
  const int my_n = ctl.my_count;
  const int wg_pairs = my_n == -2 ? (npairs / (nmt * ntn)) * (nmt * ntn) : npairs;
  auto next_tile = [&](int it) -> int {
    if (my_n == -2) {
      const int t = pair + it * wg_pairs;
      return pair < wg_pairs && t < total ? t : -1;
    }
    if (my_n >= 0) return it < my_n ? ctl.my_tiles[it] : -1;
    const int t = pair + it * npairs;
    return t < total ? t : -1;
  };

  // Coordinates of a tile (its local index within group g): K chunk c, m and n
  // tiles, and its k-block range [kb0, kb1).  Weight-gradient tiles are
  // numbered chunk by chunk, so the tiles reading the same rows run together.
  struct TileInfo {
    int c, m, n, kb0, kb1;
  };
  auto tile_info = [&](int g, int local) -> TileInfo {
    TileInfo t;
    if (Tr::row_tiles) {
      t.c = 0;
      t.m = local / ntn;
      t.n = local - t.m * ntn;
      t.kb0 = 0;
      t.kb1 = (p.K + kBKm - 1) / kBKm;
    } else {
      const int per_chunk = nmt * ntn;
      t.c = local / per_chunk;
      const int r = local - t.c * per_chunk;
      t.m = r / ntn;
      t.n = r - t.m * ntn;
      const int nkb = (ctl.pnrows[g] + kBK - 1) / kBK;
      const int csz = (nkb + ctl.nchunk[g] - 1) / ctl.nchunk[g];
      t.kb0 = t.c * csz;
      t.kb1 = min(t.kb0 + csz, nkb);
    }
    return t;
  };

  if (warp == 0) {
    // ===================== TMA producer (lane 0 of both CTAs) =====================
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_normal();
      const uint64_t pol_b = Tr::row_tiles ? l2_policy_evict_last() : l2_policy_evict_normal();
      const uint32_t pair_tx = 2u * static_cast<uint32_t>(kStageBytes);
      int stage = 0;
      uint32_t phase = 0;
      int pos = 0, issued = 0;
      bool ok = true;
      for (int it = 0, tile = next_tile(0); tile >= 0 && ok; tile = next_tile(++it)) {
        while (tile >= ctl.tile_prefix[pos + 1]) ++pos;
        const int g = ctl.gorder[pos];
        const int local = tile - ctl.tile_prefix[pos];
        const TileInfo ti = tile_info(g, local);
        const int m = ti.m, n = ti.n;
        const bool routed = g < p.E;
        const CUtensorMap* mA = routed ? &mapA : &mapA_sh;
        for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
          if (!mbar_wait_cluster(smem_u32(&ctl.empty[stage]), phase ^ 1u, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = map_to_cta(smem_u32(&ctl.full[stage]), 0);
          const uint32_t sa = smem_base + stage * kStageBytes;
          const uint32_t sb = sa + kABytes;
          if (leader) mbar_arrive_expect_tx(smem_u32(&ctl.full[stage]), pair_tx);
          if (Tr::row_tiles) {
            // A: 128 rows of this CTA, K-major
            const int a0 = routed ? (kMode == kActBwd ? ctl.row0[g] : ctl.prow0[g]) : 0;
            tma_load_3d_pair(sa, mA, full_leader, 0, a0 + m * kTileM + 128 * static_cast<int>(rank),
                             kb * (kBKm / 64), pol_a);
            if (kMode == kActBwd) {
              // B = W1 (leader) / W3 (peer) columns of the tile, N-major
              const CUtensorMap* mB =
                  leader ? (routed ? &mapB0 : &mapB0_sh) : (routed ? &mapB1 : &mapB1_sh);
              const int brow = (routed ? g * p.K : 0) + kb * kBKm;
              tma_load_3d_pair(sb, mB, full_leader, 0, brow, (n * hw) / 64, pol_b);
            } else {
              // B^T rows of this CTA's half of the tile's columns, K-major
              const bool second = kMode == kDgradX && kb * kBKm >= p.K1;
              const CUtensorMap* mB = second ? (routed ? &mapB1 : &mapB1_sh) : (routed ? &mapB0 : &mapB0_sh);
              const int k0 = second ? kb * kBKm - p.K1 : kb * kBKm;
              const int brow = (routed ? g * p.b_rows : 0) + n * kTileN + half_n * static_cast<int>(rank);
              tma_load_3d_pair(sb, mB, full_leader, 0, brow, k0 / 64, pol_b);
            }
          } else {
            // kWgrad: k = rows of the group; A [rows, M] and B [rows, N] tiles, M/N-major
            const int ak0 = routed ? (p.a_padded ? ctl.prow0[g] : ctl.row0[g]) : 0;
            const int bk0 = routed ? ctl.prow0[g] : 0;
            const int mcol = m * kTileM + 128 * static_cast<int>(rank);
            const CUtensorMap* mB = routed ? &mapB0 : &mapB0_sh;
            const int ncol = n * kTileN + half_n * static_cast<int>(rank);
            tma_load_3d_pair(sa, mA, full_leader, 0, ak0 + kb * kBK, mcol / 64, pol_a);
            tma_load_3d_pair(sb, mB, full_leader, 0, bk0 + kb * kBK, ncol / 64, pol_b);
          }
          ++issued;
          if (++stage == kSt) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        int st = stage;
        uint32_t ph = phase;
        for (int i = 0; i < kSt && i < issued; ++i) {
          if (--st < 0) {
            st = kSt - 1;
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
      const uint32_t idesc = idesc_bf16_f32_ab(kTileM, kTileN, Tr::a_mn ? 1u : 0u, Tr::b_mn ? 1u : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int i = 0, pos = 0;
      bool ok = true;
      for (int tile = next_tile(0); tile >= 0 && ok; tile = next_tile(++i)) {
        while (tile >= ctl.tile_prefix[pos + 1]) ++pos;
        const TileInfo ti = tile_info(ctl.gorder[pos], tile - ctl.tile_prefix[pos]);
        const int buf = i & 1;
        const uint32_t tph = (i >> 1) & 1;
        if (!mbar_wait_cluster(smem_u32(&ctl.tempty[buf]), tph ^ 1u, abort_flag, dev_err)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * 256;
        for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
          if (!mbar_wait_cluster(smem_u32(&ctl.full[stage]), phase, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_base + stage * kStageBytes;
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBKm / 16; ++kk) {
            // K-major: atom kk / 4 (128 rows x 128 bytes), 16-wide slice kk % 4;
            // M/N-major: 64-column blocks of kBKm k-rows (LBO = one block), slice kk
            const uint64_t adesc = Tr::a_mn ? smem_desc_sw128(sa + kk * 2048, kBKm * 128, 1024)
                                            : smem_desc_sw128(sa + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
            const uint64_t bdesc = Tr::b_mn ? smem_desc_sw128(sb + kk * 2048, kBKm * 128, 1024)
                                            : smem_desc_sw128(sb + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
            umma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb != ti.kb0 || kk != 0) ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&ctl.empty[stage]), 0x3);
          if (++stage == kSt) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&ctl.tfull[buf]), 0x3);
      }
      umma_commit_pair(smem_u32(&ctl.drain), 0x1);
      volatile int local_abort = 0;
      mbar_wait_cluster(smem_u32(&ctl.drain), 0, &local_abort, dev_err);
    }
    __syncwarp();
  } else {
    // ===================== epilogue (both CTAs) =====================
    const int q = warp & 3;
    const int part = (warp - 2) >> 2;
    const int r_in_tile = 128 * static_cast<int>(rank) + q * 32 + lane;
    const uint32_t tempty_leader0 = map_to_cta(smem_u32(&ctl.tempty[0]), 0);
    const uint32_t tempty_leader1 = map_to_cta(smem_u32(&ctl.tempty[1]), 0);
    uint8_t* stage_out = smem + kSt * kStageBytes + (warp - 2) * out_boxes_of(kMode) * kOutBoxBytes;
    if constexpr (kMode == kActBwd) {
      // SwiGLU backward: per tile, warp (q, part) holds rows q*32 .. +31 of
      // this CTA and two 32-column boxes of g | u.  The h_bar rows it needs do
      // not depend on this kernel, so they are loaded a box ahead: box 1's
      // at the start of a tile, the next tile's box 0 right after box 0's
      // math (its registers are free by then), each a half-tile before use;
      // L2 is asked for the next tile's rows at the start of a tile.  The
      // output boxes rotate through the warp's three staging buffers, one
      // bulk group per box store, so a box waits only for the store issued
      // two boxes earlier to have read its buffer (g_bar and u_bar), or for
      // all of them when h is stored too.
      auto hbar_src = [&](int g_, int m_, int n_, int c) -> const uint16_t* {
        const int row = m_ * kTileM + r_in_tile;
        const int col = n_ * hw + part * (hw / 2) + 32 * c;
        if (row >= ctl.pnrows[g_] || col >= p.N) return nullptr;
        return p.hbar + static_cast<size_t>(ctl.prow0[g_] + row) * p.N + col;
      };
      int pos = 0, i = 0;
      int tile = next_tile(0);
      int g = 0, m = 0, n = 0;
      if (tile >= 0) {
        while (tile >= ctl.tile_prefix[pos + 1]) ++pos;
        g = ctl.gorder[pos];
        const TileInfo ti = tile_info(g, tile - ctl.tile_prefix[pos]);
        m = ti.m;
        n = ti.n;
      }
      uint32_t hb0[16], hb1[16];
      if (tile >= 0) {
        const uint16_t* src = hbar_src(g, m, n, 0);
        if (src != nullptr) load_bf16x32(src, hb0);
      }
      int ring = 0;  // staging buffer of the next output box
      for (; tile >= 0; ++i) {
        const int nt = next_tile(i + 1);
        int pos2 = pos, g2 = 0, m2 = 0, n2 = 0;
        if (nt >= 0) {
          while (nt >= ctl.tile_prefix[pos2 + 1]) ++pos2;
          g2 = ctl.gorder[pos2];
          const TileInfo t2 = tile_info(g2, nt - ctl.tile_prefix[pos2]);
          m2 = t2.m;
          n2 = t2.n;
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const uint16_t* src = hbar_src(g2, m2, n2, c2);
            if (src != nullptr) asm volatile("prefetch.global.L2 [%0];" ::"l"(src) : "memory");
          }
        }
        {
          const uint16_t* src = hbar_src(g, m, n, 1);
          if (src != nullptr) load_bf16x32(src, hb1);
        }
        const int buf = i & 1;
        const uint32_t tph = (i >> 1) & 1;
        const bool got = mbar_wait_cluster(smem_u32(&ctl.tfull[buf]), tph, abort_flag, dev_err);
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * 256;
        const int nvalid = ctl.pnrows[g];
        const int orow0 = ctl.prow0[g];  // output rows (padded layout / shared rows)
        const int row = m * kTileM + r_in_tile;
        const bool valid = row < nvalid;
        const int warp_row0 = m * kTileM + 128 * static_cast<int>(rank) + q * 32;
        const bool full_box = warp_row0 + kOutBoxRows <= nvalid;
        const int col0 = n * hw;
        const size_t orow = static_cast<size_t>(orow0 + (valid ? row : 0));
        bool released = false, next0 = false;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int cc = part * (hw / 2) + c2 * kOutBoxCols;
          if (col0 + cc >= p.N) break;
          uint32_t rg[32], ru[32];
          tmem_ld_32cols(taddr + cc, rg);
          tmem_ld_32cols(taddr + hw + cc, ru);
          tmem_ld_wait();
          if (c2 == 1 || col0 + cc + kOutBoxCols >= p.N) {
            // the last box is in registers: hand the accumulator back
            // before its math and stores
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(buf ? tempty_leader1 : tempty_leader0);
            released = true;
          }
          const uint32_t(&hb)[16] = c2 == 0 ? hb0 : hb1;
          uint8_t* sg = stage_out + ring * kOutBoxBytes;
          uint8_t* su = stage_out + (ring == 2 ? 0 : ring + 1) * kOutBoxBytes;
          uint8_t* sh = stage_out + (ring == 0 ? 2 : ring - 1) * kOutBoxBytes;
          if (full_box) {
            // the stores that last read these buffers are done reading
            if (want_h)
              bulk_wait_group_read0();
            else
              bulk_wait_group_read1();
            __syncwarp();
          }
          // 16-byte chunk v of the row: columns 8 v .. 8 v + 7 of the box
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t og[4], ou[4], oh[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int j = 4 * v + jj;
              float gb[2], ub[2], hv[2];
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const float gg = __uint_as_float(rg[2 * j + t]);
                const float uu = __uint_as_float(ru[2 * j + t]);
                const float hh = t ? bf16_hi(hb[j]) : bf16_lo(hb[j]);
                const float e = __expf(-gg);
                const float sig = __fdividef(1.0f, 1.0f + e);
                const float silu = __fdividef(gg, 1.0f + e);  // the forward's expression
                hv[t] = silu * uu;
                // silu'(g) = sigmoid(g) (1 + g (1 - sigmoid(g)))
                gb[t] = hh * uu * (sig * (1.0f + gg * (1.0f - sig)));
                ub[t] = hh * silu;
              }
              og[jj] = pack_bf16x2(gb[0], gb[1]);
              ou[jj] = pack_bf16x2(ub[0], ub[1]);
              oh[jj] = pack_bf16x2(hv[0], hv[1]);
            }
            if (full_box) {
              const int sw = lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4);
              *reinterpret_cast<uint4*>(sg + sw) = make_uint4(og[0], og[1], og[2], og[3]);
              *reinterpret_cast<uint4*>(su + sw) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
              if (want_h) *reinterpret_cast<uint4*>(sh + sw) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
            } else if (valid) {
              uint16_t* gdst = p.gu + orow * (2 * p.N) + col0 + cc + 8 * v;
              *reinterpret_cast<uint4*>(gdst) = make_uint4(og[0], og[1], og[2], og[3]);
              *reinterpret_cast<uint4*>(gdst + p.N) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
              if (want_h)
                *reinterpret_cast<uint4*>(p.h + orow * p.N + col0 + cc + 8 * v) =
                    make_uint4(oh[0], oh[1], oh[2], oh[3]);
            }
          }
          if (full_box) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int r0 = orow0 + warp_row0;
              tma_store_2d(&mapC, smem_u32(sg), col0 + cc, r0);
              bulk_commit_group();
              tma_store_2d(&mapC, smem_u32(su), p.N + col0 + cc, r0);
              bulk_commit_group();
              if (want_h) {
                tma_store_2d(&mapC2, smem_u32(sh), col0 + cc, r0);
                bulk_commit_group();
              }
            }
            ring = want_h ? ring : (ring == 0 ? 2 : ring - 1);
          }
          if (c2 == 0 && nt >= 0) {
            // box 0's h_bar registers are free: the next tile's box 0 rows
            const uint16_t* src = hbar_src(g2, m2, n2, 0);
            if (src != nullptr) load_bf16x32(src, hb0);
            next0 = true;
          }
        }
        if (!next0 && nt >= 0) {  // this warp had no box in this tile
          const uint16_t* src = hbar_src(g2, m2, n2, 0);
          if (src != nullptr) load_bf16x32(src, hb0);
        }
        if (!released) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(buf ? tempty_leader1 : tempty_leader0);
        }
        tile = nt;
        pos = pos2;
        g = g2;
        m = m2;
        n = n2;
      }
    } else {
      int pos = 0, i = 0;
      for (int tile = next_tile(0); tile >= 0; tile = next_tile(++i)) {
        while (tile >= ctl.tile_prefix[pos + 1]) ++pos;
        const int g = ctl.gorder[pos];
        const int local = tile - ctl.tile_prefix[pos];
        const TileInfo ti = tile_info(g, local);
        const int m = ti.m, n = ti.n;
        const bool routed = g < p.E;
        const int buf = i & 1;
        const uint32_t tph = (i >> 1) & 1;
        const bool got = mbar_wait_cluster(smem_u32(&ctl.tfull[buf]), tph, abort_flag, dev_err);
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * 256;
        const int cols_per_part = hw / 2;
        if (Tr::row_tiles) {
          const int nvalid = ctl.pnrows[g];
          const int orow0 = ctl.prow0[g];  // output rows (padded layout / shared rows)
          const int row = m * kTileM + r_in_tile;
          const bool valid = row < nvalid;
          const int warp_row0 = m * kTileM + 128 * static_cast<int>(rank) + q * 32;
          const bool full_box = warp_row0 + kOutBoxRows <= nvalid;
          const int col0 = n * hw;
          constexpr int kChunks = kTileN / 2 / kOutBoxCols;
          // All of this warp's accumulator columns are read in one burst with a
          // single wait, and the accumulator is handed back before packing and
          // storing (a wait after every 32-column box holds the MMAs back).
          uint32_t acc[kChunks][32];
#pragma unroll
          for (int c2 = 0; c2 < kChunks; ++c2) tmem_ld_32cols(taddr + part * cols_per_part + c2 * kOutBoxCols, acc[c2]);
          tmem_ld_wait();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(buf ? tempty_leader1 : tempty_leader0);
#pragma unroll
          for (int c2 = 0; c2 < kChunks; ++c2) {
            const int cc = part * cols_per_part + c2 * kOutBoxCols;
            if (col0 + cc >= p.N) break;
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              packed[j] = pack_bf16x2(__uint_as_float(acc[c2][2 * j]), __uint_as_float(acc[c2][2 * j + 1]));
            if (full_box) {
              bulk_wait_group_read0();
              __syncwarp();
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4* dst = reinterpret_cast<uint4*>(stage_out + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4));
                *dst = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&mapC, smem_u32(stage_out), col0 + cc, orow0 + warp_row0);
                bulk_commit_group();
              }
            } else if (valid) {
              store_bf16x32(p.C + static_cast<size_t>(orow0 + row) * p.N + col0 + cc, packed);
            }
          }
        } else {
          // kWgrad: fp32 rows m * 256 + r (< M), columns n * 256 + cc (< N);
          // a split group's chunk goes to its partial slot.  Each 32 x 16 box
          // is staged with the 64-byte swizzle (conflict-free 16-byte writes)
          // and written by one TMA store; rows past M are clipped by the map.
          const bool empty_k = ti.kb1 <= ti.kb0;
          const bool split = ctl.nchunk[g] > 1;
          const int warp_row0 = m * kTileM + 128 * static_cast<int>(rank) + q * 32;
          const bool any_row = warp_row0 < p.M;
          // all of this warp's columns in one burst, then the accumulator is released
          constexpr int kBoxes = kTileN / 2 / 32;
          uint32_t acc[kBoxes][32];
          if (any_row) {
#pragma unroll
            for (int b = 0; b < kBoxes; ++b) tmem_ld_32cols(taddr + part * cols_per_part + 32 * b, acc[b]);
            tmem_ld_wait();
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(buf ? tempty_leader1 : tempty_leader0);
#pragma unroll
          for (int b = 0; b < kBoxes; ++b) {
            const int cc = part * cols_per_part + 32 * b;
            const int col = n * kTileN + cc;
            if (col >= p.N || !any_row) break;
            const uint32_t(&ra)[32] = acc[b];
            const CUtensorMap* om;
            int x, z;
            if (split) {
              om = &mapC5;
              x = col;
              z = ctl.pslot[g] + ti.c;
            } else {
              const bool second = col >= p.n_split;
              om = routed ? (second ? &mapC2 : &mapC) : (second ? &mapC4 : &mapC3);
              x = second ? col - p.n_split : col;
              z = routed ? g : 0;
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              bulk_wait_group_read0();  // the previous box's store has read the buffer
              __syncwarp();
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int j = 16 * hh + 4 * v;
                const uint4 val = empty_k ? make_uint4(0u, 0u, 0u, 0u)
                                          : make_uint4(ra[j], ra[j + 1], ra[j + 2], ra[j + 3]);
                *reinterpret_cast<uint4*>(stage_out + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4)) = val;
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(om, smem_u32(stage_out), x + kWOutCols * hh, warp_row0, z);
                bulk_commit_group();
              }
            }
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// Weight gradients of the split groups: the chunk partials of group g added
// in chunk order, split by column into the two outputs.  Block (x, g) covers
// 1024 consecutive floats of [M, N].
__global__ void __launch_bounds__(256) wgrad_reduce_kernel(const float* __restrict__ part,
                                                           const int32_t* __restrict__ offsets, int E,
                                                           int T_shared, int M, int N, int n_split,
                                                           float* w_a, float* w_b, float* ws_a, float* ws_b) {
  griddep_wait();
  griddep_launch_dependents();
  const int g = blockIdx.y;
  auto nchunk = [&](int h) {
    const int rows = h < E ? ((offsets[h + 1] - offsets[h] + 63) & ~63) : T_shared;
    const int nkb = (rows + kBK - 1) / kBK;
    return max(1, (nkb + kMaxChunkKb - 1) / kMaxChunkKb);
  };
  const int nc = nchunk(g);
  if (nc <= 1) return;
  int slot = 0;
  for (int h = 0; h < g; ++h) {
    const int c = nchunk(h);
    slot += c > 1 ? c : 0;
  }
  const size_t mn = static_cast<size_t>(M) * N;
  const size_t i4 = (static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x) * 4;
  if (i4 >= mn) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = 0; c < nc; ++c) {
    const float4 v = *reinterpret_cast<const float4*>(part + (slot + c) * mn + i4);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const int row = static_cast<int>(i4 / N), col = static_cast<int>(i4 % N);
  const bool routed = g < E;
  const bool second = col >= n_split;
  float* base = routed ? (second ? w_b : w_a) : (second ? ws_b : ws_a);
  const int ncols = second ? N - n_split : n_split;
  const int c0 = second ? col - n_split : col;
  *reinterpret_cast<float4*>(base + (routed ? static_cast<size_t>(g) * M * ncols : 0) +
                             static_cast<size_t>(row) * ncols + c0) = acc;
}

// Per-device launch state: co-resident CTA pairs per mode, error word address.
struct BwdDevice {
  int pairs[4] = {0, 0, 0, 0};
  unsigned int* dev_err = nullptr;
  bool ready = false;
};
BwdDevice g_bwd_dev[64];
std::mutex g_bwd_mu;

template <int kMode>
cudaError_t mode_setup(int sms, int* pairs) {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_bwd_kernel<kMode>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes_of(kMode));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes_of(kMode);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaOccupancyMaxActiveClusters(pairs, grouped_gemm_bwd_kernel<kMode>, &cfg);
  if (e != cudaSuccess) return e;
  return *pairs >= 1 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t bwd_setup(BwdDevice* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_bwd_mu);
  BwdDevice& bd = g_bwd_dev[dev];
  if (!bd.ready) {
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = mode_setup<kDgradW2>(sms, &bd.pairs[0])) != cudaSuccess) return e;
    if ((e = mode_setup<kActBwd>(sms, &bd.pairs[1])) != cudaSuccess) return e;
    if ((e = mode_setup<kDgradX>(sms, &bd.pairs[2])) != cudaSuccess) return e;
    if ((e = mode_setup<kWgrad>(sms, &bd.pairs[3])) != cudaSuccess) return e;
    if ((e = device_error_address(&bd.dev_err)) != cudaSuccess) return e;
    bd.ready = true;
  }
  *out = bd;
  return cudaSuccess;
}

template <int kMode>
cudaError_t launch_mode(const CUtensorMap (&m)[kMaps], BwdArgs a, cudaStream_t s, bool pdl) {
  BwdDevice bd;
  cudaError_t e = bwd_setup(&bd);
  if (e != cudaSuccess) return e;
  a.dev_err = bd.dev_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * bd.pairs[kMode], 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes_of(kMode);
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
  e = cudaLaunchKernelEx(&cfg, grouped_gemm_bwd_kernel<kMode>, m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7],
                         m[8], m[9], m[10], a);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

BwdArgs base_args(const BwdLayout& L, const int32_t* offsets) {
  BwdArgs a = {};
  a.offsets = offsets;
  a.E = L.d.E;
  a.S = L.d.T * L.d.k;
  a.S_pad = L.S_pad;
  a.T_shared = L.shared ? L.d.T : 0;
  return a;
}

}  // namespace

int bwd_padded_rows(const moe_dims& d) { return d.T * d.k + 64 * d.E; }

size_t bwd_wgrad_part_floats(const moe_dims& d, bool shared) {
  // a split group has nchunk < 2 nkb / kMaxChunkKb chunks
  const size_t kb = (static_cast<size_t>(d.T) * d.k + 64 * d.E) / kBK + (shared ? (d.T + kBK - 1) / kBK : 0);
  const size_t slots = kb / (kMaxChunkKb / 2) + 2;
  return slots * 2 * static_cast<size_t>(d.D) * d.F;
}

cudaError_t launch_bwd_dgrad_w2(const BwdLayout& L, const int32_t* offsets, const uint16_t* ybar,
                                const uint16_t* d_out, const uint16_t* W2, const uint16_t* Ws2,
                                uint16_t* hbar, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const uint64_t rows = static_cast<uint64_t>(L.S_pad) + (L.shared ? d.T : 0);
  CUtensorMap m[kMaps];
  cudaError_t e;
  // K-major operands as {64, rows, K / 64} block views: one box of 128 rows
  // and a stage's 64-deep atoms per operand
  constexpr uint32_t na = bk_of(kDgradW2) / 64;
  if ((e = tensor_map_blocks(&m[0], ybar, L.S_pad, d.D, na, 128)) != cudaSuccess) return e;
  if ((e = tensor_map_blocks(&m[2], W2, static_cast<uint64_t>(d.E) * d.F, d.D, na, 128)) != cudaSuccess) return e;
  if (L.shared) {
    if ((e = tensor_map_blocks(&m[1], d_out, d.T, d.D, na, 128)) != cudaSuccess) return e;
    if ((e = tensor_map_blocks(&m[4], Ws2, d.F, d.D, na, 128)) != cudaSuccess) return e;
  } else {
    m[1] = m[0];
    m[4] = m[2];
  }
  m[3] = m[2];
  m[5] = m[4];
  if ((e = tensor_map_2d(&m[6], hbar, rows, d.F, kOutBoxRows, kOutBoxCols)) != cudaSuccess) return e;
  BwdArgs a = base_args(L, offsets);
  a.K = d.D;
  a.N = d.F;
  a.b_rows = d.F;
  a.C = hbar;
  m[7] = m[6];
  m[8] = m[9] = m[10] = m[6];
  return launch_mode<kDgradW2>(m, a, s, pdl);
}

cudaError_t launch_bwd_act(const BwdLayout& L, const int32_t* offsets, const uint16_t* x_sorted,
                           const uint16_t* x, const uint16_t* W1, const uint16_t* W3,
                           const uint16_t* Ws1, const uint16_t* Ws3, const uint16_t* hbar,
                           uint16_t* gu, uint16_t* h, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const int S = d.T * d.k;
  CUtensorMap m[kMaps];
  cudaError_t e;
  constexpr uint32_t kb1 = bk_of(kActBwd);
  if ((e = tensor_map_blocks(&m[0], x_sorted, S, d.D, kb1 / 64, 128)) != cudaSuccess) return e;
  if ((e = tensor_map_blocks(&m[2], W1, static_cast<uint64_t>(d.E) * d.D, d.F, 2, kb1)) != cudaSuccess) return e;
  if ((e = tensor_map_blocks(&m[3], W3, static_cast<uint64_t>(d.E) * d.D, d.F, 2, kb1)) != cudaSuccess) return e;
  if (L.shared) {
    if ((e = tensor_map_blocks(&m[1], x, d.T, d.D, kb1 / 64, 128)) != cudaSuccess) return e;
    if ((e = tensor_map_blocks(&m[4], Ws1, d.D, d.F, 2, kb1)) != cudaSuccess) return e;
    if ((e = tensor_map_blocks(&m[5], Ws3, d.D, d.F, 2, kb1)) != cudaSuccess) return e;
  } else {
    m[1] = m[0];
    m[4] = m[2];
    m[5] = m[3];
  }
  const uint64_t rows = static_cast<uint64_t>(L.S_pad) + (L.shared ? d.T : 0);
  if ((e = tensor_map_2d(&m[6], gu, rows, 2 * d.F, kOutBoxRows, kOutBoxCols)) != cudaSuccess) return e;
  if (h != nullptr) {
    if ((e = tensor_map_2d(&m[7], h, rows, d.F, kOutBoxRows, kOutBoxCols)) != cudaSuccess) return e;
  } else {
    m[7] = m[6];
  }
  BwdArgs a = base_args(L, offsets);
  a.K = d.D;
  a.N = d.F;
  a.hbar = hbar;
  a.gu = gu;
  a.h = h;
  m[8] = m[9] = m[10] = m[6];
  return launch_mode<kActBwd>(m, a, s, pdl);
}

cudaError_t launch_bwd_dgrad_x(const BwdLayout& L, const int32_t* offsets, const uint16_t* gu,
                               const uint16_t* W1, const uint16_t* W3, const uint16_t* Ws1,
                               const uint16_t* Ws3, uint16_t* xbar, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const uint64_t rows = static_cast<uint64_t>(L.S_pad) + (L.shared ? d.T : 0);
  CUtensorMap m[kMaps];
  cudaError_t e;
  constexpr uint32_t nx = bk_of(kDgradX) / 64;
  if ((e = tensor_map_blocks(&m[0], gu, L.S_pad, 2 * d.F, nx, 128)) != cudaSuccess) return e;
  if ((e = tensor_map_blocks(&m[2], W1, static_cast<uint64_t>(d.E) * d.D, d.F, nx, 128)) != cudaSuccess) return e;
  if ((e = tensor_map_blocks(&m[3], W3, static_cast<uint64_t>(d.E) * d.D, d.F, nx, 128)) != cudaSuccess) return e;
  if (L.shared) {
    const uint16_t* gu_sh = gu + static_cast<size_t>(L.S_pad) * 2 * d.F;
    if ((e = tensor_map_blocks(&m[1], gu_sh, d.T, 2 * d.F, nx, 128)) != cudaSuccess) return e;
    if ((e = tensor_map_blocks(&m[4], Ws1, d.D, d.F, nx, 128)) != cudaSuccess) return e;
    if ((e = tensor_map_blocks(&m[5], Ws3, d.D, d.F, nx, 128)) != cudaSuccess) return e;
  } else {
    m[1] = m[0];
    m[4] = m[2];
    m[5] = m[3];
  }
  if ((e = tensor_map_2d(&m[6], xbar, rows, d.D, kOutBoxRows, kOutBoxCols)) != cudaSuccess) return e;
  BwdArgs a = base_args(L, offsets);
  a.K = 2 * d.F;
  a.K1 = d.F;
  a.N = d.D;
  a.b_rows = d.D;
  a.C = xbar;
  m[7] = m[6];
  m[8] = m[9] = m[10] = m[6];
  return launch_mode<kDgradX>(m, a, s, pdl);
}

cudaError_t launch_bwd_wgrad(const BwdLayout& L, const int32_t* offsets, const uint16_t* A,
                             int a_padded, int M, const uint16_t* A_sh, const uint16_t* B, int N,
                             const uint16_t* B_sh, int n_split, float* w_a, float* w_b, float* ws_a,
                             float* ws_b, float* part, cudaStream_t s, bool pdl) {
  const moe_dims& d = L.d;
  const int S = d.T * d.k;
  CUtensorMap m[kMaps];
  cudaError_t e;
  if ((e = tensor_map_blocks(&m[0], A, a_padded ? L.S_pad : S, M, 2)) != cudaSuccess) return e;
  if ((e = tensor_map_blocks(&m[2], B, L.S_pad, N, 2)) != cudaSuccess) return e;
  if (L.shared) {
    if ((e = tensor_map_blocks(&m[1], A_sh, d.T, M, 2)) != cudaSuccess) return e;
    if ((e = tensor_map_blocks(&m[4], B_sh, d.T, N, 2)) != cudaSuccess) return e;
  } else {
    m[1] = m[0];
    m[4] = m[2];
  }
  m[3] = m[2];
  m[5] = m[4];
  // fp32 outputs as {columns, M, group or slot}: 16 x 32 boxes, rows past M clipped
  const int nb = N - n_split;
  const uint64_t slots = bwd_wgrad_part_floats(d, L.shared) / (2 * static_cast<uint64_t>(d.D) * d.F);
  if ((e = tensor_map_f32_3d(&m[6], w_a, n_split, M, d.E, kWOutCols, kOutBoxRows)) != cudaSuccess) return e;
  // nb == 0 (one output, no second half): its maps are never used
  if (nb > 0) {
    if ((e = tensor_map_f32_3d(&m[7], w_b, nb, M, d.E, kWOutCols, kOutBoxRows)) != cudaSuccess) return e;
  } else {
    m[7] = m[6];
  }
  if (L.shared) {
    if ((e = tensor_map_f32_3d(&m[8], ws_a, n_split, M, 1, kWOutCols, kOutBoxRows)) != cudaSuccess) return e;
    if (nb > 0) {
      if ((e = tensor_map_f32_3d(&m[9], ws_b, nb, M, 1, kWOutCols, kOutBoxRows)) != cudaSuccess) return e;
    } else {
      m[9] = m[8];
    }
  } else {
    m[8] = m[6];
    m[9] = m[7];
  }
  if ((e = tensor_map_f32_3d(&m[10], part, N, M, slots, kWOutCols, kOutBoxRows)) != cudaSuccess) return e;
  BwdArgs a = base_args(L, offsets);
  a.M = M;
  a.N = N;
  a.a_padded = a_padded;
  a.n_split = n_split;
  a.w_a = w_a;
  a.w_b = w_b;
  a.ws_a = ws_a;
  a.ws_b = ws_b;
  a.part = part;
  e = launch_mode<kWgrad>(m, a, s, pdl);
  if (e != cudaSuccess) return e;
  const size_t mn4 = (static_cast<size_t>(M) * N / 4 + 255) / 256;
  const dim3 grid(static_cast<unsigned>(mn4), d.E + (L.shared ? 1 : 0));
  return launch_kernel(wgrad_reduce_kernel, grid, dim3(256), 0, s, true, static_cast<const float*>(part), offsets,
                       d.E, L.shared ? d.T : 0, M, N, n_split, w_a, w_b, ws_a, ws_b);
}

}  // namespace moe
