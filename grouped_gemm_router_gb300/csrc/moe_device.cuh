// Device-side building blocks for sm_103a: mbarriers, TMA tensor loads,
// tcgen05 (5th-generation tensor core) MMA / TMEM access, and the bounded
// waits every persistent kernel of this library uses.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MOE_DEV __device__ __forceinline__

// Bit set in the device error word (defined in grouped_gemm.cu, read and
// cleared by moe_device_error) when an on-chip wait times out.
#define MOE_DEVERR_TIMEOUT 1u

// A wait on an on-chip barrier is abandoned after this long.
#define MOE_WAIT_TIMEOUT_NS 2000000000ull

MOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEV uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
MOE_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

MOE_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

MOE_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

MOE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with parity `parity` of barrier `bar` to complete.
// Gives up when *abort is set by another thread or after timeout_ns; in the
// second case it sets *abort and the device error word.  Returns false when
// it gave up.
MOE_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int* dev_err,
                       uint64_t timeout_ns = MOE_WAIT_TIMEOUT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        *abort = 1;
        atomicOr(dev_err, MOE_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Same as mbar_try_wait with acquire semantics at cluster scope (for barriers
// that receive arrivals from the peer CTA of a cluster).
MOE_DEV bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait as mbar_wait, at cluster scope.
MOE_DEV bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort,
                               unsigned int* dev_err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > MOE_WAIT_TIMEOUT_NS) {
        *abort = 1;
        atomicOr(dev_err, MOE_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Arrive on a barrier given by its shared::cluster address (possibly in the
// peer CTA), release at cluster scope.
MOE_DEV void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// ---------------------------------------------------------------------------
// Clusters
// ---------------------------------------------------------------------------
MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

MOE_DEV uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

MOE_DEV uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// shared::cluster address of the variable at shared::cta address `addr` in
// the CTA of rank `rank` of this cluster.
MOE_DEV uint32_t map_to_cta(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// All threads of all CTAs of the cluster.
MOE_DEV void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), 2-D tiles into shared memory
// ---------------------------------------------------------------------------
MOE_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Loads the box at coordinates (c0 = innermost, c1) into shared memory at
// `dst`, signalling `bar` with the byte count.  c0 * element size must be a
// multiple of 16 bytes.
MOE_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                         int32_t c1, uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(cache_policy)
      : "memory");
}

// As tma_load_2d for a CTA pair: `bar` is a shared::cluster address, which may
// be the barrier of the peer CTA.
MOE_DEV void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                              int32_t c1, uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(cache_policy)
      : "memory");
}

// As tma_load_2d_pair for a 3-D tensor map (coordinates c0 = innermost, c1, c2).
MOE_DEV void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                              int32_t c1, int32_t c2, uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(cache_policy)
      : "memory");
}

// Stores the 2-D box at coordinates (c0, c1) from shared memory at `src`
// (bulk async group of the executing thread).  c0 * element size must be a
// multiple of 16 bytes and neither coordinate may be negative.
MOE_DEV void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}

// As tma_store_2d for a 3-D tensor map; elements outside the tensor are not written.
MOE_DEV void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1, int32_t c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(src)
               : "memory");
}

MOE_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until no bulk group of this thread still reads shared memory.
MOE_DEV void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until at most one bulk group of this thread still reads shared memory.
MOE_DEV void bulk_wait_group_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Waits until all bulk groups of this thread have completed.
MOE_DEV void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Makes generic-proxy shared-memory writes visible to the async proxy (TMA).
MOE_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

MOE_DEV uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MOE_DEV uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads
// ---------------------------------------------------------------------------
// Whole warp: allocate `ncols` TMEM columns, base address written to smem.
MOE_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

MOE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// CTA-pair forms (cta_group::2): both CTAs of the pair allocate / free the
// same columns of their own TMEM together.
MOE_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

MOE_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// One MMA over the CTA pair: A rows split between the two CTAs (M / 2 each),
// B columns split (N / 2 each), D rows in each CTA's own TMEM.
MOE_DEV void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at shared::cta offset `bar` in every CTA of
// `cta_mask` when the pair MMAs issued so far by this thread complete.
MOE_DEV void umma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(cta_mask)
      : "memory");
}

MOE_DEV void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

MOE_DEV void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] x B[smem desc], bf16 inputs, fp32 accumulate.
MOE_DEV void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when all previously issued tcgen05.mma of this thread
// have completed.
MOE_DEV void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

MOE_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Warp-collective: thread i receives TMEM lane (lane field of taddr) + i,
// 32 consecutive 32-bit columns starting at the column field of taddr.
MOE_DEV void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor for a tile written by TMA with 128-byte
// swizzling (8 rows x 128 bytes per swizzle atom, atoms 1024-byte aligned).
//   lbo: byte distance between atoms along the leading dimension
//   sbo: byte distance between 8-row groups along the strided dimension
MOE_DEV uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: bf16 A and B, fp32 D,
// A K-major, B K-major (b_mn_major = 0) or N-major (1), shape M x N.
MOE_DEV uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn_major) {
  uint32_t d = 0;
  d |= 1u << 4;                 // D format: f32
  d |= 1u << 7;                 // A format: bf16
  d |= 1u << 10;                // B format: bf16
  d |= b_mn_major << 16;        // B major-ness
  d |= (N >> 3) << 17;          // N / 8
  d |= (M >> 4) << 24;          // M / 16
  return d;
}

// As idesc_bf16_f32 with the major-ness of A chosen too: A K-major
// (a_mn_major = 0) or M-major (1, the transpose of a row-major [K, M] tile).
MOE_DEV uint32_t idesc_bf16_f32_ab(uint32_t M, uint32_t N, uint32_t a_mn_major, uint32_t b_mn_major) {
  return idesc_bf16_f32(M, N, b_mn_major) | (a_mn_major << 15);
}

// ---------------------------------------------------------------------------
// Small helpers
// ---------------------------------------------------------------------------
MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

MOE_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

MOE_DEV uint32_t lane_id() { return threadIdx.x & 31u; }

// One epilogue warp's 32 rows x 32 fp32 columns (lane = row; v holds the
// row's 32 values as bits) stored as two boxes of 16 columns through the
// warp's 2 KB staging buffer with the 64-byte swizzle (16-byte chunk c of
// row r at chunk c ^ ((r / 2) % 4)) and TMA stores at (col, row0, 0) of a
// 3-D fp32 tensor map with a {16, 32, 1} box.  Waits first until the
// warp's earlier stores have read the buffer.
MOE_DEV void store_box_f32_tma(const CUtensorMap* map, uint8_t* stage, const uint32_t (&v)[32], int col,
                               int row0) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4* dst = reinterpret_cast<uint4*>(stage + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
      *dst = make_uint4(v[16 * half + 4 * c], v[16 * half + 4 * c + 1], v[16 * half + 4 * c + 2],
                        v[16 * half + 4 * c + 3]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                       reinterpret_cast<uint64_t>(map)),
                   "r"(col + 16 * half), "r"(row0), "r"(0), "r"(static_cast<uint32_t>(__cvta_generic_to_shared(stage)))
                   : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
  }
}

// The same 32 fp32 values of one row stored straight to global memory
// (rows of a box that crosses the end of a group).
MOE_DEV void store_row_f32(float* dst, const uint32_t (&v)[32]) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int c = 0; c < 8; ++c)
    d4[c] = make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]), __uint_as_float(v[4 * c + 2]),
                        __uint_as_float(v[4 * c + 3]));
}

// Programmatic dependent launch: wait until the preceding kernel of the
// stream has completed and its writes are visible (returns at once when this
// kernel was not launched as a programmatic dependent) ...
MOE_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// ... and allow the next kernel of the stream to start launching now.
MOE_DEV void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

MOE_DEV bool elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}
