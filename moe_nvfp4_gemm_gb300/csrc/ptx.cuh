// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// (tiled tensor and plain bulk copies), tcgen05 (TMEM alloc, copy, block-scaled
// MMA, commit, loads) and shared-memory / instruction descriptors.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define DEVI __device__ __forceinline__

namespace nvfp4 {

// Device-side status codes (mirrors nvfp4_status in nvfp4.h).
enum : int32_t { kStatusTimeout = -7, kStatusBadOffsets = -8 };

// A wait that has not completed after this long gives up and reports a timeout (the
// default; every launch passes its own limit).
constexpr uint64_t kWatchdogNs = 2000000000ull;

DEVI uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

DEVI uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One lane of a converged warp (elect.sync). Issuing tcgen05 and TMA operations
// from a converged warp through an elected lane keeps their operands warp-uniform.
DEVI bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ---- mbarrier ---------------------------------------------------------------

DEVI void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

DEVI void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

DEVI void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

DEVI void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

DEVI bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Waits for the phase with the given parity to complete. Gives up (returns
// false) when *abort becomes non-zero or after limit_ns, in which case it sets
// *abort so that every other role of the CTA stops too.
DEVI bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
}

// Warp-collective wait: every lane polls, the result is the same in all lanes.
DEVI bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int32_t* abort, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, limit_ns)) != 0;
}

// Named CTA barrier `id` over `nthreads` threads (whole warps). Used in lockstep by
// two warps that run exactly the same number of iterations: it has no time-out.
DEVI void named_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// named_sync that also returns the AND of `v` over all participating threads
// (bar.red.and.pred): hands one warp's verdict to another without touching memory.
DEVI bool named_sync_and(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %3, 0;\n\t"
      "bar.red.and.pred po, %1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// ---- programmatic dependent launch ---------------------------------------------

// Blocks until the grids this one depends on have completed and their memory is
// visible (returns at once when the launch had no programmatic dependency).
DEVI void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel in the stream start launching (its own griddep_wait still
// orders its reads after this grid's completion).
DEVI void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- TMA ----------------------------------------------------------------------

DEVI void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

DEVI uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

DEVI uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

DEVI void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t y,
                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// 2-D tiled TMA store shared -> global, tracked by this thread's bulk async-group.
// Elements of the box outside the tensor are not written.
DEVI void tma_store_2d(const CUtensorMap* m, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
DEVI void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until this thread's bulk stores have finished reading shared memory.
DEVI void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until this thread's bulk stores are complete.
DEVI void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA) reads of them.
DEVI void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// The same loads without an L2 cache hint: createpolicy costs the issuing warp about
// a microsecond, so latency-bound kernels issue their first ring without one.
DEVI void tma_load_2d_plain(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
DEVI void bulk_load_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// L2 prefetches: no shared memory is written and nothing completes on a barrier; a later
// load of the same bytes finds them in L2. A prefetch returns no data, so issuing it
// before a dependency wait cannot read stale values: the L2 is the point of coherence
// for every later read of this GPU.
DEVI void tma_prefetch_2d(const CUtensorMap* m, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y)
               : "memory");
}
// `bytes` from src, both multiples of 16.
DEVI void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Four rows (r0..r3) of a 2-D tensor whose map has a one-row box, `x` the first
// column: 4 x box-width bytes land contiguously at dst (swizzled like a tile load).
DEVI void tma_gather4(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t r0, int32_t r1, int32_t r2,
                      int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

// Bulk copy from this CTA's shared memory into another CTA's of the cluster, completing
// `bytes` on the mbarrier at `bar_cluster` there; tracked by this thread's bulk group.
DEVI void bulk_copy_to_cluster(uint32_t dst_cluster, const void* src, uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

// Plain bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
DEVI void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---- clusters ------------------------------------------------------------------

DEVI uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

DEVI void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
DEVI uint32_t mapa_shared(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}

// Relaxed arrive on an mbarrier of any CTA in the cluster. Used only to hand a
// drained TMEM accumulator back to the MMA issuer: the tcgen05.ld reads are already
// complete (tcgen05.wait::ld) when the arrive executes, so no memory needs to be
// released, and a release-ordered arrive at cluster scope measured ~1,200 cycles
// against ~100 for this one, on the critical path of every tile.
DEVI void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 2-D tiled TMA load issued for a CTA pair: lands in this CTA's shared memory and
// signals the mbarrier at `bar_cluster` (this CTA's or its peer's).
DEVI void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int32_t x, int32_t y,
                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// ---- tcgen05 --------------------------------------------------------------------

DEVI void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

DEVI void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrives once on `bar` when every tcgen05 operation this thread issued so far is done.
DEVI void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 rows x 16 bytes from shared memory into TMEM columns [col, col+4) of lanes
// 0-31, replicated into all four 32-lane groups.
DEVI void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T, FP4 E2M1 operands with UE4M3 scales per 16 K.
DEVI void tc_mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                      uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T with A pair-wise 2:4 sparse (4:8 on FP4): K = 128 per
// instruction, A holds 64 kept values a row; `meta_tmem` holds each row's 16 index nibbles
// (lane = row, two columns, group g at nibble g % 8 of column g / 8); one UE4M3 scale per 32
// K elements of each operand (4 per row, the same TMEM tiles as a dense K = 64 step).
DEVI void tc_mma_nvf4_sp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t meta_tmem,
                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %7, 0;\n\t"
      "tcgen05.mma.sp.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, [%3], %4, [%5], [%6], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(meta_tmem), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 128 rows x 32 bytes from shared memory into TMEM lanes 0-127, columns [col, col+8).
// Source layout: rows in groups of 8, each row's 32 bytes as two 16-byte halves,
// (r/8)*256 + (half)*128 + (r%8)*16 (no swizzle; leading offset 128, stride 256).
DEVI void tc_cp_128x256b(uint32_t taddr, uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 16;
  d |= static_cast<uint64_t>(256 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns.
DEVI void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

DEVI void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// CTA-pair forms: allocation by one warp of each CTA of the pair; MMA, scale copy
// and commit issued by one thread of the even CTA, acting on both CTAs.
DEVI void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

DEVI void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

DEVI void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

DEVI void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

DEVI void tc_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

DEVI void tc_mma_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand tile written by TMA with the
// 128-byte swizzle (8-row x 128-byte atoms, 1024 bytes apart). Tile base must be
// 1024-byte aligned; a K offset inside the atom is added to the start address.
DEVI uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: next 8-row group
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
  return d;
}

// Descriptor for a 512-byte scale chunk (32 rows x 16 bytes, no swizzle,
// 8-row core matrices 128 bytes apart) read by tcgen05.cp.
DEVI uint64_t desc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor for kind::mxf4nvf4: A and B E2M1, K-major, UE4M3
// scales (scale-factor ids 0), dense, shape M x N x 64.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// The same with the sparsity flag (bit 2): A pair-wise sparse, shape M x N x 128.
__host__ __device__ constexpr uint32_t idesc_nvf4_sp(int M, int N) { return idesc_nvf4(M, N) | (1u << 2); }

DEVI uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

DEVI void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// 32-byte store (one full sector); p must be 32-byte aligned.
DEVI void st_global_v8(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Drains NC accumulator columns (one TMEM lane quarter, starting at taddr) of one
// warp into registers, releases the accumulator through `release` (called by the
// whole warp after the loads completed), then scales by alpha and stores bf16
// to yrow[col0 .. col0 + NC), columns >= N skipped in groups of 8. With `wide`
// (N % 16 == 0 and y 32-byte aligned) each lane writes whole 32-byte sectors.
template <int NC, typename Release>
DEVI void drain_accumulator(uint32_t taddr, float alpha, uint16_t* yrow, bool row_ok, int col0, int N, bool wide,
                            Release release) {
  static_assert(NC % 16 == 0, "column groups of 16");
  uint32_t r[NC];
#pragma unroll
  for (int c = 0; c < NC; c += 32) tmem_ld32(taddr + c, r + c);
  tmem_ld_wait();
  tc_fence_before();
  __syncwarp();
  release();
  if (row_ok) {
#pragma unroll
    for (int c = 0; c < NC; c += 16) {
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        w[j] = pack_bf16x2(__uint_as_float(r[c + 2 * j]) * alpha, __uint_as_float(r[c + 2 * j + 1]) * alpha);
      if (wide && col0 + c + 16 <= N) {
        st_global_v8(yrow + col0 + c, w);
      } else {
        if (col0 + c < N) st_global_v4(yrow + col0 + c, w[0], w[1], w[2], w[3]);
        if (col0 + c + 8 < N) st_global_v4(yrow + col0 + c + 8, w[4], w[5], w[6], w[7]);
      }
    }
  }
}

// As drain_accumulator, but the bf16 rows leave through TMA stores: the warp
// writes each 32-row x 64-column block into its 4 KB shared-memory buffer `buf`
// (1024-byte aligned, 128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8),
// which keeps the 32 lanes' writes at 4 wavefronts) and lane 0 stores it to
// y[row0 .. row0 + 32) x [col0 + 64 j ..) through tmY (box 64 x 32, clipped at the
// tensor's edges). The stores leave the load/store unit free and write whole
// 128-byte lines, so they do not compete with the TMA operand loads the way 32
// rows of scattered sector writes per instruction do.
template <int NC, typename Release>
DEVI void drain_accumulator_tma(uint32_t taddr, float alpha, uint8_t* buf, const CUtensorMap* tmY, int col0, int row0,
                                Release release) {
  static_assert(NC % 64 == 0, "64-column store boxes");
  const int lane = threadIdx.x & 31;
  uint32_t r[NC];
#pragma unroll
  for (int c = 0; c < NC; c += 32) tmem_ld32(taddr + c, r + c);
  tmem_ld_wait();
  tc_fence_before();
  __syncwarp();
  release();
  const uint32_t row_addr = smem_u32(buf) + lane * 128;
#pragma unroll
  for (int j = 0; j < NC / 64; ++j) {
    if (lane == 0) bulk_wait_group_read0();  // the previous box has left the buffer
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t* v = r + j * 64 + c * 8;
      const uint32_t a = row_addr + ((c ^ (lane & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                   "r"(pack_bf16x2(__uint_as_float(v[0]) * alpha, __uint_as_float(v[1]) * alpha)),
                   "r"(pack_bf16x2(__uint_as_float(v[2]) * alpha, __uint_as_float(v[3]) * alpha)),
                   "r"(pack_bf16x2(__uint_as_float(v[4]) * alpha, __uint_as_float(v[5]) * alpha)),
                   "r"(pack_bf16x2(__uint_as_float(v[6]) * alpha, __uint_as_float(v[7]) * alpha))
                   : "memory");
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmY, buf, col0 + j * 64, row0);
      bulk_commit_group();
    }
  }
}

DEVI void report_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace nvfp4
