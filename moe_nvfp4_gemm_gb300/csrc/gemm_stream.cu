// Weight-streaming NVFP4 GEMM for small token counts: decode-M dense layers and
// the grouped MoE path (per-expert GEMMs over routed tokens).
//
// Operations: "NVFP4 linear layer" (kernelindex, operation header), y = x @ W^T;
// MoE decode shape from "The Moment of Recalibration" (magik.net, Input
// Knowledge: 256 experts, top-8) and "The Moment of Synthesis" (magik.net,
// Reasoning: ~32 x 2048 x 6144 per expert, grouped GEMM as the lever for small
// per-expert M; persistent grouped GEMM in the Broader Narrative Arc of "The
// Moment of Recalibration").
//
// Swap-AB: the MMA's M side (128 TMEM lanes) holds 128 weight rows, its N side
// holds the tokens (padded to 16), so no token is padded to 128 rows. One TMA
// stream reads each weight tile once; the tokens come from L2.
//   dense decode: grid = (N/128) x S CTAs in clusters of S along K; each CTA
//     reduces its K slice in TMEM, the S partials are summed through DSMEM.
//   batched decode (k_gemm_batched): the dense decode body over a list of independent
//     GEMMs in one launch, each problem's CTAs as a single call's grid would be.
//   grouped: a persistent grid walks (token tile, weight tile) items built by
//     k_grouped_prep (ragged per-expert counts, empty experts skipped); each
//     item streams one expert's 128-row weight tile over all of K. Epilogues: bf16,
//     SwiGLU (bf16, or NVFP4 with the caller's global scale).
// Two warps issue each stage's copies (weight tile + scales; token rows + scales), each
// with its own expected bytes on the stage's barrier.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "nvfp4_quant.cuh"
#include "ptx.cuh"

namespace nvfp4 {


// One ring stage: the 128-row weight tile (128 bytes a row), the token tile (one 128-byte
// box a row; two for the sparse form, whose stage spans 512 K elements), the 2 KB of weight
// and token scales, and for the sparse form the 4 KB metadata tile.
struct StreamLayout {
  int stage_bytes, x_off, xbox, sfw_off, sfx_off, meta_off;
  __host__ __device__ StreamLayout(int x_rows, bool sparse = false) {
    x_off = 16384;
    xbox = x_rows * 128;
    sfw_off = x_off + (sparse ? 2 : 1) * xbox;
    sfx_off = sfw_off + 2048;
    meta_off = sfx_off + 2048;
    stage_bytes = meta_off + (sparse ? 4096 : 0);
  }
};

DEVI uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

struct Item {
  int wt;      // 128-row weight tile
  int e;       // expert (0 for dense)
  int row0;    // first token row
  int rows;    // token rows (<= x_rows)
  int slab;    // grouped scale slab
  int kb0, kb1;
};

template <bool GROUPED>
DEVI bool get_item(const StreamArgs& p, int i, int n_items, int NT, int KB, Item& it) {
  if (i >= n_items) return false;
  if (GROUPED) {
    const int tile = i / NT;
    const int4 t = __ldg(p.tiles + tile);
    it.wt = i % NT;
    it.e = t.x;
    it.row0 = t.y;
    it.rows = t.z;
    it.slab = t.w;
    it.kb0 = 0;
    it.kb1 = KB;
  } else {
    it.wt = i / p.split;
    const int sp = i % p.split;
    it.e = 0;
    it.row0 = 0;
    it.rows = p.M;
    it.slab = 0;
    // 32-bit arithmetic (KB * split <= 2^23 * 8 for every accepted K): a 64-bit division
    // costs the producer ~0.3 us on its way to the first load
    it.kb0 = (KB * sp) / p.split;
    it.kb1 = (KB * (sp + 1)) / p.split;
  }
  return true;
}

// Item i of a role's sequence (i, i + stride, ...). Grouped: `desc` holds item i's tile
// descriptor, loaded one item ahead; after filling `it` the load for item i + stride is
// issued into it, so that no role waits for a global load at an item boundary (a role
// that stalls there stops freeing ring slots, and the weight stream loses requests in
// flight).
template <bool GROUPED>
DEVI bool next_item(const StreamArgs& p, int i, int stride, int n_items, int NT, int KB, int4& desc, Item& it) {
  if (!GROUPED) return get_item<false>(p, i, n_items, NT, KB, it);
  if (i >= n_items) return false;
  it.wt = i % NT;
  it.e = desc.x;
  it.row0 = desc.y;
  it.rows = desc.z;
  it.slab = desc.w;
  it.kb0 = 0;
  it.kb1 = KB;
  if (i + stride < n_items) desc = __ldg(p.tiles + (i + stride) / NT);
  return true;
}

template <bool GROUPED>
DEVI int4 first_desc(const StreamArgs& p, int first, int n_items, int NT) {
  return (GROUPED && first < n_items) ? __ldg(p.tiles + first / NT) : make_int4(0, 0, 0, 0);
}

// Warp roles: 0 weight producer (each stage's weight tile and scales), 1 MMA issuer, 2-5
// epilogue, 6 stage waiter (waits for a stage's bytes and hands it to the MMA warp through
// a named barrier, so that the MMA-issuing warp itself never waits on an mbarrier per
// stage), 7 token producer (each stage's token rows and scales).
constexpr int kStreamThreads = 256;
constexpr int kStreamWaiterWarp = 6;
constexpr int kStreamTokenWarp = 7;  // token rows and their scales
constexpr uint32_t kStreamHandoffBarrier = 1;
constexpr uint32_t kStreamEpilogueBarrier = 2;  // the 4 epilogue warps

// VARIANT: bit 0 SwiGLU epilogue (with bit 3: emitting NVFP4), bit 1 token gather in the load
// stage (grouped only);
// bit 2 pair-wise 2:4 sparse weights (dense or plain grouped path): the weight tile holds compressed
// values, a stage spans 512 K elements (four K = 128 sparse MMAs) and carries the metadata
// tile. Compiled separately so that the plain kernels carry none of them.
// The kernel body; `cta` is this CTA's index among the CTAs of its problem (blockIdx.x
// for a single GEMM or the grouped kernel, the index within its GEMM in a batched launch).
template <bool GROUPED, int VARIANT>
DEVI void stream_body(const CUtensorMap& tmW, const CUtensorMap& tmX, const StreamArgs& p, const int cta) {
  constexpr bool SPARSE = (VARIANT & 4) != 0;
  constexpr int KSTAGE = SPARSE ? 512 : 256;  // K elements per stage
  constexpr int KMMA = KSTAGE / 4;            // K elements per MMA
  constexpr int SF_COLS = SPARSE ? 40 : 32;   // TMEM columns per stage: scales (+ metadata)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const StreamLayout L(p.x_rows, SPARSE);
  const int STAGES = p.stages;
  // Split-K (dense, S = p.split > 1): CTA rank r of a cluster owns tokens
  // [r * m_own, (r + 1) * m_own). Its partial sums leave from `part` = [token][128 rows]
  // fp32, which reuses the stage ring (one item per CTA; every stage has been consumed
  // when the epilogue runs), so each owner's block is contiguous, and arrive in the
  // owner's `recv` = [source rank][token - r * m_own][128].
  const int S = GROUPED ? 1 : p.split;
  const int m_own = (p.M + S - 1) / S;  // token slots per owner
  float* part = reinterpret_cast<float*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * L.stage_bytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [2]
  uint64_t* tempty = tfull + 2;      // [2]
  uint64_t* drain = tempty + 2;
  uint64_t* red_bar = drain + 1;     // all S partials of this CTA's tokens have landed
  volatile uint64_t* policies = red_bar + 1;  // [2] L2 cache policies (weights, tokens) once published
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_bar + 3);
  volatile uint32_t* policies_ready = tmem_slot + 2;
  float* recv = reinterpret_cast<float*>(smem + STAGES * L.stage_bytes + 512);
  // grouped with a token gather: the x rows (token indices) of the producer's current item
  int32_t* tok_idx = reinterpret_cast<int32_t*>(smem + STAGES * L.stage_bytes + 512);
  // grouped SwiGLU emitting NVFP4: one [32 tokens][16 columns] bf16 transpose tile per
  // epilogue warp, after the token indices
  uint16_t* xpose = reinterpret_cast<uint16_t*>(smem + STAGES * L.stage_bytes + 512 + grouped_extra_bytes(p.x_rows));
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t wd = p.watchdog_ns;
  const int N = p.N, K = p.K;
  const int NT = (N + 127) / 128;
  const int KB = (K + KSTAGE - 1) / KSTAGE;
  // 512-byte scale tiles per 128 rows: one per MMA step (weights over stored values)
  const int64_t KC4 = K / KMMA;
  const int64_t KMC = (K + 511) / 512;  // sparse: 4 KB metadata tiles per 128 weight rows

  // Where an item's tiles come from (computed once per item).
  struct Src {
    int32_t wrow0, row0;
    int n16;
    const uint8_t* sfw;
    const uint8_t* sfx;
    const uint8_t* meta;
  };
  auto item_src = [&](const Item& it) {
    Src r;
    r.wrow0 = it.e * N + it.wt * 128;
    r.row0 = it.row0;
    r.n16 = (it.rows + 15) >> 4;
    r.sfw = p.sfw + it.e * p.sfw_stride + static_cast<int64_t>(it.wt) * KC4 * 512;
    r.sfx = p.sfx + static_cast<int64_t>(it.slab) * KC4 * 512;
    r.meta = SPARSE ? p.meta + it.e * p.meta_stride + static_cast<int64_t>(it.wt) * KMC * 4096 : nullptr;
    return r;
  };
  // The token tiles and their scales of stage st_idx = K block kb (sparse: two boxes per row).
  auto issue_x = [&](uint8_t* st, uint64_t* bar, int kb, const Src& src, bool hint, uint64_t pol_x) {
    const int nsub = min(4, (K - kb * KSTAGE) / KMMA);
#pragma unroll
    for (int bx = 0; bx < (SPARSE ? 2 : 1); ++bx)
      for (int j = 0; j < src.n16; ++j) {
        uint8_t* dst = st + L.x_off + bx * L.xbox + j * 2048;
        const int32_t kx = kb * (KSTAGE / 2) + bx * 128;
        if (hint)
          tma_load_2d(dst, &tmX, bar, kx, src.row0 + j * 16, pol_x);
        else
          tma_load_2d_plain(dst, &tmX, bar, kx, src.row0 + j * 16);
      }
    if (hint)
      bulk_load(st + L.sfx_off, src.sfx + kb * 2048, nsub * 512, bar, pol_x);
    else
      bulk_load_plain(st + L.sfx_off, src.sfx + kb * 2048, nsub * 512, bar);
  };
  // Weight warp: requests stage st_idx = K block kb of an item, the 128-row weight tile and
  // its scales (and metadata), with their expected bytes on the stage's barrier, which
  // counts two arrivals: this one and the token warp's (issue_tokens).
  auto issue_stage = [&](int st_idx, int kb, const Src& src, bool hint, uint64_t pol_w) {
    const int32_t wrow0 = src.wrow0;
    const uint8_t* sfw = src.sfw;
    const int nsub = min(4, (K - kb * KSTAGE) / KMMA);
    uint8_t* st = smem + st_idx * L.stage_bytes;
    uint64_t* bar = &full[st_idx];
    mbar_arrive_expect_tx(bar, 16384 + nsub * 512 + (SPARSE ? 4096 : 0));
    if (hint) {
      tma_load_2d(st, &tmW, bar, kb * 128, wrow0, pol_w);
      bulk_load(st + L.sfw_off, sfw + kb * 2048, nsub * 512, bar, pol_w);
      if (SPARSE) bulk_load(st + L.meta_off, src.meta + kb * 4096, 4096, bar, pol_w);
    } else {
      tma_load_2d_plain(st, &tmW, bar, kb * 128, wrow0);
      bulk_load_plain(st + L.sfw_off, sfw + kb * 2048, nsub * 512, bar);
      if (SPARSE) bulk_load_plain(st + L.meta_off, src.meta + kb * 4096, 4096, bar);
    }
  };
  // Token warp: the token rows of stage st_idx (one tile load per 16 rows, or with a token
  // gather four rows per tile::gather4 from the one-row-box map of x) and their scales,
  // with their own expected bytes on the stage's barrier.
  auto issue_tokens = [&](int st_idx, int kb, const Src& src, bool hint, uint64_t pol_x) {
    const int nsub = min(4, (K - kb * KSTAGE) / KMMA);
    uint8_t* st = smem + st_idx * L.stage_bytes;
    uint64_t* bar = &full[st_idx];
    mbar_arrive_expect_tx(bar, (SPARSE ? 2 : 1) * src.n16 * 2048 + nsub * 512);
    if (GROUPED && (VARIANT & 2)) {
      for (int j = 0; j < src.n16 * 4; ++j)
        tma_gather4(st + L.x_off + j * 512, &tmX, bar, kb * 128, tok_idx[4 * j], tok_idx[4 * j + 1],
                    tok_idx[4 * j + 2], tok_idx[4 * j + 3]);
      if (hint)
        bulk_load(st + L.sfx_off, src.sfx + kb * 2048, nsub * 512, bar, pol_x);
      else
        bulk_load_plain(st + L.sfx_off, src.sfx + kb * 2048, nsub * 512, bar);
    } else {
      issue_x(st, bar, kb, src, hint, pol_x);
    }
  };
  // Dense path: the first ring of this CTA's (single) item is requested by thread 0
  // straight after the barriers exist, ahead of TMEM allocation and the CTA-wide
  // barrier; under a programmatic dependency only the weights (the token tiles may
  // come from the previous kernel).
  Item first_it;
  int n_pre = 0;
  if (!GROUPED) {
    get_item<false>(p, cta, NT * p.split, NT, KB, first_it);
    n_pre = min(STAGES, first_it.kb1 - first_it.kb0);
  }

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmW);  // first, so that the descriptors are fetched while the barriers are set up
    prefetch_tmap(&tmX);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);  // the weight warp and the token warp arrive
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // one elected lane per epilogue warp
    }
    mbar_init(drain, 1);
    mbar_init(red_bar, 1);
    *abort_flag = 0;
    *policies_ready = 0;
    fence_mbar_init();
    if (S > 1) {
      const int mine = min(m_own, p.M - static_cast<int>(cluster_rank()) * m_own);  // tokens this CTA owns
      if (mine > 0) mbar_arrive_expect_tx(red_bar, static_cast<uint32_t>(S * mine * 512));
    }
    const Src src = item_src(first_it);
    // Weights kept in L2: the first ring carries the evict_last hint as well (its policy
    // costs this thread ~0.6 us), so that none of the matrix is left at normal priority.
    const uint64_t keep = p.w_keep ? policy_evict_last() : 0;
    // The CTA's weight slice is prefetched into L2 first: under a programmatic dependency
    // those reads overlap the tail of the previous kernel, and the ring's loads then find
    // the bytes in L2 (the first ring itself when the weights are requested directly).
    {
      const int npf = GROUPED ? 0 : min(p.l2_prefetch, first_it.kb1 - first_it.kb0);
      for (int j = p.pdl == 1 ? n_pre : 0; j < npf; ++j) {
        const int kb = first_it.kb0 + j;
        tma_prefetch_2d(&tmW, kb * 128, src.wrow0);
        bulk_prefetch_l2(src.sfw + kb * 2048, min(4, (K - kb * KSTAGE) / KMMA) * 512);
        if (SPARSE) bulk_prefetch_l2(src.meta + kb * 4096, 4096);
      }
    }
    if (p.pdl == 2) griddep_wait();  // set-up-only overlap: no load before the previous kernel completes
    for (int j = 0; j < n_pre; ++j)
      if (!(cta == 0 && j + 1 == p.drop_stage))  // test hook: stage withheld
        issue_stage(j, first_it.kb0 + j, src, p.w_keep != 0, keep);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every CTA's reduction barrier is initialised (published by thread 0's
  // fence.mbarrier_init.release.cluster) before any CTA of the cluster sends partials;
  // only the sending warp waits, at the very end. The arrive itself is relaxed: a
  // release at cluster scope would hold the producer's first loads for ~1 us.
  if (S > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // With a programmatic dependency the prologue above overlapped the previous kernel.
  // The grouped path reads the tile list the preparation kernel just wrote, so every
  // warp waits here; the dense path's producer first requests its first weight tiles.
  if (GROUPED && p.pdl) griddep_wait();
  int n_items, first, stride;
  if (GROUPED) {
    n_items = __ldg(p.n_tiles) * NT;
    first = cta;
    stride = gridDim.x;
  } else {
    n_items = NT * p.split;
    first = cta;
    stride = n_items;  // one item per CTA
  }
  const uint32_t sf_base = tmem + p.acc_bufs * p.acc_cols;

  float dense_alpha = 0.0f;  // epilogue warps: g_a * g_b of the dense path
  if (warp == 0) {
    // The first ring goes out without L2 hints; createpolicy costs ~0.6 us, so an idle
    // epilogue warp builds the policies and the producer picks them up once published.
    uint64_t pol_w = 0;
    bool have_pol = false;
    int issued = 0;
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[16];
    for (int i = 0; i < 16; ++i) issued_phase[i] = -1;
    // Under a programmatic dependency in the set-up-only form no weight is requested before
    // the previous kernel completes; with NVFP4_TUNE_PDL = 1 the weights go out at once.
    if (p.pdl == 2) griddep_wait();
    Item it;
    int4 desc = first_desc<GROUPED>(p, first, n_items, NT);
    for (int i = first; next_item<GROUPED>(p, i, stride, n_items, NT, KB, desc, it) && !*abort_flag; i += stride) {
      const Src src = item_src(it);
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        if (!mbar_wait_warp(&empty[s], ph ^ 1, abort_flag, wd)) break;
        if (!have_pol && issued >= STAGES && *policies_ready) {
          __threadfence_block();
          pol_w = policies[0];
          have_pol = true;
        }
        const bool pre = issued < n_pre;  // requested in the prologue
        ++issued;
        const bool withheld = cta == 0 && issued == p.drop_stage;  // test hook
        if (!pre && !withheld && elect_one()) issue_stage(s, kb, src, have_pol, pol_w);
        __syncwarp();
        issued_phase[s] = ph;
        if (++s == STAGES) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    if (p.pdl) griddep_launch_dependents();
    for (int i = 0; i < STAGES; ++i)
      if (issued_phase[i] >= 0) {
        volatile int32_t dummy = 0;
        mbar_wait_warp(&full[i], issued_phase[i], &dummy, wd);
      }
  } else if (warp == kStreamTokenWarp) {
    // Requests every stage's token rows and their scales, in the weight warp's item and
    // stage order (two warps issue a stage's copies in about half the time one does; with
    // one, the issuing thread limited each CTA's weight stream, and on the decode path the
    // first ring left ~1 us after the CTA started). The token rows and scales may come
    // from the previous kernel in the stream: under a programmatic dependency this warp
    // waits for it first.
    if (p.pdl) griddep_wait();
    {
      uint64_t pol_x = 0;
      bool have_pol = false;
      int issued = 0;
      int s = 0;
      uint32_t ph = 0;
      int issued_phase[16];
      for (int j = 0; j < 16; ++j) issued_phase[j] = -1;
      Item it;
      auto load_tokens = [&](const Item& x) {
        return make_int4(__ldg(p.row_token + x.row0 + min(lane, x.rows - 1)),
                         __ldg(p.row_token + x.row0 + min(lane + 32, x.rows - 1)),
                         __ldg(p.row_token + x.row0 + min(lane + 64, x.rows - 1)),
                         __ldg(p.row_token + x.row0 + min(lane + 96, x.rows - 1)));
      };
      int4 tok_regs = make_int4(0, 0, 0, 0);
      bool tok_ready = false;
      int4 desc = first_desc<GROUPED>(p, first, n_items, NT);
      for (int i = first; next_item<GROUPED>(p, i, stride, n_items, NT, KB, desc, it) && !*abort_flag;
           i += stride) {
        const Src src = item_src(it);
        if (VARIANT & 2) {
          // this item's token rows (loaded during the previous item, four per lane); rows past
          // the tile's count repeat its last row (their accumulator columns are never stored),
          // indices clamped into x (prep reports bad ones)
          if (!tok_ready) tok_regs = load_tokens(it);
          tok_idx[lane] = min(max(tok_regs.x, 0), p.T - 1);
          tok_idx[lane + 32] = min(max(tok_regs.y, 0), p.T - 1);
          tok_idx[lane + 64] = min(max(tok_regs.z, 0), p.T - 1);
          tok_idx[lane + 96] = min(max(tok_regs.w, 0), p.T - 1);
          __syncwarp();
          Item nx;  // start the next item's index loads now; they land while this item streams
          tok_ready = get_item<GROUPED>(p, i + stride, n_items, NT, KB, nx);
          if (tok_ready) tok_regs = load_tokens(nx);
        }
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (!mbar_wait_warp(&empty[s], ph ^ 1, abort_flag, wd)) break;
          if (!have_pol && issued >= STAGES && *policies_ready) {
            __threadfence_block();
            pol_x = policies[1];
            have_pol = true;
          }
          ++issued;
          if (elect_one()) issue_tokens(s, kb, src, have_pol, pol_x);
          __syncwarp();
          issued_phase[s] = ph;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // Its copies in flight land before the CTA leaves (after an abort the stage's barrier
      // may never complete: the wait is bounded).
      for (int j = 0; j < STAGES; ++j)
        if (issued_phase[j] >= 0) {
          volatile int32_t dummy = 0;
          mbar_wait_warp(&full[j], issued_phase[j], &dummy, wd);
        }
    }
  } else if (warp == kStreamWaiterWarp) {
    // Owns every wait in front of the MMA warp (the item's accumulator buffer being
    // free, then each stage's bytes) and hands the verdict over through bar.red, so
    // the MMA warp touches neither an mbarrier nor shared memory between issues.
    // Same item and stage sequence as the MMA warp, also after an abort, so that
    // the named barrier (no time-out) always pairs.
    int s = 0, buf = 0;
    uint32_t ph = 0;
    uint32_t acc_ph[2] = {0, 0};
    Item it;
    int4 desc = first_desc<GROUPED>(p, first, n_items, NT);
    for (int i = first; next_item<GROUPED>(p, i, stride, n_items, NT, KB, desc, it); i += stride) {
      const bool item_ok =
          __all_sync(0xffffffffu, *abort_flag == 0) && mbar_wait_warp(&tempty[buf], acc_ph[buf] ^ 1, abort_flag, wd);
      acc_ph[buf] ^= 1;
      buf = (buf + 1 == p.acc_bufs) ? 0 : buf + 1;
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        const bool ok =
            item_ok && __all_sync(0xffffffffu, *abort_flag == 0) && mbar_wait_warp(&full[s], ph, abort_flag, wd);
        named_sync_and(kStreamHandoffBarrier, 64, ok);
        if (++s == STAGES) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    int s = 0, buf = 0;
    Item it;
    int4 desc = first_desc<GROUPED>(p, first, n_items, NT);
    for (int i = first; next_item<GROUPED>(p, i, stride, n_items, NT, KB, desc, it); i += stride) {
      const int n_mma = ((it.rows + 15) >> 4) * 16;
      const uint32_t idesc = SPARSE ? idesc_nvf4_sp(128, n_mma) : idesc_nvf4(128, n_mma);
      const uint32_t acc = tmem + buf * p.acc_cols;
      bool item_ok = true;
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        const bool ok = named_sync_and(kStreamHandoffBarrier, 64, true);
        item_ok = item_ok && ok;
        tc_fence_after();
        if (ok) {
          if (elect_one()) {
            // Fully unrolled: a data-dependent trip count here makes the elected lane
            // issue each tcgen05 instruction on its own, far more slowly.
            const int nsub = min(4, (K - kb * KSTAGE) / KMMA);
            const uint32_t w_addr = smem_u32(smem + s * L.stage_bytes);
            const uint32_t x_addr = w_addr + L.x_off;
            const uint32_t sf_col = sf_base + s * SF_COLS;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (kk < nsub) {
                tc_cp_32x128b_x4(sf_col + kk * 4, desc_sf(w_addr + L.sfw_off + kk * 512));
                tc_cp_32x128b_x4(sf_col + 16 + kk * 4, desc_sf(w_addr + L.sfx_off + kk * 512));
              }
            if (SPARSE) tc_cp_128x256b(sf_col + 32, w_addr + L.meta_off);  // 8 columns: 2 per MMA
            const uint64_t wdesc = desc_sw128(w_addr), xdesc = desc_sw128(x_addr);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (kk < nsub) {
                if (SPARSE) {
                  // 32 stored bytes of each weight row per MMA; the token rows' 64 bytes (128 K
                  // elements) at offset 0 or 64 of box kk / 2
                  const uint64_t xd = desc_sw128(x_addr + (kk >> 1) * L.xbox) + (kk & 1) * 4;
                  tc_mma_nvf4_sp(acc, wdesc + 2 * kk, xd, idesc, sf_col + 32 + 2 * kk, sf_col + kk * 4,
                                 sf_col + 16 + kk * 4, (kb != it.kb0) || (kk != 0));
                } else {
                  tc_mma_nvf4(acc, wdesc + 2 * kk, xdesc + 2 * kk, idesc, sf_col + kk * 4, sf_col + 16 + kk * 4,
                              (kb != it.kb0) || (kk != 0));
                }
              }
            tc_commit(&empty[s]);
          }
          __syncwarp();
        }
        if (++s == STAGES) s = 0;
      }
      if (item_ok) {
        if (elect_one()) tc_commit(&tfull[buf]);
        __syncwarp();
      }
      buf = (buf + 1 == p.acc_bufs) ? 0 : buf + 1;
    }
    if (p.pdl) griddep_launch_dependents();
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    volatile int32_t dummy = 0;
    mbar_wait_warp(drain, 0, &dummy, wd);
  } else {
    if (warp == 2) {
      // Weights are read once per call: evict_first keeps them from displacing the token
      // tiles (evict_last) and other data, unless the caller asks to keep them in L2.
      const uint64_t pw = p.w_keep ? policy_evict_last() : policy_evict_first(), px = policy_evict_last();
      if (lane == 0) {
        policies[0] = pw;
        policies[1] = px;
        __threadfence_block();
        *policies_ready = 1;
      }
      __syncwarp();
    }
    if (!GROUPED && p.pdl) griddep_wait();  // the global scales may come from the previous kernel
    const int q = warp & 3;
    const float ga = __ldg(p.ga);
    const float gq = (VARIANT & 8) ? __ldg(p.g_out) : 1.0f;  // NVFP4 output: the caller's global scale
    const float gq_inv = __frcp_rn(gq);
    const float gb0 = GROUPED ? 0.0f : __ldg(p.gb);  // dense: read while the mainloop runs
    dense_alpha = ga * gb0;
    int buf = 0;
    uint32_t acc_ph[2] = {0, 0};
    Item it;
    int4 desc = first_desc<GROUPED>(p, first, n_items, NT);
    for (int i = first; next_item<GROUPED>(p, i, stride, n_items, NT, KB, desc, it); i += stride) {
      if (!mbar_wait_warp(&tfull[buf], acc_ph[buf], abort_flag, wd)) break;
      tc_fence_after();
      const float alpha = ga * (GROUPED ? __ldg(p.gb + it.e) : gb0);
      const int wrow = it.wt * 128 + q * 32 + lane;  // output column
      const int n_mma = ((it.rows + 15) >> 4) * 16;
      const bool has_k = it.kb1 > it.kb0;
      const uint32_t tbase = tmem + buf * p.acc_cols + (static_cast<uint32_t>(q * 32) << 16);
      if (GROUPED) {
        // 32 columns (token rows) at a time: drained, scaled and stored; the accumulator
        // is released after the last chunk while the other buffer keeps the MMAs busy
        for (int c = 0; c < n_mma; c += 32) {
          uint32_t r[32];
          tmem_ld32(tbase + c, r);
          tmem_ld_wait();
          if (VARIANT & 8) {
            // SwiGLU emitting NVFP4. The even lanes' bf16 silu(gate) * up of this chunk's tokens
            // go to the warp's transpose tile ([token][16 output columns]: this warp's 32 weight
            // rows are 16 gate/up pairs, one whole 16-element block of every token row); then
            // lane l quantises token c + l's block with the stand-alone quantiser's device code
            // and the caller's global scale, so the codes equal nvfp4_quantize of the bf16
            // output of the plain SwiGLU epilogue.
            uint16_t* tt = xpose + q * 512;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c + j < it.rows) {
                const float v = __uint_as_float(r[j]) * alpha;
                const float up = __shfl_xor_sync(0xffffffffu, v, 1);
                if ((lane & 1) == 0) {
                  const float act = v / (1.0f + __expf(-v));
                  tt[j * 16 + (lane >> 1)] = __bfloat16_as_ushort(__float2bfloat16_rn(act * up));
                }
              }
            __syncwarp();
            if (c + lane < it.rows) {
              const uint4 h0 = *reinterpret_cast<const uint4*>(tt + lane * 16);
              const uint4 h1 = *reinterpret_cast<const uint4*>(tt + lane * 16 + 8);
              const uint32_t w[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
              uint32_t sc;
              uint2 pk;
              quantize_block(w, gq, gq_inv, sc, pk);
              const int64_t row = it.row0 + c + lane;
              const int cb = it.wt * 4 + q;        // 16-column block of the N / 2 outputs
              const int64_t kc4o = N >> 7;         // 512-byte scale tiles per 128 rows
              *reinterpret_cast<uint2*>(p.q_out + row * (N >> 2) + cb * 8) = pk;
              p.sf_out[((row >> 7) * kc4o + (cb >> 2)) * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4 + (cb & 3)] =
                  static_cast<uint8_t>(sc);
            }
            __syncwarp();
          } else if (VARIANT & 1) {
            // Weight rows 2c and 2c + 1 (gate and up of output column c) sit in adjacent
            // lanes: the even lane takes its partner's value and writes silu(gate) * up.
            const int n_out = N >> 1;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c + j < it.rows) {
                const float v = __uint_as_float(r[j]) * alpha;
                const float up = __shfl_xor_sync(0xffffffffu, v, 1);
                if ((lane & 1) == 0 && wrow < N) {
                  const float act = v / (1.0f + __expf(-v));
                  p.y[static_cast<int64_t>(it.row0 + c + j) * n_out + (wrow >> 1)] =
                      __bfloat16_as_ushort(__float2bfloat16_rn(act * up));
                }
              }
          } else if (wrow < N) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c + j < it.rows)
                p.y[static_cast<int64_t>(it.row0 + c + j) * N + wrow] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[j]) * alpha));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (elect_one()) mbar_arrive(&tempty[buf]);
        __syncwarp();
      } else {
        // one item per CTA: drain 32 columns at a time (fewer live registers)
        for (int c = 0; c < n_mma; c += 32) {
          uint32_t r[32];
          tmem_ld32(tbase + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tok = c + j;
            if (tok < it.rows) {
              if (S > 1)
                part[tok * 128 + q * 32 + lane] = has_k ? __uint_as_float(r[j]) : 0.0f;
              else if (wrow < N)
                p.y[static_cast<int64_t>(it.row0 + tok) * N + wrow] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[j]) * alpha));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (elect_one()) mbar_arrive(&tempty[buf]);
        __syncwarp();
      }
      acc_ph[buf] ^= 1;
      buf = (buf + 1 == p.acc_bufs) ? 0 : buf + 1;
    }
    if (p.pdl) griddep_launch_dependents();
  }

  if (!GROUPED && S > 1 && warp >= 2 && warp < kStreamWaiterWarp) {
    // One-way split-K reduction: each CTA sends owner o the block of o's tokens
    // (one bulk copy into o's recv slot for this rank, completing bytes on o's
    // red_bar), then the owners sum their S slots locally. No cluster-wide barrier
    // sits between the last MMA and the stores.
    fence_proxy_async_shared();  // this thread's part[] writes, before the bulk copies read them
    named_sync(kStreamEpilogueBarrier, 128);
    const uint32_t rank = cluster_rank();
    if (warp == 2) {
      asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
      if (lane == 0) {
        for (int o = 0; o < S; ++o) {
          const int n_o = min(m_own, p.M - o * m_own);
          if (n_o <= 0) continue;
          const uint32_t dst = mapa_shared(smem_u32(recv + static_cast<int>(rank) * m_own * 128), o);
          bulk_copy_to_cluster(dst, part + o * m_own * 128, static_cast<uint32_t>(n_o * 512),
                               mapa_shared(smem_u32(red_bar), o));
        }
        bulk_commit_group();
        bulk_wait_group_read0();  // part[] may be released once the copies have read it
      }
      __syncwarp();
    }
    const int mine = min(m_own, p.M - static_cast<int>(rank) * m_own);
    // Every CTA sends its partials, also after an abort (then garbage), and each owner waits
    // for all of them whatever its own state: no CTA may leave while a peer's copy into its
    // shared memory is in flight. A sender that aborted sends once its own waits gave up (one
    // limit after they began), so the owner's wait allows four limits before it gives up.
    volatile int32_t no_abort = 0;
    const bool received = mine > 0 && mbar_wait_warp(red_bar, 0, &no_abort, 4 * wd);
    if (mine > 0 && !received) *abort_flag = 1;
    if (received && !*abort_flag) {
      const int q = warp & 3;
      const int wrow = (cta / S) * 128 + q * 32 + lane;
      const float alpha = dense_alpha;
      for (int idx = 0; idx < mine; ++idx) {
        float v = 0.0f;
        for (int c = 0; c < S; ++c) v += recv[(c * m_own + idx) * 128 + q * 32 + lane];  // fixed rank order
        const int tok = static_cast<int>(rank) * m_own + idx;
        if (wrow < N) p.y[static_cast<int64_t>(tok) * N + wrow] = __bfloat16_as_ushort(__float2bfloat16_rn(v * alpha));
      }
    }
  }

  // Every thread that arrived on the cluster barrier also waits on it before the
  // CTA-wide barrier below (the sending warp already did). Leaving arrivals without a
  // wait let the __syncthreads that follows complete before all warps reached it.
  if (S > 1 && !(warp == 2)) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
  if (threadIdx.x == 0 && *abort_flag) report_status(p.status, kStatusTimeout);
}

template <bool GROUPED, int VARIANT = 0>
__global__ void __launch_bounds__(kStreamThreads, 2)
    k_gemm_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                  const StreamArgs p) {
  stream_body<GROUPED, VARIANT>(tmW, tmX, p, static_cast<int>(blockIdx.x));
}

// Several independent decode-M GEMMs in one launch (same M, their own weights, inputs,
// outputs, N and K): CTAs [cta_base[g], cta_base[g + 1]) run GEMM g exactly as a single
// call's grid would, with the launch's split-K cluster size (every GEMM's CTA count is a
// multiple of it, so no cluster spans two GEMMs).
__global__ void __launch_bounds__(kStreamThreads, 2)
    k_gemm_batched(const __grid_constant__ BatchParams bp, const __grid_constant__ StreamArgs p) {
  const int b = static_cast<int>(blockIdx.x);
  int g = 0;
  while (g + 1 < bp.count && b >= bp.cta_base[g + 1]) ++g;
  StreamArgs q = p;
  q.sfw = bp.sfw[g];
  q.sfx = bp.sfx[g];
  q.ga = bp.ga[g];
  q.gb = bp.gb[g];
  q.y = bp.y[g];
  q.N = bp.N[g];
  q.K = bp.K[g];
  stream_body<false, 0>(bp.w[g], bp.x[g], q, b - bp.cta_base[g]);
}

// ---- grouped preparation ------------------------------------------------------------

// Validates expert_offsets, lists the token tiles (<= tile_rows rows of one
// expert each; experts without rows get none) and gathers each tile's token
// scales into its own slab in the 128-row tiled layout, rows starting at 0.
// With xg: also copies packed token row row_token[r] of x_tok to row r of xg
// (the routed rows in expert order), so the GEMM reads them as plain tiles.
// Workspace: [0] n_tiles, [16..) int4 tiles[max_tiles], then the slabs (then xg).
__global__ void __launch_bounds__(256) k_grouped_prep(const int32_t* __restrict__ offsets,
                                                      const int32_t* __restrict__ row_token, int T, int E, int M_total,
                                                      int K, int kc4, int tile_rows,
                                                      const uint8_t* __restrict__ sfx, int32_t* n_tiles_out,
                                                      int4* __restrict__ tiles, uint8_t* __restrict__ slabs,
                                                      int32_t* status, const uint8_t* __restrict__ x_tok,
                                                      uint8_t* __restrict__ xg) {
  extern __shared__ int32_t sh[];  // offsets[E+1], tile_base[E+1]
  int32_t* off = sh;
  int32_t* tbase = sh + (E + 1);
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    off[e] = offsets[e];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (off[e + 1] < off[e]) bad = 1;
  if (threadIdx.x == 0 && (off[0] != 0 || off[E] != M_total)) bad = 1;
  __syncthreads();
  if (bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      *n_tiles_out = 0;
      report_status(status, kStatusBadOffsets);
    }
    return;
  }
  {
    // tile bases: an exclusive scan of the experts' tile counts, each thread summing a
    // contiguous run of experts, the runs combined across the block
    __shared__ int warp_sum[8];
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, static_cast<int>(threadIdx.x) * per), e1 = min(E, e0 + per);
    int mine = 0;
    for (int e = e0; e < e1; ++e) mine += (off[e + 1] - off[e] + tile_rows - 1) / tile_rows;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = mine;  // inclusive scan within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < wid; ++w) before += warp_sum[w];
    int acc = before + incl - mine;
    for (int e = e0; e < e1; ++e) {
      tbase[e] = acc;
      acc += (off[e + 1] - off[e] + tile_rows - 1) / tile_rows;
    }
    if (threadIdx.x == blockDim.x - 1) tbase[E] = before + incl;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const int cnt = off[e + 1] - off[e];
      for (int t = 0; t * tile_rows < cnt; ++t)
        tiles[tbase[e] + t] = make_int4(e, off[e] + t * tile_rows, min(tile_rows, cnt - t * tile_rows), tbase[e] + t);
    }
    if (threadIdx.x == 0) *n_tiles_out = tbase[E];
  }
  // One warp per routed row m at a time: its expert (binary search over the offsets), its
  // tile and row within the tile, and its source row; then the lanes gather the row's
  // scale words (one 4-byte word = four consecutive 16-element blocks) into the tile's
  // slab and, with xg, copy its packed row 16 bytes per lane and step.
  const int64_t KC4 = kc4;    // 512-byte scale tiles per 128 rows (K / 64; K / 128 for 32-element blocks)
  const int64_t C = K / 32;  // 16-byte chunks per packed row of K / 2 bytes
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); m < M_total; m += warps) {
    int lo = 0, hi = E;  // expert e with off[e] <= m < off[e+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (off[mid] <= m) lo = mid; else hi = mid;
    }
    while (off[lo + 1] <= m) ++lo;  // skip empty experts sharing the same offset
    const int j = m - off[lo];
    const int64_t tile = tbase[lo] + j / tile_rows;
    const int r = j % tile_rows;
    int src = m;  // the row of x (and of its scales) this routed row reads
    if (row_token) {
      src = __ldg(row_token + m);
      if (src < 0 || src >= T) {  // reported, and clamped so that nothing is read out of bounds
        if (lane == 0) report_status(status, kStatusBadOffsets);
        src = src < 0 ? 0 : T - 1;
      }
    }
    const uint8_t* sfx_row = sfx + (static_cast<int64_t>(src / 128) * KC4) * 512 + (src % 32) * 16 + ((src % 128) / 32) * 4;
    uint8_t* slab_row = slabs + tile * KC4 * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4;
    for (int64_t c4 = lane; c4 < KC4; c4 += 32)
      *reinterpret_cast<uint32_t*>(slab_row + c4 * 512) = *reinterpret_cast<const uint32_t*>(sfx_row + c4 * 512);
    if (xg) {
      const uint4* from = reinterpret_cast<const uint4*>(x_tok) + static_cast<int64_t>(src) * C;
      uint4* to = reinterpret_cast<uint4*>(xg) + static_cast<int64_t>(m) * C;
      for (int64_t ch = lane; ch < C; ch += 32) to[ch] = __ldg(from + ch);
    }
  }
}

// ---- host launchers -------------------------------------------------------------------

template <bool GROUPED, int VARIANT>
static cudaError_t launch_stream_t(const CUtensorMap& tmW, const CUtensorMap& tmX, const StreamArgs& a, int grid,
                                   cudaStream_t st) {
  // grouped: the token indices of a tile (the token gather); dense: the reduction's receive area
  const int smem = stream_smem_bytes(a.stages, a.x_rows,
                                     GROUPED ? grouped_extra_bytes(a.x_rows, (VARIANT & 8) != 0)
                                             : stream_recv_bytes(a.M, a.split),
                                     (VARIANT & 4) != 0);
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(k_gemm_stream<GROUPED, VARIANT>));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  if (!GROUPED && a.split > 1) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = a.split;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  if (a.pdl) {
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  e = cudaLaunchKernelEx(&cfg, k_gemm_stream<GROUPED, VARIANT>, tmW, tmX, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Receive area of the one-way split-K reduction: S slots of ceil(M / S) tokens x 128 fp32.
int stream_recv_bytes(int M, int split) { return split > 1 ? split * ((M + split - 1) / split) * 512 : 0; }

int stream_smem_bytes(int stages, int x_rows, int recv_bytes, bool sparse) {
  return stages * StreamLayout(x_rows, sparse).stage_bytes + recv_bytes + 1024 + 512;
}

cudaError_t launch_batched(const BatchParams& bp, const StreamArgs& a, int grid, cudaStream_t st) {
  const int smem = stream_smem_bytes(a.stages, a.x_rows, stream_recv_bytes(a.M, a.split));
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(k_gemm_batched));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  if (a.split > 1) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = a.split;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  if (a.pdl) {
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  return cudaLaunchKernelEx(&cfg, k_gemm_batched, bp, a);
}

cudaError_t launch_stream(const CUtensorMap& tmW, const CUtensorMap& tmX, const StreamArgs& a, bool grouped, int grid,
                          cudaStream_t st) {
  if (!grouped) return a.meta ? launch_stream_t<false, 4>(tmW, tmX, a, grid, st) : launch_stream_t<false, 0>(tmW, tmX, a, grid, st);
  if ((a.row_token || a.swiglu) && a.meta) return cudaErrorInvalidValue;  // no entry point combines them
  if (a.row_token && a.swiglu) return cudaErrorInvalidValue;
  if (a.meta) return launch_stream_t<true, 4>(tmW, tmX, a, grid, st);
  if (a.row_token) return launch_stream_t<true, 2>(tmW, tmX, a, grid, st);
  if (a.swiglu && a.q_out) return launch_stream_t<true, 9>(tmW, tmX, a, grid, st);
  if (a.swiglu) return launch_stream_t<true, 1>(tmW, tmX, a, grid, st);
  return launch_stream_t<true, 0>(tmW, tmX, a, grid, st);
}

cudaError_t launch_grouped_prep(const int32_t* offsets, const int32_t* row_token, int T, int E, int M_total, int K,
                                int kc4, int tile_rows, const uint8_t* sfx,
                                int32_t* n_tiles, int4* tiles, uint8_t* slabs, int32_t* status, int grid,
                                cudaStream_t st, const uint8_t* x_tok, uint8_t* xg) {
  const int smem = 2 * (E + 1) * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(k_grouped_prep));
    if (e != cudaSuccess) return e;
  }
  k_grouped_prep<<<grid, 256, smem, st>>>(offsets, row_token, T, E, M_total, K, kc4, tile_rows, sfx, n_tiles,
                                          tiles, slabs, status, x_tok, xg);
  return cudaGetLastError();
}

}  // namespace nvfp4
