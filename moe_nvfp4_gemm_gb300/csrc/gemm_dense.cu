// Dense NVFP4 GEMM for large M: y[M,N] = bf16((x^ . W^T^) * g_a * g_b).
//
// Operation: "NVFP4 linear layer" (kernelindex, operation header): y = x @ W^T,
// both operands FP4 with FP8 E4M3FN scales per 16 elements.
//
// Two persistent, warp-specialised tcgen05 kernels share one structure:
//   warp 0      TMA producer: K-major 128-byte-swizzled data tiles (256 K per
//               stage) and the matching 512-byte scale tiles into a STAGES-deep
//               shared-memory ring;
//   warp 1      allocates TMEM; copies each stage's scales into TMEM (tcgen05.cp)
//               and issues 4 block-scaled MMAs (K = 64 each) into the accumulator;
//   warps 2-9   epilogue: each warp drains one TMEM lane quarter and half of the
//               tile's columns into registers, releases the accumulator, then
//               scales by g_a * g_b, converts to bf16 and stores.
// Warps issue TMA and tcgen05 operations converged, through one elected lane.
// Every wait is bounded (globaltimer watchdog) and reports a timeout status.
//
//   k_gemm_dense       one CTA per SM, 128 x BN tiles (tcgen05 cta_group::1)
//   k_gemm_dense_pair  CTA pairs, 256 x 256 tiles (cta_group::2): each CTA loads
//                      its 128 rows of A and of B, the even CTA issues the MMAs
//                      for both SMs (which read B from both CTAs' shared memory);
//                      per SM this halves the operand traffic per FLOP and makes
//                      the scale copies free. The default large-M kernel.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "nvfp4_quant.cuh"
#include "ptx.cuh"

namespace nvfp4 {

constexpr int kDenseThreads = 320;  // producer, MMA, 8 epilogue warps
// CTA-pair kernel: + one warp that waits for each stage's TMA bytes and hands the
// stage to the MMA warp through a named barrier. An mbarrier wait in the MMA-issuing
// warp stalls the tensor pipe (hundreds of cycles per wait, measured on GB300); the
// named-barrier handoff does not.
constexpr int kPairThreads = 352;
constexpr int kWaiterWarp = 10;
constexpr uint32_t kStageHandoffBarrier = 1;

template <int BN, int STAGES>
struct DenseCfg {
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int GROUPS = BN / 128;  // 128-row scale tiles of B per stage
  static constexpr int SFA_BYTES = 4 * 512;
  static constexpr int SFB_BYTES = GROUPS * 4 * 512;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SF_COLS = 16 + 16 * GROUPS;  // TMEM scale columns per stage
  static constexpr int TMEM_COLS = 512;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static_assert(BN + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kDenseThreads, 1)
    k_gemm_dense(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const DenseArgs p) {
  using C = DenseCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t wd = p.watchdog_ns;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 8);  // one elected lane per epilogue warp
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int M = p.M, N = p.N, K = p.K;
  const int mt = (M + 127) / 128, nt = (N + BN - 1) / BN, tiles = mt * nt;
  const int KB = (K + 255) / 256;
  const int64_t KC4 = K / 64;  // 512-byte scale tiles per 128 rows
  const int n_rowblk = (N + 127) / 128;

  if (warp == 0) {
    const uint64_t pol = policy_evict_last();
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[STAGES];
    for (int i = 0; i < STAGES; ++i) issued_phase[i] = -1;
    int issued = 0;
    for (int t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
      int m_blk, n_blk;
      tile_coords(t, mt, nt, p.raster, m_blk, n_blk);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_warp(&empty[s], ph ^ 1, abort_flag, wd)) break;
        const bool withheld = blockIdx.x == 0 && ++issued == p.drop_stage;  // test hook
        if (!withheld && elect_one()) {
          const int nsub = min(4, (K - kb * 256) / 64);
          uint8_t* st = smem + s * C::STAGE_BYTES;
          int ngroups = 0;
#pragma unroll
          for (int g = 0; g < C::GROUPS; ++g) ngroups += (n_blk * C::GROUPS + g < n_rowblk) ? 1 : 0;
          mbar_arrive_expect_tx(&full[s], C::A_BYTES + C::B_BYTES + nsub * 512 * (1 + ngroups));
          tma_load_2d(st, &tmA, &full[s], kb * 128, m_blk * 128, pol);
          tma_load_2d(st + C::A_BYTES, &tmB, &full[s], kb * 128, n_blk * BN, pol);
          bulk_load(st + C::A_BYTES + C::B_BYTES, p.sfa + (m_blk * KC4 + kb * 4) * 512, nsub * 512, &full[s], pol);
#pragma unroll
          for (int g = 0; g < C::GROUPS; ++g) {
            const int rb = n_blk * C::GROUPS + g;
            if (rb < n_rowblk)
              bulk_load(st + C::A_BYTES + C::B_BYTES + C::SFA_BYTES + g * 2048, p.sfb + (rb * KC4 + kb * 4) * 512,
                        nsub * 512, &full[s], pol);
          }
        }
        __syncwarp();
        issued_phase[s] = ph;
        if (++s == STAGES) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    // Let every copy this CTA started land before shared memory is released.
    for (int i = 0; i < STAGES; ++i)
      if (issued_phase[i] >= 0) {
        volatile int32_t dummy = 0;
        mbar_wait_warp(&full[i], issued_phase[i], &dummy, wd);
      }
  } else if (warp == 1) {
    const uint32_t idesc = idesc_nvf4(128, BN);
    int s = 0;
    uint32_t ph = 0, acc_ph = 0;
    for (int t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
      if (!mbar_wait_warp(tempty, acc_ph ^ 1, abort_flag, wd)) break;
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_warp(&full[s], ph, abort_flag, wd)) break;
        tc_fence_after();
        if (elect_one()) {
          const int nsub = min(4, (K - kb * 256) / 64);
          const uint32_t a_addr = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + C::A_BYTES;
          const uint32_t sfa_addr = b_addr + C::B_BYTES;
          const uint32_t sfb_addr = sfa_addr + C::SFA_BYTES;
          const uint32_t sf_col = tmem + BN + s * C::SF_COLS;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            if (kk < nsub) {
              tc_cp_32x128b_x4(sf_col + kk * 4, desc_sf(sfa_addr + kk * 512));
#pragma unroll
              for (int g = 0; g < C::GROUPS; ++g)
                tc_cp_32x128b_x4(sf_col + 16 + kk * 4 * C::GROUPS + g * 4, desc_sf(sfb_addr + g * 2048 + kk * 512));
            }
          const uint64_t adesc = desc_sw128(a_addr), bdesc = desc_sw128(b_addr);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            if (kk < nsub)
              tc_mma_nvf4(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, sf_col + kk * 4,
                          sf_col + 16 + kk * 4 * C::GROUPS, (kb | kk) != 0);
          tc_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == STAGES) {
          s = 0;
          ph ^= 1;
        }
      }
      if (elect_one()) tc_commit(tfull);
      __syncwarp();
      acc_ph ^= 1;
    }
    // All MMAs issued by this warp complete before TMEM is released.
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    volatile int32_t dummy = 0;
    mbar_wait_warp(drain, 0, &dummy, wd);
  } else {
    const int q = warp & 3;         // TMEM lane quarter this warp may read
    const int h = (warp - 2) >> 2;  // which half of the tile's columns
    const float alpha = __ldg(p.ga) * __ldg(p.gb);
    const bool wide = N % 16 == 0 && (reinterpret_cast<uintptr_t>(p.y) & 31) == 0;
    uint32_t acc_ph = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
      int m_blk, n_blk;
      tile_coords(t, mt, nt, p.raster, m_blk, n_blk);
      if (!mbar_wait_warp(tfull, acc_ph, abort_flag, wd)) break;
      tc_fence_after();
      const int row = m_blk * 128 + q * 32 + lane;
      drain_accumulator<BN / 2>(tmem + (static_cast<uint32_t>(q * 32) << 16) + h * (BN / 2), alpha,
                                p.y + static_cast<int64_t>(row) * N, row < M, n_blk * BN + h * (BN / 2), N, wide,
                                [&] {
                                  if (elect_one()) mbar_arrive(tempty);
                                  __syncwarp();
                                });
      acc_ph ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag) report_status(p.status, kStatusTimeout);
}

// ---- CTA-pair kernel: 256 x 256 tiles on two SMs -----------------------------------------

struct PairCfg {
  static constexpr int STAGES = 5;
  static constexpr int A_BYTES = 128 * 128;
  static constexpr int B_BYTES = 128 * 128;
  static constexpr int SFA_BYTES = 2048;
  static constexpr int SFB_BYTES = 4096;  // scales of all 256 B rows, in both CTAs
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SF_COLS = 16 + 32;
  static constexpr int TMEM_COLS = 512;
  static constexpr int OUT_BYTES = 8 * 4096;  // one 32 x 64 bf16 store box per epilogue warp
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + 256;
  static_assert(256 + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(STAGE_BYTES % 1024 == 0, "swizzled buffers stay 1024-byte aligned");
};

// QOUT: the epilogue quantises the bf16 results to NVFP4 (codes, tiled block scales)
// with the caller's global scale instead of writing bf16.
template <bool QOUT>
__global__ void __launch_bounds__(kPairThreads, 1)
    k_gemm_dense_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                      const __grid_constant__ CUtensorMap tmY, const DenseArgs p) {
  using C = PairCfg;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_buf = smem + STAGES * C::STAGE_BYTES;  // 1024-byte aligned: STAGE_BYTES is a multiple of 1024
  uint64_t* full = reinterpret_cast<uint64_t*>(out_buf + C::OUT_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t wd = p.watchdog_ns;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 16);  // one elected lane per epilogue warp, both CTAs
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSFA);
    prefetch_tmap(&tmSFB);
    prefetch_tmap(&tmY);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int M = p.M, N = p.N, K = p.K;
  const int mt = (M + 255) / 256, nt = (N + 255) / 256, tiles = mt * nt;
  const int KB = (K + 255) / 256;
  const int KC4 = K / 64;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    const uint64_t pol = policy_evict_last();
    griddep_wait();  // launched as a programmatic dependent: loads wait for the previous kernel
    int s = 0;
    uint32_t ph = 0;
    int issued_phase[STAGES];
    for (int i = 0; i < STAGES; ++i) issued_phase[i] = -1;
    int issued = 0;
    for (int t = pair; t < tiles && !*abort_flag; t += npairs) {
      int m_blk, n_blk;
      tile_coords(t, mt, nt, p.raster, m_blk, n_blk);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_warp(&empty[s], ph ^ 1, abort_flag, wd)) break;
        // test hook: the even CTA of the first pair withholds its expect-tx arrival and
        // loads, so that stage's barrier never completes
        const bool withheld = blockIdx.x == 0 && ++issued == p.drop_stage;
        if (!withheld && elect_one()) {
          uint8_t* st = smem + s * C::STAGE_BYTES;
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
          tma_load_2d_pair(st, &tmA, bar, kb * 128, m_blk * 256 + rank * 128, pol);
          tma_load_2d_pair(st + C::A_BYTES, &tmB, bar, kb * 128, n_blk * 256 + rank * 128, pol);
          tma_load_2d_pair(st + C::A_BYTES + C::B_BYTES, &tmSFA, bar, 0, (m_blk * 2 + rank) * KC4 + kb * 4, pol);
          tma_load_2d_pair(st + C::A_BYTES + C::B_BYTES + C::SFA_BYTES, &tmSFB, bar, 0, (n_blk * 2) * KC4 + kb * 4,
                           pol);
          tma_load_2d_pair(st + C::A_BYTES + C::B_BYTES + C::SFA_BYTES + 2048, &tmSFB, bar, 0,
                           (n_blk * 2 + 1) * KC4 + kb * 4, pol);
        }
        __syncwarp();
        issued_phase[s] = ph;
        if (++s == STAGES) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    griddep_launch_dependents();  // this CTA's loads are all issued: let the next kernel set up
    // The even CTA's full barriers count both CTAs' bytes: let them all land.
    if (leader)
      for (int i = 0; i < STAGES; ++i)
        if (issued_phase[i] >= 0) {
          volatile int32_t dummy = 0;
          mbar_wait_warp(&full[i], issued_phase[i], &dummy, wd);
        }
  } else if (warp == kWaiterWarp) {
    // Owns every wait in front of the MMA warp: the accumulator being free at the
    // start of each tile, then each stage's bytes landing. The verdict (false after
    // an abort or a time-out) reaches the MMA warp through bar.red, so the MMA
    // warp touches neither an mbarrier nor shared memory between its issues. Both
    // warps run exactly tiles x KB iterations (also after an abort) so that the
    // named barrier, which cannot time out, always pairs.
    if (leader) {
      int s = 0;
      uint32_t ph = 0, acc_ph = 0;
      for (int t = pair; t < tiles; t += npairs) {
        const bool tile_ok =
            __all_sync(0xffffffffu, *abort_flag == 0) && mbar_wait_warp(tempty, acc_ph ^ 1, abort_flag, wd);
        acc_ph ^= 1;
        for (int kb = 0; kb < KB; ++kb) {
          const bool ok =
              tile_ok && __all_sync(0xffffffffu, *abort_flag == 0) && mbar_wait_warp(&full[s], ph, abort_flag, wd);
          named_sync_and(kStageHandoffBarrier, 64, ok);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (leader) {
      const uint32_t idesc = idesc_nvf4(256, 256);
      int s = 0;
      for (int t = pair; t < tiles; t += npairs) {
        bool tile_ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          const bool ok = named_sync_and(kStageHandoffBarrier, 64, true);
          tile_ok = tile_ok && ok;
          tc_fence_after();
          if (ok) {
            if (elect_one()) {
              // Fully unrolled: a data-dependent trip count here makes the elected
              // lane issue each tcgen05 instruction on its own, far more slowly.
              const int nsub = min(4, (K - kb * 256) / 64);
              const uint32_t a_addr = smem_u32(smem + s * C::STAGE_BYTES);
              const uint32_t b_addr = a_addr + C::A_BYTES;
              const uint32_t sfa_addr = b_addr + C::B_BYTES;
              const uint32_t sfb_addr = sfa_addr + C::SFA_BYTES;
              const uint32_t sf_col = tmem + 256 + s * C::SF_COLS;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                if (kk < nsub) {
                  tc_cp_32x128b_x4_pair(sf_col + kk * 4, desc_sf(sfa_addr + kk * 512));
                  tc_cp_32x128b_x4_pair(sf_col + 16 + kk * 8, desc_sf(sfb_addr + kk * 512));
                  tc_cp_32x128b_x4_pair(sf_col + 16 + kk * 8 + 4, desc_sf(sfb_addr + 2048 + kk * 512));
                }
              const uint64_t adesc = desc_sw128(a_addr), bdesc = desc_sw128(b_addr);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                if (kk < nsub)
                  tc_mma_nvf4_pair(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, sf_col + kk * 4, sf_col + 16 + kk * 8,
                                   (kb | kk) != 0);
              tc_commit_pair(&empty[s], 3);
            }
            __syncwarp();
          }
          if (++s == STAGES) s = 0;
        }
        if (tile_ok) {
          if (elect_one()) tc_commit_pair(tfull, 3);
          __syncwarp();
        }
      }
      if (elect_one()) tc_commit_pair(drain, 1);
      __syncwarp();
      volatile int32_t dummy = 0;
      mbar_wait_warp(drain, 0, &dummy, wd);
    }
  } else {
    const int q = warp & 3, h = (warp - 2) >> 2;
    griddep_wait();  // reads the global scales, writes y
    const float alpha = __ldg(p.ga) * __ldg(p.gb);
    uint8_t* buf = out_buf + (warp - 2) * 4096;
    const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
    float g_q = 1.0f, g_q_inv = 1.0f;
    if (QOUT) {
      g_q = __ldg(p.g_out);
      g_q_inv = __frcp_rn(g_q);
    }
    uint32_t acc_ph = 0;
    for (int t = pair; t < tiles; t += npairs) {
      int m_blk, n_blk;
      tile_coords(t, mt, nt, p.raster, m_blk, n_blk);
      if (!mbar_wait_warp(tfull, acc_ph, abort_flag, wd)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128;
      const int row0 = m_blk * 256 + rank * 128 + q * 32;
      const int col0 = n_blk * 256 + h * 128;
      if (QOUT) {
        // Each thread owns one output row's 128 columns = 8 blocks of 16: block amax,
        // E4M3 scale and E2M1 codes are thread-local (the stand-alone quantiser's recipe
        // on the same bf16 values the plain epilogue would store).
        uint32_t r[128];
#pragma unroll
        for (int c = 0; c < 128; c += 32) tmem_ld32(taddr + c, r + c);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (elect_one()) mbar_arrive_cluster(tempty_leader);
        __syncwarp();
        uint32_t wb[64];  // the 128 results as bf16 pairs (the fp32 values are dead after this)
#pragma unroll
        for (int j = 0; j < 64; ++j)
          wb[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * alpha, __uint_as_float(r[2 * j + 1]) * alpha);
        const int row = row0 + lane;
        const int Nc4 = N / 64;  // 4-block scale groups per row (N % 64 == 0)
        const int pad_rows = (M + 127) / 128 * 128;
        if (row < pad_rows) {
          uint32_t sw[2] = {0u, 0u};
#pragma unroll
          for (int bp = 0; bp < 4; ++bp) {  // pairs of blocks: 32 columns, 16 bytes of codes
            uint2 packed[2];
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const int blk = bp * 2 + hb;
              uint32_t w[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = wb[blk * 8 + j];
              uint32_t sc = 0;
              packed[hb] = make_uint2(0u, 0u);
              if (row < M) quantize_block(w, g_q, g_q_inv, sc, packed[hb]);
              sw[blk >> 2] |= sc << ((blk & 3) * 8);
            }
            if (row < M && col0 + bp * 32 < N)
              st_global_v4(p.q_out + static_cast<int64_t>(row) * (N / 2) + (col0 + bp * 32) / 2, packed[0].x,
                           packed[0].y, packed[1].x, packed[1].y);
          }
          // scale bytes (row, c .. c + 3) of the 128 x 4 tile layout form one word
#pragma unroll
          for (int gi = 0; gi < 2; ++gi) {
            const int cg = col0 / 64 + gi;  // 4-block group index
            if (cg < Nc4) {
              const int64_t off = (static_cast<int64_t>(row / 128) * Nc4 + cg) * 512 + (row % 32) * 16 +
                                  ((row % 128) / 32) * 4;
              *reinterpret_cast<uint32_t*>(p.sf_out + off) = sw[gi];
            }
          }
        }
      } else {
        drain_accumulator_tma<128>(taddr, alpha, buf, &tmY, col0, row0, [&] {
          if (elect_one()) mbar_arrive_cluster(tempty_leader);
          __syncwarp();
        });
      }
      acc_ph ^= 1;
    }
    if (lane == 0) bulk_wait_group0();  // this warp's stores are complete before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still read its shared memory or signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag) report_status(p.status, kStatusTimeout);
}

// ---- host launchers ---------------------------------------------------------------------------

template <int BN, int STAGES>
static cudaError_t launch_dense_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const DenseArgs& a, int grid,
                                  cudaStream_t st) {
  using C = DenseCfg<BN, STAGES>;
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(k_gemm_dense<BN, STAGES>));
  if (e != cudaSuccess) return e;
  k_gemm_dense<BN, STAGES><<<grid, kDenseThreads, C::SMEM_BYTES, st>>>(tmA, tmB, a);
  return cudaGetLastError();
}

// bn selects the tile width (128 or 256); grid is the persistent CTA count.
cudaError_t launch_dense(const CUtensorMap& tmA, const CUtensorMap& tmB, const DenseArgs& a, int bn, int grid,
                         cudaStream_t st) {
  if (bn == 256) return launch_dense_t<256, 4>(tmA, tmB, a, grid, st);
  return launch_dense_t<128, 6>(tmA, tmB, a, grid, st);
}

// grid: an even number of CTAs (two per 256 x 256 tile in flight).
cudaError_t launch_dense_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                              const CUtensorMap& tmSFB, const CUtensorMap& tmY, const DenseArgs& a, int grid,
                              cudaStream_t st, bool quantized_out) {
  auto kernel = quantized_out ? k_gemm_dense_pair<true> : k_gemm_dense_pair<false>;
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(kernel));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = PairCfg::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch, set-up only: barrier and TMEM set-up and descriptor
  // prefetch overlap the previous kernel's tail; every memory access waits for it
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmSFA, tmSFB, tmY, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace nvfp4
