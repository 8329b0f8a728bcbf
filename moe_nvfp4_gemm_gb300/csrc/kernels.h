// Launch interfaces shared by the C ABI (capi.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

struct DenseArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* ga;
  const float* gb;
  uint16_t* y;
  int M, N, K;
  int32_t* status;
  // NVFP4 output (k_gemm_dense_pair<true>): codes [M, N/2], tiled scales of [M, N], with
  // the caller's global scale; y is not written
  uint8_t* q_out;
  uint8_t* sf_out;
  const float* g_out;
  uint64_t watchdog_ns;  // limit of every pipeline wait
  int drop_stage;        // test hook: k >= 1 withholds the k-th stage CTA 0 loads (0: none)
  // tile order: 0 m-blocks fastest; -1 n-blocks fastest; G > 0 bands of G m-blocks, m fastest
  // inside a band (the band's B tiles are read by G CTA pairs at about the same time)
  int raster;
};

// Tile t of an mt x nt grid of output tiles in the order `raster` selects.
__host__ __device__ inline void tile_coords(int t, int mt, int nt, int raster, int& m_blk, int& n_blk) {
  if (raster < 0) {
    m_blk = t / nt;
    n_blk = t % nt;
  } else if (raster == 0 || raster >= mt) {
    m_blk = t % mt;
    n_blk = t / mt;
  } else {
    const int band = t / (raster * nt);
    const int first = band * raster;
    const int rows = mt - first < raster ? mt - first : raster;
    const int local = t - band * raster * nt;
    m_blk = first + local % rows;
    n_blk = local / rows;
  }
}

struct StreamArgs {
  const uint8_t* sfw;      // weight scales (grouped: expert e at sfw + e * sfw_stride)
  int64_t sfw_stride;
  const uint8_t* sfx;      // dense: token scales; grouped: scale slabs per token tile
  const float* ga;
  const float* gb;         // grouped: gb[e]
  uint16_t* y;
  const int4* tiles;       // grouped: (expert, first row, rows, slab)
  const int32_t* n_tiles;  // grouped: device count of tiles
  int32_t* status;
  int M;                   // dense: tokens; grouped: M_total
  int N, K;
  int split;               // dense: cluster size along K
  int stages;
  int x_rows;              // token rows reserved per stage (multiple of 16)
  int acc_cols;            // TMEM columns per accumulator buffer
  int acc_bufs;
  int tmem_cols;
  int pdl;                 // launched with programmatic stream serialization
  int swiglu;              // grouped: weight rows interleave gate/up; y[t, c] = silu(gate) * up, N / 2 wide
  const int32_t* row_token;  // grouped: routed row r reads token row row_token[r] of x (null: row r)
  int T;                     // grouped with row_token: rows of x
  int w_keep;                // weights loaded L2 evict_last (kept resident across calls), else evict_first
  uint64_t watchdog_ns;      // limit of every pipeline wait
  int drop_stage;            // test hook: k >= 1 withholds the k-th stage CTA 0 loads (0: none)
  const uint8_t* meta;       // pair-wise 2:4 sparse weights: tiled metadata (null: dense weights)
  int64_t meta_stride;       // grouped: bytes of metadata per expert
  int l2_prefetch;           // dense: K blocks of the CTA's weight slice prefetched into L2 at entry
  // grouped SwiGLU emitting NVFP4: codes [M, N/4] and tiled scales of [M, N/2] with the
  // caller's global scale g_out; y is not written
  uint8_t* q_out;
  uint8_t* sf_out;
  const float* g_out;
};


// A batched decode launch: up to kMaxBatch GEMMs sharing M (and the launch's split-K,
// stage count and token rows); tensor maps and pointers per GEMM, passed as kernel
// parameters.
constexpr int kMaxBatch = 8;
struct BatchParams {
  CUtensorMap w[kMaxBatch];  // weights [N, K/2], 128-row boxes
  CUtensorMap x[kMaxBatch];  // activations [M, K/2], 16-row boxes
  const uint8_t* sfw[kMaxBatch];
  const uint8_t* sfx[kMaxBatch];
  const float* ga[kMaxBatch];
  const float* gb[kMaxBatch];
  uint16_t* y[kMaxBatch];
  int N[kMaxBatch], K[kMaxBatch];
  int cta_base[kMaxBatch + 1];  // first CTA of each GEMM; cta_base[count] = grid
  int count;
};

// Token rows of one expert per grouped work item: up to 128 (MMA N <= 128); 64 bounds the
// tile count that the workspace is sized for, so either size fits the same workspace.
constexpr int kGroupTile = 64;
constexpr int kGroupTileMax = 128;

cudaError_t launch_amax(const uint16_t* x, int64_t n, float* amax_out, float* g_out, float* partial,
                        int max_partials, cudaStream_t st);
cudaError_t launch_quantize(const uint16_t* x, int64_t M, int64_t K, const float* g, uint8_t* q, uint8_t* sf,
                            cudaStream_t st);
cudaError_t launch_encode(int which, const float* v, int64_t n, uint8_t* out, cudaStream_t st);
cudaError_t launch_prune_pairs(const uint16_t* w, int64_t N, int64_t K, uint16_t* c, uint8_t* meta, int sms,
                               cudaStream_t st);
cudaError_t launch_quantize_b32(const uint16_t* x, int64_t M, int64_t K, const float* g, uint8_t* q, uint8_t* sf,
                                cudaStream_t st);
cudaError_t launch_dense(const CUtensorMap& tmA, const CUtensorMap& tmB, const DenseArgs& a, int bn, int grid,
                         cudaStream_t st);
cudaError_t launch_dense_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                              const CUtensorMap& tmSFB, const CUtensorMap& tmY, const DenseArgs& a, int grid,
                              cudaStream_t st, bool quantized_out = false);
cudaError_t launch_stream(const CUtensorMap& tmW, const CUtensorMap& tmX, const StreamArgs& a, bool grouped,
                          int grid, cudaStream_t st);
cudaError_t launch_batched(const BatchParams& bp, const StreamArgs& a, int grid, cudaStream_t st);
cudaError_t launch_grouped_prep(const int32_t* offsets, const int32_t* row_token, int T, int E, int M_total, int K,
                                int kc4, int tile_rows, const uint8_t* sfx,
                                int32_t* n_tiles, int4* tiles, uint8_t* slabs, int32_t* status, int grid,
                                cudaStream_t st, const uint8_t* x_tok = nullptr, uint8_t* xg = nullptr);
int stream_smem_bytes(int stages, int x_rows, int recv_bytes, bool sparse = false);
// shared memory after the ring for one tile's token indices (and with qout the epilogue's
// NVFP4 transpose tiles, 1 KB per epilogue warp)
__host__ __device__ inline int grouped_extra_bytes(int x_rows, bool qout = false) {
  return (x_rows * 4 > 256 ? x_rows * 4 : 256) + (qout ? 4 * 1024 : 0);
}
int stream_recv_bytes(int M, int split);

// Raises `func`'s dynamic shared-memory limit to the opt-in maximum, once per
// (kernel, device); later calls only look the pair up.
cudaError_t allow_max_smem(const void* func);

}  // namespace nvfp4
