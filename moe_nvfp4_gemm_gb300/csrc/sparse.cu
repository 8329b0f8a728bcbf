// Pair-wise 2:4 sparse NVFP4: weight pruning + compression, and the 32-element-block
// quantiser of the dense operand.
//
// "FP4 structured sparsity" is named as a kernel-level lever in "The Moment of
// Recalibration" (magik.net, The Broader Narrative Arc); the pages give no format. The
// sparse block-scaled tensor-core MMA on FP4 keeps two of the four pairs of neighbouring
// elements in every group of 8 K elements (4:8 pair-wise), reads a 4-bit index nibble per
// group, and applies one scale per 32 K elements of each operand (16 stored values of the
// compressed one). The library's readings:
//   - pruning keeps the two pairs with the largest |w_2j| + |w_2j+1| (one fp32 addition;
//     ties to the lower pair index); the kept pairs are stored in increasing index order;
//   - nibble = i0 | i1 << 2 for kept pair indices i0 < i1, metadata tiled per 128 rows x
//     512 K elements (4 KB: row r's 32 bytes at (r%128/8)*256 + (b/16)*128 + (r%8)*16 + b%16);
//   - the compressed [N, K/2] values are an ordinary NVFP4 tensor (nvfp4_amax, nvfp4_quantize);
//   - the dense operand is quantised by the NVFP4 recipe with 32-element blocks.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "nvfp4_quant.cuh"
#include "ptx.cuh"

namespace nvfp4 {

// Top two of four pair scores, ties to the lower index; returns the nibble i0 | i1 << 2.
DEVI uint32_t top2_nibble(const float (&sc)[4]) {
  int best = 0;
#pragma unroll
  for (int j = 1; j < 4; ++j)
    if (sc[j] > sc[best]) best = j;
  int second = best == 0 ? 1 : 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j != best && sc[j] > sc[second]) second = j;
  const int i0 = min(best, second), i1 = max(best, second);
  return static_cast<uint32_t>(i0 | (i1 << 2));
}

DEVI uint32_t bf16_at(const uint4& v, int i) {  // element i (0..7) of 8 packed bf16
  const uint32_t w = i < 2 ? v.x : (i < 4 ? v.y : (i < 6 ? v.z : v.w));
  return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// One thread per 16 K elements of a row (two groups of 8 -> one metadata byte, 8 kept values).
__global__ void __launch_bounds__(256) k_prune_pairs(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                     uint16_t* __restrict__ c, uint8_t* __restrict__ meta) {
  const int64_t per_row = K / 16;
  const int64_t kmc = (K + 511) / 512;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < N * per_row;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i / per_row, b = i % per_row;
    const uint4* src = reinterpret_cast<const uint4*>(w + n * K + b * 16);
    const uint4 v[2] = {__ldg(src), __ldg(src + 1)};
    uint32_t out[4];
    uint32_t byte = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float sc[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        sc[j] = __fadd_rn(fabsf(__uint_as_float(bf16_at(v[h], 2 * j) << 16)),
                          fabsf(__uint_as_float(bf16_at(v[h], 2 * j + 1) << 16)));
      const uint32_t nib = top2_nibble(sc);
      const int i0 = nib & 3, i1 = nib >> 2;
      out[2 * h] = bf16_at(v[h], 2 * i0) | (bf16_at(v[h], 2 * i0 + 1) << 16);
      out[2 * h + 1] = bf16_at(v[h], 2 * i1) | (bf16_at(v[h], 2 * i1 + 1) << 16);
      byte |= nib << (4 * h);
    }
    *reinterpret_cast<uint4*>(c + n * (K / 2) + b * 8) = make_uint4(out[0], out[1], out[2], out[3]);
    const int64_t r = n % 128, bb = b % 32;
    meta[((n / 128) * kmc + b / 32) * 4096 + (r / 8) * 256 + (bb / 16) * 128 + (r % 8) * 16 + bb % 16] =
        static_cast<uint8_t>(byte);
  }
}

// 32-element blocks: one CTA = 128 rows x 256 columns; thread i takes row i/4 and the
// 32-element block i%4 of each 128-column group (64 bytes), as the 16-element quantiser
// lays out its work; each 512-byte scale tile (128 rows x 4 blocks) leaves as one write.
constexpr int kQ32Groups = 2;  // 128-column groups per CTA

__global__ void __launch_bounds__(512) k_quantize_b32(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                      const float* __restrict__ gptr, uint8_t* __restrict__ q,
                                                      uint8_t* __restrict__ sf) {
  __shared__ uint32_t tile[kQ32Groups][128];
  const int r_local = threadIdx.x >> 2;
  const int c_local = threadIdx.x & 3;
  const int64_t row = static_cast<int64_t>(blockIdx.y) * 128 + r_local;
  const int64_t kc4 = K / 128;  // 512-byte scale tiles per 128 rows
  const int64_t grp0 = static_cast<int64_t>(blockIdx.x) * kQ32Groups;
  const float g = __ldg(gptr);
  const float g_inv = __frcp_rn(g);
  uint4 v[kQ32Groups][4];
#pragma unroll
  for (int t = 0; t < kQ32Groups; ++t)
    if (row < M && grp0 + t < kc4) {
      const uint4* src = reinterpret_cast<const uint4*>(x + row * K + ((grp0 + t) * 4 + c_local) * 32);
#pragma unroll
      for (int u = 0; u < 4; ++u) v[t][u] = __ldg(src + u);
    }
#pragma unroll
  for (int t = 0; t < kQ32Groups; ++t) {
    uint32_t s = 0;
    if (row < M && grp0 + t < kc4) {
      const uint32_t w0[8] = {v[t][0].x, v[t][0].y, v[t][0].z, v[t][0].w, v[t][1].x, v[t][1].y, v[t][1].z, v[t][1].w};
      const uint32_t w1[8] = {v[t][2].x, v[t][2].y, v[t][2].z, v[t][2].w, v[t][3].x, v[t][3].y, v[t][3].z, v[t][3].w};
      uint2 p0, p1;
      quantize_block32(w0, w1, g, g_inv, s, p0, p1);
      *reinterpret_cast<uint4*>(q + row * (K / 2) + ((grp0 + t) * 4 + c_local) * 16) = make_uint4(p0.x, p0.y, p1.x, p1.y);
    }
    reinterpret_cast<uint8_t*>(tile[t])[(r_local & 31) * 16 + (r_local >> 5) * 4 + c_local] = static_cast<uint8_t>(s);
  }
  __syncthreads();
  const int t = threadIdx.x >> 7;
  if (t < kQ32Groups && grp0 + t < kc4) {
    uint32_t* out = reinterpret_cast<uint32_t*>(sf + (static_cast<int64_t>(blockIdx.y) * kc4 + grp0 + t) * 512);
    out[threadIdx.x & 127] = tile[t][threadIdx.x & 127];
  }
}

cudaError_t launch_prune_pairs(const uint16_t* w, int64_t N, int64_t K, uint16_t* c, uint8_t* meta, int sms,
                               cudaStream_t st) {
  const int64_t items = N * (K / 16);
  int64_t blocks = (items + 255) / 256;
  if (blocks > 8 * sms) blocks = 8 * sms;
  if (blocks < 1) blocks = 1;
  k_prune_pairs<<<static_cast<int>(blocks), 256, 0, st>>>(w, N, K, c, meta);
  return cudaGetLastError();
}

cudaError_t launch_quantize_b32(const uint16_t* x, int64_t M, int64_t K, const float* g, uint8_t* q, uint8_t* sf,
                                cudaStream_t st) {
  dim3 grid(static_cast<unsigned>((K / 128 + kQ32Groups - 1) / kQ32Groups), static_cast<unsigned>((M + 127) / 128));
  k_quantize_b32<<<grid, 512, 0, st>>>(x, M, K, g, q, sf);
  return cudaGetLastError();
}

}  // namespace nvfp4
