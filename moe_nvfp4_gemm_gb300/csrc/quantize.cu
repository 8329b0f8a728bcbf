// bf16 -> NVFP4 quantisation: the tensor-wide amax / global scale and the
// per-16-element block quantiser (E4M3 block scale + packed E2M1 codes, scales
// written in the 128-row x 4-column tiled layout).
//
// Formats: "NVFP4 linear layer" (kernelindex, operation header) - FP4 values
// with FP8 E4M3FN scales, one per 16 elements; "The 3.7 PFLOPS Revelation"
// (magik.net, Input Knowledge item 2) - two FP4 values per byte, [rows, K/2].
// Recipe (the pages fix none; this is the library's stated reading):
//   g = amax / 2688 (1 if amax == 0); s = E4M3_rn_sat((amax_blk / 6) / g);
//   q = E2M1_rn_sat(x / (E4M3(s) * g)), sign kept; q = 0 when s == 0.
// Every float step is one IEEE round-to-nearest operation (true division).
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "nvfp4_quant.cuh"
#include "ptx.cuh"

namespace nvfp4 {

// ---- amax ------------------------------------------------------------------------

constexpr int kAmaxUnroll = 4;  // 16-byte loads in flight per thread

// Per-CTA partial maxima of |x|. CTA b sweeps one contiguous range of 16-byte vectors,
// each thread keeping kAmaxUnroll loads in flight (a warp reads 2 KB contiguous per
// step); maxima are taken on bf16 pairs with their sign bits cleared, which is exact.
// (A grid-stride sweep with one load in flight per thread took 14.5 us on the prefill
// activations from HBM; this one 11.8 us.)
__global__ void __launch_bounds__(256) k_amax_partial(const uint16_t* __restrict__ x, int64_t n,
                                                      float* __restrict__ partial) {
  // Launched with programmatic stream serialization: the CTAs may start while the previous
  // kernel in the stream finishes, and wait for it here before reading x.
  griddep_wait();
  // the one-CTA final reduction may launch now; it waits for this grid's completion
  griddep_launch_dependents();
  const int64_t nvec = n / 8;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t bd = blockDim.x;
  const int64_t per = (nvec + gridDim.x - 1) / gridDim.x;
  const int64_t b0 = blockIdx.x * per, b1 = min(nvec, b0 + per);
  uint32_t m2 = 0;  // running maximum of |x| on bf16 pairs
  int64_t i = b0 + threadIdx.x;
  for (; i + (kAmaxUnroll - 1) * bd < b1; i += kAmaxUnroll * bd) {
    uint4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) v[u] = __ldg(xv + i + u * bd);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(w[j] & 0x7FFF7FFFu));
    }
  }
  for (; i < b1; i += bd) {
    const uint4 v = __ldg(xv + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(w[j] & 0x7FFF7FFFu));
  }
  float m = fmaxf(bf16lo(m2), bf16hi(m2));
  if (blockIdx.x == gridDim.x - 1)  // elements past the last whole vector
    for (int64_t t = nvec * 8 + threadIdx.x; t < n; t += bd)
      m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[t]) << 16)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) partial[blockIdx.x] = m;
  }
}

// Reduces the partial maxima; writes amax and the decode-direction global scale.
__global__ void __launch_bounds__(256) k_amax_final(const float* __restrict__ partial, int np,
                                                    float* amax_out, float* g_out) {
  griddep_wait();  // launched programmatically behind k_amax_partial: its partials are complete
  // the next kernel in the stream may launch now (one CTA here holds no resources it needs);
  // a kernel that waits for this one's completion still sees amax and g
  griddep_launch_dependents();
  float m = 0.0f;
  for (int i = threadIdx.x; i < np; i += blockDim.x) m = fmaxf(m, partial[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    m = fmaxf(m, red[0]);
    if (amax_out) *amax_out = m;
    if (g_out) *g_out = (m == 0.0f) ? 1.0f : __fdiv_rn(m, 2688.0f);
  }
}

// ---- block quantiser -----------------------------------------------------------

constexpr int kQuantTiles = 2;     // 64-column groups (512-byte scale tiles) per CTA
constexpr int kQuantThreads = 256;  // 64 rows x 4 blocks of 16 elements
constexpr int kQuantRows = kQuantThreads / 4;

// One CTA = 64 rows x (64 * kQuantTiles) columns, two CTAs (consecutive in x) per 128-row
// group, so that the grid covers the scale tensor's padding rows, which are written 0
// (rows >= M load and quantise nothing); thread i handles row i/4 and
// 16-element block i%4 of each 64-column group. All of a thread's loads are issued
// before any arithmetic (64 bytes in flight per thread); a warp reads 8 rows x 128
// contiguous bytes per group. The four threads of a row combine their scale bytes with
// two shuffles and one of them stores the 4-byte word, so no CTA barrier is needed. Small
// CTAs at 40 registers keep six per SM resident (48 warps), which hides more of the
// loads' and the arithmetic's latency than larger CTAs or more blocks per thread
// (measured on the prefill activations, 4096 x 8192: 20.2-20.5 us against 22.9 us for
// 128-row CTAs with four blocks per thread and the scale tile staged in shared memory).
__global__ void __launch_bounds__(kQuantThreads, 6) k_quantize(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                               const float* __restrict__ gptr,
                                                               uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  // Launched with programmatic stream serialization (set-up overlap only): wait for the
  // previous kernel in the stream before any memory access.
  griddep_wait();
  const int r_local = threadIdx.x >> 2;
  const int c_local = threadIdx.x & 3;
  const int64_t row = static_cast<int64_t>(blockIdx.y) * 128 + (blockIdx.x & 1) * kQuantRows + r_local;
  const int64_t kc4 = K / 64;
  const int64_t col4_0 = static_cast<int64_t>(blockIdx.x >> 1) * kQuantTiles;
  const float g = __ldg(gptr);
  const float g_inv = __frcp_rn(g);
  uint4 v[kQuantTiles][2];
#pragma unroll
  for (int t = 0; t < kQuantTiles; ++t) {
    if (row < M && col4_0 + t < kc4) {
      const uint4* src = reinterpret_cast<const uint4*>(x + row * K + ((col4_0 + t) * 4 + c_local) * 16);
      v[t][0] = __ldg(src);
      v[t][1] = __ldg(src + 1);
    }
  }
#pragma unroll
  for (int t = 0; t < kQuantTiles; ++t) {
    const bool ok = row < M && col4_0 + t < kc4;
    uint32_t s = 0;
    if (ok) {
      const uint32_t w[8] = {v[t][0].x, v[t][0].y, v[t][0].z, v[t][0].w,
                             v[t][1].x, v[t][1].y, v[t][1].z, v[t][1].w};
      uint2 packed;
      quantize_block(w, g, g_inv, s, packed);
      *reinterpret_cast<uint2*>(q + row * (K / 2) + ((col4_0 + t) * 4 + c_local) * 8) = packed;
    }
    // the row's four scale bytes (blocks c_local = 0..3 of this group) as one word; in the
    // tiled layout scale byte (r, c) of a 512-byte tile sits at (r % 32) * 16 + (r / 32) * 4 + c
    uint32_t word = s << (8 * c_local);
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    if (c_local == 0 && col4_0 + t < kc4)
      *reinterpret_cast<uint32_t*>(sf + ((row / 128) * kc4 + col4_0 + t) * 512 + (row % 32) * 16 +
                                   ((row % 128) / 32) * 4) = word;
  }
}

// Elementwise encoders, exposed for exhaustive checks of the device conversions.
__global__ void k_encode_e2m1(const float* __restrict__ v, int64_t n, uint8_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = static_cast<uint8_t>(e2m1x2_encode(v[i], 0.0f) & 0xF);
}

__global__ void k_encode_e4m3(const float* __restrict__ v, int64_t n, uint8_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = static_cast<uint8_t>(e4m3_encode(v[i]));
}

// ---- host launchers ----------------------------------------------------------------

// A launch with programmatic stream serialization (the kernel waits for its predecessor
// with griddepcontrol.wait before touching memory).
static cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, cudaStream_t st) {
  static cudaLaunchAttribute attr = [] {
    cudaLaunchAttribute a = {};
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
  }();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cfg;
}

cudaError_t launch_amax(const uint16_t* x, int64_t n, float* amax_out, float* g_out, float* partial,
                        int max_partials, cudaStream_t st) {
  int64_t want = (n / 8 + 255) / 256;
  int grid = static_cast<int>(want < 1 ? 1 : (want > max_partials ? max_partials : want));
  // Both kernels are launched with programmatic stream serialization: each one's launch
  // overlaps the end of the kernel before it, and each waits (griddepcontrol.wait) for that
  // kernel to complete before it reads memory.
  cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(256), st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_amax_partial, x, n, partial);
  if (e != cudaSuccess) return e;
  cfg = pdl_config(dim3(1), dim3(256), st);
  return cudaLaunchKernelEx(&cfg, k_amax_final, static_cast<const float*>(partial), grid, amax_out, g_out);
}

cudaError_t launch_quantize(const uint16_t* x, int64_t M, int64_t K, const float* g, uint8_t* q,
                            uint8_t* sf, cudaStream_t st) {
  dim3 grid(static_cast<unsigned>((K / 64 + kQuantTiles - 1) / kQuantTiles * 2), static_cast<unsigned>((M + 127) / 128));
  cudaLaunchConfig_t cfg = pdl_config(grid, dim3(kQuantThreads), st);
  return cudaLaunchKernelEx(&cfg, k_quantize, x, M, K, g, q, sf);
}

cudaError_t launch_encode(int which, const float* v, int64_t n, uint8_t* out, cudaStream_t st) {
  int64_t want = (n + 255) / 256;
  int grid = static_cast<int>(want < 1 ? 1 : (want > 65535 ? 65535 : want));
  if (which == 0)
    k_encode_e2m1<<<grid, 256, 0, st>>>(v, n, out);
  else
    k_encode_e4m3<<<grid, 256, 0, st>>>(v, n, out);
  return cudaGetLastError();
}

}  // namespace nvfp4
