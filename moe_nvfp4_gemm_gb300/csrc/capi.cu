// C ABI: argument validation, TMA descriptor encoding, plan selection and
// launches. Declarations and the contract of every entry point: include/nvfp4.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "nvfp4.h"
#include "kernels.h"
#include "ptx.cuh"


using namespace nvfp4;

cudaError_t nvfp4::allow_max_smem(const void* func) {
  static std::mutex mu;
  static const void* seen_fn[64];
  static int seen_dev[64];
  static int n_seen = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < n_seen; ++i)
    if (seen_fn[i] == func && seen_dev[i] == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  if (e != cudaSuccess) return e;
  if (n_seen < 64) {
    seen_fn[n_seen] = func;
    seen_dev[n_seen] = dev;
    ++n_seen;
  }
  return cudaSuccess;
}

namespace {

constexpr int kAmaxPartials = 1024;
constexpr int kGroupTileRows = kGroupTile;
constexpr int kSmemLimit = 232448;

thread_local int g_last_launches = 0;

struct Tune {
  int dense_bn = 0, dense_grid = 0, stream_max_m = 0, stream_split = 0, stream_stages = 0, grouped_grid = 0,
      grouped_stages = 0, dense_kernel = 0, pdl = 0, weight_l2 = 0, dense_raster = 0, watchdog_us = 0, withhold_stage = 0,
      stream_l2_prefetch = 0, grouped_tile_rows = 0;
} g_tune;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DevInfo {
  int sms = 0;
  bool ok = false;
};

int device_info(DevInfo& d) {
  static DevInfo cache[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev].sms == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    cache[dev].sms = sms;
    cache[dev].ok = (major == 10 && minor == 3);
  }
  d = cache[dev];
  return d.ok ? NVFP4_OK : NVFP4_ERR_ARCH;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D uint8 view [rows, cols] (cols bytes contiguous), 128-byte-swizzled boxes of
// 128 bytes x box_rows; out-of-range elements read as zero.
int encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return NVFP4_ERR_CUDA;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// Scale tensor viewed as [chunks][128] uint32 (one 512-byte tile per row); boxes of
// four consecutive tiles (the scales of one 256-element K block of 128 rows).
int encode_sf(CUtensorMap* m, const void* base, uint64_t chunks) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return NVFP4_ERR_CUDA;
  cuuint64_t dims[2] = {128, chunks};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 4};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// bf16 output [rows, cols] (cols contiguous) for TMA stores: boxes of 64 columns
// (128 bytes, 128-byte swizzle) x 32 rows; elements outside the tensor are not written.
int encode_out(CUtensorMap* m, void* base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return NVFP4_ERR_CUDA;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// Programmatic-dependent-launch mode of the streaming kernels: 0 off, 1 weights requested
// before the dependency wait, 2 set-up overlap only (the default).
int stream_pdl_mode() { return g_tune.pdl == 0 ? 2 : (g_tune.pdl < 0 ? 0 : g_tune.pdl); }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

// K blocks of each decode CTA's weight slice prefetched into L2 at entry. By default as many
// as keep the prefetches of all resident CTAs (two per SM) within 48 MB of the 126 MB L2:
// the whole slice of one N = K = 8192 call (37.7 MB), but only part of each slice when a
// batched launch's resident CTAs stream far more, where prefetching everything would evict
// prefetched lines before their loads (measured: 8 batched N = K = 8192 GEMMs, M = 1,
// 7.16 us per matrix with whole slices, 6.31 us without prefetch, 6.35 us with 8 blocks).
// With the weights requested before the launch dependency (NVFP4_TUNE_PDL = 1) the first
// ring already overlaps the previous kernel, and prefetching the rest measured slower
// (9.7 against 8.5 us at M = 1): none by default then.
int stream_l2_prefetch(int64_t grid, int sms, int64_t block_bytes) {
  if (g_tune.stream_l2_prefetch != 0) return g_tune.stream_l2_prefetch < 0 ? 0 : g_tune.stream_l2_prefetch;
  if (stream_pdl_mode() == 1) return 0;
  const int64_t resident = grid < 2 * sms ? grid : 2 * int64_t(sms);
  return static_cast<int>((int64_t(48) << 20) / (resident * block_bytes));
}
uint64_t watchdog_ns() { return g_tune.watchdog_us ? uint64_t(g_tune.watchdog_us) * 1000u : kWatchdogNs; }

int64_t pad16(int64_t v) { return (v + 15) / 16 * 16; }

int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

}  // namespace

extern "C" {

const char* nvfp4_status_string(int s) {
  switch (s) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "NVFP4_ERR_UNSUPPORTED_SHAPE";
    case NVFP4_ERR_ALIGNMENT: return "NVFP4_ERR_ALIGNMENT";
    case NVFP4_ERR_ARCH: return "NVFP4_ERR_ARCH";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
    case NVFP4_ERR_WORKSPACE: return "NVFP4_ERR_WORKSPACE";
    case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
    case NVFP4_ERR_BAD_OFFSETS: return "NVFP4_ERR_BAD_OFFSETS";
    default: return "NVFP4_UNKNOWN_STATUS";
  }
}

int64_t nvfp4_scale_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return (rows + 127) / 128 * 128 * ((K / 16 + 3) / 4 * 4);
}

int nvfp4_last_launch_count(void) { return g_last_launches; }

int nvfp4_tune(int key, int value) {
  switch (key) {
    case NVFP4_TUNE_DENSE_BN:
      if (value != 0 && value != 128 && value != 256) return NVFP4_ERR_INVALID_ARG;
      g_tune.dense_bn = value;
      return NVFP4_OK;
    case NVFP4_TUNE_DENSE_GRID:
      if (value < 0) return NVFP4_ERR_INVALID_ARG;
      g_tune.dense_grid = value;
      return NVFP4_OK;
    case NVFP4_TUNE_STREAM_MAX_M:
      if (value < -1 || value > 128) return NVFP4_ERR_INVALID_ARG;
      g_tune.stream_max_m = value;
      return NVFP4_OK;
    case NVFP4_TUNE_STREAM_SPLIT:
      if (value < 0 || value > 8) return NVFP4_ERR_INVALID_ARG;
      g_tune.stream_split = value;
      return NVFP4_OK;
    case NVFP4_TUNE_STREAM_STAGES:
      if (value != 0 && (value < 2 || value > 16)) return NVFP4_ERR_INVALID_ARG;
      g_tune.stream_stages = value;
      return NVFP4_OK;
    case NVFP4_TUNE_GROUPED_GRID:
      if (value < 0) return NVFP4_ERR_INVALID_ARG;
      g_tune.grouped_grid = value;
      return NVFP4_OK;
    case NVFP4_TUNE_GROUPED_STAGES:
      if (value != 0 && (value < 2 || value > 16)) return NVFP4_ERR_INVALID_ARG;
      g_tune.grouped_stages = value;
      return NVFP4_OK;
    case NVFP4_TUNE_DENSE_KERNEL:
      if (value < 0 || value > 2) return NVFP4_ERR_INVALID_ARG;
      g_tune.dense_kernel = value;
      return NVFP4_OK;
    case NVFP4_TUNE_PDL:
      if (value < -1 || value > 2) return NVFP4_ERR_INVALID_ARG;
      g_tune.pdl = value;
      return NVFP4_OK;
    case NVFP4_TUNE_WEIGHT_L2:
      if (value < 0 || value > 1) return NVFP4_ERR_INVALID_ARG;
      g_tune.weight_l2 = value;
      return NVFP4_OK;
    case NVFP4_TUNE_WATCHDOG_US:
      if (value < 0) return NVFP4_ERR_INVALID_ARG;
      g_tune.watchdog_us = value;
      return NVFP4_OK;
    case NVFP4_TUNE_TEST_WITHHOLD_STAGE:
      if (value < 0) return NVFP4_ERR_INVALID_ARG;
      g_tune.withhold_stage = value;
      return NVFP4_OK;
    case NVFP4_TUNE_STREAM_L2_PREFETCH:
      if (value < -1) return NVFP4_ERR_INVALID_ARG;
      g_tune.stream_l2_prefetch = value;
      return NVFP4_OK;
    case NVFP4_TUNE_GROUPED_TILE_ROWS:
      if (value != 0 && value != 64 && value != 128) return NVFP4_ERR_INVALID_ARG;
      g_tune.grouped_tile_rows = value;
      return NVFP4_OK;
    case NVFP4_TUNE_DENSE_RASTER:
      if (value < -1 || value > 1024) return NVFP4_ERR_INVALID_ARG;
      g_tune.dense_raster = value;
      return NVFP4_OK;

    default:
      return NVFP4_ERR_INVALID_ARG;
  }
}

size_t nvfp4_amax_workspace_bytes(int64_t n) {
  (void)n;
  return kAmaxPartials * sizeof(float);
}

int nvfp4_amax(const uint16_t* x, int64_t n, float* amax_out, float* g_out, void* workspace, size_t workspace_bytes,
               void* stream) {
  g_last_launches = 0;
  if (n < 0 || (n > 0 && !x)) return NVFP4_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < nvfp4_amax_workspace_bytes(n)) return NVFP4_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(workspace)) return NVFP4_ERR_ALIGNMENT;
  DevInfo d;
  int rc = device_info(d);
  if (rc) return rc;
  rc = from_cuda(launch_amax(x, n, amax_out, g_out, static_cast<float*>(workspace), kAmaxPartials,
                             static_cast<cudaStream_t>(stream)));
  g_last_launches = 2;
  return rc;
}

int nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, const float* g, uint8_t* q, uint8_t* sf, void* stream) {
  g_last_launches = 0;
  if (M < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
  if (K % 64 != 0 || M > kMaxDim || K > kMaxDim || (M + 127) / 128 > 65535 || K / 64 > kMaxDim)
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || K == 0) return NVFP4_OK;
  if (!x || !g || !q || !sf) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return NVFP4_ERR_ALIGNMENT;
  DevInfo d;
  int rc = device_info(d);
  if (rc) return rc;
  rc = from_cuda(launch_quantize(x, M, K, g, q, sf, static_cast<cudaStream_t>(stream)));
  g_last_launches = 1;
  return rc;
}

int nvfp4_encode_e2m1(const float* v, int64_t n, uint8_t* out, void* stream) {
  if (n < 0 || (n > 0 && (!v || !out))) return NVFP4_ERR_INVALID_ARG;
  if (n == 0) return NVFP4_OK;
  DevInfo d;
  int rc = device_info(d);
  if (rc) return rc;
  return from_cuda(launch_encode(0, v, n, out, static_cast<cudaStream_t>(stream)));
}

int nvfp4_encode_e4m3(const float* v, int64_t n, uint8_t* out, void* stream) {
  if (n < 0 || (n > 0 && (!v || !out))) return NVFP4_ERR_INVALID_ARG;
  if (n == 0) return NVFP4_OK;
  DevInfo d;
  int rc = device_info(d);
  if (rc) return rc;
  return from_cuda(launch_encode(1, v, n, out, static_cast<cudaStream_t>(stream)));
}

size_t nvfp4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  (void)M;
  (void)N;
  (void)K;
  return 0;
}

static int check_gemm_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N <= 0 || K <= 0) return NVFP4_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % 8 != 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return NVFP4_OK;
}

int nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b, const uint8_t* sfb,
               const float* gb, uint16_t* y, int64_t M, int64_t N, int64_t K, void* workspace,
               size_t workspace_bytes, int32_t* dev_status, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  g_last_launches = 0;
  int rc = check_gemm_shape(M, N, K);
  if (rc) return rc;
  if (M == 0) return NVFP4_OK;
  if (!a || !sfa || !ga || !b || !sfb || !gb || !y) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(y))
    return NVFP4_ERR_ALIGNMENT;
  DevInfo d;
  rc = device_info(d);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  const int max_m = g_tune.stream_max_m == 0 ? 128 : g_tune.stream_max_m;
  if (M <= max_m) {
    // weight streaming: W on the MMA's 128-lane side, the M tokens on its N side
    CUtensorMap tmW, tmX;
    if ((rc = encode_2d(&tmW, b, N, K / 2, 128))) return rc;
    if ((rc = encode_2d(&tmX, a, M, K / 2, 16))) return rc;
    const int NT = static_cast<int>((N + 127) / 128);
    const int KB = static_cast<int>((K + 255) / 256);
    StreamArgs s = {};
    s.sfw = sfb;
    s.sfw_stride = 0;
    s.sfx = sfa;
    s.ga = ga;
    s.gb = gb;
    s.y = y;
    s.status = dev_status;
    s.M = static_cast<int>(M);
    s.N = static_cast<int>(N);
    s.K = static_cast<int>(K);
    s.x_rows = static_cast<int>(pad16(M));
    s.acc_cols = (s.x_rows + 31) / 32 * 32;  // the epilogue reads 32-column chunks
    s.acc_bufs = 1;
    int split = g_tune.stream_split;
    if (split == 0) {
      split = (2 * d.sms) / NT;
      split = split < 1 ? 1 : (split > 8 ? 8 : split);
    }
    if (split > KB) split = KB;
    s.split = split;
    s.pdl = stream_pdl_mode();
    s.w_keep = g_tune.weight_l2;
    s.watchdog_ns = watchdog_ns();
    s.drop_stage = g_tune.withhold_stage;
    s.l2_prefetch = stream_l2_prefetch(int64_t(NT) * split, d.sms, 16384 + 2048);
    const int stage_bytes = stream_smem_bytes(1, s.x_rows, 0) - 1536;
    const int recv_bytes = stream_recv_bytes(s.M, split);
    int stages = g_tune.stream_stages;
    if (stages == 0) {
      stages = (110 * 1024 - 1536 - recv_bytes) / stage_bytes;  // two CTAs per SM
      const int tmem_room = (256 - s.acc_cols) / 32;
      if (stages > tmem_room) stages = tmem_room;
      if (stages < 2) stages = 2;
    }
    // the outgoing split-K partials (split x ceil(M / split) x 128 fp32) reuse the stage ring
    while (split > 1 && stages * stage_bytes < recv_bytes) ++stages;
    if (stream_smem_bytes(stages, s.x_rows, recv_bytes) > kSmemLimit) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    s.stages = stages;
    s.tmem_cols = pow2_at_least(s.acc_cols + 32 * stages);
    if (s.tmem_cols > 512) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    rc = from_cuda(launch_stream(tmW, tmX, s, false, NT * split, st));
    g_last_launches = 1;
    return rc;
  }

  const int kernel = g_tune.dense_kernel ? g_tune.dense_kernel : 2;
  if (kernel == 2) {
    // CTA pairs, 256 x 256 tiles
    CUtensorMap tmA, tmB, tmSFA, tmSFB, tmY;
    if ((rc = encode_2d(&tmA, a, M, K / 2, 128))) return rc;
    if ((rc = encode_2d(&tmB, b, N, K / 2, 128))) return rc;
    if ((rc = encode_sf(&tmSFA, sfa, nvfp4_scale_bytes(M, K) / 512))) return rc;
    if ((rc = encode_sf(&tmSFB, sfb, nvfp4_scale_bytes(N, K) / 512))) return rc;
    if ((rc = encode_out(&tmY, y, M, N))) return rc;
    DenseArgs da = {sfa, sfb, ga, gb, y, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), dev_status};
    da.raster = g_tune.dense_raster;
    da.watchdog_ns = watchdog_ns();
    da.drop_stage = g_tune.withhold_stage;
    const int64_t tiles = ((M + 255) / 256) * ((N + 255) / 256);
    int pairs = (g_tune.dense_grid ? g_tune.dense_grid : d.sms) / 2;
    if (pairs > tiles) pairs = static_cast<int>(tiles);
    if (pairs < 1) pairs = 1;
    rc = from_cuda(launch_dense_pair(tmA, tmB, tmSFA, tmSFB, tmY, da, 2 * pairs, st));
    g_last_launches = 1;
    return rc;
  }
  int bn = g_tune.dense_bn ? g_tune.dense_bn : (N <= 128 ? 128 : 256);
  CUtensorMap tmA, tmB;
  if ((rc = encode_2d(&tmA, a, M, K / 2, 128))) return rc;
  if ((rc = encode_2d(&tmB, b, N, K / 2, bn))) return rc;
  DenseArgs da = {sfa, sfb, ga, gb, y, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), dev_status};
  da.raster = g_tune.dense_raster;
  da.watchdog_ns = watchdog_ns();
  da.drop_stage = g_tune.withhold_stage;
  const int64_t tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
  int grid = g_tune.dense_grid ? g_tune.dense_grid : d.sms;
  if (grid > tiles) grid = static_cast<int>(tiles);
  rc = from_cuda(launch_dense(tmA, tmB, da, bn, grid, st));
  g_last_launches = 1;
  return rc;
}

int nvfp4_gemm_quantize_out(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                            const uint8_t* sfb, const float* gb, const float* g_out, uint8_t* q_out, uint8_t* sf_out,
                            int64_t M, int64_t N, int64_t K, int32_t* dev_status, void* stream) {
  g_last_launches = 0;
  int rc = check_gemm_shape(M, N, K);
  if (rc) return rc;
  if (N % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // whole 4-block scale groups per row
  if (M == 0) return NVFP4_OK;
  if (!a || !sfa || !ga || !b || !sfb || !gb || !g_out || !q_out || !sf_out) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(q_out) ||
      !aligned16(sf_out))
    return NVFP4_ERR_ALIGNMENT;
  DevInfo d;
  rc = device_info(d);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap tmA, tmB, tmSFA, tmSFB, tmY;
  if ((rc = encode_2d(&tmA, a, M, K / 2, 128))) return rc;
  if ((rc = encode_2d(&tmB, b, N, K / 2, 128))) return rc;
  if ((rc = encode_sf(&tmSFA, sfa, nvfp4_scale_bytes(M, K) / 512))) return rc;
  if ((rc = encode_sf(&tmSFB, sfb, nvfp4_scale_bytes(N, K) / 512))) return rc;
  tmY = tmA;  // unused by the quantising epilogue
  DenseArgs da = {sfa, sfb, ga, gb, nullptr, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                  dev_status, q_out, sf_out, g_out};
  da.raster = g_tune.dense_raster;
  da.watchdog_ns = watchdog_ns();
  da.drop_stage = g_tune.withhold_stage;
  const int64_t tiles = ((M + 255) / 256) * ((N + 255) / 256);
  int pairs = (g_tune.dense_grid ? g_tune.dense_grid : d.sms) / 2;
  if (pairs > tiles) pairs = static_cast<int>(tiles);
  if (pairs < 1) pairs = 1;
  rc = from_cuda(launch_dense_pair(tmA, tmB, tmSFA, tmSFB, tmY, da, 2 * pairs, st, true));
  g_last_launches = 1;
  return rc;
}

// ---- pair-wise 2:4 sparse weights ------------------------------------------------------------

int64_t nvfp4_sparse_meta_bytes(int64_t N, int64_t K) {
  if (N < 0 || K < 0) return 0;
  return (N + 127) / 128 * ((K + 511) / 512) * 4096;
}

int64_t nvfp4_scale_bytes_b32(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return (rows + 127) / 128 * 128 * ((K / 32 + 3) / 4 * 4);
}

int nvfp4_prune_pairs(const uint16_t* w, int64_t N, int64_t K, uint16_t* c_out, uint8_t* meta_out, void* stream) {
  g_last_launches = 0;
  if (N < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
  if (K % 128 != 0 || N > kMaxDim || K > kMaxDim) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (N == 0 || K == 0) return NVFP4_OK;
  if (!w || !c_out || !meta_out) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(c_out)) return NVFP4_ERR_ALIGNMENT;
  DevInfo d;
  int rc = device_info(d);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // padding of the tiled metadata (rows up to a multiple of 128, K up to 512) reads as zero
  if (N % 128 != 0 || K % 512 != 0) {
    if ((rc = from_cuda(cudaMemsetAsync(meta_out, 0, static_cast<size_t>(nvfp4_sparse_meta_bytes(N, K)), st))))
      return rc;
  }
  rc = from_cuda(launch_prune_pairs(w, N, K, c_out, meta_out, d.sms, st));
  g_last_launches = 1;
  return rc;
}

int nvfp4_quantize_b32(const uint16_t* x, int64_t M, int64_t K, const float* g, uint8_t* q, uint8_t* sf,
                       void* stream) {
  g_last_launches = 0;
  if (M < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
  if (K % 128 != 0 || M > kMaxDim || K > kMaxDim || (M + 127) / 128 > 65535) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || K == 0) return NVFP4_OK;
  if (!x || !g || !q || !sf) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return NVFP4_ERR_ALIGNMENT;
  DevInfo d;
  int rc = device_info(d);
  if (rc) return rc;
  rc = from_cuda(launch_quantize_b32(x, M, K, g, q, sf, static_cast<cudaStream_t>(stream)));
  g_last_launches = 1;
  return rc;
}

int nvfp4_sparse_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b_c, const uint8_t* sfb_c,
                      const uint8_t* meta, const float* gb, uint16_t* y, int64_t M, int64_t N, int64_t K,
                      int32_t* dev_status, void* stream) {
  g_last_launches = 0;
  int rc = check_gemm_shape(M, N, K);
  if (rc) return rc;
  if (K % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return NVFP4_OK;
  if (!a || !sfa || !ga || !b_c || !sfb_c || !meta || !gb || !y) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b_c) || !aligned16(sfb_c) || !aligned16(meta) ||
      !aligned16(y))
    return NVFP4_ERR_ALIGNMENT;
  DevInfo d;
  rc = device_info(d);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // weight streaming (swap-AB): the compressed weights on the MMA's 128-lane side, up to 128
  // token rows on its N side; larger M runs as one launch per 128-row chunk
  CUtensorMap tmW;
  if ((rc = encode_2d(&tmW, b_c, N, K / 4, 128))) return rc;
  const int NT = static_cast<int>((N + 127) / 128);
  const int KB = static_cast<int>((K + 511) / 512);
  const int64_t chunk_sf = (K / 128) * 512;  // x scale bytes per 128 rows
  int launches = 0;
  for (int64_t m0 = 0; m0 < M; m0 += 128) {
    const int Mc = static_cast<int>(M - m0 < 128 ? M - m0 : 128);
    CUtensorMap tmX;
    if ((rc = encode_2d(&tmX, a + m0 * (K / 2), Mc, K / 2, 16))) return rc;
    StreamArgs s = {};
    s.sfw = sfb_c;
    s.sfx = sfa + (m0 / 128) * chunk_sf;
    s.ga = ga;
    s.gb = gb;
    s.y = y + m0 * N;
    s.status = dev_status;
    s.M = Mc;
    s.N = static_cast<int>(N);
    s.K = static_cast<int>(K);
    s.meta = meta;
    s.x_rows = static_cast<int>(pad16(Mc));
    s.acc_cols = (s.x_rows + 31) / 32 * 32;
    s.acc_bufs = 1;
    int split = g_tune.stream_split;
    if (split == 0) {
      split = (2 * d.sms) / NT;
      split = split < 1 ? 1 : (split > 8 ? 8 : split);
    }
    if (split > KB) split = KB;
    s.split = split;
    s.pdl = stream_pdl_mode();
    s.w_keep = g_tune.weight_l2;
    s.watchdog_ns = watchdog_ns();
    s.drop_stage = g_tune.withhold_stage;
    s.l2_prefetch = stream_l2_prefetch(int64_t(NT) * split, d.sms, 16384 + 2048 + 4096);
    const int stage_bytes = stream_smem_bytes(1, s.x_rows, 0, true) - 1536;
    const int recv_bytes = stream_recv_bytes(s.M, split);
    int stages = g_tune.stream_stages;
    if (stages == 0) {
      stages = (110 * 1024 - 1536 - recv_bytes) / stage_bytes;  // two CTAs per SM
      const int tmem_room = (256 - s.acc_cols) / 40;
      if (stages > tmem_room) stages = tmem_room;
      if (stages < 2) stages = 2;
    }
    while (split > 1 && stages * stage_bytes < recv_bytes) ++stages;
    if (stream_smem_bytes(stages, s.x_rows, recv_bytes, true) > kSmemLimit) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    s.stages = stages;
    s.tmem_cols = pow2_at_least(s.acc_cols + 40 * stages);
    if (s.tmem_cols > 512) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    rc = from_cuda(launch_stream(tmW, tmX, s, false, NT * split, st));
    ++launches;
    g_last_launches = launches;
    if (rc) return rc;
  }
  return NVFP4_OK;
}

static int64_t grouped_max_tiles(int32_t E, int64_t M_total) { return (M_total + kGroupTileRows - 1) / kGroupTileRows + E; }

static int64_t grouped_slab_offset(int32_t E, int64_t M_total) {
  return (16 + grouped_max_tiles(E, M_total) * 16 + 255) / 256 * 256;
}

int nvfp4_gemm_batched(const nvfp4_gemm_problem* problems, int32_t count, int64_t M, int32_t* dev_status,
                       void* stream) {
  g_last_launches = 0;
  if (!problems || count < 1 || count > NVFP4_MAX_BATCH || M < 0) return NVFP4_ERR_INVALID_ARG;
  for (int g = 0; g < count; ++g) {
    const int rc = check_gemm_shape(M, problems[g].N, problems[g].K);
    if (rc) return rc;
  }
  if (M > 128) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // the weight-streaming kernel's token range
  if (M == 0) return NVFP4_OK;
  for (int g = 0; g < count; ++g) {
    const nvfp4_gemm_problem& q = problems[g];
    if (!q.a || !q.sfa || !q.ga || !q.b || !q.sfb || !q.gb || !q.y) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(q.a) || !aligned16(q.sfa) || !aligned16(q.b) || !aligned16(q.sfb) || !aligned16(q.y))
      return NVFP4_ERR_ALIGNMENT;
  }
  DevInfo d;
  int rc = device_info(d);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // One split-K cluster size for the launch, chosen from all GEMMs' 128-row weight tiles
  // as a single call chooses it from its own; no GEMM splits finer than its K blocks.
  int64_t tiles = 0;
  int min_kb = 1 << 30;
  for (int g = 0; g < count; ++g) {
    tiles += (problems[g].N + 127) / 128;
    const int kb = static_cast<int>((problems[g].K + 255) / 256);
    if (kb < min_kb) min_kb = kb;
  }
  int split = g_tune.stream_split;
  if (split == 0) {
    const int64_t sp = (2 * static_cast<int64_t>(d.sms)) / tiles;
    split = static_cast<int>(sp < 1 ? 1 : (sp > 8 ? 8 : sp));
  }
  if (split > min_kb) split = min_kb;
  if (tiles * split > (int64_t(1) << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;

  BatchParams bp = {};  // kernel parameters: copied by the launch
  int cta = 0;
  for (int g = 0; g < count; ++g) {
    const nvfp4_gemm_problem& q = problems[g];
    if ((rc = encode_2d(&bp.w[g], q.b, q.N, q.K / 2, 128))) return rc;
    if ((rc = encode_2d(&bp.x[g], q.a, M, q.K / 2, 16))) return rc;
    bp.sfw[g] = q.sfb;
    bp.sfx[g] = q.sfa;
    bp.ga[g] = q.ga;
    bp.gb[g] = q.gb;
    bp.y[g] = q.y;
    bp.N[g] = static_cast<int>(q.N);
    bp.K[g] = static_cast<int>(q.K);
    bp.cta_base[g] = cta;
    cta += static_cast<int>((q.N + 127) / 128) * split;
  }
  bp.cta_base[count] = cta;
  bp.count = count;

  StreamArgs s = {};
  s.sfw_stride = 0;
  s.status = dev_status;
  s.M = static_cast<int>(M);
  s.x_rows = static_cast<int>(pad16(M));
  s.acc_cols = (s.x_rows + 31) / 32 * 32;
  s.acc_bufs = 1;
  s.split = split;
  s.pdl = stream_pdl_mode();
  s.w_keep = g_tune.weight_l2;
  s.watchdog_ns = watchdog_ns();
  s.drop_stage = g_tune.withhold_stage;
  s.l2_prefetch = stream_l2_prefetch(cta, d.sms, 16384 + 2048);
  const int stage_bytes = stream_smem_bytes(1, s.x_rows, 0) - 1536;
  const int recv_bytes = stream_recv_bytes(s.M, split);
  int stages = g_tune.stream_stages;
  if (stages == 0) {
    stages = (110 * 1024 - 1536 - recv_bytes) / stage_bytes;  // two CTAs per SM
    const int tmem_room = (256 - s.acc_cols) / 32;
    if (stages > tmem_room) stages = tmem_room;
    if (stages < 2) stages = 2;
  }
  while (split > 1 && stages * stage_bytes < recv_bytes) ++stages;
  if (stream_smem_bytes(stages, s.x_rows, recv_bytes) > kSmemLimit) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  s.stages = stages;
  s.tmem_cols = pow2_at_least(s.acc_cols + 32 * stages);
  if (s.tmem_cols > 512) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  rc = from_cuda(launch_batched(bp, s, cta, st));
  g_last_launches = 1;
  return rc;
}

size_t nvfp4_grouped_gemm_workspace_bytes(int32_t E, int64_t M_total, int64_t N, int64_t K) {
  (void)N;
  if (E <= 0 || M_total < 0 || K <= 0) return 0;
  return static_cast<size_t>(grouped_slab_offset(E, M_total) + grouped_max_tiles(E, M_total) * (K / 64) * 512);
}

// The gather entry's larger workspace: the plain one (rounded up to 256 bytes), then the
// routed rows copied out of the token activations, [M_total, K/2].
static size_t gathered_rows_offset(int32_t E, int64_t M_total, int64_t N, int64_t K) {
  return (nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K) + 255) / 256 * 256;
}

size_t nvfp4_grouped_gemm_gather_workspace_bytes(int32_t E, int64_t M_total, int64_t N, int64_t K) {
  if (E <= 0 || M_total < 0 || K <= 0) return 0;
  return gathered_rows_offset(E, M_total, N, K) + static_cast<size_t>(M_total) * static_cast<size_t>(K / 2);
}

// row_token (null: none): routed row r reads row row_token[r] of the T-row activations a.
// meta (null: dense weights): pair-wise 2:4 sparse experts, b / sfb their compressed codes and
// scales, a / sfa the routed rows in 32-element blocks.
static int grouped_impl(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b, const uint8_t* sfb,
                        const float* gb, const int32_t* expert_offsets, int32_t E, int64_t M_total, int64_t N,
                        int64_t K, uint16_t* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream, int swiglu, const int32_t* row_token = nullptr, int64_t T = 0,
                        const uint8_t* meta = nullptr, uint8_t* q_out = nullptr, uint8_t* sf_out = nullptr,
                        const float* g_out = nullptr) {
  g_last_launches = 0;
  const bool sparse = meta != nullptr;
  if (sparse && K % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (row_token && M_total > 0 && (T <= 0 || T > kMaxDim)) return NVFP4_ERR_INVALID_ARG;
  if (E <= 0) return NVFP4_ERR_INVALID_ARG;
  int rc = check_gemm_shape(M_total, N, K);
  if (rc) return rc;
  if (static_cast<int64_t>(E) * N > kMaxDim || E > 16384) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  // routed rows are indexed with 32-bit integers on the device, with headroom for the
  // preparation kernel's grid stride
  if (M_total > (int64_t(1) << 30)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (M_total == 0) return NVFP4_OK;
  const bool qout = q_out != nullptr;
  if (!a || !sfa || !ga || !b || !sfb || !gb || !expert_offsets || (!qout && !y)) return NVFP4_ERR_INVALID_ARG;
  if (qout && (!sf_out || !g_out)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || (!qout && !aligned16(y)) ||
      (qout && (!aligned16(q_out) || !aligned16(sf_out))))
    return NVFP4_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K))
    return NVFP4_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return NVFP4_ERR_ALIGNMENT;
  DevInfo d;
  rc = device_info(d);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (qout && M_total % 128 != 0) {
    // The scale tensor's padding rows (up to a multiple of 128) read as zero: the last
    // 128-row group's scale tiles are cleared first, then the kernel writes its rows' bytes.
    const int64_t kc4o = (N / 2) / 64;
    if ((rc = from_cuda(cudaMemsetAsync(sf_out + (M_total / 128) * kc4o * 512, 0, kc4o * 512, st)))) return rc;
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* n_tiles = reinterpret_cast<int32_t*>(ws);
  int4* tiles = reinterpret_cast<int4*>(ws + 16);
  uint8_t* slabs = ws + grouped_slab_offset(E, M_total);
  // Token gather: with room for the routed rows the preparation kernel copies them out
  // (M_total x K/2 bytes, a few microseconds) and the GEMM reads them as plain tiles;
  // otherwise the GEMM's load stage fetches them four rows per tile::gather4.
  uint8_t* xg = nullptr;
  if (row_token && workspace_bytes >= nvfp4_grouped_gemm_gather_workspace_bytes(E, M_total, N, K))
    xg = ws + gathered_rows_offset(E, M_total, N, K);
  // token rows per work item: up to 128, so that a heavily routed expert streams its
  // weights ceil(rows / 128) times
  const int tile_rows = g_tune.grouped_tile_rows ? g_tune.grouped_tile_rows : kGroupTileMax;
  // one warp per routed row and step (eight per block)
  const int64_t prep_blocks = (M_total + 7) / 8;
  int prep_grid = static_cast<int>(prep_blocks < 4 * d.sms ? prep_blocks : 4 * d.sms);
  if (prep_grid < 1) prep_grid = 1;
  rc = from_cuda(launch_grouped_prep(expert_offsets, row_token, static_cast<int>(T), E, static_cast<int>(M_total),
                                     static_cast<int>(K), static_cast<int>(sparse ? K / 128 : K / 64), tile_rows, sfa,
                                     n_tiles,
                                     tiles, slabs, dev_status, prep_grid, st, xg ? a : nullptr, xg));
  g_last_launches = 1;
  if (rc) return rc;

  CUtensorMap tmW, tmX;
  if ((rc = encode_2d(&tmW, b, static_cast<uint64_t>(E) * N, sparse ? K / 4 : K / 2, 128))) return rc;
  if (xg) {
    if ((rc = encode_2d(&tmX, xg, M_total, K / 2, 16))) return rc;
    row_token = nullptr;  // the GEMM reads the copied rows
  } else if (row_token) {
    if ((rc = encode_2d(&tmX, a, T, K / 2, 1))) return rc;  // one-row boxes for tile::gather4
  } else if ((rc = encode_2d(&tmX, a, M_total, K / 2, 16))) {
    return rc;
  }
  StreamArgs s = {};
  s.row_token = row_token;
  s.T = static_cast<int>(T);
  s.sfw = sfb;
  s.sfw_stride = nvfp4_scale_bytes(N, sparse ? K / 2 : K);
  s.meta = meta;
  s.meta_stride = sparse ? nvfp4_sparse_meta_bytes(N, K) : 0;
  s.sfx = slabs;
  s.ga = ga;
  s.gb = gb;
  s.y = y;
  s.tiles = tiles;
  s.n_tiles = n_tiles;
  s.status = dev_status;
  s.M = static_cast<int>(M_total);
  s.N = static_cast<int>(N);
  s.K = static_cast<int>(K);
  s.split = 1;
  s.pdl = stream_pdl_mode();
  s.w_keep = g_tune.weight_l2;
  s.watchdog_ns = watchdog_ns();
  s.drop_stage = g_tune.withhold_stage;
  s.x_rows = tile_rows;
  s.acc_cols = tile_rows;
  s.acc_bufs = 2;
  s.swiglu = swiglu;
  s.q_out = q_out;
  s.sf_out = sf_out;
  s.g_out = g_out;
  const int sf_cols = sparse ? 40 : 32;  // TMEM columns per stage: scales (+ metadata)
  const int stage_bytes = stream_smem_bytes(1, s.x_rows, 0, sparse) - 1536;
  int stages = g_tune.grouped_stages;
  if (stages == 0) stages = (kSmemLimit - 1536 - grouped_extra_bytes(tile_rows, qout)) / stage_bytes;
  const int tmem_room = (512 - 2 * s.acc_cols) / sf_cols;
  if (stages > tmem_room) stages = tmem_room;
  if (stages > 16) stages = 16;
  if (stream_smem_bytes(stages, s.x_rows, grouped_extra_bytes(tile_rows, qout), sparse) > kSmemLimit)
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  s.stages = stages;
  s.tmem_cols = pow2_at_least(2 * s.acc_cols + sf_cols * stages);
  const int grid = g_tune.grouped_grid ? g_tune.grouped_grid : d.sms;
  rc = from_cuda(launch_stream(tmW, tmX, s, true, grid, st));
  g_last_launches = 2;
  return rc;
}

int nvfp4_grouped_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b, const uint8_t* sfb,
                       const float* gb, const int32_t* expert_offsets, int32_t E, int64_t M_total, int64_t N,
                       int64_t K, uint16_t* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       void* stream) {
  return grouped_impl(a, sfa, ga, b, sfb, gb, expert_offsets, E, M_total, N, K, y, workspace, workspace_bytes,
                      dev_status, stream, 0);
}

int nvfp4_grouped_gemm_gather(const uint8_t* a_tok, const uint8_t* sfa_tok, const float* ga, const uint8_t* b,
                              const uint8_t* sfb, const float* gb, const int32_t* expert_offsets,
                              const int32_t* row_token, int32_t E, int64_t T, int64_t M_total, int64_t N, int64_t K,
                              uint16_t* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream) {
  if (!row_token && M_total > 0) return NVFP4_ERR_INVALID_ARG;
  return grouped_impl(a_tok, sfa_tok, ga, b, sfb, gb, expert_offsets, E, M_total, N, K, y, workspace, workspace_bytes,
                      dev_status, stream, 0, row_token, T);
}

int nvfp4_grouped_sparse_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b_c,
                              const uint8_t* sfb_c, const uint8_t* meta, const float* gb,
                              const int32_t* expert_offsets, int32_t E, int64_t M_total, int64_t N, int64_t K,
                              uint16_t* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream) {
  if (!meta && M_total > 0) return NVFP4_ERR_INVALID_ARG;
  if (meta && !aligned16(meta)) return NVFP4_ERR_ALIGNMENT;
  return grouped_impl(a, sfa, ga, b_c, sfb_c, gb, expert_offsets, E, M_total, N, K, y, workspace, workspace_bytes,
                      dev_status, stream, 0, nullptr, 0, meta);
}

int nvfp4_grouped_gemm_swiglu(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b_gu,
                              const uint8_t* sfb_gu, const float* gb, const int32_t* expert_offsets, int32_t E,
                              int64_t M_total, int64_t N_gu, int64_t K, uint16_t* y, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return grouped_impl(a, sfa, ga, b_gu, sfb_gu, gb, expert_offsets, E, M_total, N_gu, K, y, workspace,
                      workspace_bytes, dev_status, stream, 1);
}

int nvfp4_grouped_gemm_swiglu_quantize_out(const uint8_t* a, const uint8_t* sfa, const float* ga,
                                           const uint8_t* b_gu, const uint8_t* sfb_gu, const float* gb,
                                           const int32_t* expert_offsets, int32_t E, int64_t M_total, int64_t N_gu,
                                           int64_t K, const float* g_out, uint8_t* q_out, uint8_t* sf_out,
                                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                           void* stream) {
  g_last_launches = 0;
  if (N_gu > 0 && N_gu % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;  // whole 16-element output blocks per warp
  if (M_total > 0 && !q_out) return NVFP4_ERR_INVALID_ARG;
  return grouped_impl(a, sfa, ga, b_gu, sfb_gu, gb, expert_offsets, E, M_total, N_gu, K, nullptr, workspace,
                      workspace_bytes, dev_status, stream, 1, nullptr, 0, nullptr, q_out, sf_out, g_out);
}

}  // extern "C"

// ---- allocation-free grouped GEMM ------------------------------------------------------------

// Scratch of nvfp4_grouped_gemm_noalloc: one copy on every device that loads this
// library, held until the process exits. In host code this name is only a stand-in;
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_grouped_scratch[NVFP4_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_dev_ptr[64];  // per device: device address of g_grouped_scratch, or null
}  // namespace

extern "C" int nvfp4_grouped_gemm_noalloc(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                                          const uint8_t* sfb, const float* gb, const int32_t* expert_offsets,
                                          int32_t E, int64_t M_total, int64_t N, int64_t K, uint16_t* y,
                                          int32_t* dev_status, void* stream) {
  g_last_launches = 0;
  if (nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K) > NVFP4_NOALLOC_SCRATCH_BYTES)
    return NVFP4_ERR_WORKSPACE;  // problem too large for the fixed scratch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NVFP4_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_dev_ptr[dev]) {
      // first call on this device (which is current): look the array's address up once
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_grouped_scratch) != cudaSuccess || !ptr) return NVFP4_ERR_CUDA;
      g_scratch_dev_ptr[dev] = ptr;
    }
    scratch = g_scratch_dev_ptr[dev];
  }
  return nvfp4_grouped_gemm(a, sfa, ga, b, sfb, gb, expert_offsets, E, M_total, N, K, y, scratch,
                            NVFP4_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
