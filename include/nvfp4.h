/*
 * nvfp4.h - C ABI of the GB300 (sm_103a) NVFP4 block-scaled GEMM library.
 *
 * What is computed (the pages are cited by title and section):
 *   "NVFP4 linear layer" (kernelindex, operation header): y = x @ W^T, where x
 *   and W are FP4 (E2M1) values with FP8 E4M3FN scale factors, one scale per 16
 *   consecutive K elements (sf_vec_size = 16, sf_k = K/16, in_features_half = K/2).
 *   "The 3.7 PFLOPS Revelation" (magik.net, Input Knowledge item 2): two FP4
 *   values per byte, so data tensors are [rows, K/2] and scale tensors [rows, K/16].
 *   "The Moment of Recalibration" (magik.net, Input Knowledge) and "The Moment of
 *   Synthesis" (magik.net, Reasoning): MoE layers of 256 experts with top-8
 *   routing, each expert a small GEMM; grouped GEMM is the remedy.
 *
 * Conventions taken by this library where the pages are silent:
 *   - Packed FP4: byte j of a row holds element 2j in bits 0-3 and 2j+1 in bits 4-7.
 *   - Scale tensors are tiled: scale (r, c), c = k/16, lives at byte
 *       ((r/128) * ceil(Kc/4) + c/4) * 512 + (r%32) * 16 + ((r%128)/32) * 4 + c%4,
 *     Kc = K/16; the tensor has nvfp4_scale_bytes(rows, K) bytes, padding 0.
 *   - Each tensor carries one FP32 global scale g in the decode direction:
 *     value = E2M1(code) * E4M3(scale) * g. Quantisation uses g = amax/(6*448).
 *   - y = bf16_rn((sum_k x^ w^) * g_a * g_b), accumulated in fp32 on the GPU.
 *
 * General rules for every entry point:
 *   - Tensor arguments are DEVICE pointers owned by the caller; bf16 tensors are
 *     passed as uint16_t bit patterns; scalars such as g are device fp32.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls only
 *     enqueue work: they never synchronise and never allocate.
 *   - The return value is NVFP4_OK or a negative nvfp4_status for arguments
 *     rejected on the host (nothing is enqueued then) or a failed launch
 *     (NVFP4_ERR_CUDA). Errors found on the device (malformed expert offsets, a
 *     wait that timed out) are written to *dev_status when dev_status is not
 *     NULL; the caller zeroes it beforehand and reads it after synchronising.
 *   - Shapes: K % 64 == 0, N % 8 == 0, M >= 0, all sizes < 2^31 (grouped calls: at
 *     most 2^30 routed rows, E <= 16384 experts, E * N < 2^31). Data, scale and
 *     output base pointers are 16-byte aligned (TMA). M == 0 is a no-op.
 *   - The device must be compute capability 10.3 (GB300, sm_103a).
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = -1,     /* null pointer, negative size */
  NVFP4_ERR_UNSUPPORTED_SHAPE = -2, /* K % 64, N % 8, size limits */
  NVFP4_ERR_ALIGNMENT = -3,       /* a base pointer is not 16-byte aligned */
  NVFP4_ERR_ARCH = -4,            /* current device is not sm_103 */
  NVFP4_ERR_CUDA = -5,            /* a CUDA call or launch failed */
  NVFP4_ERR_WORKSPACE = -6,       /* workspace missing or too small */
  NVFP4_ERR_TIMEOUT = -7,         /* device: a pipeline wait gave up (watchdog) */
  NVFP4_ERR_BAD_OFFSETS = -8      /* device: expert_offsets not 0..M_total, non-decreasing */
} nvfp4_status;

/* Human-readable name of a status code. Never NULL. */
const char* nvfp4_status_string(int status);

/* Bytes of a tiled scale tensor for `rows` rows and K elements per row:
 * ceil(rows/128)*128 * ceil(K/64)*4. Returns 0 for invalid sizes. */
int64_t nvfp4_scale_bytes(int64_t rows, int64_t K);

/*
 * Tensor-wide amax of a bf16 tensor and its global scale. Not on the pages
 * (they quantise "ahead of execution": "Blackwell NVFP4 GEMM" case page, What is
 * this?); the recipe is the library's reading: g = amax / 2688 (6 * 448), and
 * g = 1 when amax == 0.
 *   x          device bf16 [n], 16-byte aligned
 *   amax_out   device fp32 scalar, written (may be NULL)
 *   g_out      device fp32 scalar, written (may be NULL)
 *   workspace  device scratch of nvfp4_amax_workspace_bytes(n) bytes, 16-byte aligned
 */
size_t nvfp4_amax_workspace_bytes(int64_t n);
int nvfp4_amax(const uint16_t* x, int64_t n, float* amax_out, float* g_out, void* workspace,
               size_t workspace_bytes, void* stream);

/*
 * bf16 -> NVFP4 block quantisation (the secondary path; the pages exclude
 * quantisation from their timings: "Blackwell NVFP4 GEMM" case page, What is this?).
 * Per row r and 16-element block b, with g = *global_scale (device fp32, > 0):
 *   s = E4M3_rn_satfinite((amax_b / 6) / g), q = E2M1_rn_satfinite(x / (E4M3(s) * g)),
 *   all codes 0 when s == 0; every step one IEEE fp32 round-to-nearest-even op.
 *   x        device bf16 [M, K] row-major, 16-byte aligned
 *   q_out    device u8 [M, K/2]
 *   sf_out   device u8, nvfp4_scale_bytes(M, K) bytes, tiled layout (padding written 0)
 * Bit-exact with the library's CPU oracle.
 */
int nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, const float* global_scale, uint8_t* q_out,
                   uint8_t* sf_out, void* stream);

/*
 * Dense NVFP4 GEMM, y = x @ W^T ("NVFP4 linear layer", kernelindex, operation header).
 *   a, sfa, ga   x: packed [M, K/2], tiled scales nvfp4_scale_bytes(M, K), fp32 global scale
 *   b, sfb, gb   W: packed [N, K/2], tiled scales nvfp4_scale_bytes(N, K), fp32 global scale
 *   y            bf16 [M, N] row-major, written
 *   workspace    may be NULL when nvfp4_gemm_workspace_bytes() returns 0 (it does today)
 * Small M (decode) runs a weight-streaming split-K kernel, large M a persistent
 * tcgen05 tile kernel; the result agrees with the oracle within
 * |y - y_ref| <= 4e-3 |y_ref| + 1e-5 sum_k |x^_k w^_k|.
 */
size_t nvfp4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
int nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b, const uint8_t* sfb,
               const float* gb, uint16_t* y, int64_t M, int64_t N, int64_t K, void* workspace,
               size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * NVFP4 GEMM whose epilogue emits NVFP4 instead of bf16: y = bf16(x^ . W^T^ * g_a * g_b)
 * as in nvfp4_gemm, then each 16-column block of y quantised with the caller's global
 * scale by the nvfp4_quantize recipe (the quantisation-overhead remark of "Blackwell
 * NVFP4 GEMM", What is this?: a layer chain otherwise re-reads y to quantise it).
 *   g_out    device fp32, decode-direction global scale of the output (for example from
 *            calibration, or nvfp4_amax of an earlier batch); blocks whose values exceed
 *            the range it allows saturate, as in nvfp4_quantize
 *   q_out    [M, N/2] packed E2M1 codes, written
 *   sf_out   nvfp4_scale_bytes(M, N) bytes in the 128 x 4 tiled layout, written
 *            (padding rows up to a multiple of 128 written as zero)
 * N must be a multiple of 64. Codes and scales equal nvfp4_quantize applied to the bf16
 * values nvfp4_gemm returns for the same operands (bit for bit).
 */
int nvfp4_gemm_quantize_out(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                            const uint8_t* sfb, const float* gb, const float* g_out, uint8_t* q_out, uint8_t* sf_out,
                            int64_t M, int64_t N, int64_t K, int32_t* dev_status, void* stream);

/*
 * Grouped (MoE) NVFP4 GEMM: for each expert e and each row m with
 * expert_offsets[e] <= m < expert_offsets[e+1], y[m, :] = x[m, :] @ W_e^T
 * ("The Moment of Synthesis", magik.net, Reasoning: grouped GEMM over the
 * per-expert GEMMs of ~16-32 tokens each).
 *   a, sfa, ga       routed tokens, rows sorted by expert: packed [M_total, K/2],
 *                    one tiled scale tensor over M_total rows, one global scale
 *   b, sfb, gb       expert weights: packed [E, N, K/2]; scales [E] x nvfp4_scale_bytes(N, K)
 *                    bytes back to back; gb device fp32 [E]
 *   expert_offsets   device int32 [E+1], 0 = offsets[0] <= ... <= offsets[E] = M_total;
 *                    checked on the device (NVFP4_ERR_BAD_OFFSETS in *dev_status, y untouched)
 *   y                bf16 [M_total, N], written
 *   workspace        device scratch of nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K)
 *                    bytes, 256-byte aligned, contents need no initialisation
 * Experts with no rows read none of their weights. Routing, the token gather
 * and the weighted combine are the caller's.
 */
size_t nvfp4_grouped_gemm_workspace_bytes(int32_t E, int64_t M_total, int64_t N, int64_t K);
int nvfp4_grouped_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                       const uint8_t* sfb, const float* gb, const int32_t* expert_offsets, int32_t E,
                       int64_t M_total, int64_t N, int64_t K, uint16_t* y, void* workspace,
                       size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * Grouped GEMM with the token gather fused into its load stage: routed row r (rows sorted
 * by expert as in nvfp4_grouped_gemm) multiplies token row_token[r] of the T-row
 * activations, so tokens are quantised once and never permuted in memory ("The Moment
 * of Synthesis", magik.net, Reasoning: top-8 routing sends each token to 8 experts).
 *   a_tok, sfa_tok   activations [T, K/2] and their tiled scales over T rows
 *   row_token        device int32 [M_total], values in [0, T); a value outside it is
 *                    reported as NVFP4_ERR_BAD_OFFSETS in *dev_status (its row's output is
 *                    then unspecified; nothing is read out of bounds)
 *   y                bf16 [M_total, N], routed-row order
 *   workspace        nvfp4_grouped_gemm_gather_workspace_bytes(E, M_total, N, K) bytes: the
 *                    preparation kernel then copies the routed rows out (M_total x K/2 bytes,
 *                    a few microseconds) and the GEMM reads them as plain tiles (fastest).
 *                    With only nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K) bytes the
 *                    GEMM's load stage fetches the rows itself with TMA tile::gather4 (four
 *                    token rows per instruction; no copy, more issue work per stage).
 * Other arguments as nvfp4_grouped_gemm. Either way the result equals nvfp4_grouped_gemm
 * on the gathered rows bit for bit.
 */
size_t nvfp4_grouped_gemm_gather_workspace_bytes(int32_t E, int64_t M_total, int64_t N, int64_t K);
int nvfp4_grouped_gemm_gather(const uint8_t* a_tok, const uint8_t* sfa_tok, const float* ga, const uint8_t* b,
                              const uint8_t* sfb, const float* gb, const int32_t* expert_offsets,
                              const int32_t* row_token, int32_t E, int64_t T, int64_t M_total, int64_t N, int64_t K,
                              uint16_t* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream);

/*
 * MoE gate/up projection with the SwiGLU activation fused into the epilogue:
 * y[m, c] = silu(gate[m, c]) * up[m, c], silu(v) = v / (1 + exp(-v)), where gate and
 * up are the grouped GEMM's outputs for expert e's weight rows 2c and 2c + 1
 * ("The Moment of Synthesis", magik.net, Reasoning: the per-expert N = 2048 x 2 fused
 * gate+up projection feeding a K = 2048 down projection). Arguments as
 * nvfp4_grouped_gemm with:
 *   b_gu, sfb_gu     packed [E, N_gu, K/2] with gate and up rows interleaved row by row
 *                    (row 2c gate row c, row 2c + 1 up row c; quantise the interleaved
 *                    matrix), scales of that matrix; N_gu = 2 I, a multiple of 8
 *   y                bf16 [M_total, N_gu / 2], written
 *   workspace        nvfp4_grouped_gemm_workspace_bytes(E, M_total, N_gu, K) bytes
 * The activation runs in fp32 on g_a * g_b * accumulator values before the one bf16
 * rounding of the product; the result agrees with the oracle within the bound the
 * GEMM tolerance of each factor implies:
 * (1 + 2^-8) (1.1 t_g (|u| + t_u) + |silu(g)| t_u) + 2^-8 |y|.
 */
int nvfp4_grouped_gemm_swiglu(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b_gu,
                              const uint8_t* sfb_gu, const float* gb, const int32_t* expert_offsets, int32_t E,
                              int64_t M_total, int64_t N_gu, int64_t K, uint16_t* y, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * The same gate/up projection with SwiGLU, emitting NVFP4 for the down projection instead
 * of bf16 ("The Moment of Synthesis", magik.net, Reasoning: the gate+up output feeds the
 * K = 2048 down-projection grouped GEMM). The epilogue forms each output's bf16 value exactly
 * as nvfp4_grouped_gemm_swiglu does and quantises it with the caller's global scale g_out
 * (a calibrated activation scale: a tensor-wide amax cannot exist before the outputs do)
 * by the recipe of nvfp4_quantize. So the codes and scales equal, bit for bit,
 * nvfp4_quantize(nvfp4_grouped_gemm_swiglu(...), g_out).
 *   g_out      device fp32 [1], decode-direction global scale of the output
 *   q_out      device u8 [M_total, N_gu / 4], packed E2M1 codes
 *   sf_out     device u8, nvfp4_scale_bytes(M_total, N_gu / 2) bytes, tiled E4M3 scales;
 *              the padding rows up to a multiple of 128 are written 0
 *   N_gu       a multiple of 128 (each epilogue warp then owns whole 16-element blocks)
 * Other arguments as nvfp4_grouped_gemm_swiglu (no y). Returns
 * NVFP4_ERR_UNSUPPORTED_SHAPE for N_gu not a multiple of 128, NVFP4_ERR_INVALID_ARG for a
 * null q_out, sf_out or g_out, otherwise as nvfp4_grouped_gemm.
 */
int nvfp4_grouped_gemm_swiglu_quantize_out(const uint8_t* a, const uint8_t* sfa, const float* ga,
                                           const uint8_t* b_gu, const uint8_t* sfb_gu, const float* gb,
                                           const int32_t* expert_offsets, int32_t E, int64_t M_total, int64_t N_gu,
                                           int64_t K, const float* g_out, uint8_t* q_out, uint8_t* sf_out,
                                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                           void* stream);

/*
 * Pair-wise 2:4 sparse NVFP4 ("FP4 structured sparsity", named as a kernel-level lever in
 * "The Moment of Recalibration", magik.net, The Broader Narrative Arc; the pages give no
 * format). The sparse block-scaled tensor-core MMA on FP4 keeps two of the four pairs of
 * neighbouring K elements in every group of 8 (4:8 pair-wise), reads one index nibble per
 * group and applies one scale per 32 K elements of each operand. Formats:
 *   - compressed weights c [N, K/2]: the kept pairs of each group in increasing index order,
 *     quantised as an ordinary NVFP4 tensor (nvfp4_amax + nvfp4_quantize over [N, K/2]:
 *     codes [N, K/4] bytes, 16-element-block scales nvfp4_scale_bytes(N, K/2));
 *   - metadata: per group the nibble i0 | i1 << 2 of the kept pair indices (i0 < i1), tiled
 *     per 128 rows x 512 K elements into 4096-byte tiles, row r's 32 bytes (groups 2b in the
 *     low nibble of byte b) at (r%128/8)*256 + (b/16)*128 + (r%8)*16 + b%16; padding zero;
 *     nvfp4_sparse_meta_bytes(N, K) bytes;
 *   - activations quantised with 32-element blocks (nvfp4_quantize_b32).
 * K must be a multiple of 128.
 */

/* Bytes of the tiled metadata of an [N, K] weight. */
int64_t nvfp4_sparse_meta_bytes(int64_t N, int64_t K);
/* Bytes of a tiled scale tensor with 32-element blocks: ceil(rows/128)*128 * ceil(K/128)*4. */
int64_t nvfp4_scale_bytes_b32(int64_t rows, int64_t K);

/*
 * Prunes and compresses a dense bf16 weight: in each group of 8 K elements the two pairs
 * with the largest |w_2j| + |w_2j+1| (one fp32 addition; ties to the lower pair index)
 * are kept. Bit-exact with the library's CPU oracle.
 *   w         device bf16 [N, K] row-major, 16-byte aligned
 *   c_out     device bf16 [N, K/2], written
 *   meta_out  device u8, nvfp4_sparse_meta_bytes(N, K) bytes, tiled as above, written
 */
int nvfp4_prune_pairs(const uint16_t* w, int64_t N, int64_t K, uint16_t* c_out, uint8_t* meta_out, void* stream);

/*
 * nvfp4_quantize with 32-element blocks (the activation operand of nvfp4_sparse_gemm):
 * s = E4M3_rn_satfinite((amax_32 / 6) / g), q = E2M1_rn_satfinite(x / (E4M3(s) * g)).
 *   q_out   [M, K/2]; sf_out nvfp4_scale_bytes_b32(M, K) bytes (128 x 4 tiles over K/32)
 * Bit-exact with the library's CPU oracle.
 */
int nvfp4_quantize_b32(const uint16_t* x, int64_t M, int64_t K, const float* global_scale, uint8_t* q_out,
                       uint8_t* sf_out, void* stream);

/*
 * y = x @ W^T with W pair-wise 2:4 sparse, on the sparse tensor cores (tcgen05.mma.sp).
 *   a, sfa, ga      x: packed [M, K/2], 32-element-block scales nvfp4_scale_bytes_b32(M, K)
 *   b_c, sfb_c, gb  compressed W: codes [N, K/4], scales nvfp4_scale_bytes(N, K/2), global scale
 *   meta            tiled metadata, nvfp4_sparse_meta_bytes(N, K) bytes
 *   y               bf16 [M, N], written
 * A weight-streaming kernel (the weights' bytes are 39 % fewer than dense NVFP4's); M above
 * 128 runs as one launch per 128 rows. The result agrees with the oracle within
 * |y - y_ref| <= 4e-3 |y_ref| + 1e-5 sum_k |x^_k w^_k|.
 */
int nvfp4_sparse_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b_c,
                      const uint8_t* sfb_c, const uint8_t* meta, const float* gb, uint16_t* y, int64_t M, int64_t N,
                      int64_t K, int32_t* dev_status, void* stream);

/*
 * Grouped (MoE) form of nvfp4_sparse_gemm: rows expert_offsets[e] .. expert_offsets[e+1]-1
 * of x (sorted by expert, quantised with nvfp4_quantize_b32 over the M_total rows) use
 * expert e's pair-wise 2:4 sparse weight. Experts with no rows read none of their bytes.
 *   b_c, sfb_c, gb   compressed experts: codes [E, N, K/4]; scales [E] x nvfp4_scale_bytes(N, K/2)
 *                    bytes back to back; gb device fp32 [E]
 *   meta             [E] x nvfp4_sparse_meta_bytes(N, K) bytes of tiled metadata, back to back
 *   workspace        nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K) bytes, 256-byte aligned
 * Other arguments and the device-side offset checks as nvfp4_grouped_gemm; K % 128 == 0.
 */
int nvfp4_grouped_sparse_gemm(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b_c,
                              const uint8_t* sfb_c, const uint8_t* meta, const float* gb,
                              const int32_t* expert_offsets, int32_t E, int64_t M_total, int64_t N, int64_t K,
                              uint16_t* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream);

/*
 * Allocation-free variant of nvfp4_grouped_gemm. The pages have no counterpart;
 * it exists for callers that cannot call cudaMalloc at the point where they run
 * the MoE layer: runtimes that hand kernels a fixed memory budget and offer no
 * allocator, and plugins or extensions that must not reach into the host
 * program's allocator (whose pools and bookkeeping they do not own).
 *
 * Same arguments and result as nvfp4_grouped_gemm, minus the workspace: the
 * scratch (tile list and per-tile activation scales) lives in one array of
 * NVFP4_NOALLOC_SCRATCH_BYTES (16 MiB) compiled into the library, present on
 * every device that loads the library until the process exits.
 *   - Returns NVFP4_ERR_WORKSPACE when nvfp4_grouped_gemm_workspace_bytes(E,
 *     M_total, N, K) exceeds NVFP4_NOALLOC_SCRATCH_BYTES (256 experts with 4096
 *     routed rows and K = 6144 need 15.0 MiB and fit).
 *   - The first call on a device looks up the array's device address with that
 *     device current (cudaGetSymbolAddress) and caches it; make that first call
 *     before any stream capture. Every call also makes the CUDA runtime calls
 *     nvfp4_grouped_gemm makes: cudaGetDevice, cudaGetLastError after each
 *     launch, the device-attribute queries of the first call on a device, and
 *     cudaFuncSetAttribute (maximum dynamic shared memory) at the first launch
 *     of each kernel variant on a device; none of them allocates.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents. The kernels write every scratch byte they read, so nothing needs
 *     clearing between calls, but calls that overlap on the GPU (unordered streams)
 *     race on it: order them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define NVFP4_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int nvfp4_grouped_gemm_noalloc(const uint8_t* a, const uint8_t* sfa, const float* ga, const uint8_t* b,
                               const uint8_t* sfb, const float* gb, const int32_t* expert_offsets, int32_t E,
                               int64_t M_total, int64_t N, int64_t K, uint16_t* y, int32_t* dev_status,
                               void* stream);

/*
 * Several independent decode-M GEMMs in one launch: y_g = x_g @ W_g^T for g < count, every
 * problem as nvfp4_gemm computes it ("NVFP4 linear layer", kernelindex, operation header),
 * sharing M (1..128, the decode range: the weight-streaming kernel) but with its own
 * operands, N and K. One launch streams all the weights, so the fixed costs of a decode
 * call (launch, first-load latency, split-K reduction, tail) are paid once and overlap
 * other problems' streaming, instead of once per GEMM ("The Moment of Recalibration", Input
 * Knowledge Required: decode-size GEMMs far below the part's rates). Each problem's outputs are
 * within the GEMM tolerance of the oracle; the split-K cluster size is chosen for the whole
 * launch, so a problem's result may differ in the last bf16 place from a single
 * nvfp4_gemm call of it (bit for bit equal when both use the same split).
 *   problems  host array [count], read during the call only; every pointer a device address
 *             as for nvfp4_gemm (a [M, K/2], sfa, ga [1], b [N, K/2], sfb, gb [1], y [M, N])
 *   count     1..NVFP4_MAX_BATCH
 * Returns NVFP4_ERR_INVALID_ARG (no problems, count out of range, M < 0, a null pointer),
 * NVFP4_ERR_UNSUPPORTED_SHAPE (M > 128, or a shape nvfp4_gemm rejects),
 * NVFP4_ERR_ALIGNMENT, or NVFP4_OK (nothing launched when M == 0). dev_status as for
 * nvfp4_gemm (NVFP4_ERR_TIMEOUT when a pipeline wait gave up).
 */
#define NVFP4_MAX_BATCH 8
typedef struct nvfp4_gemm_problem {
  const uint8_t* a;
  const uint8_t* sfa;
  const float* ga;
  const uint8_t* b;
  const uint8_t* sfb;
  const float* gb;
  uint16_t* y;
  int64_t N;
  int64_t K;
} nvfp4_gemm_problem;
int nvfp4_gemm_batched(const nvfp4_gemm_problem* problems, int32_t count, int64_t M, int32_t* dev_status,
                       void* stream);

/*
 * Elementwise device encoders used by the quantiser, for exhaustive checks:
 * fp32 -> E2M1 code (round to nearest even, saturating, sign kept) and
 * fp32 -> E4M3FN code (round to nearest even, saturating to +-448).
 *   v device fp32 [n]; out device u8 [n].
 */
int nvfp4_encode_e2m1(const float* v, int64_t n, uint8_t* out, void* stream);
int nvfp4_encode_e4m3(const float* v, int64_t n, uint8_t* out, void* stream);

/*
 * Process-wide tuning overrides (0 restores the automatic choice). Used by the
 * tests to force each kernel path and by benchmark sweeps. Not thread-safe with
 * concurrent GEMM calls.
 *   NVFP4_TUNE_DENSE_BN        dense tile width: 128 or 256
 *   NVFP4_TUNE_DENSE_GRID      persistent CTAs of the dense kernel
 *   NVFP4_TUNE_STREAM_MAX_M    largest M sent to the weight-streaming kernel (<= 128;
 *                              -1 sends every M to the tile kernel)
 *   NVFP4_TUNE_STREAM_SPLIT    split-K cluster size of the streaming kernel (1..8)
 *   NVFP4_TUNE_STREAM_STAGES   pipeline depth of the streaming kernel (2..16)
 *   NVFP4_TUNE_GROUPED_GRID    persistent CTAs of the grouped kernel
 *   NVFP4_TUNE_GROUPED_STAGES  pipeline depth of the grouped kernel (2..16)
 *   NVFP4_TUNE_DENSE_KERNEL    large-M kernel: 1 single-CTA 128 x BN tiles, 2 CTA-pair
 *                              256 x 256 tiles (the default)
 *   NVFP4_TUNE_PDL             programmatic dependent launch of the decode-M and grouped
 *                              kernels. 2 (and 0, the default): their set-up (barriers, TMEM,
 *                              descriptor prefetch) overlaps the tail of the previous kernel in
 *                              the stream; every memory access waits for that kernel to
 *                              complete, so stream order is kept in all cases. 1: in addition
 *                              the decode kernel requests its first weight tiles before that
 *                              wait; only valid when the previous kernel does not write the
 *                              weights (b, sfb) of the call (activations, scales and outputs
 *                              are still ordered after it). -1: plain stream order.
 *   NVFP4_TUNE_WEIGHT_L2       L2 residency of the weights (b, sfb) read by the decode-M and
 *                              grouped kernels. 0 (default): streamed, loaded with the
 *                              evict_first priority so a read-once matrix displaces nothing.
 *                              1: kept, loaded with the evict_last priority, so a matrix that
 *                              fits in L2 and is called again stays resident while other
 *                              weights stream past it (the "L2 cache pinning" of magik.net,
 *                              "The Moment of Recalibration", The Broader Narrative Arc). Lines
 *                              keep the priority they were last loaded with; a later call with
 *                              0 on the same matrix demotes them again. Results are unchanged.
 *   NVFP4_TUNE_DENSE_RASTER    order in which the persistent large-M kernels walk the output
 *                              tiles: 0 (default) m-blocks fastest, -1 n-blocks fastest, G > 0
 *                              bands of G m-blocks (m fastest inside a band). Results unchanged.
 *   NVFP4_TUNE_WATCHDOG_US     limit, in microseconds, after which a GEMM kernel's pipeline
 *                              wait gives up, stops the CTA's other roles, frees its tensor
 *                              memory and reports NVFP4_ERR_TIMEOUT in *dev_status (0: the
 *                              default, 2 s). Applies to the launches that follow.
 *   NVFP4_TUNE_STREAM_L2_PREFETCH  decode-M kernels: K blocks (of 256 K elements, 512 when
 *                              sparse) of each CTA's weight slice prefetched into L2 when the
 *                              CTA starts, ahead of the launch-dependency wait. 0 (default): as
 *                              many as keep the prefetches of all resident CTAs within 48 MB
 *                              of L2 (the whole slice for one N = K = 8192 call), none under
 *                              NVFP4_TUNE_PDL = 1 (the first ring is then requested early); -1: none;
 *                              k > 0: k blocks. A prefetch moves no data into the kernel, so
 *                              results and stream order are unchanged.
 *   NVFP4_TUNE_GROUPED_TILE_ROWS  token rows of one expert per grouped work item: 128 (the
 *                              default) or 64. An expert with r routed rows streams its weights
 *                              ceil(r / tile rows) times. Results are unchanged.
 *   NVFP4_TUNE_TEST_WITHHOLD_STAGE  test hook for the timeout path: k >= 1 makes the first CTA
 *                              of each GEMM kernel withhold the loads of the k-th pipeline stage
 *                              it would request, so that stage never arrives and the waits run
 *                              into the watchdog (the result is then unspecified). 0: off.
 * Returns NVFP4_OK or NVFP4_ERR_INVALID_ARG.
 */
enum {
  NVFP4_TUNE_DENSE_BN = 1,
  NVFP4_TUNE_DENSE_GRID = 2,
  NVFP4_TUNE_STREAM_MAX_M = 3,
  NVFP4_TUNE_STREAM_SPLIT = 4,
  NVFP4_TUNE_STREAM_STAGES = 5,
  NVFP4_TUNE_GROUPED_GRID = 6,
  NVFP4_TUNE_GROUPED_STAGES = 7,
  NVFP4_TUNE_DENSE_KERNEL = 8,
  NVFP4_TUNE_PDL = 9,
  NVFP4_TUNE_WEIGHT_L2 = 10,
  NVFP4_TUNE_DENSE_RASTER = 11,
  NVFP4_TUNE_WATCHDOG_US = 12,
  NVFP4_TUNE_TEST_WITHHOLD_STAGE = 13,
  NVFP4_TUNE_STREAM_L2_PREFETCH = 14,
  NVFP4_TUNE_GROUPED_TILE_ROWS = 15
};
int nvfp4_tune(int key, int value);

/* Number of kernel launches the last GEMM / grouped GEMM / quantize / amax call
 * on this host thread enqueued (for launch accounting in benchmarks). */
int nvfp4_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */
