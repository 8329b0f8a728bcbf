/*
 * NVFP4 oracle: a plain, slow CPU statement of what the NVFP4 path computes.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library calls this code; it is
 * loaded by the tests, by __graft_entry__.smoke() and by bench.py's CPU
 * baseline leg, and by nothing else. It shares no code with the CUDA path.
 *
 * What it follows (the pages are cited by title and section):
 *  - "NVFP4 linear layer" (kernelindex, operation header): y = x . W^T, x and W
 *    FP4 (E2M1) with FP8 E4M3FN scale factors, one per 16 consecutive elements
 *    (sf_vec_size = 16, sf_k = K/16, in_features_half = K/2).
 *  - "The 3.7 PFLOPS Revelation" (magik.net, Input Knowledge item 2): two FP4
 *    values per byte, data tensors [rows, K/2], scale tensors [rows, K/16].
 *  - The per-tensor FP32 global scale, the quantisation recipe and the 128x4
 *    scale tile layout are not on the pages; the readings taken are:
 *      g = amax / (6 * 448) (1.0 when amax == 0), decode direction;
 *      s = E4M3_rne_satfinite((amax_block / 6) / g), fp32 divisions in that order;
 *      q = E2M1_rne_satfinite(x / (E4M3(s) * g)), fp32, sign kept; all-zero
 *          codes when s == 0;
 *      low nibble holds the even K element;
 *      scale (r, c) lives at ((r/128)*(Kc4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4,
 *          Kc4 = ceil(Kc/4), padding bytes 0.
 *  - GEMM reference: the sum over k of the fully decoded products in float64,
 *    times g_a * g_b; an exact integer mode (every decoded product is an
 *    integer multiple of 2^-20) pins it.
 *
 * Every float32 step is written as a separate C float operation; this file is
 * compiled with -ffp-contract=off and without fast-math so that each one is a
 * single IEEE round-to-nearest-even operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- value tables (format definitions) ---------------------------------- */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0. */
double nvo_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* E4M3FN: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0; no
 * infinities; S.1111.111 is NaN; exponent 0 is subnormal (m/8) * 2^-6. */
double nvo_e4m3_value(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Nearest of the ascending magnitudes mags[0..n-1] (code i has magnitude
 * mags[i]); a tie goes to the even code; a >= mags[n-1] saturates. a >= 0. */
static int nearest_code(double a, const double* mags, int n) {
  if (a >= mags[n - 1]) return n - 1;
  int lo = 0;
  while (lo + 1 < n && mags[lo + 1] <= a) lo++;
  if (mags[lo] == a) return lo;
  double dl = a - mags[lo], dh = mags[lo + 1] - a; /* exact: both are short dyadics */
  if (dl < dh) return lo;
  if (dh < dl) return lo + 1;
  return (lo & 1) ? lo + 1 : lo;
}

static double g_e2m1_mag[8];
static double g_e4m3_mag[127];
static int g_tables_ready = 0;

static void init_tables(void) {
  if (g_tables_ready) return;
  for (int i = 0; i < 8; i++) g_e2m1_mag[i] = nvo_e2m1_value(i);
  for (int i = 0; i < 127; i++) g_e4m3_mag[i] = nvo_e4m3_value(i);
  g_tables_ready = 1;
}

/* E2M1 round-to-nearest-even, saturating to +-6, sign kept (so -0.1 -> 0x8). */
int nvo_e2m1_encode(float v) {
  init_tables();
  int sign = signbit(v) ? 8 : 0;
  return sign | nearest_code(fabs((double)v), g_e2m1_mag, 8);
}

/* E4M3FN round-to-nearest-even, saturating to +-448 (0x7E / 0xFE). */
int nvo_e4m3_encode(float t) {
  init_tables();
  int sign = signbit(t) ? 0x80 : 0;
  return sign | nearest_code(fabs((double)t), g_e4m3_mag, 127);
}

/* Array forms of the two encoders (used by the exhaustive format tests). */
void nvo_e2m1_encode_n(const float* v, int64_t n, uint8_t* out) {
  init_tables();
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)nvo_e2m1_encode(v[i]);
}

void nvo_e4m3_encode_n(const float* v, int64_t n, uint8_t* out) {
  init_tables();
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)nvo_e4m3_encode(v[i]);
}

/* ---- layouts ------------------------------------------------------------- */

static inline float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

int64_t nvo_scale_bytes(int64_t rows, int64_t K) {
  int64_t kc = K / 16;
  return ((rows + 127) / 128) * 128 * (((kc + 3) / 4) * 4);
}

/* Byte offset of scale (row r, scale column c) in the tiled scale tensor. */
int64_t nvo_sf_offset(int64_t r, int64_t c, int64_t K) {
  int64_t kc4 = (K / 16 + 3) / 4;
  return ((r / 128) * kc4 + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* Tiled scale tensor -> linear [rows, K/16] and back. */
void nvo_sf_unswizzle(const uint8_t* sf, int64_t rows, int64_t K, uint8_t* lin) {
  int64_t kc = K / 16;
  for (int64_t r = 0; r < rows; r++)
    for (int64_t c = 0; c < kc; c++) lin[r * kc + c] = sf[nvo_sf_offset(r, c, K)];
}

void nvo_sf_swizzle(const uint8_t* lin, int64_t rows, int64_t K, uint8_t* sf) {
  int64_t kc = K / 16;
  memset(sf, 0, (size_t)nvo_scale_bytes(rows, K));
  for (int64_t r = 0; r < rows; r++)
    for (int64_t c = 0; c < kc; c++) sf[nvo_sf_offset(r, c, K)] = lin[r * kc + c];
}

/* ---- quantisation -------------------------------------------------------- */

float nvo_amax_bf16(const uint16_t* x, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; i++) {
    float a = fabsf(bf16_to_f32(x[i]));
    if (a > m) m = a;
  }
  return m;
}

float nvo_global_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  return amax / 2688.0f; /* 6 * 448 */
}

/* x: bf16 [M, K] row-major. q: [M, K/2]. sf: nvo_scale_bytes(M, K) bytes. */
void nvo_quantize(const uint16_t* x, int64_t M, int64_t K, float g, uint8_t* q, uint8_t* sf) {
  init_tables();
  memset(sf, 0, (size_t)nvo_scale_bytes(M, K));
  int64_t kc = K / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < M; r++) {
    for (int64_t c = 0; c < kc; c++) {
      const uint16_t* blk = x + r * K + c * 16;
      float amax = 0.0f;
      for (int i = 0; i < 16; i++) {
        float a = fabsf(bf16_to_f32(blk[i]));
        if (a > amax) amax = a;
      }
      float t1 = amax / 6.0f;
      float t = t1 / g;
      int s = nvo_e4m3_encode(t) & 0x7F;
      uint8_t codes[16];
      if (s == 0) {
        memset(codes, 0, 16);
      } else {
        float dec = (float)nvo_e4m3_value(s);
        float d = dec * g;
        for (int i = 0; i < 16; i++) {
          float v = bf16_to_f32(blk[i]) / d;
          codes[i] = (uint8_t)nvo_e2m1_encode(v);
        }
      }
      for (int j = 0; j < 8; j++)
        q[r * (K / 2) + c * 8 + j] = (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
      sf[nvo_sf_offset(r, c, K)] = (uint8_t)s;
    }
  }
}

/* Fully decoded row: out[k] = E2M1(code k) * E4M3(scale k/16), float64. */
static void decode_row(const uint8_t* q, const uint8_t* sf, int64_t r, int64_t K, double* out) {
  for (int64_t k = 0; k < K; k++) {
    uint8_t byte = q[r * (K / 2) + k / 2];
    int code = (k & 1) ? (byte >> 4) : (byte & 15);
    out[k] = nvo_e2m1_value(code) * nvo_e4m3_value(sf[nvo_sf_offset(r, k / 16, K)]);
  }
}

void nvo_dequantize(const uint8_t* q, const uint8_t* sf, float g, int64_t rows, int64_t K,
                    double* out) {
  for (int64_t r = 0; r < rows; r++) {
    decode_row(q, sf, r, K, out + r * K);
    for (int64_t k = 0; k < K; k++) out[r * K + k] *= (double)g;
  }
}

/* ---- GEMM ----------------------------------------------------------------- */

/*
 * y[i, j] = (sum_k A^[rows[i], k] * B^[cols[j], k]) * ga * gb, float64, where ^
 * means the decoded value E2M1 * E4M3 (global scales excluded inside the sum).
 * absdot[i, j] = sum_k |A^ B^| * |ga * gb| (the tolerance's magnitude term).
 * rows / cols may be NULL (all rows of A / all rows of B).
 */
void nvo_gemm_f64(const uint8_t* a, const uint8_t* sfa, float ga, const uint8_t* b,
                  const uint8_t* sfb, float gb, int64_t M, int64_t N, int64_t K,
                  const int64_t* rows, int64_t nr, const int64_t* cols, int64_t nc, double* y,
                  double* absdot) {
  init_tables();
  if (!rows) nr = M;
  if (!cols) nc = N;
  double* bd = (double*)malloc(sizeof(double) * (size_t)nc * (size_t)K);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nc; j++) decode_row(b, sfb, cols ? cols[j] : j, K, bd + j * K);
#pragma omp parallel
  {
    double* ad = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < nr; i++) {
      decode_row(a, sfa, rows ? rows[i] : i, K, ad);
      for (int64_t j = 0; j < nc; j++) {
        double s = 0.0, sa = 0.0;
        const double* bj = bd + j * K;
        for (int64_t k = 0; k < K; k++) {
          double p = ad[k] * bj[k];
          s += p;
          sa += fabs(p);
        }
        y[i * nc + j] = s * (double)ga * (double)gb;
        if (absdot) absdot[i * nc + j] = sa * fabs((double)ga * (double)gb);
      }
    }
    free(ad);
  }
  free(bd);
}

/* Integer forms: E2M1 value = e2 / 2, E4M3 value = s9 * 2^-9 (finite codes). */
static int e2m1_twice(int code) {
  static const int mag2[8] = {0, 1, 2, 3, 4, 6, 8, 12};
  return (code & 8) ? -mag2[code & 7] : mag2[code & 7];
}

static int64_t e4m3_times_512(int code, int* nan_flag) {
  int e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) {
    *nan_flag = 1;
    return 0;
  }
  int64_t mag = (e == 0) ? m : ((int64_t)(8 + m) << (e - 1));
  return (code & 0x80) ? -mag : mag;
}

/*
 * Exact mode: S[i, j] = sum_k e2(a) * s9(sa) * e2(b) * s9(sb) as a 128-bit
 * integer (so the real sum is S * 2^-20), returned as hi (signed) / lo words.
 * Returns 1 if a NaN scale code was met, else 0.
 */
int nvo_gemm_exact(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                   int64_t M, int64_t N, int64_t K, int64_t* hi, uint64_t* lo) {
  int nan_flag = 0;
  for (int64_t i = 0; i < M; i++) {
    for (int64_t j = 0; j < N; j++) {
      __int128 s = 0;
      for (int64_t k = 0; k < K; k++) {
        uint8_t ab = a[i * (K / 2) + k / 2], bb = b[j * (K / 2) + k / 2];
        int ca = (k & 1) ? (ab >> 4) : (ab & 15), cb = (k & 1) ? (bb >> 4) : (bb & 15);
        int64_t xa = e2m1_twice(ca) * e4m3_times_512(sfa[nvo_sf_offset(i, k / 16, K)], &nan_flag);
        int64_t xb = e2m1_twice(cb) * e4m3_times_512(sfb[nvo_sf_offset(j, k / 16, K)], &nan_flag);
        s += (__int128)xa * (__int128)xb;
      }
      hi[i * N + j] = (int64_t)(s >> 64);
      lo[i * N + j] = (uint64_t)s;
    }
  }
  return nan_flag;
}

/*
 * Grouped: rows offsets[e] .. offsets[e+1]-1 of a use expert e's weights
 * b + e*N*K/2, scales sfb + e*nvo_scale_bytes(N, K), global scale gb[e].
 * rows (indices into 0..M_total-1) may be NULL for all rows; cols likewise.
 * Returns 1 if the offsets are malformed (not monotone from 0 to M_total).
 */
int nvo_grouped_gemm_f64(const uint8_t* a, const uint8_t* sfa, float ga, const uint8_t* b,
                         const uint8_t* sfb, const float* gb, const int32_t* offsets, int32_t E,
                         int64_t M_total, int64_t N, int64_t K, const int64_t* rows, int64_t nr,
                         const int64_t* cols, int64_t nc, double* y, double* absdot) {
  if (offsets[0] != 0 || offsets[E] != M_total) return 1;
  for (int32_t e = 0; e < E; e++)
    if (offsets[e + 1] < offsets[e]) return 1;
  if (!rows) nr = M_total;
  if (!cols) nc = N;
  int64_t wbytes = N * (K / 2), sbytes = nvo_scale_bytes(N, K);
  int64_t* pick = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nr > 0 ? nr : 1));
  int64_t* where = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nr > 0 ? nr : 1));
  double* ty = (double*)malloc(sizeof(double) * (size_t)(nr > 0 ? nr : 1) * (size_t)nc);
  double* ta = (double*)malloc(sizeof(double) * (size_t)(nr > 0 ? nr : 1) * (size_t)nc);
  for (int32_t e = 0; e < E; e++) {
    int64_t cnt = 0;
    for (int64_t i = 0; i < nr; i++) {
      int64_t m = rows ? rows[i] : i;
      if (offsets[e] <= m && m < offsets[e + 1]) {
        pick[cnt] = m;
        where[cnt] = i;
        cnt++;
      }
    }
    if (cnt == 0) continue;
    nvo_gemm_f64(a, sfa, ga, b + e * wbytes, sfb + e * sbytes, gb[e], M_total, N, K, pick, cnt,
                 cols, nc, ty, ta);
    for (int64_t t = 0; t < cnt; t++) {
      memcpy(y + where[t] * nc, ty + t * nc, sizeof(double) * (size_t)nc);
      if (absdot) memcpy(absdot + where[t] * nc, ta + t * nc, sizeof(double) * (size_t)nc);
    }
  }
  free(pick);
  free(where);
  free(ty);
  free(ta);
  return 0;
}

/* ---- pair-wise 2:4 sparsity (weights) ---------------------------------------
 *
 * The structured sparsity of the sparse tensor-core MMA on FP4 data: in every group of
 * 8 consecutive K elements (4 pairs of neighbours 2j, 2j+1) two pairs are kept ("FP4
 * structured sparsity", "The Moment of Recalibration", The Broader Narrative Arc; the
 * pages give no format, the readings are the library's):
 *   - pruning of a dense bf16 W: keep the two pairs with the largest score
 *     |w_2j| + |w_2j+1| (one fp32 addition), a tie going to the lower pair index;
 *   - compression: the kept pairs in increasing index order, [N, K/2] values;
 *   - metadata: per group the nibble i0 | i1 << 2 (i0 < i1, the kept pair indices);
 *     byte b of a row holds groups 2b (low nibble) and 2b + 1, [N, K/16] bytes;
 *   - the compressed values are quantised as an ordinary [N, K/2] NVFP4 tensor
 *     (16-element blocks over stored values = 32 logical K elements);
 *   - the dense operand (activations) carries one scale per 32 K elements.
 */

static void top2_pairs(const uint16_t* grp, int* i0, int* i1) {
  float sc[4];
  for (int j = 0; j < 4; j++) sc[j] = fabsf(bf16_to_f32(grp[2 * j])) + fabsf(bf16_to_f32(grp[2 * j + 1]));
  int best = 0;
  for (int j = 1; j < 4; j++)
    if (sc[j] > sc[best]) best = j;
  int second = -1;
  for (int j = 0; j < 4; j++)
    if (j != best && (second < 0 || sc[j] > sc[second])) second = j;
  *i0 = best < second ? best : second;
  *i1 = best < second ? second : best;
}

/* w: bf16 [N, K] (K % 8 == 0). c: bf16 [N, K/2]. meta: [N, K/16] bytes. */
void nvo_prune_pairs(const uint16_t* w, int64_t N, int64_t K, uint16_t* c, uint8_t* meta) {
  memset(meta, 0, (size_t)(N * (K / 16)));
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; n++)
    for (int64_t g = 0; g < K / 8; g++) {
      const uint16_t* grp = w + n * K + g * 8;
      int i0, i1;
      top2_pairs(grp, &i0, &i1);
      uint16_t* out = c + n * (K / 2) + g * 4;
      out[0] = grp[2 * i0];
      out[1] = grp[2 * i0 + 1];
      out[2] = grp[2 * i1];
      out[3] = grp[2 * i1 + 1];
      meta[n * (K / 16) + g / 2] |= (uint8_t)((i0 | (i1 << 2)) << (4 * (g & 1)));
    }
}

/* Tiled metadata: per 128 rows and 512 K elements (32 bytes a row) one 4096-byte tile,
 * rows in groups of 8 with each row's 32 bytes as two 16-byte halves:
 * byte b of row r at (r%128/8)*256 + (b/16)*128 + (r%8)*16 + b%16. */
int64_t nvo_meta_tiled_bytes(int64_t N, int64_t K) { return (N + 127) / 128 * ((K + 511) / 512) * 4096; }

int64_t nvo_meta_offset(int64_t n, int64_t b, int64_t K) {
  int64_t kmc = (K + 511) / 512, r = n % 128, bb = b % 32;
  return ((n / 128) * kmc + b / 32) * 4096 + (r / 8) * 256 + (bb / 16) * 128 + (r % 8) * 16 + bb % 16;
}

void nvo_meta_tile(const uint8_t* lin, int64_t N, int64_t K, uint8_t* tiled) {
  memset(tiled, 0, (size_t)nvo_meta_tiled_bytes(N, K));
  for (int64_t n = 0; n < N; n++)
    for (int64_t b = 0; b < K / 16; b++) tiled[nvo_meta_offset(n, b, K)] = lin[n * (K / 16) + b];
}

void nvo_meta_untile(const uint8_t* tiled, int64_t N, int64_t K, uint8_t* lin) {
  for (int64_t n = 0; n < N; n++)
    for (int64_t b = 0; b < K / 16; b++) lin[n * (K / 16) + b] = tiled[nvo_meta_offset(n, b, K)];
}

/* Scale tensors with `bs`-element blocks (16 or 32): the same 128 x 4 tiles over K/bs columns. */
int64_t nvo_scale_bytes_bs(int64_t rows, int64_t K, int64_t bs) {
  int64_t kc = K / bs;
  return ((rows + 127) / 128) * 128 * (((kc + 3) / 4) * 4);
}

static int64_t sf_offset_bs(int64_t r, int64_t c, int64_t K, int64_t bs) {
  int64_t kc4 = (K / bs + 3) / 4;
  return ((r / 128) * kc4 + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* The quantisation recipe of nvo_quantize with 32-element blocks. */
void nvo_quantize_b32(const uint16_t* x, int64_t M, int64_t K, float g, uint8_t* q, uint8_t* sf) {
  init_tables();
  memset(sf, 0, (size_t)nvo_scale_bytes_bs(M, K, 32));
  int64_t kc = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < M; r++) {
    for (int64_t c = 0; c < kc; c++) {
      const uint16_t* blk = x + r * K + c * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; i++) {
        float a = fabsf(bf16_to_f32(blk[i]));
        if (a > amax) amax = a;
      }
      float t1 = amax / 6.0f;
      float t = t1 / g;
      int s = nvo_e4m3_encode(t) & 0x7F;
      uint8_t codes[32];
      if (s == 0) {
        memset(codes, 0, 32);
      } else {
        float dec = (float)nvo_e4m3_value(s);
        float d = dec * g;
        for (int i = 0; i < 32; i++) {
          float v = bf16_to_f32(blk[i]) / d;
          codes[i] = (uint8_t)nvo_e2m1_encode(v);
        }
      }
      for (int j = 0; j < 16; j++)
        q[r * (K / 2) + c * 16 + j] = (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
      sf[sf_offset_bs(r, c, K, 32)] = (uint8_t)s;
    }
  }
}

/* Decoded logical row of a compressed sparse weight: zeros at pruned positions,
 * kept element k = E2M1(stored code) * E4M3(scale of its 16-element stored block). */
static void decode_sparse_row(const uint8_t* cq, const uint8_t* csf, const uint8_t* meta, int64_t n, int64_t K,
                              double* out) {
  const int64_t Ks = K / 2;
  for (int64_t k = 0; k < K; k++) out[k] = 0.0;
  for (int64_t g = 0; g < K / 8; g++) {
    int nib = (meta[n * (K / 16) + g / 2] >> (4 * (g & 1))) & 15;
    int pi[2] = {nib & 3, nib >> 2};
    for (int h = 0; h < 2; h++)
      for (int e = 0; e < 2; e++) {
        int64_t st = 4 * g + 2 * h + e;                 /* stored index */
        int64_t k = 8 * g + 2 * pi[h] + e;              /* its logical K position */
        uint8_t byte = cq[n * (Ks / 2) + st / 2];
        int code = (st & 1) ? (byte >> 4) : (byte & 15);
        out[k] = nvo_e2m1_value(code) * nvo_e4m3_value(csf[sf_offset_bs(n, st / 16, Ks, 16)]);
      }
  }
}

/*
 * Sparse GEMM: y[i, j] = (sum_k X^[rows[i], k] * W^[cols[j], k]) * gx * gw in float64, X^
 * decoded with 32-element blocks (scales xsf), W^ the decoded logical weight (cq [N, K/4]
 * bytes of compressed codes, csf its 16-element-block scales over K/2, meta [N, K/16]).
 * absdot as in nvo_gemm_f64.
 */
void nvo_sparse_gemm_f64(const uint8_t* xq, const uint8_t* xsf, float gx, const uint8_t* cq, const uint8_t* csf,
                         const uint8_t* meta, float gw, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                         int64_t nr, const int64_t* cols, int64_t nc, double* y, double* absdot) {
  init_tables();
  if (!rows) nr = M;
  if (!cols) nc = N;
  double* wd = (double*)malloc(sizeof(double) * (size_t)nc * (size_t)K);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nc; j++) decode_sparse_row(cq, csf, meta, cols ? cols[j] : j, K, wd + j * K);
#pragma omp parallel
  {
    double* xd = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < nr; i++) {
      int64_t m = rows ? rows[i] : i;
      for (int64_t k = 0; k < K; k++) {
        uint8_t byte = xq[m * (K / 2) + k / 2];
        int code = (k & 1) ? (byte >> 4) : (byte & 15);
        xd[k] = nvo_e2m1_value(code) * nvo_e4m3_value(xsf[sf_offset_bs(m, k / 32, K, 32)]);
      }
      for (int64_t j = 0; j < nc; j++) {
        double s = 0.0, sa = 0.0;
        const double* wj = wd + j * K;
        for (int64_t k = 0; k < K; k++) {
          double p = xd[k] * wj[k];
          s += p;
          sa += fabs(p);
        }
        y[i * nc + j] = s * (double)gx * (double)gw;
        if (absdot) absdot[i * nc + j] = sa * fabs((double)gx * (double)gw);
      }
    }
    free(xd);
  }
  free(wd);
}

int nvo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
