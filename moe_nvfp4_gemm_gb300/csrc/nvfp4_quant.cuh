// The NVFP4 block-quantisation recipe as device functions, shared by the stand-alone
// quantiser (quantize.cu) and the GEMM epilogue that emits NVFP4 (gemm_dense.cu), so
// that both produce identical codes and scales from identical bf16 inputs.
//
// Formats: "NVFP4 linear layer" (kernelindex, operation header) - FP4 values
// with FP8 E4M3FN scales, one per 16 elements; "The 3.7 PFLOPS Revelation"
// (magik.net, Input Knowledge item 2) - two FP4 values per byte.
// Recipe (the pages fix none; this is the library's stated reading):
//   s = E4M3_rn_sat((amax_blk / 6) / g);  q = E2M1_rn_sat(x / (E4M3(s) * g)), sign kept;
//   q = 0 when s == 0. Every float step is one IEEE round-to-nearest operation.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace nvfp4 {

DEVI uint32_t e4m3_encode(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  return r & 0xFFu;
}

DEVI float e4m3_decode(uint32_t code) {
  uint32_t h2;
  uint16_t in = static_cast<uint16_t>(code & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Two E2M1 codes in one byte: `lo` in bits 0-3, `hi` in bits 4-7.
DEVI uint32_t e2m1x2_encode(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

DEVI float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
DEVI float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed pair of fp32 (Blackwell's f32x2 datapath: two IEEE round-to-nearest
// operations per instruction, lane by lane).
DEVI uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
DEVI void f2_split(uint64_t v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
DEVI uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
DEVI uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// v with the sign bit of x: the quotient of a nonzero x already has x's sign, and a
// zero x (either sign) must keep its own (the correction step below yields +0 for -0).
DEVI float with_sign_of(float v, float x) {
  return __uint_as_float((__float_as_uint(v) & 0x7FFFFFFFu) | (__float_as_uint(x) & 0x80000000u));
}
// Eight E2M1 codes, element 2j in the low nibble of byte j.
DEVI uint32_t e2m1x8_encode(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Correctly rounded x / d without a division instruction, given y = RN(1 / d):
//   q0 = RN(x y);  q1 = RN(q0 + RN(x - q0 d) y);  q2 = RN(q1 + (x - q1 d) y)  (fma each).
// Why q2 = RN(x / d), with u = 2^-24 and no over- or underflow:
//   y = (1 + h) / d and q0 = (x / d)(1 + e), |h| <= u, |e| <= 2u + u^2. The remainder's exact
//   value is -x e; its rounding adds (1 + r), |r| <= u. So q0 + RN(x - q0 d) y =
//   (x / d)(1 - e (r + h + r h)), within 5 u^2 relative of x / d, and q1, its rounding, is
//   within half an ulp plus 5 u^2 of x / d: one of the two floats around it (faithful).
//   For a faithful q1 the remainder x - q1 d is a float (one fma computes it exactly), and
//   Markstein's theorem (P. Markstein, "Computation of elementary functions on the IBM
//   RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990: a faithful quotient and a
//   reciprocal within half an ulp give the correctly rounded quotient after one such
//   correction) makes q2 = RN(x / d).
// One correction alone is not enough: q0 itself can be two ulps off when the quotient's
// significand is close to 2, and then the theorem does not apply.
// Range: x, the quotient and d in [1e-30, 1e30] in magnitude keep d, y and every quotient
// normal and the remainders representable: x - q d is a multiple of ulp(q) ulp(d) >=
// 2^(e - 47) for 2^e <= |x| < 2^(e+1), hence of 2^-149 once |x| >= 2^-102 (~2e-31), so
// even a subnormal remainder is exact. Elsewhere the IEEE division.
DEVI float div_rn_by(float x, float d, float y) {
  const float q0 = __fmul_rn(x, y);
  const float ax = fabsf(x), aq = fabsf(q0);
  if (!(ax >= 1e-30f && ax <= 1e30f && aq >= 1e-30f && aq <= 1e30f && d >= 1e-30f && d <= 1e30f))
    return __fdiv_rn(x, d);
  const float q1 = __fmaf_rn(__fmaf_rn(-q0, d, x), y, q0);
  return __fmaf_rn(__fmaf_rn(-q1, d, x), y, q1);
}

// Largest |x| of 16 bf16 values (8 packed pairs), exact.
DEVI float block_amax16(const uint32_t (&w)[8]) {
  // |x| of both halves at once (sign bits cleared), maximum on the bf16 pairs (exact)
  uint32_t m2 = w[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int j = 1; j < 8; ++j) asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(w[j] & 0x7FFF7FFFu));
  return fmaxf(bf16lo(m2), bf16hi(m2));
}

// E4M3 code of a block with maximum |x| amax: E4M3_rn_sat(RN(RN(amax / 6) / g)); g_inv = RN(1 / g).
DEVI uint32_t block_scale_code(float amax, float g, float g_inv) {
  // 0x3e2aaaab = RN(1 / 6)
  const float t = amax == 0.0f ? 0.0f : div_rn_by(div_rn_by(amax, 6.0f, __uint_as_float(0x3e2aaaabu)), g, g_inv);
  return e4m3_encode(t);
}

// E2M1 codes of 16 bf16 values (8 packed pairs) with block scale code s (0: all codes 0);
// amax is the largest |x| of the block the scale belongs to (it bounds the quotients).
DEVI uint2 block_codes16(const uint32_t (&w)[8], uint32_t s, float g, float amax) {
  uint32_t packed[2] = {0u, 0u};
  if (s != 0) {
    const float d = __fmul_rn(e4m3_decode(s), g);
    // x / d correctly rounded without a division per element, by the two corrections of
    // div_rn_by, two elements per instruction. The block-wide guard bounds d and the
    // largest quotient; an element with |x| < 2^-102 or a quotient below 2^-126 may lose
    // exactness, but its quotient is then below 2^-102 / 1e-30 < 0.2 (or 2^-126), so its
    // code is 0 (with x's sign, restored below) whatever the rounding. Blocks outside the
    // guard take IEEE division.
    const float y = __frcp_rn(d);
    const bool fast = d > 1e-30f && d < 1e30f && __fmul_rn(amax, y) < 1e30f;
    const uint64_t yy = f2(y, y), nd = f2(-d, -d);
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // eight elements (one output word) at a time
      float v[8];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float lo = bf16lo(w[h * 4 + jj]), hi = bf16hi(w[h * 4 + jj]);
        if (fast) {
          const uint64_t xx = f2(lo, hi);
          const uint64_t q0 = f2_mul(xx, yy);
          const uint64_t q1 = f2_fma(f2_fma(q0, nd, xx), yy, q0);  // faithful
          const uint64_t rem = f2_fma(q1, nd, xx);                  // x - q1 d, exact
          f2_split(f2_fma(rem, yy, q1), v[2 * jj], v[2 * jj + 1]);
          v[2 * jj] = with_sign_of(v[2 * jj], lo);
          v[2 * jj + 1] = with_sign_of(v[2 * jj + 1], hi);
        } else {
          v[2 * jj] = __fdiv_rn(lo, d);
          v[2 * jj + 1] = __fdiv_rn(hi, d);
        }
      }
      packed[h] = e2m1x8_encode(v);
    }
  }
  return make_uint2(packed[0], packed[1]);
}

// One 16-element block: scale code s and 8 bytes of packed codes. g_inv = RN(1 / g),
// computed once per thread.
DEVI void quantize_block(const uint32_t (&w)[8], float g, float g_inv, uint32_t& s, uint2& packed_out) {
  const float amax = block_amax16(w);
  s = block_scale_code(amax, g, g_inv);
  packed_out = block_codes16(w, s, g, amax);
}

// One 32-element block (the dense operand of the pair-wise sparse GEMM): one scale from the
// amax of all 32 values, then the codes of both halves with it.
DEVI void quantize_block32(const uint32_t (&w0)[8], const uint32_t (&w1)[8], float g, float g_inv, uint32_t& s,
                           uint2& p0, uint2& p1) {
  const float amax = fmaxf(block_amax16(w0), block_amax16(w1));
  s = block_scale_code(amax, g, g_inv);
  p0 = block_codes16(w0, s, g, amax);
  p1 = block_codes16(w1, s, g, amax);
}

}  // namespace nvfp4
