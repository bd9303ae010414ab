// f16 operands for the tensor-core routes that round a weight (the 4-bit
// prefill and MUL_MAT_ID, and the Q8 route above the decode sizes).
//
// A weight w = q * s + m is formed once in f16: one round-to-nearest-even,
// so |w16 - w| <= 2^-11 |w| while |w| lies in f16's normal range.  The
// tensor cores' kind::f16 MMA takes A and B of one type, so the activations
// are f16 too.  bf16 activations have f16's precision (8 significant bits
// fit in 11) but not its range, so each activation row is first multiplied
// by a power of two that puts its largest magnitude in [2^14, 2^15):
//   * no scaled value can overflow f16 (whose largest finite value is 65504);
//   * a bf16 value is exact in f16 whenever its scaled magnitude is at least
//     2^-17 (its 8 significant bits then sit on f16's grid), which holds for
//     every element within a factor 2^31 of its row's largest one;
//   * the row's results are multiplied back by the inverse power of two,
//     which is exact in fp32.
// Products of two f16 values are exact in fp32 (22 significant bits), so the
// only other error is the fp32 accumulation.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qmm_device.cuh"

namespace qmm {

// Largest f16 magnitude: a weight block whose |m| + 15|s| (or 127|s| for
// 8-bit codes) exceeds it cannot be formed in f16, and the call reports
// QMM_ERR_RANGE.
constexpr float kF16Max = 65504.0f;

// Power-of-two factors for an activation row whose largest magnitude has the
// bf16 bit pattern `amax_bits` (sign cleared): `down` scales the row into
// [2^14, 2^15) before the f16 conversion, `up` = 1 / down scales the results
// back.  An all-zero or non-finite row keeps factor 1.
QMM_DEV void f16_row_scale(uint32_t amax_bits, float& down, float& up) {
  if (amax_bits == 0u || amax_bits >= 0x7F80u) {
    down = 1.0f;
    up = 1.0f;
    return;
  }
  const uint32_t f = amax_bits << 16;   // the fp32 bits of the same value
  const int eb = (int)(f >> 23);
  // floor(log2(amax)); bf16 subnormals are fp32 subnormals
  const int e = eb != 0 ? eb - 127 : (31 - __clz((int)(f & 0x7FFFFFu))) - 149;
  const int sh = min(14 - e, 126);       // e <= 127, so sh >= -113
  down = __uint_as_float((uint32_t)(127 + sh) << 23);
  up = __uint_as_float((uint32_t)(127 - sh) << 23);
}

// Per-halfword maximum of |bf16| bit patterns: for non-NaN values the order
// of magnitudes is the unsigned order of the patterns with the sign cleared.
QMM_DEV uint32_t bf16x2_absmax_bits(uint32_t acc, uint32_t w) { return __vmaxu2(acc, w & 0x7FFF7FFFu); }
QMM_DEV uint32_t bf16x2_absmax_fold(uint32_t acc) { return max(acc & 0xFFFFu, acc >> 16); }

// Two bf16 values times `down`, rounded to f16 (exact in the cases above).
QMM_DEV uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float down) {
  const float lo = __uint_as_float(w << 16) * down;
  const float hi = __uint_as_float(w & 0xFFFF0000u) * down;
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

QMM_DEV uint4 bf16x8_to_f16x8_scaled(uint4 v, float down) {
  return make_uint4(bf16x2_to_f16x2_scaled(v.x, down), bf16x2_to_f16x2_scaled(v.y, down),
                    bf16x2_to_f16x2_scaled(v.z, down), bf16x2_to_f16x2_scaled(v.w, down));
}

// Two 4-bit codes of one q4 word as an f16x2 pair (1024 + q0, 1024 + q1):
// code 2i sits in bits [4i, 4i+4) and code 2i+1 in bits [16+4i, 16+4i+4).
// 1024 is 0x6400 in f16, whose unit in the last place is 1.
QMM_DEV uint32_t q4_pair_biased_f16(uint32_t word, int i) {
  uint32_t r;
  const uint32_t w = word >> (4 * i);
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(0x000F000Fu), "r"(0x64006400u));
  return r;
}

// q * s + m in f16 from a (1024 + q) pair and f16x2 pairs (s, s), (m, m):
// the subtraction is exact, the fma rounds once.
QMM_DEV uint32_t dequant2_f16(uint32_t q2_biased, uint32_t s2, uint32_t m2) {
  __half2 q = *reinterpret_cast<__half2*>(&q2_biased);
  const uint32_t c1024 = 0x64006400u;
  q = __hsub2(q, *reinterpret_cast<const __half2*>(&c1024));
  const __half2 w = __hfma2(q, *reinterpret_cast<__half2*>(&s2), *reinterpret_cast<__half2*>(&m2));
  return *reinterpret_cast<const uint32_t*>(&w);
}

// A block's (scale, min) bf16 pair (scale in the low half) as the f16x2
// operands (s, s) and (m, m) of dequant2_f16.  Both conversions are exact
// while |s| and |m| lie in f16's normal range.  `wmax` tracks the largest
// |m| + 15 |s| seen, the bound on the block's weights.
QMM_DEV void q4_pair_to_f16(uint32_t pair, uint32_t& s2, uint32_t& m2, float& wmax) {
  const float s = __uint_as_float(pair << 16), m = __uint_as_float(pair & 0xFFFF0000u);
  wmax = fmaxf(wmax, fmaf(15.0f, fabsf(s), fabsf(m)));
  const __half2 h = __floats2half2_rn(s, m);
  const uint32_t u = *reinterpret_cast<const uint32_t*>(&h);
  s2 = __byte_perm(u, 0, 0x1010);
  m2 = __byte_perm(u, 0, 0x3232);
}

}  // namespace qmm
