// Device-side helpers shared by the kernels: loads, legacy MMA wrappers, the
// exact int8 epilogue and the error-status word.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "qmm.h"

#define QMM_DEV __device__ __forceinline__

namespace qmm {

// First error wins: a 0 in the caller's status word becomes `code`.
QMM_DEV void set_status(int32_t* st, int32_t code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

QMM_DEV uint4 ldg128(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Read-once stream (weights): do not allocate in L1.
QMM_DEV uint4 ldg128_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

QMM_DEV uint32_t ldg32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// Two fp32 lanes in one 64-bit register, for the packed f32x2 arithmetic of
// sm_100+ (each lane rounds exactly as the scalar instruction would).
QMM_DEV uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
QMM_DEV void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
QMM_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
QMM_DEV uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
QMM_DEV uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// int8 byte i of word xw (already XORed with 0x80808080) as fp32: the byte
// becomes the low mantissa byte of 2^23, and 2^23 + 128 is subtracted (exact).
QMM_DEV float s8_byte_to_f32(uint32_t xw, int i) {
  return __uint_as_float(__byte_perm(xw, 0x4B000000u, 0x7540u + (uint32_t)i)) - 8388736.0f;
}

QMM_DEV uint32_t u4_get(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// D = A(16x32 s8, row) * B(32x8 s8, col) + D, exact int32 accumulation.
QMM_DEV void mma_s8_16832(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D with fp32 accumulation.
// Four biased bytes (code + 128 each) as two f16x2 pairs of the codes,
// exactly: each byte becomes the low mantissa byte of 1024 (f16 0x6400), and
// 1024 + 128 is subtracted.  lo holds bytes 0 and 1 (byte 0 in the low half).
QMM_DEV void biased4_to_f16(uint32_t u, uint32_t& lo, uint32_t& hi) {
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140u);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342u);
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(l), "r"(0x64806480u));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(h), "r"(0x64806480u));
}

// No side effects beyond d: not volatile, so independent MMAs may be
// interleaved by the compiler to hide each one's latency.
QMM_DEV void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                           uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D with fp32 accumulation.
QMM_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                            uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

QMM_DEV float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
QMM_DEV float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two 4-bit codes of one q4 word as a bf16x2 pair (128 + q0, 128 + q1):
// code 2i sits in bits [4i, 4i+4) and code 2i+1 in bits [16+4i, 16+4i+4).
QMM_DEV uint32_t q4_pair_biased(uint32_t word, int i) {
  uint32_t r;
  const uint32_t w = word >> (4 * i);
  // r = (w & 0x000F000F) | 0x43004300 in one lop3
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(0x000F000Fu), "r"(0x43004300u));
  return r;
}

// ---------------------------------------------------------------------------
// int8 epilogue.  Integer steps run modulo 2^32 (uint32): the final Y is the
// exact value whenever it fits in int32, which the API requires.
// ---------------------------------------------------------------------------
struct Int8Epi {
  int out_type;            // qmm_dtype
  const int32_t* bias;
  const float* s_x;
  int s_x_stride;          // 0 or 1
  const float* s_w;
  float s_y;
  int zp_y;
  uint32_t zAp;            // zA' (two's complement)
  uint32_t zBp;            // zB'
  uint32_t Kz;             // K * zA'
  const int32_t* col_sum;
  void* out;
  int64_t ldo;
};

QMM_DEV int32_t zp_correct(int32_t S, int32_t colsum, int32_t rowsum, const Int8Epi& e) {
  uint32_t y = (uint32_t)S - e.zAp * (uint32_t)colsum - e.zBp * ((uint32_t)rowsum - e.Kz);
  return (int32_t)y;
}

// Output conversion of one element (fp32 steps with explicit IEEE rounding),
// given the element's bias, activation scale and weight scale (0, 1 and 1
// where the epilogue has none).
QMM_DEV void int8_store_vals(const Int8Epi& e, int m, int n, int32_t Y, int32_t bias, float sx, float sw) {
  const int32_t yb = (int32_t)((uint32_t)Y + (uint32_t)bias);
  if (e.out_type == QMM_S32) {
    reinterpret_cast<int32_t*>(e.out)[(int64_t)m * e.ldo + n] = yb;
    return;
  }
  const float yf = __int2float_rn(yb);
  if (e.out_type == QMM_F32) {
    reinterpret_cast<float*>(e.out)[(int64_t)m * e.ldo + n] = __fmul_rn(__fmul_rn(yf, sx), sw);
    return;
  }
  const float mq = __fdiv_rn(__fmul_rn(sx, sw), e.s_y);
  float r = __fmul_rn(yf, mq);
  r = fminf(fmaxf(r, -1.0e9f), 1.0e9f);   // keeps the integer conversion in range
  int q = __float2int_rn(r) + e.zp_y;
  if (e.out_type == QMM_S8) {
    q = min(max(q, -128), 127);
    reinterpret_cast<int8_t*>(e.out)[(int64_t)m * e.ldo + n] = (int8_t)q;
  } else {
    q = min(max(q, 0), 255);
    reinterpret_cast<uint8_t*>(e.out)[(int64_t)m * e.ldo + n] = (uint8_t)q;
  }
}

QMM_DEV void int8_store(const Int8Epi& e, int m, int n, int32_t Y) {
  int8_store_vals(e, m, n, Y, e.bias ? e.bias[n] : 0, e.s_x ? e.s_x[e.s_x_stride ? m : 0] : 1.0f,
                  e.s_w ? e.s_w[n] : 1.0f);
}

}  // namespace qmm
