// FP8 (e4m3) rows of the paged KV cache: conversion and quantisation helpers.
//
// Source: Ultralytics glossary "PagedAttention", section "Related techniques"
// (FP8 cache quantisation stores keys and values at 8-bit precision, about
// half the bytes of 16-bit formats).  Format reading: e4m3, one fp32 scale per
// cached row (token x KV head), s = amax / 448 (1 for an all-zero row), code =
// e4m3 nearest to x / s with ties to even, saturating at +-448.  Both
// divisions are IEEE float32 (__fdiv_rn), the rounding is the hardware's
// round-to-nearest-even conversion with saturation.
//
// Pool layout (per block b and KV head h, 16 token slots, d = 128):
//   K codes: 16 rows x 128 B at ((b * h_kv + h) * 16 + r) * 128; the 16-byte
//            chunk c of row r sits at chunk position c ^ (4 * (r & 1)), so the
//            decode's 16-byte shared-memory loads of two neighbouring rows
//            fall in different banks;
//   V codes: transposed, 128 rows (one per d) x 16 B (one byte per slot) at
//            ((b * h_kv + h) * 128 + dd) * 16 + r, so that the decode's
//            value fragments (d x tokens) are plain 4-byte loads;
//   scales:  fp32 [num_blocks][h_kv][16] for K and for V.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace kvs {

constexpr float kE4m3Max = 448.0f;

// byte offset of (row r, element e) in a block-head's K code tile (d = 128)
__host__ __device__ __forceinline__ int f8_k_off(int r, int e) {
  return r * 128 + ((((e >> 4) ^ ((r & 1) << 2))) << 4) + (e & 15);
}

// four e4m3 codes (bytes, lowest first) -> two f16x2 words (lo: bytes 0,1)
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// two floats -> f16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// bf16x2 word -> f16x2 word (exact for values in f16's normal range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// two floats -> two e4m3 codes in a 16-bit value (lo in the low byte)
__device__ __forceinline__ uint32_t e4m3x2_pack(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// the row scale from the row's largest magnitude
__device__ __forceinline__ float f8_row_scale(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
}

// four values -> four codes (lowest first) under scale s
__device__ __forceinline__ uint32_t f8_quant4(float x0, float x1, float x2, float x3, float s) {
  return e4m3x2_pack(__fdiv_rn(x0, s), __fdiv_rn(x1, s)) |
         (e4m3x2_pack(__fdiv_rn(x2, s), __fdiv_rn(x3, s)) << 16);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace kvs
