// NVFP4 block codec on the device: one E4M3 scale per 16 values, E2M1 codes,
// a per-tensor (or per-row) FP32 scale.  Format from "NVFP4 KV cache vs NVFP4
// weights" (section "NVFP4 KV cache vs NVFP4 weights") and "NVFP4 KV cache
// prefill vs decode performance" (section "NVFP4 stores 4.5 bits per value
// before padding").  Rounding rule per block of 16 values x with scale g:
//   s     = amax(|x|) / (6 g)            (IEEE division)
//   byte  = E4M3(s), nearest-even, saturating at 448 (hardware cvt)
//   inv   = 1 / (g * e4m3(byte))         (correctly rounded reciprocal)
//   code  = E2M1(x * inv), nearest-even, saturating at 6, sign kept
//   zero scale byte -> all sixteen codes 0
// Every step is a single IEEE fp32 operation so the result is reproducible
// bit for bit.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace nvfp4kv {

// Exact E4M3 (non-negative) byte -> fp32.
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2 = cvt_e4m3x2_to_f16x2(byte & 0xFFu);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Quantize 16 values with scale g.  Returns the 8 packed bytes in w0 (elements
// 0..7) and w1 (elements 8..15), element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t quant_block16(const float* x, float g, uint32_t& w0, uint32_t& w1) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float six_g = __fmul_rn(6.0f, g);
  const float s_real = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, six_g);
  const uint32_t sc = cvt_e4m3x2(s_real, 0.0f) & 0xFFu;
  const float sdec = e4m3_to_f32(sc);
  if (sdec == 0.0f) {
    w0 = 0u;
    w1 = 0u;
    return sc;
  }
  const float inv = __frcp_rn(__fmul_rn(g, sdec));
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = cvt_e2m1x2(__fmul_rn(x[2 * i], inv), __fmul_rn(x[2 * i + 1], inv));
  w0 = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  w1 = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return sc;
}

// bf16 pair (packed in a 32-bit word, element 0 in the low half) -> floats.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

// Four code bytes (eight E2M1 values) -> four f16x2 words, exactly: word i
// holds byte i, its low nibble in the low half.  The bytes are taken as
// sub-registers of the word, so no shifts or masks precede the conversions.
__device__ __forceinline__ void cvt_e2m1x8_to_f16x2(uint32_t codes, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(codes));
}

// Eight E2M1 codes (one 32-bit word, element i in nibble i) times an f16x2
// scale pair -> four f16x2 words (element 2i in the low half of word i).
// Exact: every E2M1 x E4M3 product is an f16 normal (2^-10 .. 2688) with at
// most 6 significant bits.
__device__ __forceinline__ void dequant8_f16(uint32_t codes, uint32_t scale_h2, uint32_t (&out)[4]) {
  uint32_t h[4];
  cvt_e2m1x8_to_f16x2(codes, h);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&h[i]), *reinterpret_cast<const __half2*>(&scale_h2));
    out[i] = *reinterpret_cast<uint32_t*>(&r);
  }
}

// Same, to bf16x2.  The E2M1 value is produced exactly in f16 by the hardware
// conversion, moved into bf16 by re-biasing the exponent (value * 2^-112, a
// normal bf16 for every non-zero code), then multiplied by scale * 2^112
// (scale_b2 holds that product as a bf16 pair).  Both steps are exact.
__device__ __forceinline__ void dequant8_bf16(uint32_t codes, uint32_t scale_b2, uint32_t (&out)[4]) {
  uint32_t hw[4];
  cvt_e2m1x8_to_f16x2(codes, hw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t h = hw[i];
    uint32_t a = ((h & 0x7FFF7FFFu) >> 3) | (h & 0x80008000u);
    __nv_bfloat162 r =
        __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&scale_b2));
    out[i] = *reinterpret_cast<uint32_t*>(&r);
  }
}

// Block-scale byte -> bf16 pair holding scale * 2^112 (exact).
__device__ __forceinline__ uint32_t scale_bf16x2_x2p112(uint32_t byte) {
  float s = e4m3_to_f32(byte) * 5.192296858534828e33f;  // 2^112
  uint32_t b = __float_as_uint(s) >> 16;                 // exact: <= 4 significant bits
  return b | (b << 16);
}

}  // namespace nvfp4kv
