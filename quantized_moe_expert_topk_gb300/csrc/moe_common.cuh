// moe_common.cuh -- device-side element codecs and small helpers shared by the
// kernels of this library (internal header, not part of the ABI).
//
// Element formats (the OCP microscaling formats the MoE pages use:
// "vLLM/vllm/model_executor/layers/quantization/mxfp4.py",
// GptOssMxfp4MoEMethod.create_weights; "vllm.model_executor.layers.quantization.
// quark.quark_moe", QuarkNvfp4MoEMethod.create_weights):
//   e2m1   sign | 2-bit exponent (bias 1) | 1-bit mantissa; 0,.5,1,1.5,2,3,4,6
//   e4m3fn sign | 4-bit exponent (bias 7) | 3-bit mantissa; max 448, no inf
//   e8m0   2^(c-127)
// Every decode below is exact: each decoded value (and each product of an
// e2m1 code with its e8m0 or e4m3 scale) is representable in bf16 over the
// formats' usual ranges, so the tensor-core operands carry no rounding.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- enums (ABI values)
enum WFmt { W_BF16 = 0, W_FP8_TENSOR = 1, W_FP8_CHANNEL = 2, W_FP8_BLOCK128 = 3, W_MXFP4 = 4,
            W_NVFP4 = 5 };
enum AFmt { A_BF16 = 0, A_FP8_TENSOR_STATIC = 1, A_FP8_TENSOR_DYN = 2, A_FP8_TOKEN_DYN = 3,
            A_FP8_GROUP128_DYN = 4, A_NVFP4_DYN = 5, A_MXFP4_DYN = 6, A_MXFP8_DYN = 7 };
enum Act { ACT_SILU = 0, ACT_GELU = 1, ACT_SWIGLU_OAI = 2 };
enum Gate { GATE_SEPARATED = 0, GATE_INTERLEAVED = 1 };

constexpr float kFp8Max = 448.0f;
constexpr float kE2m1Max = 6.0f;
constexpr float kScaleFloor = 1e-12f;

// Device error word (first error wins).  Kernels receive its address (taken
// once on the host with cudaGetSymbolAddress) and record a code with this.
__device__ __forceinline__ void record_device_error(int *word, int code) {
  if (word) atomicCAS(word, 0, code);
}

// ---------------------------------------------------------------- decode
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// e4m3fn code -> fp32 (exact).  Normal: (1 + m/8) 2^(e-7); subnormal: m 2^-9.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float v = (e == 0) ? static_cast<float>(m) * 0.001953125f
                     : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -v : v;
}

// e2m1 nibble -> fp32 (exact).
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  float v = (e == 0) ? 0.5f * static_cast<float>(m)
                     : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (c & 8u) ? -v : v;
}

// e8m0 code -> fp32 (2^(c-127)); codes 0 and 255 are outside fp32's normal
// range and are mapped to 2^-127 (subnormal) / NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
  if (c == 0) return __uint_as_float(0x00400000u);
  if (c == 255) return __uint_as_float(0x7fc00000u);
  return __uint_as_float(c << 23);
}

// ---------------------------------------------------------------- encode
// fp32 -> e4m3fn, round-to-nearest-even, saturating to +-448 (sign kept).
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xffu;
}

// (lo, hi) fp32 -> one byte of two e2m1 codes (lo in bits 3..0), RNE, saturating at +-6.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r & 0xffu;
}

// fp8 dynamic scale of a group: fl32(max(amax, 1e-12) / 448), IEEE divide.
__device__ __forceinline__ float fp8_group_scale(float amax) {
  return __fdiv_rn(fmaxf(amax, kScaleFloor), kFp8Max);
}

// NVFP4 x16 quantiser of one group of 16 fp32 values (the decision rule of
// QuarkNvfp4MoEMethod's dynamic activations): s = e4m3(fl32(fl32(amax/6)/gs)),
// code = e2m1(fl32(v / fl32(e4m3(s) * gs))), zero codes when s decodes to 0.
// Returns s; lo / hi hold the 16 codes (element 2i in the low nibble).
__device__ __forceinline__ uint32_t nvfp4_quant16(const float (&v)[16], float gs, uint32_t &lo,
                                                  uint32_t &hi) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t s = f32_to_e4m3(__fdiv_rn(__fdiv_rn(amax, kE2m1Max), gs));
  const float sv = e4m3_to_f32(s);
  lo = hi = 0;
  if (sv != 0.f) {
    const float denom = __fmul_rn(sv, gs);
#pragma unroll
    for (int i = 0; i < 8; i += 2)
      lo |= f32x2_to_e2m1x2(__fdiv_rn(v[i], denom), __fdiv_rn(v[i + 1], denom)) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; i += 2)
      hi |= f32x2_to_e2m1x2(__fdiv_rn(v[8 + i], denom), __fdiv_rn(v[9 + i], denom)) << (4 * i);
  }
  return s;
}

// 2^e as fp32, exact for e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// OCP MX shared exponent of a block whose largest magnitude is amax (> 0):
// floor(log2(amax)) - emax (emax 2 for e2m1, 8 for e4m3), clamped to the e8m0
// range [-127, 127].  The block's codes are the RNE-saturating conversions of
// x * 2^-X, an exact scaling (X <= 125 for any finite fp32 amax, so 2^-X is a
// normal fp32).
__device__ __forceinline__ int mx_shared_exp(float amax, int emax) {
  int ex;
  frexpf(amax, &ex);  // amax = f * 2^ex, 0.5 <= f < 1: floor(log2(amax)) = ex - 1
  const int X = ex - 1 - emax;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// (lo, hi) fp32 -> two e4m3fn codes (lo in bits 7..0), RNE, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Exact f16 pairs of two e2m1 codes (one byte, element 0 in bits 3..0) or of
// two e4m3fn codes (element 0 in bits 7..0), by the hardware converts; the
// first element lands in the low half.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t b) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
      : "=r"(r) : "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t c) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)c));
  return r;
}

// Two values of a block with shared exponent X: quantised (x * 2^-X, RNE
// saturating to e2m1 when fp4, else e4m3), dequantised and multiplied by
// 2^(X + a), as an f16 pair.  The codes' f16 values are exact and so is
// their fp32 product with the power of two, so the one rounding is the final
// convert: exact wherever code * 2^(X + a) lies in f16's range (a code has at
// most 4 significant bits); below 2^-126 the product is far under f16's
// smallest subnormal and becomes 0.
__device__ __forceinline__ uint32_t mx_qdq_pair_f16(float v0, float v1, bool fp4, int X, int a) {
  const float inv = pow2f(-X);
  const float outs = X + a >= -126 ? pow2f(X + a) : 0.f;
  const uint32_t h = fp4 ? e2m1x2_to_f16x2(f32x2_to_e2m1x2(v0 * inv, v1 * inv))
                         : e4m3x2_to_f16x2(f32x2_to_e4m3x2(v0 * inv, v1 * inv));
  const float2 d = __half22float2(*reinterpret_cast<const __half2 *>(&h));
  const __half2 o = __floats2half2_rn(d.x * outs, d.y * outs);
  return *reinterpret_cast<const uint32_t *>(&o);
}

// Eight consecutive values of one 32-element OCP MX block quantised (MXFP4
// when fp4, else MXFP8) and dequantised, times 2^a, as four packed f16 pairs.
// The four consecutive lanes named by gmask hold the block's 32 values and
// call this together; the block maximum is taken across them.  Same decisions
// as the MX quantiser.
__device__ __forceinline__ uint4 mx_qdq_f16x8(const float (&v)[8], bool fp4, int a,
                                              unsigned gmask) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
  uint32_t o[4] = {0u, 0u, 0u, 0u};
  if (amax > 0.f) {
    const int X = mx_shared_exp(amax, fp4 ? 2 : 8);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = mx_qdq_pair_f16(v[2 * i], v[2 * i + 1], fp4, X, a);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// A whole 32-element block held by one thread, quantised and dequantised to
// f16 (no extra power of two); out[i] holds elements 2i, 2i + 1.
__device__ __forceinline__ void mx_qdq_f16x32(const float (&v)[32], bool fp4,
                                              uint32_t (&out)[16]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int X = amax > 0.f ? mx_shared_exp(amax, fp4 ? 2 : 8) : 0;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    out[i] = amax > 0.f ? mx_qdq_pair_f16(v[2 * i], v[2 * i + 1], fp4, X, 0) : 0u;
}

// ---------------------------------------------------------------- activations
__device__ __forceinline__ float sigmoidf_(float v) { return 1.0f / (1.0f + expf(-v)); }

__device__ __forceinline__ float act_and_mul(int act, float g, float u, float alpha, float beta,
                                             float limit) {
  if (act == ACT_SILU) return g * sigmoidf_(g) * u;
  if (act == ACT_GELU) return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f)) * u;
  // SwiGLU-OAI: clamp, then (u + beta) * g * sigmoid(alpha * g)
  if (limit > 0.0f) {
    g = fminf(g, limit);
    u = fminf(fmaxf(u, -limit), limit);
  }
  return (u + beta) * g * sigmoidf_(alpha * g);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__host__ __device__ __forceinline__ long ceil_div(long a, long b) { return (a + b - 1) / b; }

}  // namespace moe
