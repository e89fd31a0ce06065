// moe_quant.cu -- dynamic / static activation quantisers (moe_quant_act) and
// the stage-2 requantisation of the intermediate.
//
// Schemes of the AITER leaves on the page
// "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe":
// AiterFp8TensorExperts (per-tensor static or dynamic), AiterFp8ChannelExperts
// (per-token dynamic), AiterFp8BlockExperts (1x128 dynamic), and NVFP4 x16
// with an fp32 global (QuarkNvfp4MoEMethod, page
// "vllm.model_executor.layers.quantization.quark.quark_moe").
//
// Decision rules (both the scale and the codes are taken in fp32, with IEEE
// round-to-nearest divides and the hardware's RNE saturating converts):
//   fp8   scale = fl32(max(amax, 1e-12) / 448);  code = e4m3(fl32(x / scale))
//   NVFP4 s = e4m3(fl32(fl32(amax / 6) / g));   code = e2m1(fl32(x / fl32(s * g)))
//         (s == 0 gives zero codes)
//   OCP MX X = floor(log2 amax) - emax (clamped);  code = RNE-sat(x * 2^-X)
// All kernels are HBM-bound streaming passes: 16-byte loads, one warp (or
// thread) per group, codes written with 4- or 8-byte stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

template <typename InT>
__device__ __forceinline__ float load_elem(const InT *x, long i);
template <>
__device__ __forceinline__ float load_elem<uint16_t>(const uint16_t *x, long i) {
  return bf16_to_f32(x[i]);
}
template <>
__device__ __forceinline__ float load_elem<float>(const float *x, long i) {
  return x[i];
}

// Four consecutive elements (4-element aligned) in one vector load.
template <typename InT>
__device__ __forceinline__ void load4(const InT *x, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float *x, float (&v)[4]) {
  const float4 f = *reinterpret_cast<const float4 *>(x);
  v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
template <>
__device__ __forceinline__ void load4<uint16_t>(const uint16_t *x, float (&v)[4]) {
  const uint2 u = *reinterpret_cast<const uint2 *>(x);
  v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
  v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
}

// Row state of a sorted intermediate row: -1 beyond num_post_pad (skip),
// 0 padding row (zero codes), 1 live row.
__device__ __forceinline__ int row_state(const QuantArgs &a, long r) {
  if (!a.sorted_ids) return 1;
  if (r >= *a.num_post_pad) return -1;
  return a.sorted_ids[r] < a.S ? 1 : 0;
}

// ---- fp8, 1x128 groups: one warp per 4 groups of a row; 8 lanes per group,
// lane owns 16 consecutive columns (two 16-byte loads of bf16 in flight per
// lane, the maximum reduced over the group's 8 lanes).  The same arithmetic per
// element as a group per warp; a ragged last group (cols % 128) takes the
// per-element path.
template <typename InT>
__global__ void quant_fp8_group128(QuantArgs a) {
  const long warp_id = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int G = (int)ceil_div(a.cols, 128);
  const int WG = (G + 3) / 4;  // warps per row
  const long r = warp_id / WG;
  const int g = (int)(warp_id % WG) * 4 + (lane >> 3);  // this lane's group
  if (r >= a.rows) return;  // warp-uniform
  const int st = row_state(a, r);
  if (st < 0) return;  // warp-uniform
  const bool in = g < G;
  const InT *x = static_cast<const InT *>(a.x) + r * a.cols;
  uint8_t *codes = static_cast<uint8_t *>(a.codes) + r * a.cols;
  float *scales = static_cast<float *>(a.scales);
  const int c0 = g * 128 + (lane & 7) * 16;
  float v[16];
  const bool full = in && st > 0 && c0 + 15 < a.cols && (a.cols & 3) == 0;
  if (full) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[4];
      load4<InT>(x + c0 + 4 * q, f);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[4 * q + i] = f[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      v[i] = (in && st > 0 && c0 + i < a.cols) ? load_elem<InT>(x, c0 + i) : 0.f;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = fp8_group_scale(amax);
  uint32_t packed[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    packed[q] = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) packed[q] |= f32_to_e4m3(__fdiv_rn(v[4 * q + i], scale)) << (8 * i);
    if (st == 0) packed[q] = 0;
  }
  if (!in) return;
  if (c0 + 15 < a.cols && (a.cols & 15) == 0) {
    *reinterpret_cast<uint4 *>(codes + c0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  } else {
    for (int i = 0; i < 16; ++i)
      if (c0 + i < a.cols) codes[c0 + i] = (packed[i >> 2] >> (8 * (i & 3))) & 0xff;
  }
  if ((lane & 7) == 0) scales[r * G + g] = st > 0 ? scale : 0.f;
}

// ---- fp8 per row (token): one CTA of 256 threads per row.
template <typename InT>
__global__ void quant_fp8_row(QuantArgs a) {
  const long r = blockIdx.x;
  const int st = row_state(a, r);
  if (st < 0) return;
  const InT *x = static_cast<const InT *>(a.x) + r * a.cols;
  uint8_t *codes = static_cast<uint8_t *>(a.codes) + r * a.cols;
  __shared__ float red[8];
  float amax = 0.f;
  for (int c = threadIdx.x; c < a.cols; c += blockDim.x) amax = fmaxf(amax, fabsf(load_elem<InT>(x, c)));
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
  const float scale = fp8_group_scale(amax);
  for (int c = threadIdx.x; c < a.cols; c += blockDim.x) {
    codes[c] = st > 0 ? (uint8_t)f32_to_e4m3(__fdiv_rn(load_elem<InT>(x, c), scale)) : 0;
  }
  if (threadIdx.x == 0) static_cast<float *>(a.scales)[r] = st > 0 ? scale : 0.f;
}

// ---- fp8 per tensor (static or dynamic): one CTA (1024 threads) for the
// whole tensor; used by no large workload (the per-tensor scheme is rare).
template <typename InT>
__global__ void quant_fp8_tensor(QuantArgs a, int dynamic) {
  __shared__ float red[32];
  float scale;
  if (dynamic) {
    float amax = 0.f;
    for (long r = 0; r < a.rows; ++r) {
      if (row_state(a, r) <= 0) continue;
      const InT *x = static_cast<const InT *>(a.x) + r * a.cols;
      for (int c = threadIdx.x; c < a.cols; c += blockDim.x) amax = fmaxf(amax, fabsf(load_elem<InT>(x, c)));
    }
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
    scale = fp8_group_scale(amax);
  } else {
    scale = a.param[0];
  }
  for (long r = 0; r < a.rows; ++r) {
    const int st = row_state(a, r);
    if (st < 0) continue;
    const InT *x = static_cast<const InT *>(a.x) + r * a.cols;
    uint8_t *codes = static_cast<uint8_t *>(a.codes) + r * a.cols;
    for (int c = threadIdx.x; c < a.cols; c += blockDim.x) {
      codes[c] = st > 0 ? (uint8_t)f32_to_e4m3(__fdiv_rn(load_elem<InT>(x, c), scale)) : 0;
    }
  }
  if (threadIdx.x == 0) static_cast<float *>(a.scales)[0] = scale;
}

// ---- NVFP4 x16: one thread per group of 16 (8 code bytes + 1 scale byte).
template <typename InT>
__global__ void quant_nvfp4(QuantArgs a) {
  const long gid = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const int G = a.cols / 16;
  const long r = gid / G;
  const int g = (int)(gid % G);
  if (r >= a.rows) return;
  const int st = row_state(a, r);
  if (st < 0) return;
  uint8_t *codes = static_cast<uint8_t *>(a.codes) + r * (a.cols / 2) + g * 8;
  uint8_t *scales = static_cast<uint8_t *>(a.scales) + r * G + g;
  if (st == 0) {
    *reinterpret_cast<uint2 *>(codes) = make_uint2(0, 0);
    *scales = 0;
    return;
  }
  const float gs = a.sorted_ids ? a.param[a.expert_ids[r / a.BM]] : a.param[0];
  const InT *x = static_cast<const InT *>(a.x) + r * a.cols + g * 16;
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = load_elem<InT>(x, i);
  uint32_t lo, hi;
  const uint32_t s = nvfp4_quant16(v, gs, lo, hi);
  *reinterpret_cast<uint2 *>(codes) = make_uint2(lo, hi);
  *scales = (uint8_t)s;
}

// ---- OCP MX (32-element blocks, e8m0 scale): one warp per block, lane = element.
//   X = floor(log2(amax)) - emax (2 for e2m1, 8 for e4m3), clamped to [-127, 127];
//   scale code X + 127; code = RNE-saturating convert of x * 2^-X (exact scaling);
//   amax == 0: scale code 0, zero codes.
template <typename InT, bool FP4>
__global__ void quant_mx(QuantArgs a) {
  const long warp_id = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int G = a.cols / 32;
  const long r = warp_id / G;
  const int g = (int)(warp_id % G);
  if (r >= a.rows) return;
  const int st = row_state(a, r);
  if (st < 0) return;
  const float v = st > 0 ? load_elem<InT>(static_cast<const InT *>(a.x) + r * a.cols, g * 32 + lane)
                         : 0.f;
  const float amax = warp_max(fabsf(v));
  int code_x = 0;  // e8m0 scale code
  float q = 0.f;   // x * 2^-X
  if (amax > 0.f) {
    const int X = mx_shared_exp(amax, FP4 ? 2 : 8);
    code_x = X + 127;
    q = v * pow2f(-X);
  }
  uint8_t *scales = static_cast<uint8_t *>(a.scales);
  if (lane == 0) scales[r * G + g] = (uint8_t)code_x;
  if (FP4) {
    // element 2i in the low nibble: even lanes pack their pair
    const float q_hi = __shfl_down_sync(0xffffffffu, q, 1);
    if ((lane & 1) == 0)
      static_cast<uint8_t *>(a.codes)[r * (a.cols / 2) + g * 16 + (lane >> 1)] =
          (uint8_t)f32x2_to_e2m1x2(q, q_hi);
  } else {
    static_cast<uint8_t *>(a.codes)[r * a.cols + g * 32 + lane] = (uint8_t)f32_to_e4m3(q);
  }
}

// fp32 rows -> f16 of their MX quantise-dequantise.  One thread per chunk of
// 8 values: chunk c of row r is thread r * N/8 + c, and N/8 % 4 == 0, so the
// four threads of a 32-element block are four aligned consecutive lanes of
// one warp and share the row's fate.  zero_pad: padding rows get zeros
// (else they are skipped, like rows at or beyond *ntp).
__global__ void mx_qdq_rows_kernel(const float *__restrict__ src, long rows, int N,
                                   const int32_t *__restrict__ sorted_ids,
                                   const int32_t *__restrict__ ntp, int S,
                                   uint16_t *__restrict__ dst, int fp4, int zero_pad) {
  griddep_launch_dependents();
  griddep_wait();
  const int n8 = N / 8;
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long r = i / n8;
  const int c = (int)(i - r * n8);
  if (r >= rows || (ntp && r >= *ntp)) return;
  const bool live = !sorted_ids || sorted_ids[r] < S;
  if (!live && !zero_pad) return;
  const unsigned gmask = 0xFu << (threadIdx.x & 28);
  uint4 o = make_uint4(0u, 0u, 0u, 0u);
  if (live) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src + r * N) + 2 * c;
    const float4 u = s4[0], w = s4[1];
    const float f[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
    o = mx_qdq_f16x8(f, fp4 != 0, 0, gmask);
  }
  reinterpret_cast<uint4 *>(dst + r * N)[c] = o;
}

template <typename InT>
cudaError_t launch_quant_t(const QuantArgs &a, cudaStream_t stream) {
  if (a.rows <= 0 || a.cols <= 0) return cudaSuccess;
  switch (a.afmt) {
    case A_FP8_GROUP128_DYN: {
      const long warps = a.rows * ((ceil_div(a.cols, 128) + 3) / 4);
      quant_fp8_group128<InT><<<(unsigned)ceil_div(warps * 32, 256), 256, 0, stream>>>(a);
      break;
    }
    case A_FP8_TOKEN_DYN:
      quant_fp8_row<InT><<<(unsigned)a.rows, 256, 0, stream>>>(a);
      break;
    case A_FP8_TENSOR_STATIC:
    case A_FP8_TENSOR_DYN:
      quant_fp8_tensor<InT><<<1, 1024, 0, stream>>>(a, a.afmt == A_FP8_TENSOR_DYN);
      break;
    case A_NVFP4_DYN: {
      const long groups = a.rows * (a.cols / 16);
      quant_nvfp4<InT><<<(unsigned)ceil_div(groups, 128), 128, 0, stream>>>(a);
      break;
    }
    case A_MXFP4_DYN:
    case A_MXFP8_DYN: {
      const long groups = a.rows * (a.cols / 32);  // one warp each
      if (a.afmt == A_MXFP4_DYN)
        quant_mx<InT, true><<<(unsigned)ceil_div(groups * 32, 256), 256, 0, stream>>>(a);
      else
        quant_mx<InT, false><<<(unsigned)ceil_div(groups * 32, 256), 256, 0, stream>>>(a);
      break;
    }
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant(const QuantArgs &a, cudaStream_t stream) {
  return a.x_is_f32 ? launch_quant_t<float>(a, stream) : launch_quant_t<uint16_t>(a, stream);
}

cudaError_t launch_mx_qdq_rows(const float *src, long rows, int N, const int32_t *sorted_ids,
                               const int32_t *num_post_pad, int S, void *dst, int fp4,
                               int zero_pad, cudaStream_t stream, bool dependent) {
  if (rows <= 0) return cudaSuccess;
  return launch_kernel(mx_qdq_rows_kernel, dim3((unsigned)ceil_div(rows * (N / 8), 256)),
                       dim3(256), 0, stream, dependent, src, rows, N, sorted_ids, num_post_pad,
                       S, static_cast<uint16_t *>(dst), fp4, zero_pad);
}

}  // namespace moe
