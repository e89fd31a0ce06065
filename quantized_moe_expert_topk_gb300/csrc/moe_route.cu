// moe_route.cu -- fused router: logits -> top-k expert ids and weights.
//
// The apply_monolithic path (GptOssMxfp4MoEMethod / Mxfp4MoEMethod on the
// mxfp4.py page, QuarkOCP_MX_MoEMethod on the quark_moe page) hands the
// router logits together with num_expert_group, topk_group,
// e_score_correction_bias and routed_scaling_factor to the expert kernel.
// The rule implemented (stated in include/moe_experts.h, moe_route_topk):
// softmax or sigmoid scores s, choice keys c = s + bias; with groups, a group
// scores max(c) (no bias) or the sum of its two largest c (bias), and only the
// topk_group best groups stay eligible; the topk eligible experts with the
// largest keys are chosen (ties to the lower id); weights are the unbiased
// scores, optionally renormalised, times the scaling factor.  Without bias the
// keys are the logits themselves (both score functions are increasing), so
// the choice does not depend on exp rounding.
//
// One warp per token; lane l holds experts l, l+32, ... (E <= 1024).
#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int kRouteMaxGroups = 32;

struct Best {
  float key;
  int idx;
};

// a before b: larger key, then lower index; idx < 0 means "none"
__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
  if (ib < 0) return ia >= 0;
  if (ia < 0) return false;
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ Best warp_best(Best b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float k2 = __shfl_xor_sync(0xffffffffu, b.key, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, b.idx, o);
    if (better(k2, i2, b.key, b.idx)) {
      b.key = k2;
      b.idx = i2;
    }
  }
  return b;
}

__device__ __forceinline__ float warp_fmax(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_fsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int PER_LANE>
__global__ void __launch_bounds__(128)
route_kernel(const void *__restrict__ logits, int bf16_in, int M, int E, int topk, int scoring,
             int renorm, int G, int TG, const float *__restrict__ bias, float scale,
             int32_t *__restrict__ ids_out, float *__restrict__ w_out) {
  // dependent launch: the next grid (the sort) may be scheduled now; this
  // one waits for the producer of the logits before reading them
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const long t = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= M) return;  // uniform per warp

  float lg[PER_LANE], sc[PER_LANE], key[PER_LANE];
  uint32_t elig = 0;  // bit i: element i of this lane exists and may be chosen
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    if (e < E) {
      v = bf16_in ? bf16_to_f32(static_cast<const uint16_t *>(logits)[t * E + e])
                  : static_cast<const float *>(logits)[t * E + e];
      elig |= 1u << i;
    }
    lg[i] = v;
    mx = fmaxf(mx, v);
  }
  // scores: softmax numerators exp(l - max) (normalised by den) or sigmoids
  float den = 1.f;
  if (scoring == 0) {
    mx = warp_fmax(mx);
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      sc[i] = ((elig >> i) & 1u) ? expf(lg[i] - mx) : 0.f;
      part += sc[i];
    }
    den = warp_fsum(part);
  } else {
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i)
      sc[i] = ((elig >> i) & 1u) ? 1.f / (1.f + expf(-lg[i])) : 0.f;
  }
  // choice keys: the logits themselves, or score + bias
  const bool biased = bias != nullptr;
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    key[i] = !((elig >> i) & 1u) ? -INFINITY
             : biased             ? (scoring == 0 ? sc[i] / den : sc[i]) + bias[e]
                                  : lg[i];
  }

  if (G > 1) {
    // group scores: max key (no bias) or the sum of the two largest keys
    const int gs = E / G;
    float gscore[kRouteMaxGroups];
#pragma unroll
    for (int g = 0; g < kRouteMaxGroups; ++g) gscore[g] = -INFINITY;
#pragma unroll
    for (int g = 0; g < kRouteMaxGroups; ++g) {
      if (g >= G) break;
      float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i) {
        const int e = lane + 32 * i;
        if (((elig >> i) & 1u) && e / gs == g) {
          const float v = key[i];
          if (v > b1) {
            b2 = b1;
            b1 = v;
          } else if (v > b2) {
            b2 = v;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {  // merge the lanes' (largest, second) pairs
        const float o1 = __shfl_xor_sync(0xffffffffu, b1, o);
        const float o2 = __shfl_xor_sync(0xffffffffu, b2, o);
        const float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
        b1 = fmaxf(b1, o1);
        b2 = n2;
      }
      gscore[g] = biased ? b1 + b2 : b1;
    }
    // the topk_group best groups (ties to the lower group) stay eligible
    uint32_t keep = 0;
    for (int j = 0; j < TG; ++j) {
      int bg = -1;
      float bk = -INFINITY;
#pragma unroll
      for (int g = 0; g < kRouteMaxGroups; ++g)
        if (g < G && !((keep >> g) & 1u) && (bg < 0 || gscore[g] > bk)) {
          bg = g;
          bk = gscore[g];
        }
      keep |= 1u << bg;
    }
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (((elig >> i) & 1u) && !((keep >> (e / gs)) & 1u)) elig &= ~(1u << i);
    }
  }

  // top-k by key (descending, ties to the lower id)
  int my_id = -1;
  float my_s = 0.f, sel_sum = 0.f;
  for (int j = 0; j < topk; ++j) {
    Best b{-INFINITY, -1};
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (((elig >> i) & 1u) && better(key[i], e, b.key, b.idx)) {
        b.key = key[i];
        b.idx = e;
      }
    }
    b = warp_best(b);
    const int e = b.idx;  // >= 0: the host checks topk <= eligible experts
    float s = 0.f;
    if ((e & 31) == lane) {
      const int ie = e >> 5;
      elig &= ~(1u << ie);
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i)
        if (i == ie) s = sc[i];
    }
    s = __shfl_sync(0xffffffffu, s, e & 31);
    if (lane == j) {
      my_id = e;
      my_s = s;
    }
    sel_sum += s;
  }
  if (lane < topk) {
    const float w = renorm ? my_s / sel_sum : my_s / den;
    ids_out[t * topk + lane] = my_id;
    w_out[t * topk + lane] = w * scale;
  }
}

}  // namespace

cudaError_t launch_route(const void *logits, int bf16_in, int M, int E, int topk, int scoring,
                         int renorm, int G, int TG, const float *bias, float scale, int32_t *ids,
                         float *weights, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const dim3 grid((unsigned)ceil_div((long)M * 32, 128)), block(128);
  const int per_lane = (E + 31) / 32;
#define MOE_ROUTE_CASE(P)                                                                   \
  if (per_lane <= P)                                                                        \
    return launch_kernel(route_kernel<P>, grid, block, 0, st, true, logits, bf16_in, M, E, topk, \
                         scoring, renorm, G, TG, bias, scale, ids, weights);
  MOE_ROUTE_CASE(1)
  MOE_ROUTE_CASE(2)
  MOE_ROUTE_CASE(4)
  MOE_ROUTE_CASE(8)
  MOE_ROUTE_CASE(16)
  MOE_ROUTE_CASE(32)
#undef MOE_ROUTE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
