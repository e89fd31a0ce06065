// moe_gemm_generic.cu -- grouped GEMMs of the fused experts for every weight
// format (bf16, FP8 per-tensor / per-channel / 128x128 block, MXFP4, NVFP4):
//   W13 mode: gate/up GEMM over gathered token rows + activation epilogue
//   W2 mode:  down GEMM over sorted intermediate rows + router-weight
//             multiply + fp32 scatter-add into the token accumulator
// ("rocm_aiter_fused_experts" on page "vllm.model_executor.layers.fused_moe.
// experts.rocm_aiter_moe"; the reduce happens inside the experts call, as the
// leaf's TopKWeightAndReduceNoOP finalize says).
//
// Design.  Each CTA owns one sorted block of 64 rows (all rows of a block
// belong to one expert, guaranteed by the sort) and one tile of 128 output
// columns.  Operands are decoded EXACTLY to bf16 while being staged into
// shared memory: e4m3, e2m1*2^e (MXFP4) and e2m1*e4m3 (NVFP4) are all bf16
// values, so the tensor-core products are exact and the only rounding is the
// fp32 accumulation.  Scales that do not fold exactly (fp8 per-tensor and
// per-channel, NVFP4 globals, fp8 per-token activation scales) are applied
// to the fp32 accumulator in the epilogue; FP8 128x128 block scales are
// applied per 128-wide reduction block ("promotion": a partial accumulator
// per block, multiplied by a_scale[row, kb] * w_scale[col_block, kb]).
// W13 tiles pair gate and up rows so that each thread owns both halves of
// its (row, j) outputs: warp wn computes gate rows j0+16wn.. and the matching
// up rows, for either row layout (SEPARATED or INTERLEAVED).
#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = kGenericBlockM;  // 64 sorted rows per tile
constexpr int BN = 128;             // weight rows (output columns) per tile
constexpr int BK = 32;              // reduction step per pipeline stage
constexpr int LDS = BK + 8;         // smem row stride (bf16): 80 B, conflict-free ldmatrix
constexpr int THREADS = 256;

enum { MODE_W13 = 0, MODE_W2 = 1 };
// Weight kinds; WK_MX_A4 / WK_MX_A8 are MXFP4 weights with MXFP4 / MXFP8
// (OCP MX, e8m0 per 32) activations, decoded exactly to bf16 like the weights.
enum { WK_BF16 = 0, WK_FP8 = 1, WK_MXFP4 = 2, WK_NVFP4 = 3, WK_MX_A4 = 4, WK_MX_A8 = 5 };
template <int WK>
constexpr bool mx_weights() { return WK == WK_MXFP4 || WK == WK_MX_A4 || WK == WK_MX_A8; }

struct Smem {
  __nv_bfloat16 A[2][BM][LDS];
  __nv_bfloat16 B[2][BN][LDS];
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void *p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Weight row of tile column q (0..127) in n-tile `nt`; returns -1 past the end.
template <int MODE>
__device__ __forceinline__ long weight_row(const GemmArgs &a, int nt, int q) {
  if (MODE == MODE_W13) {
    const int qq = q & 31;
    const int j = nt * 64 + (q >> 5) * 16 + (qq & 15);
    const int up = qq >= 16;
    if (j >= a.N) return -1;
    return a.gate == GATE_SEPARATED ? (long)(up ? a.N + j : j) : (long)(2 * j + up);
  } else {
    const int i = nt * BN + q;
    return i < a.K ? i : -1;
  }
}

template <int MODE, int WK>
__global__ void __launch_bounds__(THREADS) gemm_kernel(GemmArgs a) {
  __shared__ __align__(16) Smem sm;
  // dependent launch: wait for the producer of the sorted rows / operands
  // (it may still be draining); the next kernel may be scheduled now
  griddep_wait();
  griddep_launch_dependents();
  const int blk = blockIdx.x;
  const int nt = blockIdx.y;
  if ((long)blk * BM >= (long)*a.num_post_pad) return;
  const int e = a.expert_ids[blk];
  if (e < 0 || e >= a.El) return;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;
  const int Kred = MODE == MODE_W13 ? a.K : a.N;  // reduction length
  const int R = MODE == MODE_W13 ? 2 * a.N : a.K;  // weight rows per expert
  const int KT = Kred / BK;
  const bool fp8_block = WK == WK_FP8 && a.wfmt == W_FP8_BLOCK128;

  // ---------------- A staging assignment: row tid/4, 8 elements at (tid%4)*8
  const int a_row = tid >> 2, a_kc = (tid & 3) * 8;
  const long a_r = (long)blk * BM + a_row;
  const int a_s = a.sorted_ids[a_r];
  const bool a_live = a_s < a.S;
  const long a_src = MODE == MODE_W13 ? (a_live ? a_s / a.T : 0) : a_r;

  // ---------------- B staging assignment: column q = tid/2, 16 elements at (tid%2)*16
  const int b_q = tid >> 1, b_kc = (tid & 1) * 16;
  const long b_wrow = weight_row<MODE>(a, nt, b_q);
  const bool b_live = b_wrow >= 0;
  const long b_row_g = (long)e * R + (b_live ? b_wrow : 0);  // global weight row

  // raw registers of one stage
  uint4 ra = make_uint4(0, 0, 0, 0);
  uint32_t ra_sc = 0;
  uint4 rb0 = make_uint4(0, 0, 0, 0), rb1 = make_uint4(0, 0, 0, 0);
  uint32_t rb_sc = 0;

  auto load_stage = [&](int kt) {
    const int k0 = kt * BK;
    // A
    if (a_live) {
      if (WK == WK_BF16 || WK == WK_MXFP4) {
        ra = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.a_codes) +
                                                   a_src * Kred + k0 + a_kc));
      } else if (WK == WK_FP8 || WK == WK_MX_A8) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(
            static_cast<const uint8_t *>(a.a_codes) + a_src * Kred + k0 + a_kc));
        ra.x = v.x; ra.y = v.y;
        if (WK == WK_MX_A8)  // one 32-element block per stage (BK == 32)
          ra_sc = static_cast<const uint8_t *>(a.a_scales)[a_src * (Kred / 32) + k0 / 32];
      } else if (WK == WK_MX_A4) {
        ra.x = __ldg(reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(a.a_codes) +
                                                        a_src * (Kred / 2) + (k0 + a_kc) / 2));
        ra_sc = static_cast<const uint8_t *>(a.a_scales)[a_src * (Kred / 32) + k0 / 32];
      } else {
        ra.x = __ldg(reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(a.a_codes) +
                                                        a_src * (Kred / 2) + (k0 + a_kc) / 2));
        ra_sc = static_cast<const uint8_t *>(a.a_scales)[a_src * (Kred / 16) + (k0 + a_kc) / 16];
      }
    }
    // B
    if (b_live) {
      if (WK == WK_BF16) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.w_codes) +
                                                         b_row_g * Kred + k0 + b_kc);
        rb0 = __ldg(p);
        rb1 = __ldg(p + 1);
      } else if (WK == WK_FP8) {
        rb0 = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(a.w_codes) +
                                                    b_row_g * Kred + k0 + b_kc));
      } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(
            static_cast<const uint8_t *>(a.w_codes) + b_row_g * (Kred / 2) + (k0 + b_kc) / 2));
        rb0.x = v.x; rb0.y = v.y;
        if (mx_weights<WK>())
          rb_sc = static_cast<const uint8_t *>(a.w_scales)[b_row_g * (Kred / 32) + k0 / 32];
        else
          rb_sc = static_cast<const uint8_t *>(a.w_scales)[b_row_g * (Kred / 16) + (k0 + b_kc) / 16];
      }
    }
  };

  auto store_stage = [&](int buf) {
    // A: 8 elements -> 16 bytes
    uint4 va;
    if (!a_live) {
      va = make_uint4(0, 0, 0, 0);
    } else if (WK == WK_BF16 || WK == WK_MXFP4) {
      va = ra;
    } else if (WK == WK_FP8 || WK == WK_MX_A8) {
      const float sc = WK == WK_MX_A8 ? e8m0_to_f32(ra_sc) : 1.f;  // exact in bf16
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t src = i < 2 ? ra.x : ra.y;
        const int sh = (i & 1) * 16;
        w[i] = pack_bf16x2(e4m3_to_f32((src >> sh) & 0xff) * sc,
                           e4m3_to_f32((src >> (sh + 8)) & 0xff) * sc);
      }
      va = make_uint4(w[0], w[1], w[2], w[3]);
    } else if (WK == WK_MX_A4) {
      const float sc = e8m0_to_f32(ra_sc);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = pack_bf16x2(e2m1_to_f32((ra.x >> (8 * i)) & 15) * sc,
                           e2m1_to_f32((ra.x >> (8 * i + 4)) & 15) * sc);
      va = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      const float sc = e4m3_to_f32(ra_sc);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = pack_bf16x2(e2m1_to_f32((ra.x >> (8 * i)) & 15) * sc,
                           e2m1_to_f32((ra.x >> (8 * i + 4)) & 15) * sc);
      va = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4 *>(&sm.A[buf][a_row][a_kc]) = va;
    // B: 16 elements -> 32 bytes
    uint4 v0, v1;
    if (!b_live) {
      v0 = v1 = make_uint4(0, 0, 0, 0);
    } else if (WK == WK_BF16) {
      v0 = rb0;
      v1 = rb1;
    } else if (WK == WK_FP8) {
      uint32_t w[8];
      const uint32_t src[4] = {rb0.x, rb0.y, rb0.z, rb0.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t s = src[i >> 1];
        const int sh = (i & 1) * 16;
        w[i] = pack_bf16x2(e4m3_to_f32((s >> sh) & 0xff), e4m3_to_f32((s >> (sh + 8)) & 0xff));
      }
      v0 = make_uint4(w[0], w[1], w[2], w[3]);
      v1 = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      const float sc = mx_weights<WK>() ? e8m0_to_f32(rb_sc) : e4m3_to_f32(rb_sc);
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t s = i < 4 ? rb0.x : rb0.y;
        const int sh = (i & 3) * 8;
        w[i] = pack_bf16x2(e2m1_to_f32((s >> sh) & 15) * sc, e2m1_to_f32((s >> (sh + 4)) & 15) * sc);
      }
      v0 = make_uint4(w[0], w[1], w[2], w[3]);
      v1 = make_uint4(w[4], w[5], w[6], w[7]);
    }
    *reinterpret_cast<uint4 *>(&sm.B[buf][b_q][b_kc]) = v0;
    *reinterpret_cast<uint4 *>(&sm.B[buf][b_q][b_kc + 8]) = v1;
  };

  float acc[2][4][4];
  float part[2][4][4];  // per-128-block partial sums (FP8 128x128 blocks only)
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[mi][ni][c] = part[mi][ni][c] = 0.f;

  // per-thread output coordinates: rows (mi, half) and tile columns (ni, c)
  long src_row[2][2];  // A source row of each accumulator row (token or sorted row)
  bool row_live[2][2];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const long r = (long)blk * BM + wm * 32 + mi * 16 + (lane >> 2) + h * 8;
      const int s = a.sorted_ids[r];
      row_live[mi][h] = s < a.S;
      src_row[mi][h] = MODE == MODE_W13 ? (s < a.S ? s / a.T : 0) : r;
    }
  long col_wrow[4][2];
#pragma unroll
  for (int ni = 0; ni < 4; ++ni)
#pragma unroll
    for (int c = 0; c < 2; ++c) col_wrow[ni][c] = weight_row<MODE>(a, nt, wn * 32 + ni * 8 + (lane & 3) * 2 + c);

  auto compute = [&](int buf) {
#pragma unroll
    for (int kk = 0; kk < BK; kk += 16) {
      uint32_t af[2][4], bfr[4][2];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
        ldmatrix_x4(af[mi], &sm.A[buf][wm * 32 + mi * 16 + (lane & 15)][kk + (lane >> 4) * 8]);
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        uint32_t r[4];
        ldmatrix_x4(r, &sm.B[buf][wn * 32 + nj * 16 + (lane & 7) + (lane >> 4) * 8]
                                [kk + ((lane >> 3) & 1) * 8]);
        bfr[2 * nj][0] = r[0];
        bfr[2 * nj][1] = r[1];
        bfr[2 * nj + 1][0] = r[2];
        bfr[2 * nj + 1][1] = r[3];
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          if (fp8_block) mma_bf16(part[mi][ni], af[mi], bfr[ni][0], bfr[ni][1]);
          else mma_bf16(acc[mi][ni], af[mi], bfr[ni][0], bfr[ni][1]);
        }
    }
  };

  auto promote = [&](int kb) {
    const int Ga = (int)ceil_div(Kred, 128);                 // A groups along the reduction
    const long RB = ceil_div(R, 128), CB = ceil_div(Kred, 128);
    const float *as = static_cast<const float *>(a.a_scales);
    const float *ws = static_cast<const float *>(a.w_scales);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float sa = row_live[mi][h] ? as[src_row[mi][h] * Ga + kb] : 0.f;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const long wr = col_wrow[ni][c];
            const float sw = wr >= 0 ? ws[((long)e * RB + wr / 128) * CB + kb] : 0.f;
            acc[mi][ni][h * 2 + c] += part[mi][ni][h * 2 + c] * (sa * sw);
            part[mi][ni][h * 2 + c] = 0.f;
          }
      }
  };

  // ---------------- main loop: register-staged double buffer
  if (KT > 0) {
    load_stage(0);
    store_stage(0);
  }
  __syncthreads();
  for (int kt = 0; kt < KT; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < KT) load_stage(kt + 1);
    compute(buf);
    if (fp8_block && (kt == KT - 1 || ((kt + 1) * BK) % 128 == 0)) promote((kt * BK) / 128);
    if (kt + 1 < KT) store_stage(buf ^ 1);
    __syncthreads();
  }

  // ---------------- epilogue
  auto row_factor = [&](int mi, int h) -> float {
    if (WK == WK_FP8) {
      if (a.afmt == A_FP8_TENSOR_STATIC || a.afmt == A_FP8_TENSOR_DYN)
        return static_cast<const float *>(a.a_scales)[0];
      if (a.afmt == A_FP8_TOKEN_DYN)
        return row_live[mi][h] ? static_cast<const float *>(a.a_scales)[src_row[mi][h]] : 0.f;
      return 1.f;
    }
    if (WK == WK_NVFP4) return MODE == MODE_W13 ? a.a_global[0] : a.a_global[e];
    return 1.f;
  };
  auto col_factor = [&](long wr) -> float {
    if (wr < 0) return 0.f;
    if (WK == WK_FP8) {
      if (a.wfmt == W_FP8_TENSOR) return static_cast<const float *>(a.w_scales)[e];
      if (a.wfmt == W_FP8_CHANNEL) return static_cast<const float *>(a.w_scales)[(long)e * R + wr];
      return 1.f;
    }
    if (WK == WK_NVFP4) return a.w_global[e];
    return 1.f;
  };
  auto col_bias = [&](long wr) -> float {
    if (!a.w_bias || wr < 0) return 0.f;
    const long i = (long)e * R + wr;
    return a.bias_f32 ? static_cast<const float *>(a.w_bias)[i]
                      : bf16_to_f32(static_cast<const uint16_t *>(a.w_bias)[i]);
  };

  if (MODE == MODE_W13) {
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const long r = (long)blk * BM + wm * 32 + mi * 16 + (lane >> 2) + h * 8;
        const float rf = row_factor(mi, h);
        // router weight on the stage-1 output (apply_router_weight_on_input)
        const float zw = (a.w_stage1 && row_live[mi][h]) ? a.topk_weights[a.sorted_ids[r]] : 1.f;
#pragma unroll
        for (int ni = 0; ni < 2; ++ni) {
          float z[2];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const long wg = col_wrow[ni][c], wu = col_wrow[ni + 2][c];
            const float g = acc[mi][ni][h * 2 + c] * rf * col_factor(wg) + col_bias(wg);
            const float u = acc[mi][ni + 2][h * 2 + c] * rf * col_factor(wu) + col_bias(wu);
            z[c] = row_live[mi][h] ? zw * act_and_mul(a.act, g, u, a.alpha, a.beta, a.limit) : 0.f;
          }
          const int j = nt * 64 + wn * 16 + ni * 8 + (lane & 3) * 2;
          if (j < a.N) {  // N is a multiple of 32, so j + 1 < N as well
            if (a.out_f32) {
              *reinterpret_cast<float2 *>(static_cast<float *>(a.out) + r * a.N + j) =
                  make_float2(z[0], z[1]);
            } else {
              *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(a.out) + r * a.N + j) =
                  pack_bf16x2(z[0], z[1]);
            }
          }
        }
      }
  } else {
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!row_live[mi][h]) continue;
        const long r = (long)blk * BM + wm * 32 + mi * 16 + (lane >> 2) + h * 8;
        const int s = a.sorted_ids[r];
        const long t = s / a.T;
        const float wt = a.w_stage1 ? 1.f : a.topk_weights[s];
        const float rf = row_factor(mi, h);
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const long wr = col_wrow[ni][c];
            if (wr < 0) continue;
            const float y = acc[mi][ni][h * 2 + c] * rf * col_factor(wr) + col_bias(wr);
            atomicAdd(a.acc + t * a.K + wr, wt * y);
          }
      }
  }
}

template <int MODE>
cudaError_t launch_mode(const GemmArgs &a, long cap_rows, cudaStream_t stream) {
  const long blocks = cap_rows / BM;
  if (blocks <= 0) return cudaSuccess;
  const long ntiles = MODE == MODE_W13 ? ceil_div(a.N, 64) : ceil_div(a.K, BN);
  dim3 grid((unsigned)blocks, (unsigned)ntiles);
  switch (a.wfmt) {
    case W_BF16: return launch_kernel(gemm_kernel<MODE, WK_BF16>, grid, dim3(THREADS), 0, stream, true, a);
    case W_FP8_TENSOR:
    case W_FP8_CHANNEL:
    case W_FP8_BLOCK128:
      return launch_kernel(gemm_kernel<MODE, WK_FP8>, grid, dim3(THREADS), 0, stream, true, a);
    case W_MXFP4:
      if (a.afmt == A_MXFP4_DYN)
        return launch_kernel(gemm_kernel<MODE, WK_MX_A4>, grid, dim3(THREADS), 0, stream, true, a);
      if (a.afmt == A_MXFP8_DYN)
        return launch_kernel(gemm_kernel<MODE, WK_MX_A8>, grid, dim3(THREADS), 0, stream, true, a);
      return launch_kernel(gemm_kernel<MODE, WK_MXFP4>, grid, dim3(THREADS), 0, stream, true, a);
    case W_NVFP4: return launch_kernel(gemm_kernel<MODE, WK_NVFP4>, grid, dim3(THREADS), 0, stream, true, a);
    default: return cudaErrorInvalidValue;
  }
}

__global__ void finalize_kernel(const float *__restrict__ acc, long n, uint16_t *__restrict__ out) {
  griddep_wait();  // the accumulator is complete (dependent launch after the w2 kernel)
  const long i = ((long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i + 3 < n) {
    const float4 v = *reinterpret_cast<const float4 *>(acc + i);
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2 *>(out + i) = o;
  } else {
    for (long k = i; k < n; ++k) {
      __nv_bfloat16 b = __float2bfloat16_rn(acc[k]);
      out[k] = *reinterpret_cast<uint16_t *>(&b);
    }
  }
}

__global__ void zero_kernel(float *__restrict__ buf, long n) {
  const long stride = (long)gridDim.x * blockDim.x;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) buf[i] = 0.f;
}

}  // namespace

cudaError_t launch_gemm_w13(const GemmArgs &a, long cap_rows, cudaStream_t stream) {
  return launch_mode<MODE_W13>(a, cap_rows, stream);
}

cudaError_t launch_gemm_w2(const GemmArgs &a, long cap_rows, cudaStream_t stream) {
  return launch_mode<MODE_W2>(a, cap_rows, stream);
}

cudaError_t launch_finalize(const float *acc, long n, void *out_bf16, cudaStream_t stream,
                            bool dependent) {
  if (n <= 0) return cudaSuccess;
  return launch_kernel(finalize_kernel, dim3((unsigned)ceil_div(ceil_div(n, 4), 256)), dim3(256), 0,
                       stream, dependent, acc, n, static_cast<uint16_t *>(out_bf16));
}

cudaError_t launch_zero(float *buf, long n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  long ctas = ceil_div(n, 256 * 8);
  if (ctas > 4 * 152) ctas = 4 * 152;
  zero_kernel<<<(unsigned)ctas, 256, 0, stream>>>(buf, n);
  return cudaGetLastError();
}

}  // namespace moe
