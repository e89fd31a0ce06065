// moe_fp8.cu -- persistent tcgen05 grouped GEMMs of the fused experts for FP8
// weights with 128 x 128 block scales and 1 x 128 dynamic activation groups
// (AiterFp8BlockExperts on page
// "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe": e4m3 weights
// with one fp32 scale per 128 x 128 block, e4m3 activations with one fp32
// scale per token and 128 columns; the intermediate is requantised the same
// way before the second GEMM).
//
// The tensor cores multiply e4m3 codes (kind::f8f6f4, fp32 accumulation in
// Tensor Memory); the block scales cannot ride in the MMA (they are arbitrary
// fp32, not powers of two), so every 128-wide reduction block is accumulated
// on its own in one of two Tensor Memory buffers and folded into registers by
// the epilogue warps as acc += partial * a_scale[row, kb] * w_scale[n-block, kb]
// ("promotion"), while the tensor cores fill the other buffer.
//
// Tiles are 128 sorted rows (one expert) x 256 weight rows; one reduction
// stage is one 128-wide block (128 bytes of codes per row).  One CTA per SM
// walks a static list of tiles (block-major: each block's n-tiles in turn);
// its stage ring runs across tile boundaries.
// Warp roles:
//   warp 0      TMA producer: the A rows (2-D TMA, 128-byte swizzle) and the
//               256 weight rows as eight 32-row boxes -- 48 KB per stage
//   warp 1      TMEM owner; lane 0 issues the stage's four MMAs into the
//               promotion buffer of the stage and commits it
//   warps 2-17  epilogue: each thread owns one row and 64 columns; per stage
//               it copies its 64 partial sums out of Tensor Memory, releases
//               the buffer and folds them in with the block scales; after the
//               tile's last stage it applies the bias and activation and
//               quantises the row's 128 outputs (one 1 x 128 group, its
//               maximum gathered from the four threads that hold it) into
//               e4m3 codes + an fp32 scale (W13), or multiplies the router
//               weight and adds into the fp32 token accumulator (W2): each
//               warp transposes its 32 rows through shared memory 32 columns
//               at a time, so that one red.add instruction covers 4 rows x 128
//               contiguous bytes instead of 32 rows x 16 bytes
//   warp 18     each stage's scales (the 128 rows' activation-group scales and
//               the block scales of the eight 32-row weight groups) into a
//               shared-memory ring, ahead of the MMAs, so that the epilogue
//               reads no scale from global memory
// Every wait is bounded; on a timeout the CTA records MOE_ERR_TIMEOUT, stops
// issuing, lets its copies and MMAs land, frees its Tensor Memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stddef.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = kTcBlockM;  // 128 sorted rows
constexpr int BN = 256;        // weight rows per tile
constexpr int BK = 128;        // reduction elements (= bytes) per stage: one scale block
// stages in the ring: W2 keeps one fewer to make room for its transposition
// buffers
template <int MODE> constexpr int ring_stages() { return MODE == 0 ? 4 : 3; }
constexpr int NSC = 8;         // stages in the scale ring
constexpr int SC_FLOATS = 136; // per scale stage: 128 rows + 8 weight groups
constexpr int STAGE_A = BM * BK;                   // 16 KB
constexpr int STAGE_B = BN * BK;                   // 32 KB
constexpr int NUM_EPI = 16;
constexpr int SCALE_WARP = 2 + NUM_EPI;             // 18
constexpr int THREADS = (3 + NUM_EPI) * 32;        // 608
constexpr int TMEM_COLS = 512;                     // two promotion buffers of 256 columns
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kErrTimeout = 5;
// m-blocks that walk the n-tiles together (1: each block walks its n-tiles in
// turn; an expert's blocks are adjacent, so they still share its weight tiles
// through L2): DeepSeek-V3 at M=4096, ms per step 3.521 / 3.550 / 3.548 /
// 3.568 for 1 / 2 / 4 / 8 (16 / 32 / 64 slower still)
constexpr int kRasterGroup = 1;


enum { MODE_W13 = 0, MODE_W2 = 1 };

template <int MODE>
struct Smem {
  static constexpr int NS = ring_stages<MODE>();
  unsigned char a[NS][STAGE_A];
  unsigned char b[NS][STAGE_B];
  uint64_t full[NS], empty[NS];
  uint64_t acc_full[2], acc_empty[2], drain;
  // scale ring: [0, 128) the rows' activation-group scales of the stage's
  // block, [128, 136) the block scales of weight group c (32 rows) = 0..7
  alignas(16) float sc[NSC][SC_FLOATS];
  uint64_t sc_full[NSC], sc_empty[NSC];
  // W13: the per-thread maxima of a row's 1 x 128 group (four threads hold
  // it), double-buffered by tile
  alignas(16) float amax_stage[MODE == 0 ? 2 : 1][BM][4];
  // W2: per epilogue warp, 32 rows x 32 columns of outputs, each row's eight
  // 16-byte units stored at unit (u ^ (row & 7)) (conflict-free both ways)
  alignas(16) float xpose[MODE == 0 ? 1 : NUM_EPI][32 * 32];
  uint64_t staged[2], freed[2];
  uint32_t tmem_base;
  int abort_flag;
};
template <int MODE> constexpr size_t smem_bytes() { return sizeof(Smem<MODE>) + 1024; }
static_assert(offsetof(Smem<0>, b) % 1024 == 0 && offsetof(Smem<1>, b) % 1024 == 0 &&
                  offsetof(Smem<0>, sc) % 16 == 0 && offsetof(Smem<1>, sc) % 16 == 0 &&
                  offsetof(Smem<0>, amax_stage) % 16 == 0 && offsetof(Smem<1>, xpose) % 16 == 0 &&
                  (SC_FLOATS * 4) % 16 == 0,
              "shared-memory layout alignment");
static_assert(smem_bytes<0>() <= 227 * 1024 && smem_bytes<1>() <= 227 * 1024,
              "shared memory per CTA");

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, int *err,
                                              volatile int *abort_flag) {
  if (*abort_flag) return false;
  if (!mbar_wait_bounded(bar, parity, kWaitCycles, err)) {
    record_device_error(err, kErrTimeout);
    *abort_flag = 1;
    return false;
  }
  return true;
}

// Activation of one (gate, up) pair with the fast exponential and divide
// intrinsics (a few fp32 ulps, far below the e4m3 intermediate's step).
__device__ __forceinline__ float act_fast(int act, float g, float u, float alpha, float beta,
                                          float limit) {
  if (act == ACT_SILU) return __fdividef(g, 1.0f + __expf(-g)) * u;
  if (act == ACT_GELU) return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f)) * u;
  if (limit > 0.0f) {
    g = fminf(g, limit);
    u = fminf(fmaxf(u, -limit), limit);
  }
  return (u + beta) * __fdividef(g, 1.0f + __expf(-alpha * g));
}

// An epilogue wait whose outcome is the same on every lane of the warp (the
// warp then leaves its loops together: its shuffles and warp barriers never
// wait for a lane that has left).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int *err,
                                          volatile int *abort_flag) {
  const bool ok = wait_or_abort(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// x / d from the reciprocal rd = 1 / d (rounded): the product, then one
// correction by its fma residual (Markstein's quotient step) -- the correctly
// rounded quotient except in rare cases, whose one-ulp difference the e4m3
// rounding that follows absorbs but at a tie.
__device__ __forceinline__ float div_by(float x, float d, float rd) {
  const float q = x * rd;
  return fmaf(fmaf(-q, d, x), rd, q);
}

__device__ __forceinline__ void red_add_v4(float *p, float x, float y, float z, float w) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x), "f"(y), "f"(z),
               "f"(w)
               : "memory");
}

__device__ __forceinline__ void tile_coords(long t, long nblocks, int ntiles, int &blk, int &nt) {
  const long span = (long)kRasterGroup * ntiles;
  const long g0 = t / span * kRasterGroup;
  const long gs = min((long)kRasterGroup, nblocks - g0);
  const long local = t - g0 * ntiles;
  blk = (int)(g0 + local % gs);
  nt = (int)(local / gs);
}

// First weight row (within the expert) of 32-row group b (0..7) of n-tile nt:
// W13 SEPARATED -> gate and up rows of outputs nt * 128 + 32 (b / 2) .. + 31
// alternate; W13 INTERLEAVED and W2 -> rows nt * 256 + 32 b as stored.
template <int MODE>
__device__ __forceinline__ long group_row(const TcArgs &a, int nt, int b) {
  if (MODE == MODE_W13 && a.gate == GATE_SEPARATED) {
    const long j = (long)nt * 128 + (b >> 1) * 32;
    return (b & 1) ? a.N + j : j;
  }
  return (long)nt * BN + 32 * b;
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
fp8b_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const TcArgs a) {
  constexpr int NS = ring_stages<MODE>();
  extern __shared__ unsigned char smem_raw[];
  Smem<MODE> &sm = *reinterpret_cast<Smem<MODE> *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = (int)ceil_div(a.C, BK);
  const long ntiles_total = a.nblocks * a.ntiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < NSC; ++s) {
      mbar_init(&sm.sc_full[s], 32);
      mbar_init(&sm.sc_empty[s], NUM_EPI);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], NUM_EPI);
      mbar_init(&sm.staged[b], NUM_EPI);
      mbar_init(&sm.freed[b], NUM_EPI);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int *abort_flag = &sm.abort_flag;
  const int ntp = *a.num_post_pad;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      long g = 0;
      for (long t = blockIdx.x; t < ntiles_total && !*abort_flag; t += gridDim.x) {
        int blk, nt;
        tile_coords(t, a.nblocks, a.ntiles, blk, nt);
        if ((long)blk * BM >= ntp) continue;
        const int e = a.expert_ids[blk];
        if (e < 0 || e >= a.El) continue;
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int s = (int)(g % NS);
          if (!wait_or_abort(&sm.empty[s], (uint32_t)(((g / NS) & 1) ^ 1), a.err, abort_flag))
            break;
          mbar_arrive_expect_tx(&sm.full[s], STAGE_A + STAGE_B);
          tma_load_2d(sm.a[s], &tmA, kt * BK, blk * BM, &sm.full[s]);
#pragma unroll
          for (int b = 0; b < 8; ++b)
            tma_load_2d(sm.b[s] + b * 4096, &tmB, kt * BK,
                        (int)((long)e * a.R + group_row<MODE>(a, nt, b)), &sm.full[s]);
        }
      }
      if (*abort_flag) {
        for (long k = g > NS ? g - NS : 0; k < g; ++k)
          mbar_wait_bounded(&sm.full[k % NS], (uint32_t)((k / NS) & 1), kWaitCycles);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_e4m3(BM, BN);
      long g = 0;
      for (long t = blockIdx.x; t < ntiles_total && !*abort_flag; t += gridDim.x) {
        int blk, nt;
        tile_coords(t, a.nblocks, a.ntiles, blk, nt);
        if ((long)blk * BM >= ntp) continue;
        const int e = a.expert_ids[blk];
        if (e < 0 || e >= a.El) continue;
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int s = (int)(g % NS), b = (int)(g & 1);
          if (!wait_or_abort(&sm.full[s], (uint32_t)((g / NS) & 1), a.err, abort_flag)) break;
          // the epilogue has folded the previous block this buffer held
          if (!wait_or_abort(&sm.acc_empty[b], (uint32_t)(((g >> 1) & 1) ^ 1), a.err, abort_flag))
            break;
          tc_fence_after();
          const uint64_t ad = umma_desc_sw128(smem_addr(sm.a[s]));
          const uint64_t bd = umma_desc_sw128(smem_addr(sm.b[s]));
#pragma unroll
          for (int j = 0; j < 4; ++j)  // 4 MMAs of 32 elements (32 bytes) each
            umma_f8(tmem + 256 * b, ad + 2 * j, bd + 2 * j, idesc, j == 0 ? 0u : 1u);
          umma_commit(&sm.empty[s]);
          umma_commit(&sm.acc_full[b]);
        }
      }
      umma_commit(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0, kWaitCycles);
    }
  } else if (warp == SCALE_WARP) {
    // ------------------------------------------------------------ scale ring
    {  // one entry per stage, in the MMAs' order
      const float *ws = static_cast<const float *>(a.w_scales);
      const long RB = ceil_div(a.R, 128), CB = KT;
      long g = 0;
      for (long t = blockIdx.x; t < ntiles_total && !*abort_flag; t += gridDim.x) {
        int blk, nt;
        tile_coords(t, a.nblocks, a.ntiles, blk, nt);
        if ((long)blk * BM >= ntp) continue;
        const int e = a.expert_ids[blk];
        if (e < 0 || e >= a.El) continue;
        const float *sa = a.a_groupscale + (long)blk * BM * a.a_groups;
        // the lanes 0-7 each own one weight group's block-scale row (none
        // past the weight's R rows); a 32-row group never crosses a block
        const float *swc = nullptr;
        if (lane < 8) {
          const long wr = group_row<MODE>(a, nt, lane);
          if (wr < a.R) swc = ws + ((long)e * RB + wr / 128) * CB;
        }
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int s = (int)(g % NSC);
          if (!wait_or_abort(&sm.sc_empty[s], (uint32_t)(((g / NSC) & 1) ^ 1), a.err, abort_flag))
            break;
#pragma unroll
          for (int i = lane; i < BM; i += 32) sm.sc[s][i] = sa[(long)i * a.a_groups + kt];
          if (lane < 8) sm.sc[s][BM + lane] = swc ? swc[kt] : 0.f;
          mbar_arrive(&sm.sc_full[s]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter of this warp
    const int cq = (warp - 2) >> 2;   // tile columns [64 cq, 64 cq + 64)
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + 64 * cq;
    const bool sep = MODE == MODE_W13 && a.gate == GATE_SEPARATED;
    long g = 0, etile = 0;
    bool ok = true;
    for (long t = blockIdx.x; t < ntiles_total && ok; t += gridDim.x) {
      int blk, nt;
      tile_coords(t, a.nblocks, a.ntiles, blk, nt);
      if ((long)blk * BM >= ntp) continue;
      const int e = a.expert_ids[blk];
      if (e < 0 || e >= a.El) continue;
      const long r = (long)blk * BM + q * 32 + lane;
      const int s_id = a.sorted_ids[r];
      const bool live = s_id < a.S;
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.f;
      for (int kt = 0; kt < KT; ++kt, ++g) {
        const int b = (int)(g & 1);
        // this block's scales from the ring: the row's activation-group
        // scale times the block scales of this thread's two weight groups
        const int s = (int)(g % NSC);
        if (!warp_wait(&sm.sc_full[s], (uint32_t)((g / NSC) & 1), a.err, abort_flag)) {
          ok = false;
          break;
        }
        const float fa = live ? sm.sc[s][q * 32 + lane] : 0.f;
        const float f0 = fa * sm.sc[s][BM + 2 * cq], f1 = fa * sm.sc[s][BM + 2 * cq + 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sc_empty[s]);
        if (!warp_wait(&sm.acc_full[b], (uint32_t)((g >> 1) & 1), a.err, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // 16 columns at a time (the 64 accumulators stay in registers)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[16];
          tmem_ld_32x32b_x16(tq + 256 * b + 16 * c, v);
          const float f = c < 2 ? f0 : f1;
#pragma unroll
          for (int i = 0; i < 16; i += 2) fma_f32x2(acc[16 * c + i], acc[16 * c + i + 1], v[i], v[i + 1], f);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[b]);  // the tensor cores may refill it
      }
      if (!ok) break;
      auto bias_of = [&](long wrow) -> float {
        if (!a.w_bias) return 0.f;
        const long i = (long)e * a.R + wrow;
        return a.bias_f32 ? static_cast<const float *>(a.w_bias)[i]
                          : bf16_to_f32(static_cast<const uint16_t *>(a.w_bias)[i]);
      };
      if constexpr (MODE == MODE_W13) {
        // outputs jbase .. jbase + 31 of the row: SEPARATED -> gate acc[i],
        // up acc[32 + i]; INTERLEAVED -> gate acc[2 i], up acc[2 i + 1]
        const int jbase = nt * 128 + 32 * cq;
        const bool in = jbase < a.N;  // N % 32 == 0: all 32 in range or none
        const float zw = (a.w_stage1 && live) ? a.topk_weights[s_id] : 1.f;
        float z[32];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const long j = jbase + i;
          const long grow = sep ? j : 2 * j, urow = sep ? a.N + j : 2 * j + 1;
          const float gv = (sep ? acc[i] : acc[2 * i]) + (in ? bias_of(grow) : 0.f);
          const float uv = (sep ? acc[32 + i] : acc[2 * i + 1]) + (in ? bias_of(urow) : 0.f);
          z[i] = (live && in) ? zw * act_fast(a.act, gv, uv, a.alpha, a.beta, a.limit) : 0.f;
          amax = fmaxf(amax, fabsf(z[i]));
        }
        // the row's 1 x 128 group maximum from its four threads
        const int sb = (int)(etile & 1);
        const uint32_t sph = (uint32_t)((etile >> 1) & 1);
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.freed[sb], sph ^ 1, kWaitCycles, a.err));
        if (ok) {
          sm.amax_stage[sb][q * 32 + lane][cq] = amax;
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.staged[sb]);
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.staged[sb], sph, kWaitCycles, a.err));
        }
        if (ok) {
          const float4 m4 = *reinterpret_cast<const float4 *>(&sm.amax_stage[sb][q * 32 + lane][0]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.freed[sb]);
          const float scale = fp8_group_scale(fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w)));
          if (in) {
            const float rs = __frcp_rn(scale);
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = f32x2_to_e4m3x2(div_by(z[4 * i], scale, rs), div_by(z[4 * i + 1], scale, rs)) |
                     (f32x2_to_e4m3x2(div_by(z[4 * i + 2], scale, rs),
                                      div_by(z[4 * i + 3], scale, rs)) << 16);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(a.out) + r * a.N + jbase);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
          if (cq == 0) a.out_scales[r * ceil_div(a.N, 128) + nt] = scale;
        } else {
          record_device_error(a.err, kErrTimeout);
          *abort_flag = 1;
        }
        ++etile;
      } else {
        // outputs i0 .. i0 + 63 of the row (token tok), 32 columns at a time
        // through this warp's transposition buffer: lane l then adds row
        // 4 j + l / 8, columns 4 (l % 8) .. + 3 of the chunk (one 128-byte
        // line per 8 lanes)
        const int tok = live ? s_id / a.T : -1;  // -1: padding row
        const float wt = live ? (a.w_stage1 ? 1.f : a.topk_weights[s_id]) : 0.f;
        const long i0 = (long)nt * BN + 64 * cq;
        float4 *xp = reinterpret_cast<float4 *>(sm.xpose[warp - 2]);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          if (i0 + 32 * ch >= a.K) break;  // warp-uniform
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = 32 * ch + 4 * u;
            const long col = i0 + c;  // K % 4 == 0: the 4 columns all in range or none
            const bool in = col < a.K;
            xp[lane * 8 + (u ^ (lane & 7))] =
                make_float4(wt * (acc[c] + (in ? bias_of(col) : 0.f)),
                            wt * (acc[c + 1] + (in ? bias_of(col + 1) : 0.f)),
                            wt * (acc[c + 2] + (in ? bias_of(col + 2) : 0.f)),
                            wt * (acc[c + 3] + (in ? bias_of(col + 3) : 0.f)));
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int rho = 4 * j + (lane >> 3), u = lane & 7;
            const int tok_r = __shfl_sync(0xffffffffu, tok, rho);
            const long col = i0 + 32 * ch + 4 * u;
            if (tok_r >= 0 && col < a.K) {
              const float4 v = xp[rho * 8 + (u ^ (rho & 7))];
              red_add_v4(a.acc + (long)tok_r * a.K + col, v.x, v.y, v.z, v.w);
            }
          }
          __syncwarp();
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

int fp8b_ntiles(int w13, int N, int K) { return w13 ? (int)ceil_div(N, 128) : (int)ceil_div(K, 256); }

bool make_tc_map_u8(CUtensorMap *tm, const void *base, long rows, long cols, int box_rows);

template <int MODE>
cudaError_t launch_fp8b_t(const CUtensorMap &ta, const CUtensorMap &tb, const TcArgs &a, int grid,
                          cudaStream_t st) {
  static int attr_dev[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_dev[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fp8b_gemm_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<MODE>());
    if (e != cudaSuccess) return e;
    attr_dev[dev] = 1;
  }
  fp8b_gemm_kernel<MODE><<<(unsigned)grid, THREADS, smem_bytes<MODE>(), st>>>(ta, tb, a);
  return cudaGetLastError();
}

cudaError_t launch_fp8b_gemm(const TcArgs &a_in, const void *a_codes, long cap_rows, int w13,
                             int sm_count, cudaStream_t st) {
  TcArgs a = a_in;
  a.ntiles = fp8b_ntiles(w13, a.N, a.K);
  const long blocks = cap_rows / BM;
  if (blocks <= 0) return cudaSuccess;
  a.nblocks = blocks;
  CUtensorMap ta, tb;
  if (!make_tc_map_u8(&ta, a_codes, cap_rows, a.C, BM)) return cudaErrorInvalidValue;
  if (!make_tc_map_u8(&tb, a.w_codes, (long)a.El * a.R, a.C, 32)) return cudaErrorInvalidValue;
  const long tiles = blocks * a.ntiles;
  const int grid = (int)(tiles < sm_count ? tiles : sm_count);
  return w13 ? launch_fp8b_t<MODE_W13>(ta, tb, a, grid, st)
             : launch_fp8b_t<MODE_W2>(ta, tb, a, grid, st);
}

}  // namespace moe
