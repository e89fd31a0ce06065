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
// walks a static list of tiles; its stage ring runs across tile boundaries.
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
//               weight and adds into the fp32 token accumulator (W2)
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
constexpr int NS = 4;          // stages in the ring
constexpr int STAGE_A = BM * BK;                   // 16 KB
constexpr int STAGE_B = BN * BK;                   // 32 KB
constexpr int NUM_EPI = 16;
constexpr int THREADS = (2 + NUM_EPI) * 32;        // 576
constexpr int TMEM_COLS = 512;                     // two promotion buffers of 256 columns
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kErrTimeout = 5;
constexpr int kRasterGroup = 8;

enum { MODE_W13 = 0, MODE_W2 = 1 };

struct Smem {
  unsigned char a[NS][STAGE_A];
  unsigned char b[NS][STAGE_B];
  uint64_t full[NS], empty[NS];
  uint64_t acc_full[2], acc_empty[2], drain;
  // W13: the per-thread maxima of a row's 1 x 128 group (four threads hold
  // it), double-buffered by tile
  alignas(16) float amax_stage[2][BM][4];
  uint64_t staged[2], freed[2];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;
static_assert(offsetof(Smem, b) % 1024 == 0 && offsetof(Smem, amax_stage) % 16 == 0,
              "shared-memory layout alignment");

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
  extern __shared__ unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = (int)ceil_div(a.C, BK);
  const long ntiles_total = a.nblocks * a.ntiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
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
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quarter of this warp
    const int cq = (warp - 2) >> 2;   // tile columns [64 cq, 64 cq + 64)
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + 64 * cq;
    const float *ws = static_cast<const float *>(a.w_scales);
    const long RB = ceil_div(a.R, 128), CB = KT;
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
      // weight scale rows of this thread's two 32-column halves (block of
      // 128 weight rows; a 32-row group never crosses a block boundary)
      const long wr0 = group_row<MODE>(a, nt, 2 * cq), wr1 = group_row<MODE>(a, nt, 2 * cq + 1);
      const float *sw0 = wr0 < a.R ? ws + ((long)e * RB + wr0 / 128) * CB : nullptr;
      const float *sw1 = wr1 < a.R ? ws + ((long)e * RB + wr1 / 128) * CB : nullptr;
      const float *sa = a.a_groupscale + r * a.a_groups;
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.f;
      float fa = live ? sa[0] : 0.f;
      float f0 = sw0 ? fa * sw0[0] : 0.f, f1 = sw1 ? fa * sw1[0] : 0.f;
      for (int kt = 0; kt < KT; ++kt, ++g) {
        const int b = (int)(g & 1);
        // the next block's scales are loaded while this one is folded
        const float fa_n = (live && kt + 1 < KT) ? sa[kt + 1] : 0.f;
        const float f0_n = (sw0 && kt + 1 < KT) ? fa_n * sw0[kt + 1] : 0.f;
        const float f1_n = (sw1 && kt + 1 < KT) ? fa_n * sw1[kt + 1] : 0.f;
        if (!wait_or_abort(&sm.acc_full[b], (uint32_t)((g >> 1) & 1), a.err, abort_flag)) {
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
        f0 = f0_n;
        f1 = f1_n;
      }
      if (!ok) break;
      auto bias_of = [&](long wrow) -> float {
        if (!a.w_bias) return 0.f;
        const long i = (long)e * a.R + wrow;
        return a.bias_f32 ? static_cast<const float *>(a.w_bias)[i]
                          : bf16_to_f32(static_cast<const uint16_t *>(a.w_bias)[i]);
      };
      if (MODE == MODE_W13) {
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
          z[i] = (live && in) ? zw * act_and_mul(a.act, gv, uv, a.alpha, a.beta, a.limit) : 0.f;
          amax = fmaxf(amax, fabsf(z[i]));
        }
        // the row's 1 x 128 group maximum from its four threads
        const int sb = (int)(etile & 1);
        const uint32_t sph = (uint32_t)((etile >> 1) & 1);
        ok = mbar_wait_bounded(&sm.freed[sb], sph ^ 1, kWaitCycles, a.err);
        if (ok) {
          sm.amax_stage[sb][q * 32 + lane][cq] = amax;
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.staged[sb]);
          ok = mbar_wait_bounded(&sm.staged[sb], sph, kWaitCycles, a.err);
        }
        if (ok) {
          const float4 m4 = *reinterpret_cast<const float4 *>(&sm.amax_stage[sb][q * 32 + lane][0]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.freed[sb]);
          const float scale = fp8_group_scale(fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w)));
          if (in) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = f32x2_to_e4m3x2(__fdiv_rn(z[4 * i], scale), __fdiv_rn(z[4 * i + 1], scale)) |
                     (f32x2_to_e4m3x2(__fdiv_rn(z[4 * i + 2], scale),
                                      __fdiv_rn(z[4 * i + 3], scale)) << 16);
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
      } else if (live) {
        const long tok = s_id / a.T;
        const float wt = a.w_stage1 ? 1.f : a.topk_weights[s_id];
        const long i0 = (long)nt * BN + 64 * cq;
        float *dst = a.acc + tok * a.K + i0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i0 + 4 * i >= a.K) break;
          float y[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) y[u] = wt * (acc[4 * i + u] + bias_of(i0 + 4 * i + u));
          red_add_v4(dst + 4 * i, y[0], y[1], y[2], y[3]);
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
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_dev[dev] = 1;
  }
  fp8b_gemm_kernel<MODE><<<(unsigned)grid, THREADS, SMEM_BYTES, st>>>(ta, tb, a);
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
