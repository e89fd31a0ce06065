// moe_tc.cu -- tcgen05 grouped GEMMs of the fused experts for prefill-sized
// batches ("rocm_aiter_fused_experts" on page "vllm.model_executor.layers.
// fused_moe.experts.rocm_aiter_moe"; weight formats of the AITER leaves there,
// GptOssMxfp4MoEMethod on the mxfp4.py page and QuarkNvfp4MoEMethod on the
// quark_moe page).
//
// One CTA computes a 128 x 128 tile: 128 sorted rows of one expert (the sort
// pads every expert to a multiple of 128) x 128 weight rows, accumulated in
// TMEM.  Operand kinds:
//   K_BF16  bf16 weights:   A (sorted bf16 rows) and B by 2-D TMA, kind::f16
//   K_FP8   e4m3 weights:   A (sorted e4m3 codes) and B by 2-D TMA, kind::f8f6f4
//   K_FP4   MXFP4 weights:  A (sorted f16 rows) by 2-D TMA; B streamed as
//                           load-time packed records (TMA bulk copy) and
//                           decoded by the eight epilogue warps into exact f16
//                           (code x group scale) in the swizzled layout,
//                           kind::f16 with f16 operands
// Every stage is 128 bytes of reduction per row (64 bf16 / 128 e4m3), i.e. one
// 128-byte swizzle atom.  Warp roles: warp 0 TMA producer; warp 1 TMEM owner,
// lane 0 issues tcgen05.mma + tcgen05.commit; warps 2-9 epilogue (tcgen05.ld,
// scales, bias, activation or router weight + red.add); for FP4 weights the
// same eight warps decode B during the main loop.  (NVFP4 weights run on the
// block-scaled kernels of moe_bs.cu; the gather below prepares their A rows.)  FP8 128x128 block scales: every 128-wide reduction block lands in
// one of two TMEM buffers and the epilogue warps fold it into registers with
// a_scale[row, kb] * w_scale[block, kb] (promotion).  Two CTAs share an SM
// (3-stage rings, 256 TMEM columns each), so one CTA's epilogue overlaps the
// other's main loop.  All waits are bounded.
//
// W13 tile rows: SEPARATED -> [gate j0..j0+31 | up j0..j0+31 | gate j0+32..63 |
// up j0+32..63]; INTERLEAVED -> the weight rows 2*j0 .. 2*j0+127 as stored
// (gate, up alternate).  Either way the gate and up of an output j sit in the
// same epilogue thread's 64 columns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = kTcBlockM;   // 128
constexpr int BN = 128;
constexpr int NS = 3;
constexpr int STAGE_A = BM * 128;
constexpr int STAGE_B = BN * 128;
constexpr int NUM_EPI = 8;   // epilogue warps; for FP4 weights they also decode B
constexpr int NUM_DEC = NUM_EPI;
constexpr int THREADS = (2 + NUM_EPI) * 32;  // 320: two CTAs per SM
constexpr int TMEM_COLS = 256;
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kErrTimeout = 5;

enum { MODE_W13 = 0, MODE_W2 = 1 };
enum { K_BF16 = 0, K_FP8 = 1, K_FP4 = 2 };

struct Smem {
  unsigned char a[NS][STAGE_A];
  unsigned char b[NS][STAGE_B];
  unsigned char raw[NS][kTcRecMaxBytes];
  uint64_t full_a[NS], full_raw[NS], full_b[NS], empty[NS], raw_empty[NS];
  uint64_t acc_full[2], acc_empty[2], done;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;  // + alignment slack

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// First weight row (within the expert) of 32-row group `b` (0..3) of n-tile nt.
template <int MODE>
__device__ __forceinline__ long group_row(const TcArgs &a, int nt, int b) {
  if (MODE == MODE_W13) {
    if (a.gate == GATE_SEPARATED) {
      const long j = (long)nt * 64 + (b >> 1) * 32;
      return (b & 1) ? a.N + j : j;
    }
    return (long)nt * 128 + 32 * b;
  }
  return (long)nt * BN + 32 * b;
}

// Swizzled byte offset of 16-byte chunk c of row n in a 128-row x 128-byte tile.
__device__ __forceinline__ uint32_t sw128(int n, int c) {
  return (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4));
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, const TcArgs &a,
                                              volatile int *abort_flag) {
  if (*abort_flag) return false;
  if (!mbar_wait_bounded(bar, parity, kWaitCycles, a.err)) {
    record_device_error(a.err, kErrTimeout);
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

constexpr int kTcRasterGroup = 1;
constexpr int kPrefetchStages = 12;  // FP4 weight records prefetched into L2 ahead

template <int MODE, int KIND>
__global__ void __launch_bounds__(THREADS, 2)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Grouped raster: groups of `mgroup` m-blocks walk the n-tiles together, m
  // fastest inside a group.  With one m-block per group (the setting used) the
  // CTAs resident at one time share one A block and stream the weight tiles of
  // its expert; an m-fastest order re-read A from DRAM once per n-tile wave.
  int nt, blk;
  {
    const long id = blockIdx.x, span = (long)a.mgroup * a.ntiles;
    const long g0 = id / span * a.mgroup;
    const long gs = min((long)a.mgroup, a.nblocks - g0);
    const long local = id - g0 * a.ntiles;
    blk = (int)(g0 + local % gs);
    nt = (int)(local / gs);
  }
  if ((long)blk * BM >= (long)*a.num_post_pad) return;  // uniform for the CTA
  const int e = a.expert_ids[blk];
  if (e < 0 || e >= a.El) return;
  const bool promote = KIND == K_FP8 && a.wfmt == W_FP8_BLOCK128;
  const int BKE = KIND == K_FP8 ? 128 : 64;  // reduction elements per stage
  const int KT = (a.C + BKE - 1) / BKE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full_a[s], 1);
      mbar_init(&sm.full_raw[s], 1);
      mbar_init(&sm.full_b[s], NUM_DEC);
      mbar_init(&sm.empty[s], 1);
      mbar_init(&sm.raw_empty[s], NUM_DEC);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], NUM_EPI);
    }
    mbar_init(&sm.done, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const long rec_stride = (long)a.rec_bytes;
      int issued = 0, issued_raw = 0;  // stages whose copies were started
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % NS;
        const uint32_t par = ((kt / NS) & 1) ^ 1;
        if (!wait_or_abort(&sm.empty[s], par, a, abort_flag)) break;
        issued = kt + 1;
        if (KIND == K_FP4) {
          mbar_arrive_expect_tx(&sm.full_a[s], STAGE_A);
          tma_load_2d(sm.a[s], &tmA, kt * BKE, blk * BM, &sm.full_a[s]);
          // the weight records of one tile are contiguous: keep the next
          // kPrefetchStages of them on their way into L2, far ahead of the
          // small shared-memory ring (the weight stream is latency-bound)
          const unsigned char *tile_rec = static_cast<const unsigned char *>(a.w_packed) +
              ((long)e * a.ntiles + nt) * KT * rec_stride;
          {
            const int p0 = kt == 0 ? 1 : kt + kPrefetchStages;
            const int p1 = min(KT, kt == 0 ? 1 + kPrefetchStages : p0 + 1);
            if (p0 < p1)
              prefetch_l2_bulk(tile_rec + p0 * rec_stride, (uint32_t)((p1 - p0) * rec_stride));
          }
          if (!wait_or_abort(&sm.raw_empty[s], par, a, abort_flag)) break;
          issued_raw = kt + 1;
          const unsigned char *src = tile_rec + kt * rec_stride;
          mbar_arrive_expect_tx(&sm.full_raw[s], (uint32_t)a.rec_bytes);
          tma_bulk_g2s(sm.raw[s], src, (uint32_t)a.rec_bytes, &sm.full_raw[s]);
        } else {
          mbar_arrive_expect_tx(&sm.full_a[s], STAGE_A + STAGE_B);
          tma_load_2d(sm.a[s], &tmA, kt * BKE, blk * BM, &sm.full_a[s]);
#pragma unroll
          for (int b = 0; b < 4; ++b)
            tma_load_2d(sm.b[s] + b * 4096, &tmB, kt * BKE,
                        (int)((long)e * a.R + group_row<MODE>(a, nt, b)), &sm.full_a[s]);
        }
      }
      if (*abort_flag) {
        // after an abort, let the copies already issued land before the CTA
        // exits (bounded; no early exit on the error word here)
        for (int kt = issued > NS ? issued - NS : 0; kt < issued; ++kt)
          mbar_wait_bounded(&sm.full_a[kt % NS], (kt / NS) & 1, kWaitCycles);
        for (int kt = issued_raw > NS ? issued_raw - NS : 0; kt < issued_raw; ++kt)
          mbar_wait_bounded(&sm.full_raw[kt % NS], (kt / NS) & 1, kWaitCycles);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = KIND == K_FP8   ? umma_idesc_e4m3(BM, BN)
                                 : KIND == K_FP4 ? umma_idesc_f16(BM, BN)
                                                 : umma_idesc_bf16(BM, BN);
      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % NS;
        const uint32_t par = (kt / NS) & 1;
        if (!wait_or_abort(&sm.full_a[s], par, a, abort_flag)) break;
        if (KIND == K_FP4 && !wait_or_abort(&sm.full_b[s], par, a, abort_flag)) break;
        tc_fence_after();
        uint32_t d = tmem;
        bool fresh = kt == 0;
        if (promote) {  // one 128-wide reduction block per stage
          const int buf = kt & 1;
          if (!wait_or_abort(&sm.acc_empty[buf], ((kt / 2) & 1) ^ 1, a, abort_flag)) break;
          tc_fence_after();
          d = tmem + buf * BN;
          fresh = true;
        }
        const uint64_t ad = umma_desc_sw128(smem_addr(sm.a[s]));
        const uint64_t bd = umma_desc_sw128(smem_addr(sm.b[s]));
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // 4 MMAs of 32 bytes of reduction each
          if (KIND == K_FP8) umma_f8(d, ad + 2 * j, bd + 2 * j, idesc, (fresh && j == 0) ? 0u : 1u);
          else umma_f16(d, ad + 2 * j, bd + 2 * j, idesc, (fresh && j == 0) ? 0u : 1u);
        }
        umma_commit(&sm.empty[s]);
        if (promote) umma_commit(&sm.acc_full[kt & 1]);
      }
      if (!promote) umma_commit(&sm.done);
    }
  } else {
    if (KIND == K_FP4) {
      // ---------------------------------------------------------- FP4 decode
      // 256 threads, 4 chunks of 8 reduction elements each per stage:
      // thread t decodes row t/2, chunks 4*(t&1) .. 4*(t&1)+3.
      const int t = threadIdx.x - 64;
      const int n = t >> 1, c0 = (t & 1) * 4;

      for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % NS;
        const uint32_t par = (kt / NS) & 1;
        if (!wait_or_abort(&sm.full_raw[s], par, a, abort_flag)) break;
        if (!wait_or_abort(&sm.empty[s], par ^ 1, a, abort_flag)) break;
        const unsigned char *rec = sm.raw[s];
        const uint4 cw = *reinterpret_cast<const uint4 *>(rec + n * 32 + c0 * 4);
        const uint32_t sc = rec[4096 + n * 2 + (c0 >> 2)];  // e8m0 of these 32 elements
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.raw_empty[s]);
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
        // the group scale 2^(sc - 127) as an f16x2 pair (exact: the e8m0 codes
        // are range-checked at load time)
        const uint32_t sh = sc >= 113 ? (sc - 112) << 10 : 1u << (sc - 103);
        const uint32_t f = sh | (sh << 16);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t hv[4];
          e2m1x8_to_f16x2x4(words[u], hv);
          uint4 o;
          o.x = hmul2_u32(hv[0], f);
          o.y = hmul2_u32(hv[1], f);
          o.z = hmul2_u32(hv[2], f);
          o.w = hmul2_u32(hv[3], f);
          *reinterpret_cast<uint4 *>(sm.b[s] + sw128(n, c0 + u)) = o;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.full_b[s]);
      }
    }
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;              // 0..7
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int h = ew >> 2;                // column half: tile columns [64h, 64h+64)
    const long r = (long)blk * BM + q * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const int s_id = a.sorted_ids[r];
    const bool live = s_id < a.S;
    float acc[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = 0.f;

    if (promote) {
      const long RB = (a.R + 127) / 128, CB = KT;
      const float *ws = static_cast<const float *>(a.w_scales);
      const float *sa_row = a.a_groupscale + r * a.a_groups;
      const float *sw_ptr[2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const long br = group_row<MODE>(a, nt, 2 * h + cc) / 128;
        sw_ptr[cc] = br < RB ? ws + ((long)e * RB + br) * CB : nullptr;
      }
      // the block scales of stage kb+2 are loaded while stage kb is promoted
      auto load_f = [&](int kb, float (&f)[2]) {
        const float sa = (live && kb < KT) ? sa_row[kb] : 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) f[cc] = (sw_ptr[cc] && kb < KT) ? sa * sw_ptr[cc][kb] : 0.f;
      };
      float f_cur[2], f_nxt[2];
      load_f(0, f_cur);
      load_f(1, f_nxt);
      for (int kb = 0; kb < KT; ++kb) {
        const int buf = kb & 1;
        float f_far[2];
        load_f(kb + 2, f_far);
        if (!wait_or_abort(&sm.acc_full[buf], (kb / 2) & 1, a, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float v[16];
            tmem_ld_32x32b_x16(trow + buf * BN + 64 * h + 32 * cc + 16 * p, v);
#pragma unroll
            for (int i = 0; i < 16; i += 2)
              fma_f32x2(acc[32 * cc + 16 * p + i], acc[32 * cc + 16 * p + i + 1], v[i], v[i + 1],
                        f_cur[cc]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          f_cur[cc] = f_nxt[cc];
          f_nxt[cc] = f_far[cc];
        }
      }
    } else if (wait_or_abort(&sm.done, 0, a, abort_flag)) {
      tc_fence_after();
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        float v[16];
        tmem_ld_32x32b_x16(trow + 64 * h + 16 * p, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[16 * p + i] = v[i];
      }
    }

    if (!*abort_flag) {
      float rf = 1.f;
      if (a.a_scalar) rf *= a.a_scalar[0];
      if (a.a_rowscale) rf *= a.a_rowscale[r];
      if (a.a_expertscale) rf *= a.a_expertscale[e];
      auto col_factor = [&](long wrow) -> float {
        if (KIND == K_FP8) {
          if (a.wfmt == W_FP8_TENSOR) return static_cast<const float *>(a.w_scales)[e];
          if (a.wfmt == W_FP8_CHANNEL)
            return static_cast<const float *>(a.w_scales)[(long)e * a.R + wrow];
          return 1.f;
        }
        if (a.wfmt == W_NVFP4) return a.w_global[e];
        return 1.f;
      };
      auto bias_of = [&](long wrow) -> float {
        if (!a.w_bias) return 0.f;
        const long i = (long)e * a.R + wrow;
        return a.bias_f32 ? static_cast<const float *>(a.w_bias)[i]
                          : bf16_to_f32(static_cast<const uint16_t *>(a.w_bias)[i]);
      };
      if (MODE == MODE_W13) {
        // router weight on the stage-1 output (apply_router_weight_on_input)
        const float zw = (a.w_stage1 && live) ? a.topk_weights[s_id] : 1.f;
        const int jbase = nt * 64 + 32 * h;
        if (jbase < a.N) {  // N % 32 == 0: the 32 outputs are all in range or none
          const bool sep = a.gate == GATE_SEPARATED;
          const bool mx_out = a.out_mode == TC_OUT_MX4_F16 || a.out_mode == TC_OUT_MX8_F16;
          float zb[32];  // MX: the 32 outputs are one OCP MX block (jbase % 32 == 0)
#pragma unroll
          for (int p = 0; p < 2; ++p) {  // 16 outputs per pass
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int ii = 16 * p + i;
              const long j = jbase + ii;
              const float gacc = sep ? acc[ii] : acc[2 * ii];
              const float uacc = sep ? acc[32 + ii] : acc[2 * ii + 1];
              const long grow = sep ? j : 2 * j;
              const long urow = sep ? a.N + j : 2 * j + 1;
              const float gv = gacc * rf * col_factor(grow) + bias_of(grow);
              const float uv = uacc * rf * col_factor(urow) + bias_of(urow);
              z[i] = live ? zw * act_and_mul(a.act, gv, uv, a.alpha, a.beta, a.limit) : 0.f;
            }
            if (mx_out) {
#pragma unroll
              for (int i = 0; i < 16; ++i) zb[16 * p + i] = z[i];
            } else if (a.out_mode == TC_OUT_F32) {
              float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + r * a.N + jbase + 16 * p);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_float4(z[4 * i], z[4 * i + 1], z[4 * i + 2], z[4 * i + 3]);
            } else if (a.out_mode == TC_OUT_F16) {
              uint32_t w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const __half2 h2 = __floats2half2_rn(z[2 * i], z[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t *>(&h2);
              }
              uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + r * a.N + jbase + 16 * p);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
              uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + r * a.N + jbase + 16 * p);
#pragma unroll
              for (int i = 0; i < 2; ++i)
                dst[i] = make_uint4(pack_bf16x2(z[8 * i], z[8 * i + 1]),
                                    pack_bf16x2(z[8 * i + 2], z[8 * i + 3]),
                                    pack_bf16x2(z[8 * i + 4], z[8 * i + 5]),
                                    pack_bf16x2(z[8 * i + 6], z[8 * i + 7]));
            }
          }
          if (mx_out) {  // quantise-dequantise the block into exact f16
            uint32_t w[16];
            mx_qdq_f16x32(zb, a.out_mode == TC_OUT_MX4_F16, w);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + r * a.N + jbase);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
      } else if (live) {
        const long t = s_id / a.T;
        const float wt = a.w_stage1 ? 1.f : a.topk_weights[s_id];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const long i0 = (long)nt * BN + 64 * h + 32 * cc;
          if (i0 >= a.K) continue;  // K % 32 == 0: a chunk is fully in or out
          float *dst = a.acc + t * a.K + i0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float y[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const long wrow = i0 + 4 * i + u;
              y[u] = wt * (acc[32 * cc + 4 * i + u] * rf * col_factor(wrow) + bias_of(wrow));
            }
            red_add_v4(dst + 4 * i, y[0], y[1], y[2], y[3]);
          }
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

// ------------------------------------------------------------------ gather
// Sorted-order activation rows for the w13 GEMM: e4m3 codes copied as they
// are (fp8 formats), e2m1 codes + scale-factor records (NVFP4, the
// block-scaled kernels: quantised here from the bf16 rows, or copied from
// moe_quant_act's output), bf16 rows, or f16 rows scaled per row by a power of
// two (MXFP4 weights), plus per-row / per-group scales.  One warp per sorted
// row.
__global__ void gather_rows_kernel(GatherArgs g) {
  const long r = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= *g.num_post_pad) return;
  const int s = g.sorted_ids[r];
  const bool live = s < g.S;
  const long t = live ? s / g.T : 0;
  if (g.x16) {  // f16 token rows converted once per token by the sort
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(g.out) + r * g.K);
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g.x16) + t * g.K);
    for (int c = lane; c < g.K / 8; c += 32) dst[c] = live ? src[c] : make_uint4(0, 0, 0, 0);
    if (lane == 0) g.rowscale[r] = live ? g.x_inv[t] : 0.f;
  } else if (g.afmt == A_BF16 && !g.to_f16) {
    uint16_t *dst = static_cast<uint16_t *>(g.out) + r * g.K;
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g.codes) + t * g.K);
    for (int c = lane; c < g.K / 8; c += 32)
      reinterpret_cast<uint4 *>(dst)[c] = live ? src[c] : make_uint4(0, 0, 0, 0);
  } else if (g.afmt == A_BF16 || g.afmt == A_MXFP4_DYN || g.afmt == A_MXFP8_DYN) {
    // f16 rows scaled by 2^a so that the row maximum lands in [2^14, 2^15)
    // (exact for bf16 values); rowscale = 2^-a.  MX formats: g.codes is the
    // bf16 x and each 32-element block is quantised and dequantised first
    // (|QDQ(x)| <= 1.75 * 2^floor(log2 max|x|) stays below 2^15 after 2^a).
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g.codes) + t * g.K);
    float amax = 0.f;
    for (int c = lane; live && c < g.K / 8; c += 32) {
      const uint4 v = src[c];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                                 fabsf(__uint_as_float(w[i] & 0xffff0000u))));
    }
    amax = warp_max(amax);
    int ex = 0, a = 0;
    if (amax > 0.f) {
      frexpf(amax, &ex);
      a = 15 - ex;
    }
    const float mul = ldexpf(1.0f, a);
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(g.out) + r * g.K);
    const int mx = g.afmt == A_MXFP4_DYN ? 1 : g.afmt == A_MXFP8_DYN ? 2 : 0;
    // chunk c holds elements 8c..8c+7 and c % 4 == lane % 4: the four lanes
    // of a 32-element block run every iteration together (K % 32 == 0)
    const unsigned gmask = 0xFu << (lane & 28);
    for (int c = lane; c < g.K / 8; c += 32) {
      uint4 o = make_uint4(0, 0, 0, 0);
      if (live) {
        const uint4 v = src[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        if (mx) {
          float f[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
          }
          o = mx_qdq_f16x8(f, mx == 1, a, gmask);
        } else {
          uint32_t q[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16) * mul,
                                                __uint_as_float(w[i] & 0xffff0000u) * mul);
            q[i] = *reinterpret_cast<const uint32_t *>(&h);
          }
          o = make_uint4(q[0], q[1], q[2], q[3]);
        }
      }
      dst[c] = o;
    }
    if (lane == 0) g.rowscale[r] = live ? ldexpf(1.0f, -a) : 0.f;
  } else if (g.afmt == A_NVFP4_DYN && g.sf_out && g.x_nvfp4) {
    // block-scaled operand quantised here from the token's bf16 row (the
    // stage-1 quantiser's rule, nvfp4_quant16): lane l takes the 16-element
    // group 32 i + l; the first lane of every four packs the step's four
    // scales into its record word (and replicas); zeros for padding rows and
    // past K
    const long KS = ceil_div(g.K, kTcBsStage);
    const int G = g.K / 16;
    const float gs = g.nv_global[0];
    const uint4 *xr = reinterpret_cast<const uint4 *>(g.x_nvfp4 + t * g.K);
    uint8_t *dst = static_cast<uint8_t *>(g.out) + r * (g.K / 2);
    uint8_t *sf = static_cast<uint8_t *>(g.sf_out);
    for (int i = 0; i < (G + 31) / 32; ++i) {  // warp-uniform
      const int grp = 32 * i + lane;
      uint32_t lo = 0, hi = 0, sb = 0;
      if (live && grp < G) {
        const uint4 u0 = xr[2 * grp], u1 = xr[2 * grp + 1];
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float v[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          v[2 * k] = __uint_as_float(w[k] << 16);
          v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
        sb = nvfp4_quant16(v, gs, lo, hi);
      }
      if (grp < G) *reinterpret_cast<uint2 *>(dst + 8 * grp) = make_uint2(lo, hi);
      const uint32_t word = sb | (__shfl_down_sync(0xffffffffu, sb, 1) << 8) |
                            (__shfl_down_sync(0xffffffffu, sb, 2) << 16) |
                            (__shfl_down_sync(0xffffffffu, sb, 3) << 24);
      if ((lane & 3) == 0 && grp < G) {
        const long o = bs_sfa_offset(r, (long)(grp / 4) * 64, KS);
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint32_t *>(sf + o + 1024 * q) = word;
      }
    }
    for (int st = (G + 3) / 4 + lane; st < KS * 4; st += 32) {  // steps past K
      const long o = bs_sfa_offset(r, (long)st * 64, KS);
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint32_t *>(sf + o + 1024 * q) = 0u;
    }
  } else if (g.afmt == A_NVFP4_DYN && g.sf_out) {
    // block-scaled operand: the codes row as it is, and its ue4m3 scales into
    // the scale-factor records of the sorted rows (zeros past K and for
    // padding rows)
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(g.out) + r * (g.K / 2));
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(g.codes) +
                                                       t * (g.K / 2));
    for (int c = lane; c < g.K / 32; c += 32) dst[c] = live ? src[c] : make_uint4(0, 0, 0, 0);
    // the four scales of a 64-element step are one aligned word of the
    // record (and of each replica): one 4-byte load, four 4-byte stores
    const long KS = ceil_div(g.K, kTcBsStage);
    const int G = g.K / 16;
    const uint8_t *sc = static_cast<const uint8_t *>(g.scales) + t * G;
    uint8_t *sf = static_cast<uint8_t *>(g.sf_out);
    for (int st = lane; st < KS * 4; st += 32) {
      uint32_t v = 0;
      if (live && 4 * st + 3 < G && (G & 3) == 0) {
        v = reinterpret_cast<const uint32_t *>(sc)[st];
      } else if (live) {
        for (int b = 0; b < 4; ++b)
          if (4 * st + b < G) v |= (uint32_t)sc[4 * st + b] << (8 * b);
      }
      const long o = bs_sfa_offset(r, (long)st * 64, KS);
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint32_t *>(sf + o + 1024 * q) = v;
    }
  } else {  // fp8 codes, copied
    uint8_t *dst = static_cast<uint8_t *>(g.out) + r * g.K;
    const uint8_t *src = static_cast<const uint8_t *>(g.codes) + t * g.K;
    for (int c = lane; c < g.K / 16; c += 32)
      reinterpret_cast<uint4 *>(dst)[c] =
          live ? reinterpret_cast<const uint4 *>(src)[c] : make_uint4(0, 0, 0, 0);
    for (int c = (g.K / 16) * 16 + lane; c < g.K; c += 32) dst[c] = live ? src[c] : 0;
    if (g.afmt == A_FP8_TOKEN_DYN && lane == 0)
      g.rowscale[r] = live ? static_cast<const float *>(g.scales)[t] : 0.f;
    if (g.afmt == A_FP8_GROUP128_DYN) {
      const int G = (g.K + 127) / 128;
      for (int c = lane; c < G; c += 32)
        g.groupscale[r * G + c] = live ? static_cast<const float *>(g.scales)[t * G + c] : 0.f;
    }
  }
}

// fp32 intermediate rows -> f16 rows scaled by 2^a (row maximum in
// [2^14, 2^15)) and rowscale = 2^-a; rows at or beyond num_post_pad are left
// alone, padding rows become zeros.  One warp per row.
__global__ void rescale_rows_kernel(const float *__restrict__ src, long cap, int N,
                                    const int32_t *__restrict__ sorted_ids,
                                    const int32_t *__restrict__ ntp, int S,
                                    uint16_t *__restrict__ dst, float *__restrict__ rowscale) {
  const long r = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= *ntp) return;
  const bool live = sorted_ids[r] < S;
  const float4 *s4 = reinterpret_cast<const float4 *>(src + r * N);
  float amax = 0.f;
  for (int c = lane; live && c < N / 4; c += 32) {
    const float4 v = s4[c];
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  amax = warp_max(amax);
  int ex = 0, a = 0;
  if (amax > 0.f) {
    frexpf(amax, &ex);
    a = 15 - ex;
  }
  const float mul = ldexpf(1.0f, a);
  uint2 *d2 = reinterpret_cast<uint2 *>(dst + r * N);
  for (int c = lane; c < N / 4; c += 32) {
    uint2 o = make_uint2(0, 0);
    if (live) {
      const float4 v = s4[c];
      const __half2 h0 = __floats2half2_rn(v.x * mul, v.y * mul);
      const __half2 h1 = __floats2half2_rn(v.z * mul, v.w * mul);
      o = make_uint2(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1));
    }
    d2[c] = o;
  }
  if (lane == 0) rowscale[r] = live ? ldexpf(1.0f, -a) : 0.f;
}

// Range of the e8m0 scale codes of a weight tensor (for the f16 decode check).
__global__ void scale_range_kernel(const uint8_t *__restrict__ s, long n, int *__restrict__ mn,
                                   int *__restrict__ mx) {
  int lo = 255, hi = 0;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int v = s[i];
    lo = min(lo, v);
    hi = max(hi, v);
  }
  atomicMin(mn, lo);
  atomicMax(mx, hi);
}

// ------------------------------------------------------------------ packing
// Load-time records of FP4 weights for the decoders: per (expert, n-tile,
// 64-wide reduction stage) [128 rows x 32 code bytes][128 rows x scale bytes],
// rows in the tile order of the kernel.  One thread per record byte.
__global__ void pack_tc_fp4_kernel(TcPackArgs p) {
  const long o = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= p.total) return;
  const long rec = o / p.rec_bytes;
  const int wb = (int)(o % p.rec_bytes);
  const int kt = (int)(rec % p.kstages);
  const long ent = rec / p.kstages;
  const int nt = (int)(ent % p.ntiles);
  const long e = ent / p.ntiles;
  const int sb = 2;  // e8m0 scale bytes per row per stage
  int n;
  bool code;
  int byte_in_row;
  if (wb < 4096) {
    code = true;
    n = wb / 32;
    byte_in_row = wb % 32;
  } else if (wb < 4096 + 128 * sb) {
    code = false;
    n = (wb - 4096) / sb;
    byte_in_row = (wb - 4096) % sb;
  } else {
    p.out[o] = 0;
    return;
  }
  // weight row of tile row n
  const int b = n >> 5;
  long row;
  bool valid;
  if (p.w13) {
    if (p.gate == GATE_SEPARATED) {
      const long j = (long)nt * 64 + (b >> 1) * 32 + (n & 31);
      valid = j < p.N;
      row = (b & 1) ? p.N + j : j;
    } else {
      row = (long)nt * 128 + n;
      valid = row < 2L * p.N;
    }
  } else {
    row = (long)nt * 128 + n;
    valid = row < p.R;
  }
  unsigned char v;
  if (code) {
    const long k2 = (long)kt * 32 + byte_in_row;  // byte index along the row (2 codes per byte)
    v = (valid && k2 < p.C / 2) ? p.codes[((long)e * p.R + row) * (p.C / 2) + k2] : 0;
  } else {
    const long grp = (long)kt * 2 + byte_in_row;
    v = (valid && grp < p.C / 32) ? p.scales[((long)e * p.R + row) * (p.C / 32) + grp] : 127;
  }
  p.out[o] = v;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D K-major tensor map with 128-byte swizzle: rows x cols elements, box
// (128 bytes of columns) x box_rows.
bool make_map(CUtensorMap *tm, const void *base, long rows, long cols, bool bytes, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int esz = bytes ? 1 : 2;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / esz), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int KIND>
cudaError_t launch_tc_t(const CUtensorMap &ta, const CUtensorMap &tb, const TcArgs &a, long blocks,
                        cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE, KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  tc_gemm_kernel<MODE, KIND><<<(unsigned)(blocks * a.ntiles), THREADS, SMEM_BYTES, st>>>(ta, tb, a);
  return cudaGetLastError();
}

}  // namespace

// 2-D K-major byte tensor map with the 128-byte swizzle (the block-scaled
// kernels' A operand: rows of packed e2m1 codes).
bool make_tc_map_u8(CUtensorMap *tm, const void *base, long rows, long cols, int box_rows) {
  return make_map(tm, base, rows, cols, true, box_rows);
}

// 2-D K-major 16-bit tensor map with the 128-byte swizzle (the weight-streaming
// kernels' slot rows).
bool make_tc_map_b16(CUtensorMap *tm, const void *base, long rows, long cols, int box_rows) {
  return make_map(tm, base, rows, cols, false, box_rows);
}

int tc_ntiles(int w13, int N, int K) { return w13 ? (int)ceil_div(N, 64) : (int)ceil_div(K, BN); }

size_t tc_packed_bytes(int w13, int nvfp4, int N, int K, int El) {
  if (nvfp4) return bs_packed_bytes(w13, N, K, El);  // block-scaled records
  const int C = w13 ? K : N;
  return (size_t)El * tc_ntiles(w13, N, K) * ceil_div(C, 64) * (4096 + 128 * 2);
}

cudaError_t launch_pack_tc_fp4(const TcPackArgs &p, cudaStream_t st) {
  if (p.total <= 0) return cudaSuccess;
  if (p.nvfp4) return launch_pack_bs(p, st);
  pack_tc_fp4_kernel<<<(unsigned)ceil_div(p.total, 256), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rescale_rows(const float *src, long cap, int N, const int32_t *sorted_ids,
                                const int32_t *ntp, int S, void *dst, float *rowscale,
                                cudaStream_t st) {
  if (cap <= 0) return cudaSuccess;
  rescale_rows_kernel<<<(unsigned)ceil_div(cap * 32, 256), 256, 0, st>>>(
      src, cap, N, sorted_ids, ntp, S, static_cast<uint16_t *>(dst), rowscale);
  return cudaGetLastError();
}

cudaError_t launch_scale_range(const uint8_t *s, long n, int *mn_mx, cudaStream_t st) {
  const int init[2] = {255, 0};
  cudaError_t e = cudaMemcpyAsync(mn_mx, init, sizeof(init), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  long blocks = ceil_div(n, 256);
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  scale_range_kernel<<<(unsigned)blocks, 256, 0, st>>>(s, n, mn_mx, mn_mx + 1);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const GatherArgs &g, long cap_rows, cudaStream_t st) {
  if (cap_rows <= 0) return cudaSuccess;
  gather_rows_kernel<<<(unsigned)ceil_div(cap_rows * 32, 256), 256, 0, st>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_tc_gemm(const TcArgs &a_in, const void *a_sorted, long cap_rows, int w13,
                           cudaStream_t st) {
  TcArgs a = a_in;
  a.ntiles = tc_ntiles(w13, a.N, a.K);
  const long blocks = cap_rows / BM;
  if (blocks <= 0) return cudaSuccess;
  if (blocks * a.ntiles > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  a.nblocks = blocks;
  a.mgroup = (int)min(blocks, (long)kTcRasterGroup);
  const int kind = a.wfmt == W_BF16 ? K_BF16 : a.wfmt == W_MXFP4 ? K_FP4 : K_FP8;
  CUtensorMap ta, tb;
  if (!make_map(&ta, a_sorted, cap_rows, a.C, kind == K_FP8, BM)) return cudaErrorInvalidValue;
  if (kind == K_FP4) {
    tb = ta;  // unused
    a.rec_bytes = 4096 + 128 * 2;
  } else if (!make_map(&tb, a.w_codes, (long)a.El * a.R, a.C, kind == K_FP8, 32)) {
    return cudaErrorInvalidValue;
  }
  if (w13) {
    switch (kind) {
      case K_BF16: return launch_tc_t<MODE_W13, K_BF16>(ta, tb, a, blocks, st);
      case K_FP8: return launch_tc_t<MODE_W13, K_FP8>(ta, tb, a, blocks, st);
      default: return launch_tc_t<MODE_W13, K_FP4>(ta, tb, a, blocks, st);
    }
  }
  switch (kind) {
    case K_BF16: return launch_tc_t<MODE_W2, K_BF16>(ta, tb, a, blocks, st);
    case K_FP8: return launch_tc_t<MODE_W2, K_FP8>(ta, tb, a, blocks, st);
    default: return launch_tc_t<MODE_W2, K_FP4>(ta, tb, a, blocks, st);
  }
}

}  // namespace moe
