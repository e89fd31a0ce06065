// moe_bs.cu -- persistent block-scaled tcgen05 grouped GEMMs of the fused
// experts for NVFP4 w4a4 prefill batches (QuarkNvfp4MoEMethod on page
// "vllm.model_executor.layers.quantization.quark.quark_moe": e2m1 codes, one
// e4m3 scale per 16 elements, an fp32 global per expert; the two GEMM stages
// of rocm_aiter_fused_experts on page
// "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe").
//
// Both operands stay in their storage format: the tensor cores multiply e2m1
// codes with their ue4m3 block scales (tcgen05.mma kind::mxf4nvf4,
// scale_vec::4X), accumulating in fp32 in Tensor Memory; the fp32 globals are
// applied in the epilogue.
//
// Tiles are 128 sorted rows (one expert; the sort pads each expert to 128) x
// 256 weight rows, reduction stages of 256 elements (128 bytes of codes per
// row).  One CTA per SM walks a static list of tiles (persistent); its stage
// ring runs across tile boundaries, so the loads of the next tile overlap the
// end of the current one.  Warp roles:
//   warp 0      TMA producer: per stage the A rows' codes (2-D TMA, 128-byte
//               swizzle), the A scale-factor record, the B record (codes
//               pre-swizzled + scale factors) -- 72 KB, one mbarrier
//   warp 1      TMEM owner; lane 0 issues each stage's four MMAs
//   warps 2-17  epilogue: each thread owns one row and 64 accumulator
//               columns; it copies them to registers, releases the
//               accumulator (the next tile's MMAs start) and then applies
//               the scales, bias, activation and NVFP4 quantiser (W13) or the
//               router weight and the fp32 reduce (W2)
//   warp 18     lane 0 copies each stage's scale factors from shared memory
//               into the stage's own Tensor Memory buffer (six tcgen05.cp
//               .128x256b: two for A, four for B; a copy instruction costs
//               the tensor pipe about the same whatever its width) as soon as
//               the stage has landed, and hands it to the MMA thread with a
//               commit on sf_full; the buffer is free again when the stage's
//               MMAs are (the producer's next copies into the stage, which
//               this warp waits for, come after that)
// Every wait is bounded; on a timeout the CTA records MOE_ERR_TIMEOUT, stops
// issuing, lets its copies and MMAs land, frees its Tensor Memory and exits.
#include <cuda.h>
#include <stddef.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = kTcBlockM;  // 128 sorted rows
constexpr int BN = 256;        // weight rows per tile
constexpr int NS = 3;          // stages in the ring
constexpr int STAGE_A = BM * 128;                  // 16 KB of A codes
constexpr int STAGE_B = BN * 128;                  // 32 KB of B codes
// B scale factors of a stage: one 4 KB .128x256b source per MMA step, row L =
// [step words of rows L % 32 + 32 w of rows 0-127 | the same for rows
// 128-255] (the layout of bs_sfa_offset with the B halves in place of the
// step pair)
constexpr int SFB_BYTES = 4 * 4096;
constexpr int NUM_EPI = 16;
constexpr int CP_WARP = 2 + NUM_EPI;               // warp 18
constexpr int THREADS = (3 + NUM_EPI) * 32;        // 608
constexpr int TMEM_COLS = 512;
// Tensor Memory columns: accumulator [0, 256); one buffer of scale factors
// (four MMA steps) per ring stage at 256 + 48 s: A at +0 (4 columns per step),
// B at +16 (8 per step: rows 0-127, then rows 128-255).  Within the 4 columns
// of a 128-row block and step, lane L column w holds the scale word of row
// L % 32 + 32 w, the same in all four lane quarters; byte b of a word scales
// the b-th 16-element block of the step.
constexpr uint32_t kAccCol = 0, kSfCol = 256, kSfBufCols = 48, kSfbOff = 16;
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kErrTimeout = 5;
// m-blocks that walk the n-tiles together: W13 (16 reduction stages per tile)
// 32, W2 (long tiles) 16 -- measured on the Mixtral NVFP4 prefill: DRAM reads
// of W13 2.09 / 1.46 / 1.11 GB for groups of 8 / 16 / 32, of W2 1.34 / 1.30 /
// 1.44 GB
template <int MODE> constexpr int kRasterGroup = MODE == 0 ? 32 : 16;
// Weight records are prefetched into L2 this many stages ahead of the ring
// (by the CTA of the first m-block of each raster group only: the others of
// the group read the same records), so the ring's copies hit L2.  Measured on
// the Mixtral NVFP4 prefill (ms per step): 1.690 / 1.650 / 1.639 / 1.647 /
// 1.659 for 0 / 2 / 4 / 8 / 16 stages.
constexpr int kPrefetchAhead = 4;

enum { MODE_W13 = 0, MODE_W2 = 1 };

struct Smem {
  unsigned char a[NS][STAGE_A];
  unsigned char b[NS][STAGE_B];
  unsigned char sfa[NS][kBsSfaRecBytes];
  unsigned char sfb[NS][SFB_BYTES];
  uint64_t full[NS], empty[NS];
  uint64_t sf_full[NS];
  uint64_t acc_full, acc_empty, drain, cp_drain;
  // W13: the scale factors of a tile's 128 intermediate columns (one 4 KB
  // .128x256b source of the W2 operand; its 32 distinct rows) are assembled
  // here and written out with 16-byte stores; double-buffered by tile
  alignas(16) unsigned char sf_stage[2][1024];  // read and written in 16-byte pieces
  uint64_t staged[2], freed[2];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;
// operand stages start on 1024-byte boundaries (128-byte swizzle atoms), the
// scale-factor sources and the staging buffer on 16-byte ones (bulk copies,
// tcgen05.cp, 16-byte shared-memory accesses)
static_assert(offsetof(Smem, b) % 1024 == 0 && offsetof(Smem, sfa) % 16 == 0 &&
                  offsetof(Smem, sfb) % 16 == 0 && offsetof(Smem, sf_stage) % 16 == 0,
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

// 32 consecutive fp32 columns of this warp's 32 lanes, without the wait.
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Tile t of the grid's list -> (m-block, n-tile): groups of kRasterGroup
// m-blocks walk the n-tiles together, m fastest, so the CTAs working at one
// time share each weight tile and each A block through L2.
template <int MODE>
__device__ __forceinline__ void tile_coords(long t, long nblocks, int ntiles, int &blk, int &nt) {
  constexpr int G = kRasterGroup<MODE>;
  const long span = (long)G * ntiles;
  const long g0 = t / span * G;
  const long gs = min((long)G, nblocks - g0);
  const long local = t - g0 * ntiles;
  blk = (int)(g0 + local % gs);
  nt = (int)(local / gs);
}

// Activation of one (gate, up) pair, fast forms (ex2-based exponential,
// approximate divide); their error (a few fp32 ulps) is far below the
// intermediate's NVFP4 step.
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

// NVFP4 x16 quantiser of the intermediate (one group of 16 outputs):
// s = e4m3(fl32(fl32(amax / 6) / g)); codes = e2m1 of v * (1 / fl32(e4m3(s) * g)).
// The element codes are decided on the product with the reciprocal (one
// divide per group): the values being quantised are the GPU's fp32 GEMM
// outputs, which already differ from an exact computation by rounding.
__device__ __forceinline__ uint32_t nvfp4_quant16_fast(const float (&v)[16], float gs,
                                                       uint32_t &lo, uint32_t &hi) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t s = f32_to_e4m3(__fdiv_rn(__fdiv_rn(amax, kE2m1Max), gs));
  const float sv = e4m3_to_f32(s);
  lo = hi = 0;
  if (sv != 0.f) {
    const float inv = __fdiv_rn(1.0f, __fmul_rn(sv, gs));
#pragma unroll
    for (int i = 0; i < 8; i += 2)
      lo |= f32x2_to_e2m1x2(v[i] * inv, v[i + 1] * inv) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; i += 2)
      hi |= f32x2_to_e2m1x2(v[8 + i] * inv, v[9 + i] * inv) << (4 * i);
  }
  return s;
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
bs_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = (int)ceil_div(a.C, kTcBsStage);
  const long ntiles_total = a.nblocks * a.ntiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < NS; ++s) mbar_init(&sm.sf_full[s], 1);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, NUM_EPI);
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.cp_drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.staged[b], NUM_EPI);
      mbar_init(&sm.freed[b], NUM_EPI);
    }
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
      long g = 0;  // stages issued
      for (long t = blockIdx.x; t < ntiles_total && !*abort_flag; t += gridDim.x) {
        int blk, nt;
        tile_coords<MODE>(t, a.nblocks, a.ntiles, blk, nt);
        if ((long)blk * BM >= ntp) continue;
        const int e = a.expert_ids[blk];
        if (e < 0 || e >= a.El) continue;
        const unsigned char *brec = static_cast<const unsigned char *>(a.w_packed) +
                                    ((long)e * a.ntiles + nt) * KT * (long)(STAGE_B + SFB_BYTES);
        const unsigned char *asf = static_cast<const unsigned char *>(a.a_sf) +
                                   (long)blk * KT * kBsSfaRecBytes;
        const bool leader = (blk % kRasterGroup<MODE>) == 0;
        if (leader && kPrefetchAhead > 0)
          prefetch_l2_bulk(brec, (uint32_t)(min(KT, kPrefetchAhead) * (STAGE_B + SFB_BYTES)));
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int s = (int)(g % NS);
          if (leader && kPrefetchAhead > 0 && kt + kPrefetchAhead < KT)
            prefetch_l2_bulk(brec + (long)(kt + kPrefetchAhead) * (STAGE_B + SFB_BYTES),
                             (uint32_t)(STAGE_B + SFB_BYTES));
          if (!wait_or_abort(&sm.empty[s], (uint32_t)(((g / NS) & 1) ^ 1), a.err, abort_flag)) {
            break;
          }
          const unsigned char *rec = brec + (long)kt * (STAGE_B + SFB_BYTES);
          mbar_arrive_expect_tx(&sm.full[s], STAGE_A + kBsSfaRecBytes + STAGE_B + SFB_BYTES);
          tma_load_2d(sm.a[s], &tmA, kt * 128, blk * BM, &sm.full[s]);
          tma_bulk_g2s(sm.sfa[s], asf + (long)kt * kBsSfaRecBytes, kBsSfaRecBytes, &sm.full[s]);
          tma_bulk_g2s(sm.b[s], rec, STAGE_B, &sm.full[s]);
          tma_bulk_g2s(sm.sfb[s], rec + STAGE_B, SFB_BYTES, &sm.full[s]);
        }
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA exits
        for (long k = g > NS ? g - NS : 0; k < g; ++k)
          mbar_wait_bounded(&sm.full[k % NS], (uint32_t)((k / NS) & 1), kWaitCycles);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_nvf4(BM, BN);
      long g = 0, tc = 0;
      for (long t = blockIdx.x; t < ntiles_total && !*abort_flag; t += gridDim.x) {
        int blk, nt;
        tile_coords<MODE>(t, a.nblocks, a.ntiles, blk, nt);
        if ((long)blk * BM >= ntp) continue;
        const int e = a.expert_ids[blk];
        if (e < 0 || e >= a.El) continue;
        // the epilogue has copied the previous tile's accumulator out
        if (!wait_or_abort(&sm.acc_empty, (uint32_t)((tc & 1) ^ 1), a.err, abort_flag)) break;
        tc_fence_after();
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int s = (int)(g % NS);
          // the stage's operands have landed (the scale-factor warp waited
          // for them) and its scale factors are in Tensor Memory buffer s
          if (!wait_or_abort(&sm.sf_full[s], (uint32_t)((g / NS) & 1), a.err, abort_flag)) break;
          tc_fence_after();
          const uint32_t sf = tmem + kSfCol + kSfBufCols * s;
          const uint64_t ad = umma_desc_sw128(smem_addr(sm.a[s]));
          const uint64_t bd = umma_desc_sw128(smem_addr(sm.b[s]));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            umma_nvf4(tmem + kAccCol, ad + 2 * j, bd + 2 * j, idesc, sf + 4 * j,
                      sf + kSfbOff + 8 * j, (kt == 0 && j == 0) ? 0u : 1u);
          umma_commit(&sm.empty[s]);
        }
        if (*abort_flag) break;
        umma_commit(&sm.acc_full);
        ++tc;
      }
      // every MMA and copy issued above has completed before Tensor Memory
      // is freed
      umma_commit(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0, kWaitCycles);
    }
  } else if (warp == CP_WARP) {
    // ------------------------------------------------------------ scale factors
    if (lane == 0) {
      long g = 0;
      for (long t = blockIdx.x; t < ntiles_total && !*abort_flag; t += gridDim.x) {
        int blk, nt;
        tile_coords<MODE>(t, a.nblocks, a.ntiles, blk, nt);
        if ((long)blk * BM >= ntp) continue;
        const int e = a.expert_ids[blk];
        if (e < 0 || e >= a.El) continue;
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int s = (int)(g % NS);
          // the stage has landed: its scale factors are in shared memory and
          // buffer s is free (the producer refilled the stage only after the
          // MMAs of its previous round completed)
          if (!wait_or_abort(&sm.full[s], (uint32_t)((g / NS) & 1), a.err, abort_flag)) break;
          tc_fence_after();
          const uint32_t sf = tmem + kSfCol + kSfBufCols * s;
          const uint32_t sfa = smem_addr(sm.sfa[s]), sfb = smem_addr(sm.sfb[s]);
#pragma unroll
          for (int p = 0; p < 2; ++p)  // A: steps 2p, 2p + 1 -> columns 8p .. 8p + 7
            tc_cp_128x256b(sf + 8 * p, sf256_smem_desc(sfa + 4096 * p));
#pragma unroll
          for (int j = 0; j < 4; ++j)  // B: step j -> columns 8j .. 8j + 7
            tc_cp_128x256b(sf + kSfbOff + 8 * j, sf256_smem_desc(sfb + 4096 * j));
          umma_commit(&sm.sf_full[s]);
        }
        if (*abort_flag) break;
      }
      // every copy issued above has completed before Tensor Memory is freed
      umma_commit(&sm.cp_drain);
      mbar_wait_bounded(&sm.cp_drain, 0, kWaitCycles);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quarter of this warp
    const int cq = (warp - 2) >> 2;     // column quarter: tile columns [64 cq, 64 cq + 64)
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + kAccCol + 64 * cq;
    long tc = 0, etile = 0;
    const float a_sc = a.a_scalar ? a.a_scalar[0] : 1.f;
    const long ks_out = ceil_div(a.N, kTcBsStage);
    for (long t = blockIdx.x; t < ntiles_total; t += gridDim.x) {
      int blk, nt;
      tile_coords<MODE>(t, a.nblocks, a.ntiles, blk, nt);
      if ((long)blk * BM >= ntp) continue;
      const int e = a.expert_ids[blk];
      if (e < 0 || e >= a.El) continue;
      const long r = (long)blk * BM + q * 32 + lane;
      const int s_id = a.sorted_ids[r];
      const bool live = s_id < a.S;
      if (!wait_or_abort(&sm.acc_full, (uint32_t)(tc & 1), a.err, abort_flag)) break;
      tc_fence_after();
      float acc[64];
      {
        uint32_t v0[32], v1[32];
        tmem_ld_x32(trow, v0);
        tmem_ld_x32(trow + 32, v1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          acc[i] = __uint_as_float(v0[i]);
          acc[32 + i] = __uint_as_float(v1[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty);  // the next tile's MMAs may start
      ++tc;

      const float wg = a.w_global[e];
      if (MODE == MODE_W13) {
        const float sc = a_sc * wg;  // stage-1 global x weight global
        const float zw = (a.w_stage1 && live) ? a.topk_weights[s_id] : 1.f;
        const int jbase = nt * 128 + 32 * cq;
        const bool sep = a.gate == GATE_SEPARATED;
        uint8_t sfq[2] = {0, 0};  // this thread's two group scales (0 past N)
        if (jbase < a.N) {  // N % 32 == 0: all 32 outputs in range or none
          const uint16_t *bias = static_cast<const uint16_t *>(a.w_bias);
          const float *bias32 = static_cast<const float *>(a.w_bias);
          uint32_t codes[4];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int ii = 16 * p + i;
              const long j = jbase + ii;
              float gv = (sep ? acc[ii] : acc[2 * ii]) * sc;
              float uv = (sep ? acc[32 + ii] : acc[2 * ii + 1]) * sc;
              if (a.w_bias) {
                const long grow = (long)e * a.R + (sep ? j : 2 * j);
                const long urow = (long)e * a.R + (sep ? a.N + j : 2 * j + 1);
                gv += a.bias_f32 ? bias32[grow] : bf16_to_f32(bias[grow]);
                uv += a.bias_f32 ? bias32[urow] : bf16_to_f32(bias[urow]);
              }
              z[i] = live ? zw * act_fast(a.act, gv, uv, a.alpha, a.beta, a.limit) : 0.f;
            }
            sfq[p] = (uint8_t)nvfp4_quant16_fast(z, a.out_global[e], codes[2 * p], codes[2 * p + 1]);
          }
          *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(a.out) + r * (a.N / 2) + jbase / 2) =
              make_uint4(codes[0], codes[1], codes[2], codes[3]);
        }
        // scale factors: this thread's two bytes into the staged source (row
        // lane, half cq / 2, word q, bytes 2 (cq % 2) + {0, 1}), then every
        // epilogue warp writes 16 of the source's 256 16-byte pieces
        const int sb = (int)(etile & 1);
        const uint32_t sph = (uint32_t)((etile >> 1) & 1);
        bool ok = mbar_wait_bounded(&sm.freed[sb], sph ^ 1, kWaitCycles, a.err);
        if (ok) {
          *reinterpret_cast<uint16_t *>(&sm.sf_stage[sb][lane * 32 + (cq >> 1) * 16 + q * 4 +
                                                        2 * (cq & 1)]) =
              (uint16_t)(sfq[0] | (sfq[1] << 8));
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.staged[sb]);
          ok = mbar_wait_bounded(&sm.staged[sb], sph, kWaitCycles, a.err);
        }
        if (ok) {
          const int ew = warp - 2;
          uint8_t *sfo = static_cast<uint8_t *>(a.out_sf) +
                         ((long)blk * ks_out + nt / 2) * kBsSfaRecBytes + (nt & 1) * 4096;
          // the tile after the last one, if the last stage's second pair has
          // no tile, gets zero scale factors
          const bool tail = nt == a.ntiles - 1 && (nt & 1) == 0;
          if (lane < 16) {
            const int x = ew * 16 + lane;                  // 0..255
            const int i = (x % 64) >> 1, half = x & 1, L = i + 32 * (x / 64);
            const long off = (L / 8) * 256 + half * 128 + (L % 8) * 16;
            *reinterpret_cast<uint4 *>(sfo + off) =
                *reinterpret_cast<const uint4 *>(&sm.sf_stage[sb][i * 32 + half * 16]);
            if (tail) *reinterpret_cast<uint4 *>(sfo + 4096 + off) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.freed[sb]);
        } else {
          record_device_error(a.err, kErrTimeout);
          *abort_flag = 1;
        }
        ++etile;
      } else if (live) {
        const long tok = s_id / a.T;
        const float wt = (a.w_stage1 ? 1.f : a.topk_weights[s_id]);
        const float sc = wt * (a.a_expertscale ? a.a_expertscale[e] : 1.f) * wg;
        const long i0 = (long)nt * BN + 64 * cq;
        if (i0 < a.K) {  // K % 32 == 0: 32-column halves are fully in or out
          float *dst = a.acc + tok * a.K + i0;
          const uint16_t *bias = static_cast<const uint16_t *>(a.w_bias);
          const float *bias32 = static_cast<const float *>(a.w_bias);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (i0 + 4 * i >= a.K) break;
            float y[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const long wrow = i0 + 4 * i + u;
              float b = 0.f;
              if (a.w_bias) {
                const long bi = (long)e * a.R + wrow;
                b = a.bias_f32 ? bias32[bi] : bf16_to_f32(bias[bi]);
              }
              y[u] = acc[4 * i + u] * sc + wt * b;
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

// Load-time records of NVFP4 weights for this kernel: per (expert, n-tile of
// 256 weight rows, 256-wide reduction stage) the 256 tile rows' codes (128
// bytes each, 128-byte swizzle: 16-byte chunk c of row n at
// (n / 8) * 1024 + (n % 8) * 128 + ((c ^ (n % 8)) * 16)), then the stage's
// scale factors as four .128x256b sources (SFB_BYTES).  W13 tile rows: SEPARATED -> eight groups of 32 rows,
// gate and up of outputs j0 + 32 i alternating; INTERLEAVED -> the rows
// 2 j0 .. 2 j0 + 255 as stored.  Zeros past the tensor.  One thread per byte.
__global__ void pack_bs_kernel(TcPackArgs p) {
  const long o = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= p.total) return;
  constexpr int REC = STAGE_B + SFB_BYTES;
  const long rec = o / REC;
  const int wb = (int)(o % REC);
  const int kt = (int)(rec % p.kstages);
  const long ent = rec / p.kstages;
  const int nt = (int)(ent % p.ntiles);
  const long e = ent / p.ntiles;
  int n;
  long k;
  const bool code = wb < STAGE_B;
  if (code) {
    n = (wb / 1024) * 8 + (wb % 1024) / 128;
    const int c = ((wb % 128) / 16) ^ (n & 7);
    k = (long)kt * 128 + c * 16 + (wb % 16);
  } else {
    // source j (MMA step), row L, byte y of its 32: half y / 16 of the tile
    // rows, scale word (y % 16) / 4 -> tile row 128 half + 32 w + L % 32
    const int w = wb - STAGE_B;
    const int j = w / 4096, x = w % 4096;
    const int L = (x / 256) * 8 + (x % 128) / 16;
    const int y = ((x % 256) / 128) * 16 + (x % 16);
    n = 128 * (y / 16) + 32 * ((y % 16) / 4) + (L % 32);
    k = (long)kt * 16 + j * 4 + (y % 4);
  }
  const int b = n >> 5;  // 32-row group 0..7
  long row;
  bool valid;
  if (p.w13) {
    if (p.gate == GATE_SEPARATED) {
      const long jj = (long)nt * 128 + (b >> 1) * 32 + (n & 31);
      valid = jj < p.N;
      row = (b & 1) ? p.N + jj : jj;
    } else {
      row = (long)nt * 256 + n;
      valid = row < 2L * p.N;
    }
  } else {
    row = (long)nt * 256 + n;
    valid = row < p.R;
  }
  unsigned char v = 0;
  if (code) {
    if (valid && k < p.C / 2) v = p.codes[((long)e * p.R + row) * (p.C / 2) + k];
  } else {
    if (valid && k < p.C / 16) v = p.scales[((long)e * p.R + row) * (p.C / 16) + k];
  }
  p.out[o] = v;
}

}  // namespace

int bs_ntiles(int w13, int N, int K) { return w13 ? (int)ceil_div(N, 128) : (int)ceil_div(K, 256); }

size_t bs_packed_bytes(int w13, int N, int K, int El) {
  const int C = w13 ? K : N;
  return (size_t)El * bs_ntiles(w13, N, K) * ceil_div(C, kTcBsStage) * (STAGE_B + SFB_BYTES);
}

cudaError_t launch_pack_bs(const TcPackArgs &p, cudaStream_t st) {
  if (p.total <= 0) return cudaSuccess;
  pack_bs_kernel<<<(unsigned)ceil_div(p.total, 256), 256, 0, st>>>(p);
  return cudaGetLastError();
}

bool make_tc_map_u8(CUtensorMap *tm, const void *base, long rows, long cols, int box_rows);

template <int MODE>
cudaError_t launch_bs_t(const CUtensorMap &ta, const TcArgs &a, int grid, cudaStream_t st) {
  static int attr_dev[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_dev[dev]) {
    cudaError_t e = cudaFuncSetAttribute(bs_gemm_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_dev[dev] = 1;
  }
  bs_gemm_kernel<MODE><<<(unsigned)grid, THREADS, SMEM_BYTES, st>>>(ta, a);
  return cudaGetLastError();
}

cudaError_t launch_bs_gemm(const TcArgs &a_in, const void *a_codes, long cap_rows, int w13,
                           int sm_count, cudaStream_t st) {
  TcArgs a = a_in;
  a.ntiles = bs_ntiles(w13, a.N, a.K);
  const long blocks = cap_rows / BM;
  if (blocks <= 0) return cudaSuccess;
  a.nblocks = blocks;
  CUtensorMap ta;
  if (!make_tc_map_u8(&ta, a_codes, cap_rows, a.C / 2, BM)) return cudaErrorInvalidValue;
  const long tiles = blocks * a.ntiles;
  const int grid = (int)(tiles < sm_count ? tiles : sm_count);
  return w13 ? launch_bs_t<MODE_W13>(ta, a, grid, st) : launch_bs_t<MODE_W2>(ta, a, grid, st);
}

}  // namespace moe
