// moe_tcd.cu -- tcgen05 grouped GEMMs for MXFP4 weights with bf16 activations
// (w4a16, GptOssMxfp4MoEMethod on the mxfp4.py page) or OCP MX activations
// dequantised to exact f16 (w4a4 / w4a8; the two GEMM stages of
// rocm_aiter_fused_experts on page
// "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe") at prefill
// batches whose experts hold more than one 128-slot block each.
//
// The tensor cores multiply f16 operands (kind::f16, fp32 accumulation in
// Tensor Memory), so the e2m1 weights are decoded to exact f16 (code x 2^e)
// on the SMs -- ALU work per weight element.  These kernels decode each
// 256-row weight stage once and multiply it with two 128-slot blocks of the
// expert (two accumulators of 128 x 256 in Tensor Memory), halving the decode
// work per FLOP against one block per decoded tile.
//   unit   (active local expert, pair of its 128-slot blocks, 256 weight rows)
//   A      the pair's sorted f16 rows (per-token power-of-two scaled x, or the
//          intermediate), 2-D TMA with the 128-byte swizzle, 16 KB per block
//   B      two load-time 128-row records (e2m1 codes + e8m0 scales of 64
//          reduction elements; MOE_LAYOUT_TC) decoded into the swizzled f16
//          layout, 32 KB
// One CTA per SM walks units u = blockIdx.x, + gridDim.x, ... (experts in
// order, their block pairs, the weight tiles fastest: the CTAs working at one
// time share the pair's rows and the weight records through L2).  Warp roles:
//   warp 0      lane 0: TMA producer (A tiles, records) into a 3-stage ring,
//               and L2 prefetches of the unit's next records; lanes 1-31
//               stage each unit's 256 biases in shared memory (two buffers)
//   warp 1      TMEM owner; lane 0 issues the stage's MMAs (4 per block) and
//               commits
//   warps 2-17  decode each stage's records (thread t: row t / 2, 32 elements)
//               during the main loop; at a unit's end they drain the two
//               accumulators (lane quarter warp % 4, 64 columns each) and
//               apply the epilogue: W13 x-scale, bias, SwiGLU-OAI (MX
//               activations: each thread's 32 outputs quantised and
//               dequantised as one MX block), f16 intermediate; W2 bias,
//               router weight, fp32 red.add.  Both write through the warp's
//               own 16 rows of decoded-weight slot 0 (free during the
//               epilogue), transposed so that one store / red.add
//               instruction covers 8 rows x 64 contiguous bytes
// Every wait is bounded; on a timeout the CTA records MOE_ERR_TIMEOUT, stops
// issuing, lets its copies and MMAs land, frees its Tensor Memory and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stddef.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128;                // slot rows per block
constexpr int BN = 256;                // weight rows per unit
constexpr int NS = 3;                  // ring stages
constexpr int STAGE_A = BM * 128;      // 16 KB of f16 rows (64 reduction elements)
constexpr int STAGE_B = BN * 128;      // 32 KB of decoded f16 weights
constexpr int REC = 4096 + 128 * 2;    // one 128-row MXFP4 record of a stage
constexpr int NUM_EPI = 16;
constexpr int THREADS = (2 + NUM_EPI) * 32;  // 576
constexpr int TMEM_COLS = 512;         // two accumulators of 256 columns
constexpr int kMaxActive = 1024;
// record stages prefetched into L2 ahead: measured on GPT-OSS-120B at M=8192,
// W13 0.963 / 0.959 / 0.952 / 0.949 ms for 8 / 16 / 24 / 32, W2 best at 16
template <int MODE> constexpr int prefetch_stages() { return MODE == 0 ? 32 : 16; }
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kErrTimeout = 5;

enum { MODE_W13 = 0, MODE_W2 = 1 };

struct Smem {
  unsigned char a[NS][2][STAGE_A];
  unsigned char b[NS][STAGE_B];
  unsigned char raw[NS][2][REC];
  // full: the stage's A tiles landed; raw_full: its weight records landed
  // (the decoders start on those without waiting for A); b_full: decoded
  uint64_t full[NS], raw_full[NS], empty[NS], b_full[NS];
  uint64_t acc_full, acc_empty, drain;
  // the unit's biases, staged by the producer warp's lanes 1-31: W13 (gate,
  // up) of its 128 outputs, W2 its 256 output rows; double-buffered by unit
  alignas(16) float bias[2][256];
  uint64_t bias_full[2], bias_empty[2];
  int unit_pre[kMaxActive + 1];  // units of the active experts before each one
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;
static_assert(offsetof(Smem, b) % 1024 == 0 && offsetof(Smem, raw) % 16 == 0 && REC % 16 == 0 &&
                  offsetof(Smem, bias) % 16 == 0,
              "shared-memory layout alignment");
constexpr int kBiasLanes = 31;  // producer-warp lanes 1-31
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

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

// A wait of the decoder / epilogue warps whose outcome is the same on every
// lane (the warp leaves its loops together: its shuffles and warp barriers
// never wait for a lane that has left).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int *err,
                                          volatile int *abort_flag) {
  const bool ok = wait_or_abort(bar, parity, err, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void red_add_v4(float *p, float x, float y, float z, float w) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x), "f"(y), "f"(z),
               "f"(w)
               : "memory");
}

// Swizzled byte offset of 16-byte chunk c of row n in a tile of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(int n, int c) {
  return (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4));
}

// Activation of one (gate, up) pair with the fast exponential and divide
// intrinsics (a few fp32 ulps, far below the f16 intermediate's step).
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

__device__ __forceinline__ float bias_value(const TcArgs &a, long i) {
  return a.bias_f32 ? static_cast<const float *>(a.w_bias)[i]
                    : bf16_to_f32(static_cast<const uint16_t *>(a.w_bias)[i]);
}

struct Unit {
  int e, blk0, nblk, nt, nrec;  // expert, first block, blocks (1 or 2), weight tile, records
};

// This CTA's units in the same order in every role.
struct Walker {
  const TcArgs *a;
  const int *pre;
  int n_act;
  long u, total;
  __device__ Walker(const TcArgs &args, const int *pre_, int n_act_)
      : a(&args), pre(pre_), n_act(n_act_), u(blockIdx.x), total(pre_[n_act_]) {}
  __device__ bool get(Unit &un) const {
    if (u >= total) return false;
    int lo = 0, hi = n_act - 1;  // the active expert whose range holds u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= u) lo = mid; else hi = mid - 1;
    }
    const int e = a->active[lo];
    const int nb = (a->counts[e] + BM - 1) / BM;
    const long local = u - pre[lo];
    const int p = (int)(local / a->ntiles);
    un.e = e;
    un.nt = (int)(local % a->ntiles);
    un.blk0 = a->offsets[e] / BM + 2 * p;
    un.nblk = min(2, nb - 2 * p);
    un.nrec = min(2, a->rec_tiles - 2 * un.nt);
    return true;
  }
  __device__ void next() { u += gridDim.x; }
};

// MXO: the W13 epilogue of OCP MX activations (the intermediate quantised and
// dequantised per 32-output block), a separate instantiation so that the
// w4a16 kernel keeps its registers
template <int MODE, bool MXO = false>
__global__ void __launch_bounds__(THREADS, 1)
tcd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = a.C / 64;  // the caller guarantees C % 64 == 0
  const int n_act = *a.n_active;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.raw_full[s], 1);
      mbar_init(&sm.empty[s], 1);
      mbar_init(&sm.b_full[s], NUM_EPI);
    }
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_empty, NUM_EPI);
    mbar_init(&sm.drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.bias_full[b], kBiasLanes);
      mbar_init(&sm.bias_empty[b], NUM_EPI);
    }
    sm.abort_flag = 0;
    mbar_fence_init();
  }
  // units before each active expert (block pairs x weight tiles), by warp 0
  if (warp == 0) {
    const int chunk = (n_act + 31) / 32;
    const int i0 = lane * chunk;
    int local = 0;
    for (int i = i0; i < i0 + chunk && i < n_act; ++i)
      local += (((a.counts[a.active[i]] + BM - 1) / BM + 1) / 2) * a.ntiles;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = i0; i < i0 + chunk && i < n_act; ++i) {
      sm.unit_pre[i] = run;
      run += (((a.counts[a.active[i]] + BM - 1) / BM + 1) / 2) * a.ntiles;
    }
    if (lane == 31) sm.unit_pre[n_act] = incl;
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
      long g = 0;
      Walker wk(a, sm.unit_pre, n_act);
      Unit un;
      while (!*abort_flag && wk.get(un)) {
        const unsigned char *rec0 = static_cast<const unsigned char *>(a.w_packed) +
                                    ((long)un.e * a.rec_tiles + 2 * un.nt) * KT * (long)REC;
        const long rec_stride = (long)KT * REC;  // the second record tile
        for (int kt = 0; kt < KT; ++kt, ++g) {
          constexpr int kPrefetch = prefetch_stages<MODE>();
          if (kt + kPrefetch < KT)
            for (int r = 0; r < un.nrec; ++r)
              prefetch_l2_bulk(rec0 + r * rec_stride + (long)(kt + kPrefetch) * REC, (uint32_t)REC);
          const int s = (int)(g % NS);
          if (!wait_or_abort(&sm.empty[s], (uint32_t)(((g / NS) & 1) ^ 1), a.err, abort_flag))
            break;
          mbar_arrive_expect_tx(&sm.raw_full[s], (uint32_t)(un.nrec * REC));
          for (int r = 0; r < un.nrec; ++r)
            tma_bulk_g2s(sm.raw[s][r], rec0 + r * rec_stride + (long)kt * REC, (uint32_t)REC,
                         &sm.raw_full[s]);
          mbar_arrive_expect_tx(&sm.full[s], (uint32_t)(un.nblk * STAGE_A));
          for (int b = 0; b < un.nblk; ++b)
            tma_load_2d(sm.a[s][b], &tmA, kt * 64, (un.blk0 + b) * BM, &sm.full[s]);
        }
        wk.next();
      }
      if (*abort_flag)  // let the copies already issued land before the CTA exits
        for (long k = g > NS ? g - NS : 0; k < g; ++k) {
          mbar_wait_bounded(&sm.raw_full[k % NS], (uint32_t)((k / NS) & 1), kWaitCycles);
          mbar_wait_bounded(&sm.full[k % NS], (uint32_t)((k / NS) & 1), kWaitCycles);
        }
    } else {
      // lanes 1-31: the biases of each unit, into buffer (unit index % 2)
      long tc = 0;
      Walker wk(a, sm.unit_pre, n_act);
      Unit un;
      while (!*abort_flag && wk.get(un)) {
        const int buf = (int)(tc & 1);
        if (!wait_or_abort(&sm.bias_empty[buf], (uint32_t)(((tc >> 1) & 1) ^ 1), a.err,
                           abort_flag))
          break;
        const long b0 = (long)un.e * a.R;
        for (int i = lane - 1; i < 256; i += kBiasLanes) {
          float v = 0.f;
          const int rr = i >> 7;  // record (128 columns) of this value
          if (a.w_bias && rr < un.nrec) {
            if (MODE == MODE_W13) {  // (gate, up) of output (2 nt + rr) 64 + (i % 128) / 2
              const long j = (long)(2 * un.nt + rr) * 64 + ((i & 127) >> 1);
              const bool up = (i & 1) != 0;
              const long row = a.gate == GATE_SEPARATED ? (up ? (long)a.N + j : j) : 2 * j + up;
              if (j < a.N) v = bias_value(a, b0 + row);
            } else {  // output row (2 nt + rr) 128 + i % 128
              const long k = (long)(2 * un.nt + rr) * 128 + (i & 127);
              if (k < a.R) v = bias_value(a, b0 + k);
            }
          }
          sm.bias[buf][i] = v;
        }
        mbar_arrive(&sm.bias_full[buf]);
        ++tc;
        wk.next();
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      long g = 0, tc = 0;
      Walker wk(a, sm.unit_pre, n_act);
      Unit un;
      while (!*abort_flag && wk.get(un)) {
        // the epilogue has drained the previous unit's accumulators
        if (!wait_or_abort(&sm.acc_empty, (uint32_t)((tc & 1) ^ 1), a.err, abort_flag)) break;
        tc_fence_after();
        const uint32_t idesc = umma_idesc_f16(BM, un.nrec * 128);
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int s = (int)(g % NS);
          const uint32_t par = (uint32_t)((g / NS) & 1);
          if (!wait_or_abort(&sm.full[s], par, a.err, abort_flag)) break;
          if (!wait_or_abort(&sm.b_full[s], par, a.err, abort_flag)) break;
          tc_fence_after();
          const uint64_t bd = umma_desc_sw128(smem_addr(sm.b[s]));
          for (int b = 0; b < un.nblk; ++b) {
            const uint64_t ad = umma_desc_sw128(smem_addr(sm.a[s][b]));
#pragma unroll
            for (int j = 0; j < 4; ++j)  // 16 reduction elements (32 bytes) each
              umma_f16(tmem + (uint32_t)(b * BN), ad + 2 * j, bd + 2 * j, idesc,
                       (kt == 0 && j == 0) ? 0u : 1u);
          }
          umma_commit(&sm.empty[s]);
        }
        if (*abort_flag) break;
        umma_commit(&sm.acc_full);
        ++tc;
        wk.next();
      }
      // every MMA issued above has completed before Tensor Memory is freed
      umma_commit(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0, kWaitCycles);
    }
  } else {
    // ------------------------------------------- decoders, then the epilogue
    const int t = threadIdx.x - 64;      // 0..511
    const int n = t >> 1, h = t & 1;     // decoded row, 32-element half
    const int rec = n >> 7, rn = n & 127;
    const int q = warp & 3;              // TMEM lane quarter
    const int cq = (warp - 2) >> 2;      // 64-column quarter of the 256 columns
    long g = 0, tc = 0;
    Walker wk(a, sm.unit_pre, n_act);
    Unit un;
    while (!__any_sync(0xffffffffu, *abort_flag != 0) && wk.get(un)) {  // warp-uniform
      for (int kt = 0; kt < KT; ++kt, ++g) {
        const int s = (int)(g % NS);
        if (!warp_wait(&sm.raw_full[s], (uint32_t)((g / NS) & 1), a.err, abort_flag)) break;
        if (rec < un.nrec) {
          const unsigned char *rp = sm.raw[s][rec];
          const uint4 cw = *reinterpret_cast<const uint4 *>(rp + rn * 32 + h * 16);
          const uint32_t sc = rp[4096 + rn * 2 + h];
          // 2^(sc - 127) as an f16x2 pair; exact: TC-packed records exist only
          // for scale codes in [106, 140] (range-checked at load time)
          const uint32_t sh = sc >= 113 ? (sc - 112) << 10 : 1u << (sc - 103);
          const uint32_t f = sh | (sh << 16);
          const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t hv[4];
            e2m1x8_to_f16x2x4(words[u], hv);
            uint4 o;
            o.x = hmul2_u32(hv[0], f);
            o.y = hmul2_u32(hv[1], f);
            o.z = hmul2_u32(hv[2], f);
            o.w = hmul2_u32(hv[3], f);
            *reinterpret_cast<uint4 *>(sm.b[s] + sw128(n, 4 * h + u)) = o;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.b_full[s]);
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;  // the warp leaves together

      // ---------------------------------------------------------- epilogue
      if (!warp_wait(&sm.acc_full, (uint32_t)(tc & 1), a.err, abort_flag)) break;
      tc_fence_after();
      const int r_rec = 2 * un.nt + (cq >> 1);  // record tile of this thread's columns
      const bool col_live = (cq >> 1) < un.nrec;
      const int bbuf = (int)(tc & 1);
      if (!warp_wait(&sm.bias_full[bbuf], (uint32_t)((tc >> 1) & 1), a.err, abort_flag)) break;
      const float *bias_s = sm.bias[bbuf];
      for (int b = 0; b < un.nblk; ++b) {
        const long r = (long)(un.blk0 + b) * BM + q * 32 + lane;  // sorted row
        float acc[64];
        {
          const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + cq * 64);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            float v[16];
            tmem_ld_32x32b_x16(taddr + 16 * p, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[16 * p + i] = v[i];
          }
        }
        const int s_id = a.sorted_ids[r];
        const bool row_live = s_id < a.S;
        if (MODE == MODE_W13) {
          const int jbase = r_rec * 64 + 32 * (cq & 1);
          // the row's 32 f16 outputs (four 16-byte units) go through this
          // warp's own 16 rows of decoded-weight slot 0 (free now, as for W2)
          // and out 8 rows x 64 contiguous bytes per store instruction
          uint4 *xp = reinterpret_cast<uint4 *>(sm.b[0] + 2048 * (warp - 2));
          const int sw_w = (lane >> 1) & 3;
          if (MXO && col_live && jbase < a.N) {  // warp-uniform
            // OCP MX activations: the 32 outputs are one MX block (jbase % 32
            // == 0), quantised and dequantised into exact f16 (the exact
            // activation, as the other f16 kernels compute it)
            const bool sep = a.gate == GATE_SEPARATED;
            const float rf = a.a_rowscale[r];
            float zb[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float gacc = sep ? acc[i] : acc[2 * i];
              const float uacc = sep ? acc[32 + i] : acc[2 * i + 1];
              zb[i] = act_and_mul(a.act, gacc * rf + bias_s[2 * (64 * (cq >> 1) + 32 * (cq & 1) + i)],
                                  uacc * rf + bias_s[2 * (64 * (cq >> 1) + 32 * (cq & 1) + i) + 1],
                                  a.alpha, a.beta, a.limit);
            }
            uint32_t w[16];
            mx_qdq_f16x32(zb, a.out_mode == TC_OUT_MX4_F16, w);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              xp[lane * 4 + (i ^ sw_w)] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          } else if (!MXO && col_live && jbase < a.N) {  // warp-uniform; N % 32 == 0
            const bool sep = a.gate == GATE_SEPARATED;
            const float rf = a.a_rowscale[r];
#pragma unroll
            for (int p = 0; p < 4; ++p) {  // 8 outputs per pass
              // the staged (gate, up) biases of these 8 outputs
              const float4 *bp = reinterpret_cast<const float4 *>(
                  bias_s + 2 * (64 * (cq >> 1) + 32 * (cq & 1) + 8 * p));
              float bgu[16];
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const float4 f = bp[v];
                bgu[4 * v] = f.x; bgu[4 * v + 1] = f.y; bgu[4 * v + 2] = f.z; bgu[4 * v + 3] = f.w;
              }
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 8; i += 2) {
                float z2[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                  const int ii = 8 * p + i + k;
                  const float gacc = sep ? acc[ii] : acc[2 * ii];
                  const float uacc = sep ? acc[32 + ii] : acc[2 * ii + 1];
                  z2[k] = act_fast(a.act, gacc * rf + bgu[2 * (i + k)],
                                   uacc * rf + bgu[2 * (i + k) + 1], a.alpha, a.beta, a.limit);
                }
                const __half2 h2 = __floats2half2_rn(z2[0], z2[1]);
                w[i >> 1] = *reinterpret_cast<const uint32_t *>(&h2);
              }
              xp[lane * 4 + (p ^ sw_w)] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          if (col_live && jbase < a.N) {  // warp-uniform: the transposed stores
            __syncwarp();
            const int live_mask = __ballot_sync(0xffffffffu, row_live);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int rho = 8 * j + (lane >> 2), u = lane & 3;
              if ((live_mask >> rho) & 1) {
                const long rr = (long)(un.blk0 + b) * BM + q * 32 + rho;
                reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + rr * a.N + jbase)[u] =
                    xp[rho * 4 + (u ^ ((rho >> 1) & 3))];
              }
            }
            __syncwarp();
          }
        } else if (col_live) {  // warp-uniform
          // outputs k0 .. k0 + 63 of the row, 16 columns at a time through
          // this warp's own 16 rows of decoded-weight slot 0 (2 KB: free now,
          // the unit's MMAs have completed and the next unit's wait for this
          // epilogue; the warp decodes into them again only after it): lane l
          // then adds row 8 j + l / 4, columns 4 (l % 4) .. + 3, so one red.add
          // covers 8 rows x 64 contiguous bytes instead of 32 rows x 16 bytes
          const int tok = row_live ? s_id / a.T : -1;  // -1: padding row
          const float wt = row_live ? (a.w_stage1 ? 1.f : a.topk_weights[s_id]) : 0.f;
          const long k0 = (long)r_rec * 128 + 64 * (cq & 1);
          float4 *xp = reinterpret_cast<float4 *>(sm.b[0] + 2048 * (warp - 2));
          const int sw_w = (lane >> 1) & 3;
#pragma unroll
          for (int c = 0; c < 4; ++c) {  // 16 outputs per chunk (K % 16 == 0)
            if (k0 + 16 * c >= a.K) break;  // warp-uniform
            const float4 *bp =
                reinterpret_cast<const float4 *>(bias_s + 128 * (cq >> 1) + 64 * (cq & 1) + 16 * c);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float4 f = bp[u];
              xp[lane * 4 + (u ^ sw_w)] = make_float4(
                  wt * (acc[16 * c + 4 * u] + f.x), wt * (acc[16 * c + 4 * u + 1] + f.y),
                  wt * (acc[16 * c + 4 * u + 2] + f.z), wt * (acc[16 * c + 4 * u + 3] + f.w));
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int rho = 8 * j + (lane >> 2), u = lane & 3;
              const int tok_r = __shfl_sync(0xffffffffu, tok, rho);
              if (tok_r >= 0) {
                const float4 v = xp[rho * 4 + (u ^ ((rho >> 1) & 3))];
                red_add_v4(a.acc + (long)tok_r * a.K + k0 + 16 * c + 4 * u, v.x, v.y, v.z, v.w);
              }
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.acc_empty);  // the next unit's MMAs may start
        mbar_arrive(&sm.bias_empty[bbuf]);
      }
      ++tc;
      wk.next();
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int MODE, bool MXO>
cudaError_t launch_tcd_t(const CUtensorMap &ta, const TcArgs &a, int grid, cudaStream_t st) {
  static int attr_dev[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_dev[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcd_gemm_kernel<MODE, MXO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_dev[dev] = 1;
  }
  tcd_gemm_kernel<MODE, MXO><<<(unsigned)grid, THREADS, SMEM_BYTES, st>>>(ta, a);
  return cudaGetLastError();
}

}  // namespace

// 2-D K-major 16-bit tensor map with the 128-byte swizzle (moe_tc.cu).
bool make_tc_map_b16(CUtensorMap *tm, const void *base, long rows, long cols, int box_rows);

bool tcd_supported(int El) { return El <= kMaxActive; }

cudaError_t launch_tcd_gemm(const TcArgs &a_in, const void *rows_f16, long cap_rows, int w13,
                            int sm_count, cudaStream_t st) {
  TcArgs a = a_in;
  a.rec_tiles = tc_ntiles(w13, a.N, a.K);          // 128-row record tiles
  a.ntiles = (a.rec_tiles + 1) / 2;                 // 256-row units
  if (cap_rows <= 0) return cudaSuccess;
  if (a.C % 64 != 0 || !a.active || !a.offsets || !a.counts || !a.n_active || !a.w_packed ||
      a.El > kMaxActive)
    return cudaErrorInvalidValue;
  CUtensorMap ta;
  if (!make_tc_map_b16(&ta, rows_f16, cap_rows, a.C, BM)) return cudaErrorInvalidValue;
  const bool mx_out = a.out_mode == TC_OUT_MX4_F16 || a.out_mode == TC_OUT_MX8_F16;
  return !w13    ? launch_tcd_t<MODE_W2, false>(ta, a, sm_count, st)
         : mx_out ? launch_tcd_t<MODE_W13, true>(ta, a, sm_count, st)
                  : launch_tcd_t<MODE_W13, false>(ta, a, sm_count, st);
}

}  // namespace moe
