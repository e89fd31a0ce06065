// moe_tcs.cu -- weight-streaming tcgen05 grouped GEMMs of the fused experts
// for MXFP4 weights with bf16 activations (w4a16, GptOssMxfp4MoEMethod on the
// mxfp4.py page; the two GEMM stages of rocm_aiter_fused_experts on page
// "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe") at batch
// sizes where a local expert holds about one to two hundred slots: too many
// for the mma.sync streaming kernels' 16-slot passes, too few to fill the
// 128-row blocks of the tcgen05 prefill kernels without padding.
//
// The weights are the MMA's M operand and an expert's slots its N operand
// (D^T = W x^T): one work unit is (active local expert, 128 weight rows), and
// a pass multiplies those rows with up to NMAX (64, 128 or 256) of the
// expert's slots at once, so each weight element is read from HBM and
// decoded once per pass, and the MMA is as wide as the pass's slot count
// (rounded up to 16) instead of a 128-row block of padded slots.
//   A = weights: load-time packed records (e2m1 codes + e8m0 scales of 128
//       rows x 64 reduction elements, one TMA bulk copy per stage) decoded by
//       the decoder warps into exact f16 (code x 2^e) in the 128-byte-swizzled
//       K-major layout; W13 rows are reordered on the way so that the gate
//       and up rows of output i are tile rows 2i and 2i + 1
//   B = the expert's slots: the sorted f16 rows (stage 1: the per-token f16
//       copy of x scaled by a power of two; stage 2: the intermediate), 2-D
//       TMA with the 128-byte swizzle, boxes of 32 rows
//   D = fp32 in Tensor Memory, 128 lanes (weight rows) x N columns (slots),
//       two buffers, so the epilogue of one pass overlaps the MMAs of the next
// Persistent CTAs (two per SM for passes of up to 128 slots, one for 256)
// walk units u = blockIdx.x, + gridDim.x, ... of the list (active expert,
// 128-row tile), tiles fastest: the CTAs working at one time share an
// expert's slot rows through L2.  Warp roles:
//   warp 0      record producer: TMA bulk copies into the record ring, and L2
//               prefetches of the unit's next records
//   warp 1      slot-row producer: 2-D TMA into the slot-row ring
//   warp 2      TMEM owner; lane 0 issues kind::f16 tcgen05.mma (M = 128,
//               N = the pass's slots, 4 per 64-element stage) and commits
//   decoders    (4 or 8 warps) records -> swizzled f16 weight tiles
//   epilogue    (4 warps) tcgen05.ld of 16 slots at a time per weight row;
//               W13: the (gate, up) pair of adjacent lanes meets with one
//               shuffle, x-scale, bias, SwiGLU-OAI, f16 intermediate; W2:
//               bias, router weight, fp32 red.add into the token accumulator
// Measured (per-role cycle counters): with passes of ~48 slots a 128 x 48 x
// 16 MMA occupies the tensor pipe for ~110 cycles, and the decoders need
// about as long per stage, so these kernels stream weights at about a third
// of HBM bandwidth; they pay off where the alternatives pad or re-stream more.
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

constexpr int BM = 128;               // weight rows per unit (the MMA's M)
constexpr int REC = 4096 + 128 * 2;   // MXFP4 record of one (unit, 64-element stage)
constexpr int STAGE_A = BM * 128;     // 16 KB of decoded f16 weights
constexpr int XBOX = 32;              // slot rows per TMA box
constexpr int NUM_EPI = 4;
constexpr int W_REC = 0, W_X = 1, W_MMA = 2, W_DEC0 = 3;
// records prefetched into L2 ahead of the ring: GPT-OSS-120B at M=2048, ms
// per step 0.7125 / 0.7157 / 0.7223 for 8 / 16 / 32
constexpr int kPrefetch = 8;
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kErrTimeout = 5;

enum { MODE_W13 = 0, MODE_W2 = 1 };

// Per pass width NMAX (slots per pass, the MMA's largest N): CTAs per SM,
// decoder warps and ring depths.  Up to 128 slots two CTAs share an SM (each
// with 256 Tensor Memory columns: two accumulators of 128), so that one CTA's
// per-stage handoffs (barrier waits, MMA issue, decode) overlap the other's;
// 256 slots need the whole Tensor Memory.
template <int NMAX> struct Cfg;
template <> struct Cfg<64> {
  static constexpr int CTAS = 2, NDEC = 4, NR = 6, NA = 3, NX = 4;
};
template <> struct Cfg<128> {
  static constexpr int CTAS = 2, NDEC = 4, NR = 6, NA = 2, NX = 3;
};
template <> struct Cfg<256> {
  static constexpr int CTAS = 1, NDEC = 8, NR = 6, NA = 3, NX = 4;
};
template <int NMAX> constexpr int threads_of() { return (W_DEC0 + Cfg<NMAX>::NDEC + NUM_EPI) * 32; }
template <int NMAX> constexpr int tmem_cols_of() { return Cfg<NMAX>::CTAS == 2 ? 256 : 512; }

template <int NMAX>
struct Smem {
  static constexpr int NR = Cfg<NMAX>::NR, NA = Cfg<NMAX>::NA, NX = Cfg<NMAX>::NX;
  unsigned char a[NA][STAGE_A];
  unsigned char x[NX][NMAX * 128];
  unsigned char raw[NR][REC];
  uint64_t raw_full[NR], raw_empty[NR];
  uint64_t a_full[NA], a_empty[NA], x_full[NX], x_empty[NX];
  uint64_t acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};
template <int NMAX> constexpr size_t smem_bytes() { return sizeof(Smem<NMAX>) + 1024; }
static_assert(offsetof(Smem<64>, x) % 1024 == 0 && offsetof(Smem<64>, raw) % 16 == 0 &&
                  offsetof(Smem<128>, x) % 1024 == 0 && offsetof(Smem<128>, raw) % 16 == 0 &&
                  offsetof(Smem<256>, x) % 1024 == 0 && offsetof(Smem<256>, raw) % 16 == 0 &&
                  REC % 16 == 0,
              "shared-memory layout alignment");
static_assert(2 * (smem_bytes<64>() + 1024) <= 228 * 1024 &&
                  2 * (smem_bytes<128>() + 1024) <= 228 * 1024 && smem_bytes<256>() <= 227 * 1024,
              "shared memory per SM");

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

// Swizzled byte offset of 16-byte chunk c of row n in a 128-byte-row tile.
__device__ __forceinline__ uint32_t sw128(int n, int c) {
  return (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4));
}

// One pass of one unit: the expert, its first sorted row, the pass's first
// slot, valid slots and MMA width.
struct Pass {
  int e, nt, row0, nv, n;
};

// Walks this CTA's units and their passes in the same order in every role.
template <int NMAX>
struct Walker {
  const TcArgs *a;
  long u, n_units;
  int p, npass, per, e, nt, off, cnt;
  __device__ Walker(const TcArgs &args, long n_units_) : a(&args), u(blockIdx.x), n_units(n_units_),
                                                         p(0), npass(0) {
    load();
  }
  __device__ void load() {
    if (u >= n_units) return;
    e = a->active[u / a->ntiles];
    nt = (int)(u % a->ntiles);
    off = a->offsets[e];
    cnt = a->counts[e];
    npass = (cnt + NMAX - 1) / NMAX;
    per = npass > 0 ? (cnt + npass - 1) / npass : 0;
    p = 0;
  }
  // the current pass (false when this CTA has no more work)
  __device__ bool get(Pass &ps) {
    while (u < n_units && p >= npass) {
      u += gridDim.x;
      load();
    }
    if (u >= n_units) return false;
    ps.e = e;
    ps.nt = nt;
    const int n0 = p * per;
    ps.nv = min(per, cnt - n0);
    ps.row0 = off + n0;
    ps.n = (ps.nv + 15) & ~15;
    return true;
  }
  __device__ bool first_pass() const { return p == 0; }
  __device__ void next() { ++p; }
};

__device__ __forceinline__ float bias_at(const TcArgs &a, int e, long row) {
  if (!a.w_bias) return 0.f;
  const long i = (long)e * a.R + row;
  return a.bias_f32 ? static_cast<const float *>(a.w_bias)[i]
                    : bf16_to_f32(static_cast<const uint16_t *>(a.w_bias)[i]);
}

template <int MODE, int NMAX>
__global__ void __launch_bounds__(threads_of<NMAX>(), Cfg<NMAX>::CTAS)
tcs_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const TcArgs a) {
  using SM = Smem<NMAX>;
  constexpr int NR = SM::NR, NA = SM::NA, NX = SM::NX;
  constexpr int NUM_DEC = Cfg<NMAX>::NDEC, W_EPI0 = W_DEC0 + NUM_DEC;
  constexpr int TMEM_COLS = tmem_cols_of<NMAX>(), ACC_COLS = TMEM_COLS / 2;
  extern __shared__ unsigned char smem_raw[];
  SM &sm = *reinterpret_cast<SM *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                   ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = a.C / 64;  // the caller guarantees C % 64 == 0

  if (threadIdx.x == 0) {
    for (int s = 0; s < NR; ++s) {
      mbar_init(&sm.raw_full[s], 1);
      mbar_init(&sm.raw_empty[s], NUM_DEC);
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&sm.a_full[s], NUM_DEC);
      mbar_init(&sm.a_empty[s], 1);
    }
    for (int s = 0; s < NX; ++s) {
      mbar_init(&sm.x_full[s], 1);
      mbar_init(&sm.x_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], NUM_EPI);
    }
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int *abort_flag = &sm.abort_flag;
  const long n_units = (long)*a.n_active * a.ntiles;

  if (warp == W_REC) {
    // ------------------------------------------------------------ records
    if (lane == 0) {
      long g = 0;
      Walker<NMAX> wk(a, n_units);
      Pass ps;
      while (!*abort_flag && wk.get(ps)) {
        const unsigned char *urec = static_cast<const unsigned char *>(a.w_packed) +
                                    ((long)ps.e * a.ntiles + ps.nt) * KT * (long)REC;
        const bool pf = wk.first_pass();  // later passes find the records in L2
        if (pf) prefetch_l2_bulk(urec, (uint32_t)(min(KT, kPrefetch) * REC));
        for (int kt = 0; kt < KT; ++kt, ++g) {
          if (pf && kt + kPrefetch < KT)
            prefetch_l2_bulk(urec + (long)(kt + kPrefetch) * REC, (uint32_t)REC);
          const int r = (int)(g % NR);
          if (!wait_or_abort(&sm.raw_empty[r], (uint32_t)(((g / NR) & 1) ^ 1), a.err, abort_flag))
            break;
          mbar_arrive_expect_tx(&sm.raw_full[r], (uint32_t)REC);
          tma_bulk_g2s(sm.raw[r], urec + (long)kt * REC, (uint32_t)REC, &sm.raw_full[r]);
        }
        wk.next();
      }
      if (*abort_flag)  // let the copies already issued land before the CTA exits
        for (long k = g > NR ? g - NR : 0; k < g; ++k)
          mbar_wait_bounded(&sm.raw_full[k % NR], (uint32_t)((k / NR) & 1), kWaitCycles);
    }
  } else if (warp == W_X) {
    // ------------------------------------------------------------ slot rows
    if (lane == 0) {
      long g = 0;
      Walker<NMAX> wk(a, n_units);
      Pass ps;
      while (!*abort_flag && wk.get(ps)) {
        const int nbox = (ps.n + XBOX - 1) / XBOX;
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int s = (int)(g % NX);
          if (!wait_or_abort(&sm.x_empty[s], (uint32_t)(((g / NX) & 1) ^ 1), a.err, abort_flag))
            break;
          mbar_arrive_expect_tx(&sm.x_full[s], (uint32_t)(nbox * XBOX * 128));
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(sm.x[s] + b * (XBOX * 128), &tmX, kt * 64, ps.row0 + b * XBOX,
                        &sm.x_full[s]);
        }
        wk.next();
      }
      if (*abort_flag)
        for (long k = g > NX ? g - NX : 0; k < g; ++k)
          mbar_wait_bounded(&sm.x_full[k % NX], (uint32_t)((k / NX) & 1), kWaitCycles);
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      long g = 0, up = 0;
      Walker<NMAX> wk(a, n_units);
      Pass ps;
      while (!*abort_flag && wk.get(ps)) {
        const int buf = (int)(up & 1);
        // the epilogue has copied this buffer's previous pass out
        if (!wait_or_abort(&sm.acc_empty[buf], (uint32_t)(((up >> 1) & 1) ^ 1), a.err, abort_flag))
          break;
        tc_fence_after();
        const uint32_t idesc = umma_idesc_f16(BM, ps.n);
        const uint32_t d = tmem + (uint32_t)(buf * ACC_COLS);
        for (int kt = 0; kt < KT; ++kt, ++g) {
          const int sa = (int)(g % NA), sx = (int)(g % NX);
          if (!wait_or_abort(&sm.a_full[sa], (uint32_t)((g / NA) & 1), a.err, abort_flag)) break;
          if (!wait_or_abort(&sm.x_full[sx], (uint32_t)((g / NX) & 1), a.err, abort_flag)) break;
          tc_fence_after();
          const uint64_t ad = umma_desc_sw128(smem_addr(sm.a[sa]));
          const uint64_t xd = umma_desc_sw128(smem_addr(sm.x[sx]));
#pragma unroll
          for (int j = 0; j < 4; ++j)  // 16 reduction elements (32 bytes) each
            umma_f16(d, ad + 2 * j, xd + 2 * j, idesc, (kt == 0 && j == 0) ? 0u : 1u);
          umma_commit(&sm.a_empty[sa]);
          umma_commit(&sm.x_empty[sx]);
        }
        if (*abort_flag) break;
        umma_commit(&sm.acc_full[buf]);
        ++up;
        wk.next();
      }
      // every MMA issued above has completed before Tensor Memory is freed
      umma_commit(&sm.drain);
      mbar_wait_bounded(&sm.drain, 0, kWaitCycles);
    }
  } else if (warp < W_EPI0) {
    // ------------------------------------------------------------ decoders
    // (row, 32-element half) pairs p = t, t + 32 NUM_DEC, ...: record row
    // n = p / 2, half h = p % 2 (one e8m0 scale), written to tile row m (W13:
    // the gate / up rows of output i at 2i / 2i + 1)
    constexpr int PAIRS = 256 / (NUM_DEC * 32);
    const int t = threadIdx.x - W_DEC0 * 32;
    int pn[PAIRS], ph[PAIRS], pm[PAIRS];
#pragma unroll
    for (int pi = 0; pi < PAIRS; ++pi) {
      const int pp = t + pi * NUM_DEC * 32;
      pn[pi] = pp >> 1;
      ph[pi] = pp & 1;
      pm[pi] = pn[pi];
      if (MODE == MODE_W13 && a.gate == GATE_SEPARATED)
        pm[pi] = 2 * ((pn[pi] >> 6) * 32 + (pn[pi] & 31)) + ((pn[pi] >> 5) & 1);
    }
    long g = 0;
    Walker<NMAX> wk(a, n_units);
    Pass ps;
    while (!*abort_flag && wk.get(ps)) {
      for (int kt = 0; kt < KT; ++kt, ++g) {
        const int r = (int)(g % NR), s = (int)(g % NA);
        if (!wait_or_abort(&sm.raw_full[r], (uint32_t)((g / NR) & 1), a.err, abort_flag)) break;
        const unsigned char *rec = sm.raw[r];
        uint4 cw[PAIRS];
        uint32_t sc[PAIRS];
#pragma unroll
        for (int pi = 0; pi < PAIRS; ++pi) {
          cw[pi] = *reinterpret_cast<const uint4 *>(rec + pn[pi] * 32 + ph[pi] * 16);
          sc[pi] = rec[4096 + pn[pi] * 2 + ph[pi]];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.raw_empty[r]);
        // the tile's previous MMAs have completed
        if (!wait_or_abort(&sm.a_empty[s], (uint32_t)(((g / NA) & 1) ^ 1), a.err, abort_flag))
          break;
#pragma unroll
        for (int pi = 0; pi < PAIRS; ++pi) {
          // 2^(sc - 127) as an f16x2 pair; exact: TC-packed records exist only
          // for scale codes in [106, 140] (range-checked at load time)
          const uint32_t sh = sc[pi] >= 113 ? (sc[pi] - 112) << 10 : 1u << (sc[pi] - 103);
          const uint32_t f = sh | (sh << 16);
          const uint32_t words[4] = {cw[pi].x, cw[pi].y, cw[pi].z, cw[pi].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t hv[4];
            e2m1x8_to_f16x2x4(words[u], hv);
            uint4 o;
            o.x = hmul2_u32(hv[0], f);
            o.y = hmul2_u32(hv[1], f);
            o.z = hmul2_u32(hv[2], f);
            o.w = hmul2_u32(hv[3], f);
            *reinterpret_cast<uint4 *>(sm.a[s] + sw128(pm[pi], 4 * ph[pi] + u)) = o;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.a_full[s]);
      }
      wk.next();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int mrow = q * 32 + lane;
    const bool up_lane = (lane & 1) != 0;
    long up = 0;
    Walker<NMAX> wk(a, n_units);
    Pass ps;
    while (wk.get(ps)) {
      const int buf = (int)(up & 1);
      if (!wait_or_abort(&sm.acc_full[buf], (uint32_t)((up >> 1) & 1), a.err, abort_flag)) break;
      tc_fence_after();
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * ACC_COLS);
      if (MODE == MODE_W13) {
        const int j = ps.nt * 64 + (mrow >> 1);  // output of this lane pair
        const bool sep = a.gate == GATE_SEPARATED;
        const float bg = bias_at(a, ps.e, sep ? j : 2L * j);
        const float bu = bias_at(a, ps.e, sep ? (long)a.N + j : 2L * j + 1);
        uint16_t *inter = static_cast<uint16_t *>(a.out);
        for (int c0 = 0; c0 < ps.n; c0 += 16) {
          float v[16];
          tmem_ld_32x32b_x16(trow + c0, v);
          // the even lane (gate row) takes slots c0 .. c0 + 7, the odd lane
          // (up row) slots c0 + 8 .. c0 + 15; each sends the other its half
          float r[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            r[i] = __shfl_xor_sync(0xffffffffu, up_lane ? v[i] : v[8 + i], 1);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int tn = c0 + (up_lane ? 8 : 0) + i;
            if (tn < ps.nv) {
              const long row = ps.row0 + tn;
              const float xs = a.a_rowscale[row];
              const float gv = (up_lane ? r[i] : v[i]) * xs + bg;
              const float uv = (up_lane ? v[8 + i] : r[i]) * xs + bu;
              const float z = act_and_mul(a.act, gv, uv, a.alpha, a.beta, a.limit);
              inter[row * a.N + j] = __half_as_ushort(__float2half_rn(z));
            }
          }
        }
      } else {
        const long k = (long)ps.nt * BM + mrow;  // output feature of this lane
        const bool kv = k < a.R;
        const float b2 = kv ? bias_at(a, ps.e, k) : 0.f;
        for (int c0 = 0; c0 < ps.n; c0 += 16) {
          float v[16];
          tmem_ld_32x32b_x16(trow + c0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tn = c0 + i;
            if (tn < ps.nv && kv) {
              const int sid = a.sorted_ids[ps.row0 + tn];
              const float w = a.w_stage1 ? 1.f : a.topk_weights[sid];
              atomicAdd(a.acc + (long)(sid / a.T) * a.K + k, w * (v[i] + b2));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
      ++up;
      wk.next();
    }
  }

  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

// 2-D K-major 16-bit tensor map with the 128-byte swizzle (boxes of 64
// elements x box_rows rows; moe_tc.cu).
bool make_tc_map_b16(CUtensorMap *tm, const void *base, long rows, long cols, int box_rows);

namespace {

template <int MODE, int NMAX>
cudaError_t launch_tcs_t(const CUtensorMap &tx, const TcArgs &a, int grid, cudaStream_t st) {
  static int attr_dev[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_dev[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcs_gemm_kernel<MODE, NMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<NMAX>());
    if (e != cudaSuccess) return e;
    attr_dev[dev] = 1;
  }
  tcs_gemm_kernel<MODE, NMAX>
      <<<(unsigned)(grid * Cfg<NMAX>::CTAS), threads_of<NMAX>(), smem_bytes<NMAX>(), st>>>(tx, a);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_tcs_w(const CUtensorMap &tx, const TcArgs &a, int nmax, int grid,
                         cudaStream_t st) {
  if (nmax <= 64) return launch_tcs_t<MODE, 64>(tx, a, grid, st);
  if (nmax <= 128) return launch_tcs_t<MODE, 128>(tx, a, grid, st);
  return launch_tcs_t<MODE, 256>(tx, a, grid, st);
}

}  // namespace

int tcs_ntiles(int w13, int N, int K) { return w13 ? (int)ceil_div(N, 64) : (int)ceil_div(K, BM); }

cudaError_t launch_tcs_gemm(const TcArgs &a_in, const void *rows_f16, long cap_rows, int w13,
                            int sm_count, cudaStream_t st) {
  TcArgs a = a_in;
  a.ntiles = tcs_ntiles(w13, a.N, a.K);
  if (cap_rows <= 0) return cudaSuccess;
  if (a.C % 64 != 0 || !a.active || !a.offsets || !a.counts || !a.n_active)
    return cudaErrorInvalidValue;
  CUtensorMap tx;
  if (!make_tc_map_b16(&tx, rows_f16, cap_rows, a.C, XBOX)) return cudaErrorInvalidValue;
  // pass width: room for the average expert's slots and a quarter more (the
  // counts are on the device; an expert with more runs several passes)
  const long avg = ((long)a.M * a.T + a.El - 1) / a.El;
  const int nmax = (int)(avg + avg / 4);
  return w13 ? launch_tcs_w<MODE_W13>(tx, a, nmax, sm_count, st)
             : launch_tcs_w<MODE_W2>(tx, a, nmax, sm_count, st);
}

}  // namespace moe
