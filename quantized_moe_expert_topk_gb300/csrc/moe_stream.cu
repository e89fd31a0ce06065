// moe_stream.cu -- weight-streaming grouped GEMMs for decode-sized batches of
// the MXFP4 layer with bf16 or OCP MX activations (few tokens per expert; the
// layer is bound by HBM reads of the weights).  Same contract as the generic
// kernels ("rocm_aiter_fused_experts" on page "vllm.model_executor.layers.
// fused_moe.experts.rocm_aiter_moe"; MXFP4 layouts and SwiGLU constants from
// "vLLM/vllm/model_executor/layers/quantization/mxfp4.py").
//
// One persistent grid (MODE_FUSED) runs both GEMMs from one work queue: all
// W13 units, then all W2 units; a W2 unit copies its expert's intermediate
// rows once that expert's W13 units have counted their epilogues done.  Very
// small batches split the W13 units along K (partials + last-arriver fixup);
// with MX activations those run the W13 and W2 grids one after the other.
//
// Work unit: (active local expert, tile of 128 weight rows, k-range).  Units
// are claimed dynamically from a global counter (persistent CTAs, four per
// SM); each unit streams its weight records once through a double-buffered
// shared-memory ring (stages of 256 reduction elements, 17 KB of weights)
// filled by TMA bulk copies (one producer warp, mbarrier full/empty pairs,
// every wait bounded, a descriptor per stage telling the consumers which
// unit/pass/k-block it holds); four consumer warps each own two m16 tiles.
//
// Arithmetic (swap-AB mma.sync m16n8k16, f16 x f16 -> fp32):
//   A = weights: e2m1 codes converted two at a time by the hardware
//       (cvt.rn.f16x2.e2m1x2) -- exact, no scale applied;
//   B = the expert's tokens (up to 16 or 32 per pass, more passes re-stream
//       the unit), already in f16 in HBM: stage-1 rows scaled per token by a power
//       of two (exact for bf16 inputs), stage-2 rows are the bounded SwiGLU-OAI
//       intermediate;
//   the e8m0 scale of each (row, 32-element group) multiplies the fp32 partial
//   of that group (two MMAs) into the accumulator.
// W13 epilogue: x-scale, bias, SwiGLU-OAI of the (gate, up) rows the packed
// layout pairs inside every m16 tile (rows 0-7 gate, 8-15 up of the same 8
// outputs), f16 intermediate (with MX activations quantised and dequantised
// per 32-output block first).  W2 epilogue: bias, router weight, fp32
// red.add into the token accumulator (the reduce of TopKWeightAndReduceNoOP).
//
// Packed weight layout (moe_prepare_weights, load time, like the pages'
// convert_weight_to_mxfp4_moe_kernel_format): records of 64 reduction
// elements per unit, [expert][unit][k64][tile(8)][512 B codes | 32 B scales];
// inside a tile the 512 code bytes are ordered so that lane L reads 16 bytes
// that hold exactly its A-fragment bytes for two 32-element groups.
#include <cuda_fp16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int CW = 4;                       // consumer warps
constexpr int MT = 2;                       // m16 tiles per consumer warp
constexpr int ROWS = CW * MT * 16;          // 128 weight rows per unit
constexpr int TILES = CW * MT;              // 8 m16 tiles per unit
constexpr int TILE_BYTES = 512 + 32;        // codes + scales of one tile, one k64 block
constexpr int REC_BYTES = TILES * TILE_BYTES;  // 4352 B per (unit, k64 block)
constexpr int S_KB = 4;                     // k64 blocks per stage (256 reduction elements)
constexpr int NS = 2;                       // pipeline stages (double buffer)
// A unit's weight records are contiguous.  The producer keeps this many stages
// beyond the one it copies requested into L2 (bulk prefetch, a hint), so the
// ring's copies find them there instead of waiting out a DRAM round trip.
// Measured on GPT-OSS-20B decode (M=64): one stage 90.0 us per grid, none
// 91.1, two 91.2, four 95.2; GPT-OSS-120B at M=512 and M=1 unchanged.
constexpr int kPrefetchStages = 1;
constexpr int XS = S_KB * 64 * 2 + 16;      // smem row stride of the token tile (528 B)
constexpr int W_STAGE = S_KB * REC_BYTES;   // 17408 B
constexpr int THREADS = (CW + 1) * 32;
// Tokens per pass TOK (n8 tiles TOK / 8): 16 at four CTAs per SM, or -- when
// the experts hold more than 32 slots each, for which 16-token passes would
// decode each weight tile three times or more -- 32 at three CTAs per SM (the
// token tiles take the shared memory and the accumulators the registers of
// the fourth).
template <int TOK> constexpr int ctas_per_sm() { return TOK == 16 ? 4 : 3; }
template <int TOK> constexpr int stage_bytes() { return W_STAGE + TOK * XS; }
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr int kErrTimeout = 5;

// MODE_FUSED: one persistent grid runs the W13 units, then the W2 units, from
// one work queue (a = W13 arguments, b = W2 arguments); the W2 units of an
// expert start their intermediate-row copies once every W13 unit of that
// expert has written its rows (a per-expert completion count).
enum { MODE_W13 = 0, MODE_W2 = 1, MODE_FUSED = 2 };
enum { F_FIRST = 1, F_LAST = 2, F_W2 = 4 };  // F_W2: a W2 unit's stage (fused grid)

struct Unit {
  int e, u, kb0, nkb, off, cnt;
};

// Stage descriptor written by the producer next to the data it loads (the
// unit's decoded fields too, so consumers start a unit without global loads).
struct StageDesc {
  int id;    // unit id, -1 = no more work
  int tok0;  // first token of this pass
  int kb;    // first k64 block of this stage within the unit's k-range
  int flags; // F_FIRST / F_LAST: first / last stage of the pass
  Unit unit;
};

template <int TOK>
struct Smem {
  unsigned char stage[NS][stage_bytes<TOK>()];
  uint64_t full[NS];
  uint64_t empty[NS];
  StageDesc desc[NS];
  // MX intermediate (MXQ): per consumer-warp pair, the two warps' per-token
  // maxima over their 16 outputs of a 32-output block (double-buffered by
  // epilogue parity) and a barrier of two arrivals
  uint64_t mx_bar[CW / 2];
  float mx_amax[2][CW][TOK];
  // per consumer warp, the epilogue operands of the pass's tokens (slot id;
  // W13: x_inv of the token, W2: router weight; W13: factor of the stage-1
  // output), loaded at the pass's first stage and read by its epilogue (in
  // shared memory rather than registers, which the main loop needs)
  int tok_sid[CW][TOK];
  float tok_f[CW][TOK], tok_zw[CW][TOK];
  int abort_flag;
};
template <int TOK> constexpr size_t smem_bytes() { return sizeof(Smem<TOK>); }
static_assert(ctas_per_sm<16>() * (smem_bytes<16>() + 1024) <= 228 * 1024 &&
                  ctas_per_sm<32>() * (smem_bytes<32>() + 1024) <= 228 * 1024,
              "shared memory per SM");

__device__ __forceinline__ Unit decode_unit(const StreamArgs &a, int id) {
  Unit r;
  const int ks = id % a.ksplit;
  const int rest = id / a.ksplit;
  r.u = rest % a.units_per_expert;
  r.e = a.active[rest / a.units_per_expert];
  const int per = (a.kblocks + a.ksplit - 1) / a.ksplit;
  r.kb0 = ks * per;
  r.nkb = min(per, a.kblocks - r.kb0);
  r.off = a.offsets[r.e];
  r.cnt = a.counts[r.e];
  return r;
}

// Byte `idx` of `w` (an e8m0 code c) as the fp32 value 2^(c-127): the byte is
// isolated (one byte permute) and multiplied by 2^23 (an integer multiply-add,
// off the integer/logic pipe) into the exponent field.  Code 0 (2^-127, below
// the fp32 normal range) reads as 0.
__device__ __forceinline__ float e8m0_byte_f32(uint32_t w, uint32_t idx) {
  return __uint_as_float(__byte_perm(w, 0u, 0x4440u | idx) * 8388608u);
}

// One k64 block of one consumer warp: MT m16 tiles x NTILES n8 token tiles
// (of the NT the accumulators hold).
template <int NTILES, int NT>
__device__ __forceinline__ void consume_k64(const unsigned char *tp0, uint32_t xs_k64, int lane,
                                            float (&acc)[MT][NT][4]) {
  const int g = lane >> 2;
  uint4 cw[MT];
  uint32_t sw[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const unsigned char *tp = tp0 + m * TILE_BYTES;
    cw[m] = *reinterpret_cast<const uint4 *>(tp + lane * 16);
    sw[m] = *reinterpret_cast<const uint32_t *>(tp + 512 + g * 4);
  }
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    // B fragments of k16 steps 2 kk and 2 kk + 1: n8 tiles in pairs (tokens
    // 16 p .. 16 p + 15) by one ldmatrix x4, an odd last tile by an x2
    uint32_t bf[2][NTILES][2];
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const int s4 = 2 * kk + s2;
#pragma unroll
      for (int p = 0; p < (NTILES + 1) / 2; ++p) {
        const uint32_t addr = xs_k64 + (p * 16 + (lane & 7) + ((lane >> 4) << 3)) * XS +
                              (s4 * 16 + ((lane >> 3) & 1) * 8) * 2;
        if (2 * p + 1 < NTILES) {
          uint32_t r[4];
          ldmatrix_x4_b16(r, addr);
          bf[s2][2 * p][0] = r[0]; bf[s2][2 * p][1] = r[1];
          bf[s2][2 * p + 1][0] = r[2]; bf[s2][2 * p + 1][1] = r[3];
        } else {
          uint32_t r[2];
          ldmatrix_x2_b16(r, addr);
          bf[s2][2 * p][0] = r[0]; bf[s2][2 * p][1] = r[1];
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      uint32_t a0[4], a1[4];
      e2m1x8_to_f16x2x4(kk == 0 ? cw[m].x : cw[m].z, a0);
      e2m1x8_to_f16x2x4(kk == 0 ? cw[m].y : cw[m].w, a1);
      // e8m0 scales of rows g and g+8 for this 32-element group
      const float f_lo = e8m0_byte_f32(sw[m], 2 * kk);
      const float f_hi = e8m0_byte_f32(sw[m], 2 * kk + 1);
      const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int n = 0; n < NTILES; ++n) {
        float part[4];
        mma_f16_16816(part, a0, bf[0][n][0], bf[0][n][1], zero);
        mma_f16_16816(part, a1, bf[1][n][0], bf[1][n][1], part);
        fma_f32x2(acc[m][n][0], acc[m][n][1], part[0], part[1], f_lo);
        fma_f32x2(acc[m][n][2], acc[m][n][3], part[2], part[3], f_hi);
      }
    }
  }
}

// SPLIT (W13 / fused): the W13 units are split along K; partials + last-arriver fixup.
// `b` holds the W2 arguments of the fused grid (unused otherwise).
// MXQ (W13 / fused, no split): the W13 epilogue quantises and dequantises the
// intermediate into OCP MX (a.out_mx: 1 MXFP4, 2 MXFP8) before its f16 store.
// A 32-output block spans the 16 outputs of two consumer warps (2w, 2w+1),
// which exchange their per-token maxima through shared memory.
template <int MODE, bool SPLIT, bool MXQ = false, int TOK = 16>
__global__ void __launch_bounds__(THREADS, ctas_per_sm<TOK>())
stream_kernel(const __grid_constant__ StreamArgs a, const __grid_constant__ StreamArgs b) {
  static_assert(TOK == 16 || (TOK == 32 && !SPLIT && !MXQ), "pass width");
  constexpr int NT = TOK / 8;  // n8 token tiles per pass
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem<TOK> &sm = *reinterpret_cast<Smem<TOK> *>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], CW);
    }
    for (int q = 0; q < CW / 2; ++q) mbar_init(&sm.mx_bar[q], 2);
    sm.abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  volatile int *abort_flag = &sm.abort_flag;


  if (warp == CW) {
    // ------------------------------------------------------------ producer
    // Claims units from a global counter (dynamic load balance), streams each
    // unit's weight records and the matching token rows into the ring, and
    // ends with a terminator stage.
    //
    // Dependent launch: the W13 grid may start while the sort grid runs, so
    // its producer waits for it before reading any of its outputs (counts,
    // offsets, the zeroed counters, the f16 copy of x).  The W2 grid starts
    // once every W13 CTA got here (so the sort is complete); its producer
    // already streams weights and waits for the W13 grid only before the
    // first copy of the intermediate rows.
    bool waited = false;
    auto wait_prior = [&]() {
      if (!waited) {
        griddep_wait();
        fence_proxy_async_global();
        if (lane == 0) griddep_launch_dependents();
        waited = true;
      }
    };
    if (MODE != MODE_W2) wait_prior();
    const int n_active = *a.n_active;
    const int n13 =  // W13 ids first
        MODE == MODE_FUSED ? n_active * a.units_per_expert * (SPLIT ? a.ksplit : 1) : 0;
    const int n_units = MODE == MODE_FUSED ? n13 + n_active * b.units_per_expert * b.ksplit
                                           : n_active * a.units_per_expert * a.ksplit;
    uint32_t it = 0;
    bool ok = true;
    auto acquire_slot = [&](int &slot) -> bool {
      slot = it % NS;
      if (!mbar_wait_bounded(&sm.empty[slot], ((it / NS) & 1) ^ 1, kWaitCycles, a.err)) {
        record_device_error(a.err, kErrTimeout);
        *abort_flag = 1;
      }
      return !*abort_flag;
    };
    while (ok) {
      int id = 0;
      if (lane == 0) id = atomicAdd(a.work_counter, 1);
      id = __shfl_sync(0xffffffffu, id, 0);
      if (id >= n_units) {
        wait_prior();  // also lets the next grid start
        int slot;
        if (acquire_slot(slot) && lane == 0) {
          sm.desc[slot] = StageDesc{-1, 0, 0, 0, Unit{0, 0, 0, 0, 0, 0}};
          mbar_arrive(&sm.full[slot]);
        }
        ++it;
        break;
      }
      // the unit's phase and the arguments of that phase
      const bool w2 = MODE == MODE_W2 || (MODE == MODE_FUSED && id >= n13);
      const bool pb = MODE == MODE_FUSED && w2;  // fields from b
      const Unit U = pb ? decode_unit(b, id - n13) : decode_unit(a, id);
      const int C = pb ? b.C : a.C;  // reduction length (K for W13, N for W2)
      // W2 in the fused grid: the intermediate rows of this expert are
      // complete once every W13 unit of it has finished every pass (one count
      // per consumer warp, from the warp that applies the epilogue: with a
      // k-split, the last arrival); those units were claimed earlier by
      // running CTAs.  The wait comes before the first copy of those rows:
      // the unit's first weight stage (and its L2 prefetch) are already in
      // flight while the W13 units finish.
      bool rows_ready = !pb;
      for (int tok0 = 0; tok0 < U.cnt && ok; tok0 += TOK) {
        const int nt = min(TOK, U.cnt - tok0);
        const unsigned char *xrow = nullptr;  // lane n < nt loads token n of this pass
        if (lane < nt) {
          const int r = U.off + tok0 + lane;
          const long src = w2 ? (long)r : (long)(a.sorted_ids[r] / a.T);
          xrow = static_cast<const unsigned char *>(pb ? b.x16 : a.x16) + src * (long)C * 2;
        }
        const int upe = pb ? b.units_per_expert : a.units_per_expert;
        const int kblocks = pb ? b.kblocks : a.kblocks;
        const unsigned char *ubase = static_cast<const unsigned char *>(pb ? b.packed : a.packed) +
            ((((long)U.e * upe + U.u) * kblocks) + U.kb0) * REC_BYTES;
        // stages 0..kPrefetchStages of this pass (all inside the unit's records)
        if (kPrefetchStages > 0 && U.nkb > 0 && lane == 0)
          prefetch_l2_bulk(ubase,
                           (uint32_t)min(U.nkb, (kPrefetchStages + 1) * S_KB) * REC_BYTES);
        for (int kb = 0; kb < U.nkb; kb += S_KB) {
          const int nkb = min(S_KB, U.nkb - kb);
          int slot;
          if (!acquire_slot(slot)) { ok = false; break; }
          unsigned char *ws = sm.stage[slot];
          const uint32_t wbytes = (uint32_t)nkb * REC_BYTES;
          // keep the next kPrefetchStages stages requested
          const int pkb = kb + kPrefetchStages * S_KB;
          if (kPrefetchStages > 0 && kb > 0 && pkb < U.nkb && lane == 0)
            prefetch_l2_bulk(ubase + (long)pkb * REC_BYTES,
                             (uint32_t)min(S_KB, U.nkb - pkb) * REC_BYTES);
          const uint32_t xbytes = (uint32_t)nkb * 128;
          if (lane == 0) {
            sm.desc[slot] = StageDesc{id, tok0, kb,
                                      (kb == 0 ? F_FIRST : 0) | (kb + S_KB >= U.nkb ? F_LAST : 0) |
                                          (pb ? F_W2 : 0),
                                      U};
            mbar_arrive_expect_tx(&sm.full[slot], wbytes + (uint32_t)nt * xbytes);
            tma_bulk_g2s(ws, ubase + (long)kb * REC_BYTES, wbytes, &sm.full[slot]);
          }
          __syncwarp();
          wait_prior();  // the token rows of W2 are the W13 grid's output
          if (!rows_ready) {
            const int need = a.units_per_expert * CW * (int)ceil_div(U.cnt, TOK);
            if (!wait_count_bounded(a.done13 + U.e, need, kWaitCycles, a.err)) {
              // the rows below are copied all the same (in bounds), so the
              // stage's barrier completes; the consumers see the abort flag
              record_device_error(a.err, kErrTimeout);
              *abort_flag = 1;
              ok = false;
            }
            fence_proxy_async_global();  // their generic stores before our TMA reads
            rows_ready = true;
          }
          if (lane < nt)
            tma_bulk_g2s(ws + W_STAGE + lane * XS, xrow + (long)(U.kb0 + kb) * 128, xbytes,
                         &sm.full[slot]);
          ++it;
          if (!ok) break;
        }
      }
    }
    // drain: every copy issued into the ring has landed before the CTA exits
    if (lane == 0) {
      const uint32_t first = it > NS ? it - NS : 0;
      for (uint32_t j = first; j < it; ++j)
        if (!mbar_wait_bounded(&sm.full[j % NS], (j / NS) & 1, kWaitCycles)) {
          record_device_error(a.err, kErrTimeout);
          break;
        }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  uint32_t it = 0;
  Unit U = {0, 0, 0, 0, 0, 0};
  int nt = 0, ntiles = 0;
  float acc[MT][NT][4];
  // this thread's tokens n * 8 + 2 t + c (n, c in {0, 1}) of the pass
  int *const tok_sid_w = sm.tok_sid[warp];
  float *const tok_f_w = sm.tok_f[warp];
  float *const tok_zw_w = sm.tok_zw[warp];
#define TOK_SID(n, c) tok_sid_w[(n) * 8 + 2 * t + (c)]
#define TOK_F(n, c) tok_f_w[(n) * 8 + 2 * t + (c)]
#define TOK_ZW(n, c) tok_zw_w[(n) * 8 + 2 * t + (c)]
  bool w2 = MODE == MODE_W2;  // phase of the current unit
  uint32_t mx_ep = 0;         // MXQ: epilogues of this warp so far (barrier parity)
  while (true) {
    const int slot = it % NS;
    if (!mbar_wait_bounded(&sm.full[slot], (it / NS) & 1, kWaitCycles, a.err)) {
      record_device_error(a.err, kErrTimeout);
      *abort_flag = 1;
    }
    if (*abort_flag) return;
    StageDesc d;
    {
      const volatile int *dv = reinterpret_cast<const volatile int *>(&sm.desc[slot]);
      d.id = dv[0];
      d.tok0 = dv[1];
      d.kb = dv[2];
      d.flags = dv[3];
    }
    if (d.id < 0) break;
    if (d.flags & F_FIRST) {
      {
        const volatile int *uv = reinterpret_cast<const volatile int *>(&sm.desc[slot].unit);
        U.e = uv[0]; U.u = uv[1]; U.kb0 = uv[2]; U.nkb = uv[3]; U.off = uv[4]; U.cnt = uv[5];
      }
      nt = min(TOK, U.cnt - d.tok0);
      ntiles = (nt + 7) >> 3;
      if (MODE == MODE_FUSED) w2 = (d.flags & F_W2) != 0;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[m][n][c] = 0.f;
      // epilogue operands of the pass's tokens (lanes 0-3 write them; the
      // epilogue reads them after the pass), loaded now so that their
      // latency hides behind the pass
      if (g == 0) {
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int tn = n * 8 + 2 * t + c;
            const int sid = tn < nt ? a.sorted_ids[U.off + d.tok0 + tn] : 0;
            // W13: x_inv of the token (times the router weight when it applies
            // to the stage-1 output); W2: the router weight (1 in that case)
            const float wr = a.w_stage1 ? (!w2 ? a.topk_weights[sid] : 1.f)
                                        : (!w2 ? 1.f : a.topk_weights[sid]);
            TOK_SID(n, c) = sid;
            TOK_F(n, c) = tn >= nt ? 0.f : !w2 ? a.x_inv[sid / a.T] : wr;
            TOK_ZW(n, c) = !w2 && tn < nt ? wr : 1.f;
          }
      }
    }
    const int nkb = min(S_KB, U.nkb - d.kb);
    const unsigned char *ws = sm.stage[slot];
    const uint32_t xs = smem_addr(ws + W_STAGE);
    const unsigned char *tw = ws + (warp * MT) * TILE_BYTES;
    if (nkb == S_KB && ntiles == NT) {
      // full stage and pass: straight-line code over the S_KB blocks, so the
      // conversions, MMAs and scale FMAs of different blocks interleave
#pragma unroll
      for (int b = 0; b < S_KB; ++b)
        consume_k64<NT, NT>(tw + b * REC_BYTES, xs + b * 128, lane, acc);
    } else if (nkb == S_KB && ntiles == 1) {
#pragma unroll
      for (int b = 0; b < S_KB; ++b)
        consume_k64<1, NT>(tw + b * REC_BYTES, xs + b * 128, lane, acc);
    } else {
      for (int b = 0; b < nkb; ++b) {
        const unsigned char *tb = tw + b * REC_BYTES;
        const uint32_t xb = xs + b * 128;
        if (ntiles == 1) consume_k64<1, NT>(tb, xb, lane, acc);
        else if (ntiles == 2) consume_k64<2, NT>(tb, xb, lane, acc);
        else if constexpr (NT == 4) {
          if (ntiles == 3) consume_k64<3, NT>(tb, xb, lane, acc);
          else consume_k64<4, NT>(tb, xb, lane, acc);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[slot]);
    ++it;
    if (!(d.flags & F_LAST)) continue;

    // -------------------------------------------------------------- epilogue
    const int tok0 = d.tok0;
    bool finish = true;  // this warp applies the activation (W13)
    if ((MODE == MODE_W13 || (MODE == MODE_FUSED && !w2)) && SPLIT) {
      // k-split: write this k-range's (gate, up) partials, already scaled by
      // the token's x_inv; the last of the ksplit arrivals for this (unit,
      // pass, warp) sums them below (no waiting: the others just move on)
      const int N = a.N;
      const int ks = d.id % a.ksplit;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int j = U.u * (TILES * 8) + (warp * MT + m) * 8 + g;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int tn = n * 8 + 2 * t + c;
            if (tn >= nt) continue;
            const float xi = TOK_F(n, c);
            float2 *dst = reinterpret_cast<float2 *>(a.hpart) +
                          ((long)ks * a.S + TOK_SID(n, c)) * N + j;
            *dst = make_float2(acc[m][n][c] * xi, acc[m][n][2 + c] * xi);
          }
      }
      __threadfence();  // the partials are visible before the count says so
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        const long cidx = (((long)(U.off + tok0) >> 4) * a.units_per_expert + U.u) * CW + warp;
        last = atomicAdd(a.fix_cnt + cidx, 1) == a.ksplit - 1;
      }
      finish = __shfl_sync(0xffffffffu, last, 0) != 0;
      if (finish) __threadfence();  // and the others' partials are visible to us
    }
    if ((MODE == MODE_W13 || (MODE == MODE_FUSED && !w2)) && finish) {
      const int N = a.N;
#pragma unroll
      for (int m = 0; m < MT && !MXQ; ++m) {
        const int j = U.u * (TILES * 8) + (warp * MT + m) * 8 + g;
        const long grow = a.gate == GATE_SEPARATED ? j : 2L * j;
        const long urow = a.gate == GATE_SEPARATED ? (long)N + j : 2L * j + 1;
        float bg = 0.f, bu = 0.f;
        if (a.bias) {
          const uint16_t *bb = static_cast<const uint16_t *>(a.bias) + (long)U.e * 2 * N;
          bg = bf16_to_f32(bb[grow]);
          bu = bf16_to_f32(bb[urow]);
        }
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int tn = n * 8 + 2 * t + c;
            if (tn >= nt) continue;
            const int r = U.off + tok0 + tn;
            const float xi = TOK_F(n, c);
            float gsum = acc[m][n][c] * xi, usum = acc[m][n][2 + c] * xi;
            if (SPLIT) {  // the sum of every k-range's partial, in k order
              gsum = usum = 0.f;
              for (int ks = 0; ks < a.ksplit; ++ks) {
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(a.hpart) +
                                        ((long)ks * a.S + TOK_SID(n, c)) * N + j);
                gsum += v.x;
                usum += v.y;
              }
            }
            const float gv = gsum + bg;
            const float uv = usum + bu;
            const float z = TOK_ZW(n, c) * act_and_mul(a.act, gv, uv, a.alpha, a.beta, a.limit);
            if (a.out_f32)
              static_cast<float *>(a.out)[(long)r * N + j] = z;
            else
              static_cast<__half *>(a.out)[(long)r * N + j] = __float2half_rn(z);
          }
      }
      if (MXQ) {
        // z of output j = (this warp's m-tile m, row g) for token (n, c)
        auto zval = [&](int m, int n, int c) -> float {
          const int j = U.u * (TILES * 8) + (warp * MT + m) * 8 + g;
          const long grow = a.gate == GATE_SEPARATED ? j : 2L * j;
          const long urow = a.gate == GATE_SEPARATED ? (long)N + j : 2L * j + 1;
          float bg = 0.f, bu = 0.f;
          if (a.bias) {
            const uint16_t *bb = static_cast<const uint16_t *>(a.bias) + (long)U.e * 2 * N;
            bg = bf16_to_f32(bb[grow]);
            bu = bf16_to_f32(bb[urow]);
          }
          const float xi = TOK_F(n, c);
          return TOK_ZW(n, c) * act_and_mul(a.act, acc[m][n][c] * xi + bg,
                                            acc[m][n][2 + c] * xi + bu, a.alpha, a.beta, a.limit);
        };
        // per token, the largest |z| of this warp's 16 outputs (the lanes of
        // one t hold the 8 g rows of both m tiles), then the pair's maximum;
        // z is computed again for the store rather than held across the wait
        float pa[2][2];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const bool in = n * 8 + 2 * t + c < nt;
            float v = in ? fmaxf(fabsf(zval(0, n, c)), fabsf(zval(1, n, c))) : 0.f;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            pa[n][c] = v;
          }
        const int buf = mx_ep & 1;
        if (g == 0)
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int c = 0; c < 2; ++c) sm.mx_amax[buf][warp][n * 8 + 2 * t + c] = pa[n][c];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.mx_bar[warp >> 1]);
        if (!mbar_wait_bounded(&sm.mx_bar[warp >> 1], mx_ep & 1, kWaitCycles, a.err)) {
          record_device_error(a.err, kErrTimeout);
          *abort_flag = 1;
        }
        if (*abort_flag) return;
        ++mx_ep;
        const bool fp4 = a.out_mx == 1;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int tn = n * 8 + 2 * t + c;
            if (tn >= nt) continue;
            const float amax = fmaxf(pa[n][c], sm.mx_amax[buf][warp ^ 1][tn]);
            uint32_t h = 0u;  // outputs j (m = 0) and j + 8 (m = 1) of this token
            if (amax > 0.f)
              h = mx_qdq_pair_f16(zval(0, n, c), zval(1, n, c), fp4,
                                  mx_shared_exp(amax, fp4 ? 2 : 8), 0);
            const long r = U.off + tok0 + tn;
            const int j0 = U.u * (TILES * 8) + warp * MT * 8 + g;
            uint16_t *dst = static_cast<uint16_t *>(a.out) + r * N;
            dst[j0] = (uint16_t)(h & 0xffffu);
            dst[j0 + 8] = (uint16_t)(h >> 16);
          }
      }
      if (MODE == MODE_FUSED) {
        // this warp's rows of this (unit, pass) are written: count it for the
        // expert (release: every lane's stores before the count)
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(a.done13 + U.e, 1);
      }
    } else if (MODE == MODE_W2 || (MODE == MODE_FUSED && (!SPLIT || w2))) {
      // (a W13 warp of a split unit that left the fixup to another arrival
      // has nothing to do here)
      const StreamArgs &w = MODE == MODE_FUSED ? b : a;  // the W2 arguments
      const int K = w.K;
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = U.u * ROWS + (warp * MT + m) * 16 + g + 8 * h;
          if (i >= K) continue;
          float bias = 0.f;
          if (w.bias && U.kb0 == 0)
            bias = bf16_to_f32(static_cast<const uint16_t *>(w.bias)[(long)U.e * K + i]);
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int tn = n * 8 + 2 * t + c;
              if (tn >= nt) continue;
              const int sidx = TOK_SID(n, c);
              const float wt = TOK_F(n, c);
              atomicAdd(w.acc + (long)(sidx / w.T) * K + i, wt * (acc[m][n][2 * h + c] + bias));
            }
        }
    }
  }
}

#undef TOK_SID
#undef TOK_F
#undef TOK_ZW

// ---------------------------------------------------------------- packing
// One thread per packed byte.
__global__ void pack_mxfp4_kernel(PackArgs p) {
  const long o = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (o >= p.total) return;
  const long rec = o / REC_BYTES;
  const int within = (int)(o % REC_BYTES);
  const int m = within / TILE_BYTES;
  const int wb = within % TILE_BYTES;
  const int kb = (int)(rec % p.kblocks);
  const long eu = rec / p.kblocks;
  const int u = (int)(eu % p.units);
  const long e = eu / p.units;
  int r16, byte_k = 0, grp = 0;
  bool is_code = wb < 512;
  if (is_code) {
    const int lane = wb / 16, bi = wb % 16;
    const int kk = bi / 8, q = (bi / 4) & 1, reg = bi & 3;
    const int gg = lane >> 2, tt = lane & 3;
    r16 = gg + 8 * (reg & 1);
    byte_k = kb * 64 + kk * 32 + q * 16 + 2 * tt + 8 * (reg >> 1);  // even element index
  } else {
    const int sb = wb - 512;
    const int gg = sb >> 2, s4 = sb & 3;
    r16 = gg + 8 * (s4 & 1);
    grp = kb * 2 + (s4 >> 1);
  }
  long row = -1;
  if (p.w13) {
    const int j = u * (TILES * 8) + m * 8 + (r16 & 7);
    const int up = r16 >= 8;
    if (j < p.N) row = p.gate == GATE_SEPARATED ? (up ? (long)p.N + j : j) : 2L * j + up;
  } else {
    const long i = (long)u * ROWS + m * 16 + r16;
    if (i < p.R) row = i;
  }
  unsigned char v;
  if (is_code) {
    v = (row >= 0 && byte_k < p.C) ? p.codes[((long)e * p.R + row) * (p.C / 2) + byte_k / 2] : 0;
  } else {
    v = (row >= 0 && grp < p.C / 32) ? p.scales[((long)e * p.R + row) * (p.C / 32) + grp] : 127;
  }
  p.out[o] = v;
}

}  // namespace

size_t stream_packed_bytes(int w13, int N, int K, int El) {
  const int units = w13 ? N / (TILES * 8) : (int)ceil_div(K, ROWS);
  const int C = w13 ? K : N;
  const int kblocks = (int)ceil_div(C, 64);
  return (size_t)El * units * kblocks * REC_BYTES;
}

cudaError_t launch_pack_mxfp4(const PackArgs &p, cudaStream_t stream) {
  if (p.total <= 0) return cudaSuccess;
  pack_mxfp4_kernel<<<(unsigned)ceil_div(p.total, 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

int stream_w13_ksplit(int M, int topk, int El, int N, int K, int sm_count) {
  // split K only when the W13 units cannot give every CTA two of them; each
  // k-range keeps at least two stages
  const long act = (long)M * topk < El ? (long)M * topk : El;
  const long units = act * (N / (TILES * 8));
  const long want = units > 0 ? ceil_div(2L * ctas_per_sm<16>() * sm_count, units) : 1;
  const long cap = (K / 64) / (2 * S_KB) > 1 ? (K / 64) / (2 * S_KB) : 1;
  return (int)(want <= 1 ? 1 : (want < cap ? want : cap));
}

long stream_w13_fixups(long cap_rows, int N) { return (cap_rows / 16) * (N / (TILES * 8)) * CW; }

int stream_units_per_expert(int w13, int N, int K) {
  return w13 ? N / (TILES * 8) : (int)ceil_div(K, ROWS);
}

cudaError_t launch_stream(const StreamArgs &a, int w13, int sm_count, cudaStream_t stream) {
  const int variant = w13 ? (a.ksplit > 1 ? 2 : 1) : 0;
  auto kern = variant == 2 ? stream_kernel<MODE_W13, true>
              : variant == 1 ? stream_kernel<MODE_W13, false>
                             : stream_kernel<MODE_W2, false>;
  static bool attr_done[3] = {false, false, false};
  if (!attr_done[variant]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes<16>());
    if (e != cudaSuccess) return e;
    attr_done[variant] = true;
  }
  const long max_units = (long)a.max_active * a.units_per_expert * a.ksplit;
  long grid = (long)ctas_per_sm<16>() * sm_count;
  if (grid > max_units) grid = max_units;
  if (grid <= 0) return cudaSuccess;
  // a programmatic dependent of the previous kernel (the sort, or the W13 grid)
  return launch_kernel(kern, dim3((unsigned)grid), dim3(THREADS), smem_bytes<16>(), stream, true,
                       a, a);
}

cudaError_t launch_stream_fused(const StreamArgs &a13, const StreamArgs &a2, int sm_count,
                                cudaStream_t stream) {
  // the MX epilogue exchanges block maxima inside one CTA: no k-split with it
  if (!a13.done13 || a13.out_f32 || (a13.out_mx && a13.ksplit != 1)) return cudaErrorInvalidValue;
  // 32-token passes: only without the k-split and the MX epilogue
  const bool wide = a13.tok_pass == 32;
  if (wide && (a13.out_mx || a13.ksplit != 1 || a2.tok_pass != 32)) return cudaErrorInvalidValue;
  const int variant = wide ? 3 : a13.out_mx ? 1 : a13.ksplit > 1 ? 2 : 0;
  auto kern = variant == 3   ? stream_kernel<MODE_FUSED, false, false, 32>
              : variant == 1 ? stream_kernel<MODE_FUSED, false, true>
              : variant == 2 ? stream_kernel<MODE_FUSED, true>
                             : stream_kernel<MODE_FUSED, false>;
  const size_t smem = wide ? smem_bytes<32>() : smem_bytes<16>();
  static bool attr_done[4] = {false, false, false, false};
  if (!attr_done[variant]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr_done[variant] = true;
  }
  const long max_units = (long)a13.max_active * a13.units_per_expert * a13.ksplit +
                         (long)a2.max_active * a2.units_per_expert * a2.ksplit;
  long grid = (long)(wide ? ctas_per_sm<32>() : ctas_per_sm<16>()) * sm_count;
  if (grid > max_units) grid = max_units;
  if (grid <= 0) return cudaSuccess;
  // a programmatic dependent of the sort
  return launch_kernel(kern, dim3((unsigned)grid), dim3(THREADS), smem, stream, true, a13, a2);
}

}  // namespace moe
