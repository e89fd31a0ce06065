// moe_align.cu -- expert sort / block padding (moe_align_block_size).
//
// The dispatch step named by moe_sorting_dispatch_policy in AiterExperts.apply
// (page "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe").  The
// pages do not print the algorithm; this kernel implements the rule stated in
// include/moe_experts.h: per local expert (ascending), the flat slot ids in
// ascending order, padded with S = M*T to a multiple of BM.
//
// One CTA of 32 warps does the sort; it is latency-bound and tiny next to the
// GEMMs.  Each warp owns a contiguous range of slots:
//   A. per-warp histograms: __match_any_sync groups the lanes holding the
//      same expert, the group leader adds the group size (no smem atomics);
//   B. per expert, an exclusive prefix over warps (stable order) and the
//      padded size; an exclusive scan over experts gives the block offsets;
//   C. each warp walks its range in order and scatters every slot to
//      offset[e] + (slots of e in earlier warps) + (rank among earlier
//      lanes of its group); the first round reuses step A's expert ids;
//   D. padding entries, expert_ids, tails.
// Only the warps that hold slots take part in B (a batch of 4 slots: 4 of
// the 32), and the block-size arithmetic is shifts for powers of two.
// Extra CTAs (blockIdx.x > 0) zero an optional fp32 buffer (the stage-2
// accumulator) so the fused path needs no separate memset launch.
//
// Large batches with caller scratch (>= kMultiMinSlots slots) run the same
// steps on NC CTAs in two grids, since every 32-slot round of a warp costs
// about the same (measured ~2000 cycles, whatever the round holds):
//   count grid:   NC CTAs, warp w of CTA c owns the (32 c + w)-th contiguous
//                 range of the slots; step A; each CTA writes its per-expert
//                 totals to scratch [NC][El];
//   scatter grid: each CTA repeats step A for its own warps, adds the totals
//                 of the CTAs before it (stable order across CTAs), then B,
//                 C and its share of D; the zeroing / conversion CTAs ride in
//                 this grid.
#include <cuda_fp16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
// multi-CTA sort: 4 rounds of 32 slots per warp, from 2 CTAs' worth of slots
constexpr long kMultiSlotsPerCta = 4L * 32 * kAlignWarps;
constexpr long kMultiMinSlots = 2 * kMultiSlotsPerCta;
constexpr int kMultiMaxCtas = 64;

// Local expert of global expert id g (-1: masked, out of range or no slot).
__device__ __forceinline__ int local_of_id(int g, const int32_t *emap, int E, int El) {
  if (g < 0 || g >= E) return -1;
  int l = emap ? emap[g] : g;
  return (l >= 0 && l < El) ? l : -1;
}

__device__ __forceinline__ int local_of(const int32_t *ids, const int32_t *emap, long s, int E,
                                        int El, long s_valid) {
  if (s >= s_valid) return -1;  // a token beyond the valid count (padded dispatch buffer)
  return local_of_id(ids[s], emap, E, El);
}

// Division by the sort's block size for the non-negative counts, offsets and
// capacities of a sort: a shift when it is a power of two (the block sizes
// the library's kernels use), else the integer divide.
struct BlockSize {
  int bm, shift;
  __device__ explicit BlockSize(int b) : bm(b), shift(-1) {
    int k = 0;
    while (k < 11 && (1 << k) < b) ++k;  // b <= 1024
    if ((1 << k) == b) shift = k;
  }
  __device__ long div(long v) const { return shift >= 0 ? v >> shift : v / bm; }
  __device__ int round_up(int v) const { return (int)(div((long)v + bm - 1) * bm); }
};

// The extra CTAs of a sort grid (index b from 0): the first zero_ctas zero
// x.zero_buf / x.zero_ints, the next conv_ctas write the per-token f16 copy
// of x.
__device__ __forceinline__ void align_extra_cta(const AlignExtras &x, int zero_ctas, int conv_ctas,
                                                int b) {
  if (b < zero_ctas) {
    // zeroing CTAs: 16-byte stores over the aligned body, scalar tail
    const long n4 = x.zero_buf ? x.zero_n / 4 : 0;
    float4 *p4 = reinterpret_cast<float4 *>(x.zero_buf);
    const long stride = (long)zero_ctas * blockDim.x;
    for (long i = (long)b * blockDim.x + threadIdx.x; i < n4; i += stride)
      p4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long i = n4 * 4 + (long)b * blockDim.x + threadIdx.x;
         x.zero_buf && i < x.zero_n; i += stride)
      x.zero_buf[i] = 0.f;
    for (long i = (long)b * blockDim.x + threadIdx.x; i < x.zero_ints_n; i += stride)
      x.zero_ints[i] = 0;
    return;
  }
  {
    // conversion CTAs: 128 threads per row of x, 8 rows per CTA; bf16 -> f16
    // scaled by 2^a so that the row maximum lands in [2^14, 2^15) (exact for
    // bf16 values).  With x_mx the values are first quantised to OCP MXFP4 /
    // MXFP8 and dequantised (|QDQ(x)| <= 1.75 * 2^floor(log2 max|x|), so the
    // same 2^a keeps them below 2^15).  Rows are 16-byte aligned (K % 32 == 0,
    // checked by the caller); up to 4 x 8 values per thread stay in registers
    // between the max pass and the convert pass.
    __shared__ float red[kAlignThreads / 128][4];
    const int k8 = x.xK / 8;
    const int tr = threadIdx.x & 127, rsub = threadIdx.x >> 7, wr = tr >> 5;
    const int lane = threadIdx.x & 31;
    const int rows_per_cta = blockDim.x / 128;
    for (int base = (b - zero_ctas) * rows_per_cta; base < x.xM;
         base += conv_ctas * rows_per_cta) {
      const int r = base + rsub;
      const bool valid = r < x.xM;
      const uint4 *xr = reinterpret_cast<const uint4 *>(x.x + (long)(valid ? r : 0) * x.xK);
      uint4 v[4];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = tr + i * 128;
        v[i] = (valid && c < k8) ? xr[c] : make_uint4(0, 0, 0, 0);
      }
      for (int c = tr + 512; valid && c < k8; c += 128) {
        const uint4 u = xr[c];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[q] << 16)),
                                   fabsf(__uint_as_float(w[q] & 0xffff0000u))));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[q] << 16)),
                                   fabsf(__uint_as_float(w[q] & 0xffff0000u))));
      }
      amax = warp_max(amax);
      if (lane == 0) red[rsub][wr] = amax;
      __syncthreads();
      amax = fmaxf(fmaxf(red[rsub][0], red[rsub][1]), fmaxf(red[rsub][2], red[rsub][3]));
      __syncthreads();
      if (!valid) continue;
      int a = 0;
      if (amax > 0.f) {
        int ex;
        frexpf(amax, &ex);  // amax = f * 2^ex, 0.5 <= f < 1
        a = 15 - ex;
      }
      const float mul = ldexpf(1.0f, a);
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__half *>(x.x16) + (long)r * x.xK);
      // the four lanes of a 32-element block (chunk c holds elements 8c..8c+7
      // and c % 4 == lane % 4) take every convert together
      const unsigned gmask = 0xFu << (lane & 28);
      auto convert = [&](const uint4 &u) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        if (x.x_mx) {  // OCP MX quantise-dequantise of the block, then 2^a
          float f[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            f[2 * q] = __uint_as_float(w[q] << 16);
            f[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
          }
          return mx_qdq_f16x8(f, x.x_mx == 1, a, gmask);
        }
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __half2 h = __floats2half2_rn(__uint_as_float(w[q] << 16) * mul,
                                              __uint_as_float(w[q] & 0xffff0000u) * mul);
          o[q] = *reinterpret_cast<const uint32_t *>(&h);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
      };
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = tr + i * 128;
        if (c < k8) dst[c] = convert(v[i]);
      }
      for (int c = tr + 512; c < k8; c += 128) dst[c] = convert(xr[c]);
      if (tr == 0) x.x_inv[r] = ldexpf(1.0f, -a);
    }
    return;
  }
}

__global__ void __launch_bounds__(kAlignThreads)
align_kernel(const int32_t *__restrict__ ids, long S, const int32_t *__restrict__ emap, int E,
             int El, int BM, int32_t *__restrict__ sorted, int32_t *__restrict__ expert_ids,
             int32_t *__restrict__ ntp, int32_t *__restrict__ counts, long cap, AlignExtras x,
             int zero_ctas, int conv_ctas) {
  // Launched as a programmatic dependent of the previous kernel (the router,
  // or whatever produced topk_ids): every CTA waits for it before reading the
  // ids or overwriting buffers it may still read.  A dependent grid (the
  // streaming GEMM) may be scheduled now: it waits for this grid's completion
  // before it reads anything written here.
  griddep_launch_dependents();
  griddep_wait();
  if (blockIdx.x > 0) {
    align_extra_cta(x, zero_ctas, conv_ctas, (int)blockIdx.x - 1);
    return;
  }
  // slots of tokens at or beyond the valid count (when given) are dropped
  long s_valid = S;
  if (x.num_valid_tokens) {
    const long n = *x.num_valid_tokens;
    const long T = x.slots_per_token;
    s_valid = n <= 0 ? 0 : (n * T < S ? n * T : S);
  }
  extern __shared__ int smem[];
  int *cnt = smem;                     // [kAlignWarps][El]  per-warp counts -> prefixes
  int *off = smem + kAlignWarps * El;  // [El + 1]           expert offsets
  int *pad = off + El + 1;             // [El]               padded sizes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  const BlockSize bs(BM);

  const long per = ceil_div(S, kAlignWarps);
  const long beg = (long)warp * per;
  const long end = beg + per < S ? beg + per : S;
  // warps that hold slots (S <= 2^30: 32-bit arithmetic); the others have
  // nothing to count or scatter, so their rows of cnt are never used
  const int nwu = per > 0 ? (int)((uint32_t)(S + per - 1) / (uint32_t)per) : 0;
  // the ids of each warp's first 32 slots, requested before the zeroing
  int g0 = -1;
  if (beg + lane < end && beg + lane < s_valid) g0 = ids[beg + lane];

  for (int i = threadIdx.x; i < nwu * El; i += blockDim.x) cnt[i] = 0;
  __syncthreads();

  // A. per-warp histogram (the first round's local experts are kept for C)
  int l0 = -1;
  for (long base = beg; base < end; base += 32) {
    const long s = base + lane;
    int l;
    if (base == beg) l = l0 = local_of_id(g0, emap, E, El);
    else l = s < end ? local_of(ids, emap, s, E, El, s_valid) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, l);
    if (l >= 0 && lane == __ffs(peers) - 1) cnt[warp * El + l] += __popc(peers);
  }
  __syncthreads();

  // B. stable prefix over warps, totals and padded sizes
  for (int e = threadIdx.x; e < El; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < nwu; ++w) {
      const int c = cnt[w * El + e];
      cnt[w * El + e] = run;
      run += c;
    }
    if (counts) counts[e] = run;
    pad[e] = bs.round_up(run);
    off[e] = run;  // live count, kept for step D
  }
  __syncthreads();
  // exclusive scan of pad[] by warp 0 (El <= 1024: 32 consecutive experts per lane)
  if (warp == 0) {
    const int chunk = (El + 31) / 32;
    const int e0 = lane * chunk;
    int local = 0;
    for (int e = e0; e < e0 + chunk && e < El; ++e) local += pad[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e0 + chunk && e < El; ++e) {
      const int p = pad[e];
      pad[e] = run;  // pad[] now holds the exclusive offsets
      run += p;
    }
    if (lane == 31) off[El] = incl;
  }
  // compact list of experts with at least one slot (ascending), by warp 1
  if (warp == 1 && x.active) {
    const int chunk = (El + 31) / 32;
    const int e0 = lane * chunk;
    int local = 0;
    for (int e = e0; e < e0 + chunk && e < El; ++e) local += off[e] > 0;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int pos = incl - local;
    for (int e = e0; e < e0 + chunk && e < El; ++e)
      if (off[e] > 0) x.active[pos++] = e;
    if (lane == 31) *x.n_active = incl;
  }
  __syncthreads();
  // pad[e] = offset of expert e, off[e] = live count of e, off[El] = total
  if (x.offsets)
    for (int e = threadIdx.x; e < El; e += blockDim.x) x.offsets[e] = pad[e];

  // C. stable scatter: expert offset + slots of the earlier warps + rank
  for (long base = beg; base < end; base += 32) {
    const long s = base + lane;
    const int l = base == beg ? l0 : (s < end ? local_of(ids, emap, s, E, El, s_valid) : -1);
    const unsigned peers = __match_any_sync(0xffffffffu, l);
    int pos = 0;
    if (l >= 0) pos = pad[l] + cnt[warp * El + l] + __popc(peers & lt_mask);
    __syncwarp();
    if (l >= 0) {
      sorted[pos] = (int32_t)s;
      if (lane == __ffs(peers) - 1) cnt[warp * El + l] += __popc(peers);
    }
    __syncwarp();
  }

  // D. padding, block -> expert table, tails
  const int total = off[El];
  for (int e = warp; e < El; e += kAlignWarps) {
    const int o = pad[e], live = off[e];
    const int padded = bs.round_up(live);
    const int ob = (int)bs.div(o), nb = (int)bs.div(padded);
    for (int i = live + lane; i < padded; i += 32) sorted[o + i] = (int32_t)S;
    for (int b = lane; b < nb; b += 32) expert_ids[ob + b] = e;
  }
  const long cap_blocks = bs.div(cap);
  for (long i = total + threadIdx.x; i < cap; i += blockDim.x) sorted[i] = (int32_t)S;
  for (long b = bs.div(total) + threadIdx.x; b < cap_blocks; b += blockDim.x) expert_ids[b] = -1;
  if (threadIdx.x == 0) {
    *ntp = total;
    if (x.counters) x.counters[0] = x.counters[1] = 0;
  }
}

// The per-warp histogram of step A over the slots [beg, end) into
// cnt[warp * El + local expert].
__device__ __forceinline__ void warp_histogram(const int32_t *ids, const int32_t *emap, int E,
                                               int El, long s_valid, long beg, long end, int *cnt,
                                               int warp, int lane) {
  for (long base = beg; base < end; base += 32) {
    const long s = base + lane;
    const int l = s < end ? local_of(ids, emap, s, E, El, s_valid) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, l);
    if (l >= 0 && lane == __ffs(peers) - 1) cnt[warp * El + l] += __popc(peers);
  }
}

__device__ __forceinline__ long valid_slots(long S, const AlignExtras &x) {
  if (!x.num_valid_tokens) return S;
  const long n = *x.num_valid_tokens;
  const long T = x.slots_per_token;
  return n <= 0 ? 0 : (n * T < S ? n * T : S);
}

// Count grid of the multi-CTA sort: per-CTA expert totals into ctot[c][El].
__global__ void __launch_bounds__(kAlignThreads)
align_count_kernel(const int32_t *__restrict__ ids, long S, const int32_t *__restrict__ emap,
                   int E, int El, int32_t *__restrict__ ctot, AlignExtras x) {
  griddep_launch_dependents();
  griddep_wait();
  const long s_valid = valid_slots(S, x);
  extern __shared__ int smem[];
  int *cnt = smem;  // [kAlignWarps][El]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kAlignWarps * El; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const long per = ceil_div(S, (long)gridDim.x * kAlignWarps);
  const long beg = ((long)blockIdx.x * kAlignWarps + warp) * per;
  const long end = beg + per < S ? beg + per : S;
  warp_histogram(ids, emap, E, El, s_valid, beg, end, cnt, warp, lane);
  __syncthreads();
  for (int e = threadIdx.x; e < El; e += blockDim.x) {
    int t = 0;
    for (int w = 0; w < kAlignWarps; ++w) t += cnt[w * El + e];
    ctot[(long)blockIdx.x * El + e] = t;
  }
}

// Scatter grid of the multi-CTA sort (CTAs nc.. are the extra CTAs).
__global__ void __launch_bounds__(kAlignThreads)
align_scatter_kernel(const int32_t *__restrict__ ids, long S, const int32_t *__restrict__ emap,
                     int E, int El, int BM, int32_t *__restrict__ sorted,
                     int32_t *__restrict__ expert_ids, int32_t *__restrict__ ntp,
                     int32_t *__restrict__ counts, long cap, AlignExtras x,
                     const int32_t *__restrict__ ctot, int nc, int zero_ctas, int conv_ctas) {
  // waits for the count grid (and so for everything before it)
  griddep_launch_dependents();
  griddep_wait();
  if ((int)blockIdx.x >= nc) {
    align_extra_cta(x, zero_ctas, conv_ctas, (int)blockIdx.x - nc);
    return;
  }
  const int c = blockIdx.x;
  const long s_valid = valid_slots(S, x);
  const BlockSize bs(BM);
  extern __shared__ int smem[];
  int *cnt = smem;                     // [kAlignWarps][El]  per-warp counts -> positions
  int *off = smem + kAlignWarps * El;  // [El + 1]           live counts, total
  int *pad = off + El + 1;             // [El]               padded sizes -> offsets
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int i = threadIdx.x; i < kAlignWarps * El; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const long per = ceil_div(S, (long)nc * kAlignWarps);
  const long beg = ((long)c * kAlignWarps + warp) * per;
  const long end = beg + per < S ? beg + per : S;
  // A. this CTA's per-warp histograms (the count grid's, again)
  warp_histogram(ids, emap, E, El, s_valid, beg, end, cnt, warp, lane);
  __syncthreads();
  // B. per expert: the slots of the CTAs before this one, then a stable
  // prefix over this CTA's warps; totals and padded sizes
  for (int e = threadIdx.x; e < El; e += blockDim.x) {
    int tot = 0, before = 0;
    for (int k = 0; k < nc; ++k) {
      const int v = ctot[(long)k * El + e];
      tot += v;
      before += k < c ? v : 0;
    }
    int run = before;
    for (int w = 0; w < kAlignWarps; ++w) {
      const int v = cnt[w * El + e];
      cnt[w * El + e] = run;
      run += v;
    }
    if (c == 0 && counts) counts[e] = tot;
    pad[e] = bs.round_up(tot);
    off[e] = tot;
  }
  __syncthreads();
  // exclusive scan of pad[] by warp 0 (El <= 1024: 32 consecutive experts per lane)
  if (warp == 0) {
    const int chunk = (El + 31) / 32;
    const int e0 = lane * chunk;
    int local = 0;
    for (int e = e0; e < e0 + chunk && e < El; ++e) local += pad[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e0 + chunk && e < El; ++e) {
      const int p = pad[e];
      pad[e] = run;
      run += p;
    }
    if (lane == 31) off[El] = incl;
  }
  // compact list of experts with at least one slot (ascending), by CTA 0's warp 1
  if (c == 0 && warp == 1 && x.active) {
    const int chunk = (El + 31) / 32;
    const int e0 = lane * chunk;
    int local = 0;
    for (int e = e0; e < e0 + chunk && e < El; ++e) local += off[e] > 0;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int pos = incl - local;
    for (int e = e0; e < e0 + chunk && e < El; ++e)
      if (off[e] > 0) x.active[pos++] = e;
    if (lane == 31) *x.n_active = incl;
  }
  __syncthreads();
  if (c == 0 && x.offsets)
    for (int e = threadIdx.x; e < El; e += blockDim.x) x.offsets[e] = pad[e];
  // C. stable scatter of this CTA's slots: expert offset + slots before + rank
  for (long base = beg; base < end; base += 32) {
    const long s = base + lane;
    const int l = s < end ? local_of(ids, emap, s, E, El, s_valid) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, l);
    int pos = 0;
    if (l >= 0) pos = pad[l] + cnt[warp * El + l] + __popc(peers & lt_mask);
    __syncwarp();
    if (l >= 0) {
      sorted[pos] = (int32_t)s;
      if (lane == __ffs(peers) - 1) cnt[warp * El + l] += __popc(peers);
    }
    __syncwarp();
  }
  // D. this CTA's share of the padding, the block -> expert table and tails
  const int total = off[El];
  const int gw = c * kAlignWarps + warp, nw = nc * kAlignWarps;
  for (int e = gw; e < El; e += nw) {
    const int o = pad[e], live = off[e];
    const int padded = bs.round_up(live);
    const int ob = (int)bs.div(o), nb = (int)bs.div(padded);
    for (int i = live + lane; i < padded; i += 32) sorted[o + i] = (int32_t)S;
    for (int b = lane; b < nb; b += 32) expert_ids[ob + b] = e;
  }
  const long gt = (long)c * blockDim.x + threadIdx.x, nt = (long)nc * blockDim.x;
  const long cap_blocks = bs.div(cap);
  for (long i = total + gt; i < cap; i += nt) sorted[i] = (int32_t)S;
  for (long b = bs.div(total) + gt; b < cap_blocks; b += nt) expert_ids[b] = -1;
  if (c == 0 && threadIdx.x == 0) {
    *ntp = total;
    if (x.counters) x.counters[0] = x.counters[1] = 0;
  }
}

}  // namespace

// CTAs of the multi-CTA sort for S slots (0: one CTA), and its scratch.
int align_multi_ctas(long S) {
  if (S < kMultiMinSlots) return 0;
  const long n = ceil_div(S, (long)kMultiSlotsPerCta);
  return (int)(n < kMultiMaxCtas ? n : kMultiMaxCtas);
}
size_t align_scratch_bytes(long S, int El) {
  return (size_t)align_multi_ctas(S) * El * sizeof(int32_t);
}

cudaError_t launch_align(const int32_t *topk_ids, int M, int T, const int32_t *expert_map, int E,
                         int El, int BM, int32_t *sorted_ids, int32_t *expert_ids,
                         int32_t *num_post_pad, int32_t *counts, long cap,
                         const AlignExtras &extra_in, cudaStream_t stream) {
  AlignExtras extra = extra_in;
  extra.slots_per_token = T;
  const size_t smem = sizeof(int) * ((size_t)kAlignWarps * El + 2 * (size_t)El + 1);
  if (smem > 48 * 1024) {
    // opt in once to the largest size these kernels can ask for (El = 1024),
    // so later calls (for instance inside a stream capture) make no attribute
    // call
    static const cudaError_t opt_in = [] {
      const int most = (int)(sizeof(int) * ((size_t)kAlignWarps * 1024 + 2 * 1024 + 1));
      cudaError_t e = cudaFuncSetAttribute(align_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, most);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(align_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 most);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(align_scatter_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, most);
      return e;
    }();
    if (opt_in != cudaSuccess) return opt_in;
  }
  int zero_ctas = 0, conv_ctas = 0;
  if ((extra.zero_buf && extra.zero_n > 0) || (extra.zero_ints && extra.zero_ints_n > 0)) {
    const long per_cta = (long)kAlignThreads * 4 * 8;
    const long n = extra.zero_buf ? extra.zero_n : 0;
    zero_ctas = (int)ceil_div(n + extra.zero_ints_n, per_cta);
    if (zero_ctas < 1) zero_ctas = 1;
    if (zero_ctas > 4 * 152) zero_ctas = 4 * 152;
  }
  if (extra.x && extra.xM > 0) {
    conv_ctas = (int)ceil_div(extra.xM, kAlignThreads / 128);
    if (conv_ctas > 2 * 152) conv_ctas = 2 * 152;
  }
  const long S = (long)M * T;
  const int nc = align_multi_ctas(S);
  if (nc > 0 && extra.scratch && extra.scratch_bytes >= align_scratch_bytes(S, El)) {
    cudaError_t e = launch_kernel(align_count_kernel, dim3(nc), dim3(kAlignThreads),
                                  sizeof(int) * (size_t)kAlignWarps * El, stream, true, topk_ids,
                                  S, expert_map, E, El, extra.scratch, extra);
    if (e != cudaSuccess) return e;
    return launch_kernel(align_scatter_kernel, dim3(nc + zero_ctas + conv_ctas),
                         dim3(kAlignThreads), smem, stream, true, topk_ids, S, expert_map, E, El,
                         BM, sorted_ids, expert_ids, num_post_pad, counts, cap, extra,
                         static_cast<const int32_t *>(extra.scratch), nc, zero_ctas, conv_ctas);
  }
  return launch_kernel(align_kernel, dim3(1 + zero_ctas + conv_ctas), dim3(kAlignThreads), smem,
                       stream, true, topk_ids, S, expert_map, E, El, BM, sorted_ids,
                       expert_ids, num_post_pad, counts, cap, extra, zero_ctas, conv_ctas);
}

}  // namespace moe

// ------------------------------------------------------------------ batched
// Batched expert-parallel input (no routing, no sort): the rows of local
// expert e are the first count[e] rows of its max_tokens-row slice, so the
// padded blocks follow from an exclusive scan of ceil(count[e] / BM) * BM.
// CTA 0 builds sorted_ids (slot e * max_tokens + i, sentinel S past count[e])
// and expert_ids; the other CTAs zero the fp32 accumulator and fill the
// per-slot weights with 1.
namespace moe {
namespace {

__global__ void __launch_bounds__(1024)
batched_align_kernel(const int32_t *__restrict__ counts_in, int El, int max_tokens, int BM,
                     int32_t *__restrict__ sorted, int32_t *__restrict__ expert_ids,
                     int32_t *__restrict__ ntp, long cap, float *__restrict__ zero_buf, long zero_n,
                     float *__restrict__ ones, int zero_ctas) {
  griddep_launch_dependents();
  griddep_wait();
  const long S = (long)El * max_tokens;
  if (blockIdx.x > 0) {
    const long stride = (long)zero_ctas * blockDim.x;
    for (long i = (long)(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < zero_n; i += stride)
      zero_buf[i] = 0.f;
    for (long i = (long)(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < S; i += stride) ones[i] = 1.f;
    return;
  }
  __shared__ int off[1025];
  __shared__ int cnt[1024];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const BlockSize bs(BM);
  for (int e = threadIdx.x; e < El; e += blockDim.x) {
    const int c = counts_in[e];
    cnt[e] = c < 0 ? 0 : (c > max_tokens ? max_tokens : c);
  }
  __syncthreads();
  // exclusive scan of the padded sizes by warp 0 (El <= 1024)
  if (warp == 0) {
    const int chunk = (El + 31) / 32;
    const int e0 = lane * chunk;
    int local = 0;
    for (int e = e0; e < e0 + chunk && e < El; ++e) local += bs.round_up(cnt[e]);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e0 + chunk && e < El; ++e) {
      off[e] = run;
      run += bs.round_up(cnt[e]);
    }
    if (lane == 31) off[El] = incl;
  }
  __syncthreads();
  const int total = off[El];
  for (int e = warp; e < El; e += blockDim.x / 32) {
    const int o = off[e], c = cnt[e];
    const int padded = bs.round_up(c);
    const int ob = (int)bs.div(o), nb = (int)bs.div(padded);
    for (int i = lane; i < padded; i += 32)
      sorted[o + i] = i < c ? (int32_t)((long)e * max_tokens + i) : (int32_t)S;
    for (int b = lane; b < nb; b += 32) expert_ids[ob + b] = e;
  }
  const long cap_blocks = bs.div(cap);
  for (long i = total + threadIdx.x; i < cap; i += blockDim.x) sorted[i] = (int32_t)S;
  for (long b = bs.div(total) + threadIdx.x; b < cap_blocks; b += blockDim.x) expert_ids[b] = -1;
  if (threadIdx.x == 0) *ntp = total;
}

}  // namespace

cudaError_t launch_batched_align(const int32_t *counts, int El, int max_tokens, int BM,
                                 int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_post_pad,
                                 long cap, float *zero_buf, long zero_n, float *ones,
                                 cudaStream_t stream) {
  const long S = (long)El * max_tokens;
  long n = zero_n > S ? zero_n : S;
  int zero_ctas = (int)ceil_div(n, 1024L * 8);
  if (zero_ctas < 1) zero_ctas = 1;
  if (zero_ctas > 4 * 152) zero_ctas = 4 * 152;
  return launch_kernel(batched_align_kernel, dim3(1 + zero_ctas), dim3(1024), 0, stream, true,
                       counts, El, max_tokens, BM, sorted_ids, expert_ids, num_post_pad, cap,
                       zero_buf, zero_n, ones, zero_ctas);
}

}  // namespace moe
