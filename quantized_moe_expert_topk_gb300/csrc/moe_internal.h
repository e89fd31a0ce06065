// moe_internal.h -- host-side declarations shared by the library's translation
// units (kernel launchers and their argument blocks).  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Launch `kern` on `stream`; with `dependent` set, as a programmatic dependent
// of the previous kernel in the stream (it may start while that kernel drains
// and must call griddepcontrol.wait before reading that kernel's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool dependent, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = dependent ? attr : nullptr;
  cfg.numAttrs = dependent ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Tile height (sorted rows per block) of the mma.sync grouped GEMMs; the
// expert sort pads every expert to a multiple of it.
constexpr int kGenericBlockM = 64;
// Tile height of the tcgen05 GEMMs (and the sort block of that path).
constexpr int kTcBlockM = 128;
// Largest packed FP4 weight record of one tcgen05 pipeline stage.
constexpr int kTcRecMaxBytes = 4096 + 128 * 4;

// Optional extra work folded into the sort launch (extra CTAs / outputs).
struct AlignExtras {
  float *zero_buf = nullptr;      // zeroed (the stage-2 accumulator)
  long zero_n = 0;
  int32_t *offsets = nullptr;     // [El] start of each expert's rows in sorted_ids
  int32_t *active = nullptr;      // [El] local experts with >= 1 slot, ascending
  int32_t *n_active = nullptr;    // [1]
  int32_t *counters = nullptr;    // [2] work counters of the streaming kernels, zeroed
  const uint16_t *x = nullptr;    // bf16 [M, K] -> x16 f16 [M, K] scaled per row by 2^a,
  void *x16 = nullptr;            //   max |x| in [2^14, 2^15) after scaling; x_inv[row] = 2^-a
  float *x_inv = nullptr;
  int xM = 0, xK = 0;
  int x_mx = 0;                   // 1 / 2: x16 holds the OCP MXFP4 / MXFP8 dequantised x
  int32_t *zero_ints = nullptr;   // also zeroed (counters of the split W13 units)
  long zero_ints_n = 0;
  const int32_t *num_valid_tokens = nullptr;  // [1]: slots of tokens >= it are dropped
  int slots_per_token = 1;                     // topk (set by launch_align)
  // scratch of the multi-CTA sort (align_scratch_bytes); null or too small:
  // the one-CTA sort
  int32_t *scratch = nullptr;
  size_t scratch_bytes = 0;
};

// The multi-CTA sort of S slots: its CTAs (0 below its size threshold: the
// one-CTA kernel) and its scratch bytes (per-CTA expert totals).
int align_multi_ctas(long S);
size_t align_scratch_bytes(long S, int El);

cudaError_t launch_align(const int32_t *topk_ids, int M, int T, const int32_t *expert_map, int E,
                         int El, int BM, int32_t *sorted_ids, int32_t *expert_ids,
                         int32_t *num_post_pad, int32_t *counts, long cap,
                         const AlignExtras &extra, cudaStream_t stream);

// Batched expert-parallel input: sorted_ids / expert_ids / num_post_pad of
// blocks of BM rows from per-expert counts (rows e * max_tokens + i, i <
// count[e]), no sort; zero_buf [zero_n] zeroed and ones [El * max_tokens] set
// to 1 (the per-slot weights) by extra CTAs.  cap = El * max_tokens + El * (BM - 1)
// rounded up to BM bounds num_post_pad.
cudaError_t launch_batched_align(const int32_t *counts, int El, int max_tokens, int BM,
                                 int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_post_pad,
                                 long cap, float *zero_buf, long zero_n, float *ones,
                                 cudaStream_t stream);

// Quantise rows of x (bf16, or fp32 when x_is_f32) into the activation format
// `afmt`.  With `sorted_ids` set, the rows are sorted intermediate rows: rows
// at or beyond *num_post_pad are skipped, padding rows get zero codes, and the
// NVFP4 global is per expert (param[expert_ids[r / BM]]).
struct QuantArgs {
  const void *x;
  int x_is_f32;
  long rows;
  int cols;
  int afmt;
  const float *param;       // static fp8 scale [1] / NVFP4 global(s)
  const int32_t *sorted_ids; // nullable
  const int32_t *expert_ids;
  const int32_t *num_post_pad;
  int S;
  int BM;
  void *codes;
  void *scales;
};
cudaError_t launch_quant(const QuantArgs &a, cudaStream_t stream);

// Failure-detection self-test (moe_selftest.cu): one bounded wait that runs
// out and records MOE_ERR_TIMEOUT in *err.
cudaError_t launch_selftest_wait(int *err, long long limit_cycles, cudaStream_t stream);

// fp32 intermediate rows -> f16 rows of their OCP MX (MXFP4 when fp4, else
// MXFP8) quantise-dequantise, no row scale (the caller guarantees the f16
// range).  With sorted_ids set, rows at or beyond *num_post_pad are skipped
// and padding rows (sorted id >= S) become zeros (zero_pad) or are skipped;
// otherwise all `rows` rows are converted.  `dependent`: launched as a
// programmatic dependent.
cudaError_t launch_mx_qdq_rows(const float *src, long rows, int N, const int32_t *sorted_ids,
                               const int32_t *num_post_pad, int S, void *dst, int fp4,
                               int zero_pad, cudaStream_t stream, bool dependent);

struct GemmArgs {
  int M, K, N, T, El, BM;
  int wfmt;     // weight format (moe_wfmt)
  int afmt;     // format of the A operand (moe_afmt; stage-2 format for w2)
  int act, gate;
  float alpha, beta, limit;
  // A operand: W13 gathers token rows (slot / T); W2 reads sorted rows.
  const void *a_codes;
  const void *a_scales;
  const float *a_global; // NVFP4 global: [1] for W13, per expert [El] for W2
  // weights
  const void *w_codes;
  const void *w_scales;
  const float *w_global;
  const void *w_bias;
  int bias_f32;
  // routing
  const int32_t *sorted_ids;
  const int32_t *expert_ids;
  const int32_t *num_post_pad;
  int S;
  // outputs
  void *out;        // W13: intermediate (bf16 or fp32 [cap, N])
  int out_f32;
  float *acc;       // W2: fp32 [M, K] accumulator
  const float *topk_weights;
  int w_stage1;     // router weight on the stage-1 output (W13 multiplies, W2 does not)
};
cudaError_t launch_gemm_w13(const GemmArgs &a, long cap_rows, cudaStream_t stream);
cudaError_t launch_gemm_w2(const GemmArgs &a, long cap_rows, cudaStream_t stream);
// Weight-streaming decode kernels (moe_stream.cu), MXFP4 w4a16.
struct StreamArgs {
  int M, K, N, T, C;              // C: reduction length (K for w13, N for w2)
  int units_per_expert, ksplit, kblocks, max_active;
  int act, gate;
  float alpha, beta, limit;
  const void *packed;             // packed weight records
  const void *bias;               // bf16 [El, R] or null
  const void *x16;                // f16 rows: x [M, K] (w13) or the intermediate [cap, N] (w2)
  const float *x_inv;             // w13: per-token inverse scale of x16
  const int32_t *sorted_ids, *offsets, *counts, *active, *n_active;
  void *out;                      // w13: f16 intermediate [cap, N] (fp32 with out_f32)
  int out_f32;                    // w13: fp32 rows for a later requantiser
  int out_mx;                     // w13 in the fused grid: 1 / 2 = OCP MXFP4 / MXFP8
                                  //   quantise-dequantise of the f16 intermediate
  float *acc;                     // w2: fp32 [M, K]
  const float *topk_weights;
  int w_stage1;                   // router weight on the stage-1 output (W13 multiplies, W2 not)
  int *err;                       // device error word
  int *work_counter;              // zero at launch; units are claimed from it
  // W13 with ksplit > 1: each k-range writes its fp32 (gate, up) partials to
  // hpart[ks][slot][N][2]; the last of the ksplit arrivals of a (unit, pass,
  // warp) -- counted in fix_cnt, zeroed by the sort -- sums them and applies
  // bias and activation
  float *hpart;
  int *fix_cnt;
  int S;                          // slots (M * T)
  // fused W13 + W2 grid (launch_stream_fused): per local expert, the count of
  // (W13 unit, pass, consumer warp) epilogues done; zeroed by the sort
  int *done13;
  // tokens per pass of the fused grid: 16 (0 reads as 16), or 32 (no k-split,
  // no MX epilogue; three CTAs per SM): both argument blocks the same
  int tok_pass;
};
// k-split of the W13 streaming units for this problem (1 = whole K per unit).
int stream_w13_ksplit(int M, int topk, int El, int N, int K, int sm_count);
// Number of fixup counters of the split W13 units for a sort capacity.
long stream_w13_fixups(long cap_rows, int N);
struct PackArgs {
  const unsigned char *codes, *scales;
  unsigned char *out;
  long total;
  int kblocks, units, w13, N, R, C, gate;
};
size_t stream_packed_bytes(int w13, int N, int K, int El);
int stream_units_per_expert(int w13, int N, int K);
cudaError_t launch_pack_mxfp4(const PackArgs &p, cudaStream_t stream);
cudaError_t launch_stream(const StreamArgs &a, int w13, int sm_count, cudaStream_t stream);
// W13 and W2 as one persistent grid: the W2 units of an expert wait, bounded,
// for its W13 units' completion count.  W13 may be split along K (not with
// the MX epilogue).
cudaError_t launch_stream_fused(const StreamArgs &a13, const StreamArgs &a2, int sm_count,
                                cudaStream_t stream);

// tcgen05 grouped GEMMs (moe_tc.cu)
// Output of the tcgen05 W13 epilogue: bf16 rows, fp32 staging rows (a
// separate requantiser follows), f16 rows (bounded SwiGLU-OAI intermediate),
// or the OCP MX quantise-dequantise of the intermediate as exact f16 values.
enum { TC_OUT_BF16 = 0, TC_OUT_F32 = 1, TC_OUT_F16 = 2, TC_OUT_MX4_F16 = 3, TC_OUT_MX8_F16 = 4 };

// Block-scaled NVFP4 operands (moe_bs.cu).  Every 256-element reduction
// stage of a 128-row block of the A operand carries an 8 KB scale-factor
// record: two 4 KB sources of tcgen05.cp .128x256b, one per pair of 64-element
// MMA steps (2p, 2p + 1).  A source is 128 rows of 32 bytes, no swizzle, in
// 8-row x 16-byte core matrices (the row's two 16-byte halves 128 bytes apart,
// 8-row groups 256 bytes apart).  Row L holds, in its first half, the scale
// words of step 2p of block rows L % 32 + 32 w (w = 0..3; byte b of word w
// scales elements [16 b, 16 b + 16) of the step) and, in its second half,
// those of step 2p + 1: rows L, L + 32, L + 64 and L + 96 hold the same bytes,
// which is the replication across the four 32-lane quarters of Tensor Memory
// that the scale factors of an M = 128 MMA need (lane L, column 4 j + w = the
// word of row L % 32 + 32 w for step j).
constexpr int kTcBsStage = 256;      // reduction elements per stage
constexpr int kBsSfaRecBytes = 8192; // 2 x 4 KB per (128-row block, stage)
// Byte offset of the scale of element j (along the reduction) of block row r
// in replica 0; the same byte is also stored at +1024, +2048 and +3072.
__host__ __device__ constexpr long bs_sfa_offset(long r, long j, long ks_count) {
  return ((r / 128) * ks_count + j / kTcBsStage) * kBsSfaRecBytes +
         ((j % kTcBsStage) / 128) * 4096 + ((r % 32) / 8) * 256 + (((j % kTcBsStage) / 64) & 1) * 128 +
         (r % 8) * 16 + ((r % 128) / 32) * 4 + (j % 64) / 16;
}
struct TcArgs {
  int M, K, N, T, El, R, C;
  int wfmt, act, gate;
  float alpha, beta, limit;
  const float *a_scalar, *a_rowscale, *a_groupscale, *a_expertscale;
  int a_groups;
  const void *w_codes, *w_scales;
  const float *w_global;
  const void *w_bias;
  int bias_f32;
  const int32_t *sorted_ids, *expert_ids, *num_post_pad;
  int S;
  void *out;
  int out_mode;          // W13 output: TC_OUT_BF16 / _F32 (staging) / _F16 /
                         // _MX4_F16 / _MX8_F16 (OCP MX quantise-dequantise into f16)
  const float *out_global;  // block-scaled NVFP4 W13: the stage-2 global per expert [El]
  float *out_scales;        // FP8-block W13: the intermediate's 1 x 128 scales [cap, ceil(N/128)]
  float *acc;
  const float *topk_weights;
  int *err;
  int w_stage1;          // router weight on the stage-1 output (W13 multiplies, W2 not)
  const void *w_packed;  // FP4 formats: load-time packed records
  const void *a_sf;      // block-scaled NVFP4: scale-factor records of the A rows
  void *out_sf;          // block-scaled NVFP4 W13: scale-factor records of the intermediate
  int ntiles;            // set by the launcher
  int rec_bytes;         // set by the launcher
  int mgroup;            // raster: m-blocks that walk the n-tiles together (launcher)
  long nblocks;          // m-blocks in the grid (launcher)
  // weight-streaming tcgen05 kernels (moe_tcs.cu): the sort's per-expert
  // sorted-row offsets and slot counts [El], the active-expert list and its length
  const int32_t *offsets, *counts, *active, *n_active;
  int rec_tiles;         // moe_tcd.cu: 128-row record tiles per expert (launcher)
};
struct GatherArgs {
  const int32_t *sorted_ids, *num_post_pad;
  int S, T, K, afmt;
  const void *codes, *scales;
  void *out;             // bf16 / f16 rows, or e4m3 codes for fp8 activations
  float *rowscale, *groupscale;
  int to_f16;            // f16 rows (FP4 weights: the f16 tensor-core kind)
  // when set: the per-token f16 copy of x made by the sort's conversion CTAs
  // (scaled by 2^a per token, x_inv = 2^-a), copied row by row
  const void *x16 = nullptr;
  const float *x_inv = nullptr;
  // block-scaled NVFP4 (afmt A_NVFP4_DYN): out receives the codes [cap, K/2]
  // and sf_out the scale-factor records of the sorted rows
  void *sf_out = nullptr;
  // when set (NVFP4): codes and scales are quantised here from the bf16 token
  // rows x_nvfp4 [M, K] with the global scale *nv_global (no quantiser pass)
  const uint16_t *x_nvfp4 = nullptr;
  const float *nv_global = nullptr;
};
cudaError_t launch_rescale_rows(const float *src, long cap, int N, const int32_t *sorted_ids,
                                const int32_t *ntp, int S, void *dst, float *rowscale,
                                cudaStream_t st);
cudaError_t launch_scale_range(const uint8_t *s, long n, int *mn_mx, cudaStream_t st);
struct TcPackArgs {
  const unsigned char *codes, *scales;
  unsigned char *out;
  long total;
  int rec_bytes, kstages, ntiles, w13, nvfp4, gate, N, R, C;
};
int tc_ntiles(int w13, int N, int K);
size_t tc_packed_bytes(int w13, int nvfp4, int N, int K, int El);
cudaError_t launch_pack_tc_fp4(const TcPackArgs &p, cudaStream_t st);
cudaError_t launch_gather_rows(const GatherArgs &g, long cap_rows, cudaStream_t st);
cudaError_t launch_tc_gemm(const TcArgs &a, const void *a_sorted, long cap_rows, int w13,
                           cudaStream_t st);
// Weight-streaming tcgen05 grouped GEMMs (moe_tcs.cu), MXFP4 w4a16 with the
// bounded SwiGLU-OAI: the weights (TC-packed records) are the MMA's M operand,
// up to 256 of an expert's sorted f16 rows (rows_f16 [cap_rows, C]) its N
// operand.  W13 writes the f16 intermediate [cap_rows, N] (a.out); W2 adds
// the router-weighted rows into a.acc.  Needs a.offsets / counts / active /
// n_active from the sort and C % 64 == 0.
// tcgen05 grouped GEMMs of MXFP4 w4a16 prefill batches whose experts hold
// more than one 128-slot block (moe_tcd.cu): each 256-row weight stage is
// decoded once for a pair of blocks.  rows_f16 [cap_rows, C]; needs the
// sort's per-expert tables (128-row blocks) and the TC-packed records.
bool tcd_supported(int El);
cudaError_t launch_tcd_gemm(const TcArgs &a, const void *rows_f16, long cap_rows, int w13,
                            int sm_count, cudaStream_t st);
int tcs_ntiles(int w13, int N, int K);
cudaError_t launch_tcs_gemm(const TcArgs &a, const void *rows_f16, long cap_rows, int w13,
                            int sm_count, cudaStream_t st);
// Persistent block-scaled NVFP4 grouped GEMMs (moe_bs.cu): A = packed e2m1
// codes [cap, C/2] + scale-factor records (a.a_sf); B = the MOE_LAYOUT_TC
// records of NVFP4 weights (a.w_packed).  W13 writes the NVFP4 intermediate
// (codes into a.out [cap, N/2], scale factors into a.out_sf); W2 adds the
// weighted outputs into a.acc.  grid = min(tiles, sm_count), one CTA per SM.
int bs_ntiles(int w13, int N, int K);
size_t bs_packed_bytes(int w13, int N, int K, int El);
cudaError_t launch_pack_bs(const TcPackArgs &p, cudaStream_t st);
cudaError_t launch_bs_gemm(const TcArgs &a, const void *a_codes, long cap_rows, int w13,
                           int sm_count, cudaStream_t st);
// Persistent FP8-block grouped GEMMs (moe_fp8.cu): A = e4m3 codes [cap, C]
// with 1 x 128 scales (a.a_groupscale, a.a_groups per row), B = the canonical
// e4m3 weights with 128 x 128 block scales.  W13 writes the intermediate as
// e4m3 codes (a.out [cap, N]) + 1 x 128 scales (a.out_scales); W2 adds the
// weighted outputs into a.acc.  grid = min(tiles, sm_count).
cudaError_t launch_fp8b_gemm(const TcArgs &a, const void *a_codes, long cap_rows, int w13,
                             int sm_count, cudaStream_t st);

// Tensor-core rate probe (moe_probe.cu): sm_count CTAs, each issuing `iters`
// MMAs of 128 x n (kind 0: f16, 1: e4m3, 2: e2m1 + ue4m3 block scales).
cudaError_t launch_mma_probe(int kind, int n, long iters, int sm_count, int *err,
                             cudaStream_t st);

cudaError_t launch_route(const void *logits, int bf16_in, int M, int E, int topk, int scoring,
                         int renorm, int G, int TG, const float *bias, float scale, int32_t *ids,
                         float *weights, cudaStream_t st);
cudaError_t launch_finalize(const float *acc, long n, void *out_bf16, cudaStream_t stream,
                            bool dependent = false);
cudaError_t launch_zero(float *buf, long n, cudaStream_t stream);

}  // namespace moe
