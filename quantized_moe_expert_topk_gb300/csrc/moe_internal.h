// moe_internal.h -- host-side declarations shared by the library's translation
// units (kernel launchers and their argument blocks).  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Tile height (sorted rows per block) of the mma.sync grouped GEMMs; the
// expert sort pads every expert to a multiple of it.
constexpr int kGenericBlockM = 64;

cudaError_t launch_align(const int32_t *topk_ids, int M, int T, const int32_t *expert_map, int E,
                         int El, int BM, int32_t *sorted_ids, int32_t *expert_ids,
                         int32_t *num_post_pad, int32_t *counts, long cap, float *zero_buf,
                         long zero_n, cudaStream_t stream);

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
};
cudaError_t launch_gemm_w13(const GemmArgs &a, long cap_rows, cudaStream_t stream);
cudaError_t launch_gemm_w2(const GemmArgs &a, long cap_rows, cudaStream_t stream);
cudaError_t launch_finalize(const float *acc, long n, void *out_bf16, cudaStream_t stream);
cudaError_t launch_zero(float *buf, long n, cudaStream_t stream);

}  // namespace moe
