/*
 * moe_experts.h -- C ABI of the GB300 (sm_103a) fused Mixture-of-Experts
 * expert computation: route -> gate/up GEMM -> activation -> down GEMM ->
 * top-k weighted reduce, with bf16, FP8 (per-tensor, per-channel, 128x128
 * block), MXFP4 and NVFP4 weights.
 *
 * The operation is the fused-experts contract of the page
 * "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe":
 * rocm_aiter_fused_experts(hidden_states, w1, w2, topk_weights, topk_ids,
 * activation, expert_mask, quant_config, ...) as called from
 * AiterExperts.apply, which writes the (M, K) result into a caller-owned
 * output.  Weight layouts follow GptOssMxfp4MoEMethod.create_weights on
 * "vLLM/vllm/model_executor/layers/quantization/mxfp4.py" and
 * QuarkNvfp4MoEMethod.create_weights on
 * "vllm.model_executor.layers.quantization.quark.quark_moe".
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or synchronises.  Work is enqueued on `stream`
 *    (a cudaStream_t passed as void*; NULL = the legacy default stream).
 *  - Arguments are validated on the host before anything is launched; a
 *    failed check returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE and enqueues nothing.  A launch failure returns
 *    MOE_ERR_CUDA.  Device-side values (ids, counts) are not validated on the
 *    host: an expert id outside [0, E) or mapped outside [0, E_l) is treated
 *    as a dropped slot, exactly like an expert-map entry of -1.
 *  - Layouts are row-major with the reduction dimension contiguous.
 *    Packed e2m1 ("fp4"): two elements per byte, element 2i in the low nibble.
 *  - Returned status codes are plain ints (moe_status).
 */
#ifndef MOE_EXPERTS_H_
#define MOE_EXPERTS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Raised whenever an entry point is added or a struct or signature changes
 * (10: moe_align_scratch_bytes and moe_align_block_size_scratch). */
#define MOE_ABI_VERSION 10

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad enum value          */
  MOE_ERR_UNSUPPORTED = 2, /* valid but unsupported combination               */
  MOE_ERR_WORKSPACE = 3,   /* workspace smaller than moe_workspace_size()     */
  MOE_ERR_CUDA = 4,        /* a CUDA launch / runtime call failed             */
  MOE_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (device word) */
} moe_status;

/* Weight formats: the AITER leaf classes' quant methods on the rocm_aiter_moe
 * page (QuantMethod NO / PER_TENSOR / PER_TOKEN / BLOCK_128x128 / BLOCK_1X32)
 * plus QuarkNvfp4MoEMethod. */
typedef enum {
  MOE_W_BF16 = 0,         /* bf16 [E_l,R,C]                                     */
  MOE_W_FP8_TENSOR = 1,   /* e4m3 [E_l,R,C], scales f32 [E_l]                   */
  MOE_W_FP8_CHANNEL = 2,  /* e4m3 [E_l,R,C], scales f32 [E_l,R]                 */
  MOE_W_FP8_BLOCK128 = 3, /* e4m3 [E_l,R,C], scales f32 [E_l,ceil(R/128),ceil(C/128)] */
  MOE_W_MXFP4 = 4,        /* e2m1 u8 [E_l,R,C/2], e8m0 u8 [E_l,R,C/32]          */
  MOE_W_NVFP4 = 5         /* e2m1 u8 [E_l,R,C/2], e4m3 u8 [E_l,R,C/16], global f32 [E_l] */
} moe_wfmt;

/* Activation (stage-1 input) formats.  Supported (weight, activation) pairs,
 * as the leaves' _supports_quant_scheme lists them:
 *   BF16 + BF16; FP8_TENSOR + FP8_TENSOR_STATIC | FP8_TENSOR_DYN;
 *   FP8_CHANNEL + FP8_TOKEN_DYN; FP8_BLOCK128 + FP8_GROUP128_DYN;
 *   MXFP4 + BF16 (w4a16), MXFP4 + MXFP4_DYN (w4a4), MXFP4 + MXFP8_DYN (w4a8)
 *   (AiterMxfp4Experts takes MXFP4 weights with bf16 or dynamically
 *   MXFP4-quantised activations; MXFP4 x MXFP8 as named by the mxfp4.py
 *   backends);
 *   NVFP4 + NVFP4_DYN.
 * The intermediate (stage-2 input) uses the same scheme: per-tensor static
 * (a2_scale) or dynamic, per-token dynamic, 1x128 dynamic, NVFP4 x16 dynamic
 * with a per-expert global, MX; bf16 for BF16 weights and MXFP4 w4a16. */
typedef enum {
  MOE_A_BF16 = 0,
  MOE_A_FP8_TENSOR_STATIC = 1, /* scale f32 [1] given                          */
  MOE_A_FP8_TENSOR_DYN = 2,    /* scale f32 [1] = amax/448 over the tensor     */
  MOE_A_FP8_TOKEN_DYN = 3,     /* scales f32 [rows]                            */
  MOE_A_FP8_GROUP128_DYN = 4,  /* scales f32 [rows, ceil(cols/128)]            */
  MOE_A_NVFP4_DYN = 5,         /* codes u8 [rows, cols/2], scales e4m3 [rows, cols/16] */
  /* OCP MX, 32-element blocks with an e8m0 scale (cols % 32 == 0): X =
   * floor(log2(amax)) - emax (2 for e2m1, 8 for e4m3) clamped to [-127, 127],
   * scale code X + 127, element = RNE-saturating e2m1 / e4m3 of x / 2^X;
   * amax == 0 gives scale code 0 and zero codes.  The stage-2 intermediate of
   * these pairs uses the same format. */
  MOE_A_MXFP4_DYN = 6,         /* codes u8 [rows, cols/2], scales e8m0 [rows, cols/32] */
  MOE_A_MXFP8_DYN = 7          /* codes e4m3 [rows, cols],  scales e8m0 [rows, cols/32] */
} moe_afmt;

/* Activations of the gated MLP (_resolve_aiter_activation; SITU is not
 * supported: its formula is not given). */
typedef enum { MOE_ACT_SILU = 0, MOE_ACT_GELU = 1, MOE_ACT_SWIGLU_OAI = 2 } moe_act;

/* Row order of w13 (gate-mode selection in rocm_aiter_fused_experts):
 * SEPARATED = [gate rows 0..N-1 ; up rows 0..N-1];
 * INTERLEAVED = gate_j at row 2j, up_j at row 2j+1. */
typedef enum { MOE_GATE_SEPARATED = 0, MOE_GATE_INTERLEAVED = 1 } moe_gate_layout;

/* One weight tensor set (w13 with R=2N, C=K; or w2 with R=K, C=N).  Device
 * pointers, caller-owned, layouts as listed under moe_wfmt. */
typedef struct {
  const void *codes;
  const void *scales;        /* NULL for MOE_W_BF16                         */
  const float *global_scale; /* MOE_W_NVFP4 only: f32 [E_l] (dequant multiplies) */
  const void *bias;          /* optional [E_l,R]: bf16, or f32 if bias_is_f32 */
  int bias_is_f32;
  const void *packed;        /* optional: the same weights repacked by moe_prepare_weights
                                (MOE_LAYOUT_STREAM, MXFP4); enables the weight-streaming
                                decode kernels */
  const void *packed_tc;     /* optional: repacked with MOE_LAYOUT_TC (MXFP4 / NVFP4);
                                enables the tcgen05 kernels for those formats */
} moe_weight_t;

typedef struct {
  int M;                  /* tokens                                              */
  int K;                  /* hidden size                                         */
  int N;                  /* intermediate size (per partition)                   */
  int topk;               /* slots per token, shared-expert slots included       */
  int num_experts;        /* E: global expert ids in topk_ids are in [0, E)      */
  int num_local_experts;  /* E_l: leading dimension of the weight tensors        */
  int wfmt, afmt, act, gate; /* moe_wfmt, moe_afmt, moe_act, moe_gate_layout     */
  float swiglu_alpha;     /* SwiGLU-OAI: z = (clamp(u)+beta) * g' * sigmoid(alpha*g') */
  float swiglu_beta;
  float swiglu_limit;     /* g' = min(g, limit), u clamped to [-limit, limit]; 0 = no clamp */
  const float *a1_scale;  /* device: FP8_TENSOR_STATIC stage-1 scale [1]; NVFP4 stage-1 global [1] */
  const float *a2_scale;  /* device: FP8_TENSOR_STATIC stage-2 scale [1]; NVFP4 stage-2 global [E_l] */
  /* apply_router_weight_on_input (doweight_stage1 of rocm_aiter_fused_experts;
   * the tkw1 path of AiterFp8ChannelExperts on the rocm_aiter_moe page moves
   * the router-weight multiply from the second GEMM's output to the first's):
   * 1 = the router weight multiplies the stage-1
   * output, z' = w * act(g, u), before the stage-2 quantiser, and the stage-2
   * reduce is unweighted: out[t] = sum_k (W2 z'_k + b2).  Requires topk == 1
   * (_assert_topk1_for_router_weight_on_input); honoured by moe_fused_experts
   * (and _noalloc); the step entry points return MOE_ERR_UNSUPPORTED with it. */
  int router_weight_on_input;
  /* num_local_tokens of rocm_aiter_fused_experts (AiterExperts.apply passes
   * expert_tokens_meta.expert_num_tokens there): device int32 [1] holding the
   * number n of valid tokens; only rows t < n of hidden_states / topk_ids take
   * part, rows t >= n of the output are written as zeros (a padded dispatch
   * buffer whose fill level is known on the device only; CUDA-graph friendly).
   * NULL = all M tokens.  Read by moe_fused_experts (and _noalloc); not with
   * MOE_A_FP8_TENSOR_DYN (its batch scale would cover the padding rows). */
  const int32_t *num_local_tokens;
  /* Kernel family of this problem (moe_path; a tuning and testing aid, read
   * per call, no process-wide state).  MOE_PATH_AUTO (0, the value of a
   * zero-initialised struct): for MXFP4 w4a16 with the bounded SwiGLU-OAI
   * (K, N multiples of 64, MOE_LAYOUT_STREAM and MOE_LAYOUT_TC weights) the
   * tcgen05 weight-streaming kernels from 64 (exclusive) to 128 slots per
   * local expert on average; otherwise the
   * mma.sync weight-streaming kernels when their conditions hold (see
   * moe_prepare_weights), else the tcgen05 kernels when M*topk >= 2048 (FP4
   * formats need MOE_LAYOUT_TC packed weights), else the generic mma.sync
   * kernels.  GENERIC, STREAM, TC and TC_STREAM force a family where it
   * applies (else the automatic choice runs).  moe_workspace_size depends
   * on it. */
  int path;
} moe_problem_t;

enum { MOE_PATH_AUTO = 0, MOE_PATH_GENERIC = 1, MOE_PATH_STREAM = 2, MOE_PATH_TC = 3,
       MOE_PATH_TC_STREAM = 4 };

/* Library / ABI identification. */
int moe_abi_version(void);
const char *moe_status_str(int status);

/* Workspace bytes moe_fused_experts needs for this problem (like the
 * workspace_shapes query of AiterExperts).  0 for an invalid problem. */
size_t moe_workspace_size(const moe_problem_t *p);

/* Entries of sorted_ids for (M, topk, E_l, block_m): every slot plus up to
 * block_m-1 padding entries per expert that has a slot, rounded up to whole
 * blocks.  expert_ids needs moe_align_capacity()/block_m entries. */
long moe_align_capacity(int M, int topk, int num_local_experts, int block_m);

/* Load-time repack of FP4 weights (the role of
 * convert_weight_to_mxfp4_moe_kernel_format on the mxfp4.py page).
 * which = 0: w13 ([E_l, 2N, K/2] codes + scales, gate/up rows per p->gate);
 * which = 1: w2.  The packed buffer (moe_packed_weight_bytes bytes, 16-B
 * aligned, caller-owned) holds the same codes and scales reordered into
 * per-tile records.  Layouts:
 *   MOE_LAYOUT_STREAM  MXFP4 with K, N multiples of 64 -> moe_weight_t.packed:
 *     the weight-streaming decode kernels, used by moe_fused_experts when both
 *     w13 and w2 carry it, the activations are bf16 (or OCP MX without the
 *     router weight on the stage-1 output), the activation is SwiGLU-OAI with
 *     0 < limit <= 64 and |beta| <= 64, and M*topk <= 64*E_l;
 *   MOE_LAYOUT_TC      MXFP4 or NVFP4 -> moe_weight_t.packed_tc: the tcgen05
 *     kernels of those formats (prefill-sized batches).  They decode into
 *     f16, so for MXFP4 every e8m0 exponent must lie in [-21, 13] (checked
 *     here; this check synchronises `stream`), else MOE_ERR_UNSUPPORTED.
 * Unsupported combinations return 0 bytes / MOE_ERR_UNSUPPORTED. */
enum { MOE_LAYOUT_STREAM = 0, MOE_LAYOUT_TC = 1 };
size_t moe_packed_weight_bytes(const moe_problem_t *p, int which, int layout);
int moe_prepare_weights(const moe_problem_t *p, int which, int layout, const moe_weight_t *w,
                        void *packed, void *stream);

/* Expert sort / block padding (the dispatch step named by
 * moe_sorting_dispatch_policy in AiterExperts.apply; the rule is this
 * library's): per local expert in ascending id, the flat slot ids t*topk+k in
 * ascending order, padded with the sentinel S = M*topk to a multiple of
 * block_m; empty experts get no block.  Tails: sorted_ids = S, expert_ids = -1.
 *   topk_ids     int32 [M, topk] (global ids)
 *   expert_map   int32 [E] global->local, -1 = dropped; NULL = identity
 *   sorted_ids   int32 [moe_align_capacity()]
 *   expert_ids   int32 [moe_align_capacity()/block_m]
 *   num_post_pad int32 [1]  total padded length
 *   expert_counts int32 [E_l] live slots per local expert (may be NULL)
 * block_m must be in [1, 1024]; E_l <= 1024. */
int moe_align_block_size(const int32_t *topk_ids, int M, int topk, const int32_t *expert_map,
                         int num_experts, int num_local_experts, int block_m,
                         int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_post_pad,
                         int32_t *expert_counts, void *stream);

/* The same sort with caller scratch: batches of 8192 slots or more then run
 * on several CTAs (the outputs are identical, bit for bit).
 *   scratch        device memory, 16-byte aligned, caller-owned, of at least
 *                  moe_align_scratch_bytes(M, topk, E_l) bytes (contents need
 *                  no initialisation and are overwritten); NULL or smaller:
 *                  the one-CTA sort of moe_align_block_size
 * moe_align_scratch_bytes returns 0 for batches that always take one CTA (and
 * for invalid arguments).  Errors as moe_align_block_size, plus
 * MOE_ERR_INVALID_ARG for a misaligned scratch pointer. */
size_t moe_align_scratch_bytes(int M, int topk, int num_local_experts);
int moe_align_block_size_scratch(const int32_t *topk_ids, int M, int topk,
                                 const int32_t *expert_map, int num_experts, int num_local_experts,
                                 int block_m, int32_t *sorted_ids, int32_t *expert_ids,
                                 int32_t *num_post_pad, int32_t *expert_counts, void *scratch,
                                 size_t scratch_bytes, void *stream);

/* Router: logits -> top-k expert ids and weights, the routing that the
 * apply_monolithic path hands to the expert kernel together with the logits
 * (GptOssMxfp4MoEMethod.apply_monolithic and Mxfp4MoEMethod.apply_monolithic
 * on "vLLM/vllm/model_executor/layers/quantization/mxfp4.py" and
 * QuarkOCP_MX_MoEMethod.apply_monolithic on the quark_moe page pass
 * router_logits, num_expert_group, topk_group, e_score_correction_bias and
 * routed_scaling_factor; the renormalised softmax top-k is the routing of the
 * GPT-OSS layers there).  The pages name the arguments but print no algorithm;
 * the rule implemented is the plain reading, per token t:
 *   s_e = softmax(logits[t])_e        (scoring MOE_SCORE_SOFTMAX)
 *       = 1 / (1 + exp(-logits[t,e])) (scoring MOE_SCORE_SIGMOID)
 *   keys: c_e = s_e + bias_e with a bias (e_score_correction_bias), else the
 *         logits themselves (same order as s, no rounding in the choice)
 *   groups (num_groups > 1; E % num_groups == 0, contiguous groups): a group
 *         scores the sum of its two largest keys with a bias, its largest key
 *         without; only the topk_group best groups (ties to the lower group)
 *         stay eligible
 *   ids:  the topk eligible experts with the largest keys, in descending key
 *         order, ties to the lower id
 *   w_j = s_{id_j} (never the bias), divided by sum_j s_{id_j} when renorm,
 *         times routed_scaling_factor.
 *   logits  f32 or bf16 (logits_bf16 != 0) [M, E];  bias f32 [E] or NULL
 *   topk_ids int32 [M, topk];  topk_weights f32 [M, topk]
 * Limits: E <= 1024, topk <= 32, num_groups <= 32 (0 or 1 = no groups),
 * topk <= topk_group * E / num_groups.  Computation in fp32. */
enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
int moe_route_topk(const void *logits, int logits_bf16, int M, int num_experts, int topk,
                   int scoring, int renorm, int num_groups, int topk_group, const float *bias,
                   float routed_scaling_factor, int32_t *topk_ids, float *topk_weights,
                   void *stream);

/* Stage-1 activation quantiser (AiterFp8TensorExperts, AiterFp8ChannelExperts,
 * AiterFp8BlockExperts, QuarkNvfp4MoEMethod).  x is bf16 [rows, cols].
 *   fp8: scale = fl32(max(amax, 1e-12) / 448); code = e4m3_rne_sat(fl32(x / scale)).
 *   NVFP4 (cols % 16 == 0): per 16 elements s = e4m3_rne_sat(fl32(fl32(amax/6)/g)),
 *     code = e2m1_rne_sat(fl32(x / fl32(e4m3(s) * g))); s == 0 gives zero codes.
 *   scale_in: device f32 [1] -- the static fp8 scale, or the NVFP4 global g.
 *   codes: u8 [rows, cols] (fp8) or [rows, cols/2] (NVFP4); scales as under moe_afmt.
 * x, codes and scales must be 16-byte aligned.  MOE_A_BF16 is rejected
 * (nothing to quantise). */
int moe_quant_act(const void *x_bf16, int rows, int cols, int afmt, const float *scale_in,
                  void *codes, void *scales, void *stream);

/* Stage-1 grouped GEMM + activation (+ stage-2 requantisation), the first of
 * the two stages rocm_aiter_fused_experts runs (the gate/up GEMM with the
 * activation and the next stage's quantisation).
 * For every sorted row r < *num_post_pad with slot s = sorted_ids[r] < S,
 * token t = s / topk, local expert e = expert_ids[r / block_m]:
 *   h = dequant(A[t]) . dequant(W13[e])^T + b13[e];  z_j = act(gate_j, up_j)
 * and writes row r of the intermediate (padding rows as zeros).
 *   a_codes / a_scales: x bf16 [M, K] for bf16 activations, else the output of
 *   moe_quant_act.  sorted_ids / expert_ids / num_post_pad: the output of
 *   moe_align_block_size with the same block_m.
 *   block_m = 64: the generic mma.sync kernels (every supported pair).
 *   block_m = 128: the tcgen05 kernels (bf16, fp8 and NVFP4 activations; FP4
 *     weights must carry their MOE_LAYOUT_TC records in packed_tc; OCP MX
 *     activations return MOE_ERR_UNSUPPORTED).
 * The intermediate (inter / inter_scales, sizes from moe_intermediate_size):
 *   bf16 weights:  bf16 [cap, N];
 *   FP8 weights:   e4m3 codes [cap, N] + the stage-2 scales (f32 [1] / [cap] /
 *                  [cap, ceil(N/128)] for tensor / token / 1x128 groups);
 *   MXFP4 w4a16:   block_m 64: bf16 [cap, N];  block_m 128: f16 [cap, N],
 *                  multiplied per row by inter_scales f32 [cap] unless the
 *                  activation is SwiGLU-OAI with 0 < limit <= 64 and
 *                  |beta| <= 64 (then the f16 values themselves, no scales);
 *   MXFP4 w4a4 / w4a8 (block_m 64): codes + e8m0 scales [cap, N/32];
 *   NVFP4:         e2m1 codes [cap, N/2] (element 2i in the low nibble) +
 *                  block_m 64: e4m3 scales [cap, N/16];  block_m 128: the
 *                  block-scaled records: for each 128-row block and each
 *                  256-column stage 8192 bytes, in which the scale of row r,
 *                  column j sits at byte (((j % 256) / 128) * 4096
 *                  + ((r % 32) / 8) * 256 + (((j % 256) / 64) % 2) * 128
 *                  + (r % 8) * 16 + ((r % 128) / 32) * 4 + (j % 64) / 16) and
 *                  again at +1024, +2048 and +3072 of its record (record
 *                  index (r / 128) * ceil(N/256) + j / 256).
 *   workspace: device scratch of moe_w13_workspace_size() bytes (block_m 64:
 *   fp32 staging of a requantised intermediate; block_m 128: the gathered
 *   rows); may be NULL when that size is 0. */
size_t moe_w13_workspace_size(const moe_problem_t *p, int block_m);
int moe_intermediate_size(const moe_problem_t *p, int block_m, size_t *inter_bytes,
                          size_t *scales_bytes);
int moe_grouped_gemm_w13_act(const moe_problem_t *p, const void *a_codes, const void *a_scales,
                             const moe_weight_t *w13, const int32_t *sorted_ids,
                             const int32_t *expert_ids, const int32_t *num_post_pad, int block_m,
                             void *inter, void *inter_scales, void *workspace, size_t ws_bytes,
                             void *stream);

/* Stage-2 grouped GEMM + top-k weighted reduce (TopKWeightAndReduceNoOP: the
 * reduce happens inside the experts computation).  For every live sorted row:
 *   y = dequant(inter[r]) . dequant(W2[e])^T + b2[e];  acc[t] += topk_weights[s] * y
 * then out_bf16 = bf16_rne(acc).  inter / inter_scales as the stage-1 call
 * with the same block_m wrote them (block_m 64: generic kernels; 128: tcgen05
 * kernels, same conditions).  acc_f32 [M, K] is caller scratch; it is zeroed
 * by this call before the reduce.  Tokens with no live slot give 0. */
int moe_grouped_gemm_w2_reduce(const moe_problem_t *p, const void *inter, const void *inter_scales,
                               const moe_weight_t *w2, const float *topk_weights,
                               const int32_t *sorted_ids, const int32_t *expert_ids,
                               const int32_t *num_post_pad, int block_m, float *acc_f32,
                               void *out_bf16, void *stream);

/* The whole fused-experts call (rocm_aiter_fused_experts): sort/pad,
 * stage-1 quantisation, w13 GEMM + activation, w2 GEMM + reduce, bf16 output.
 *   hidden_bf16  bf16 [M, K];  topk_ids int32 [M, topk];  topk_weights f32 [M, topk]
 *   expert_map   int32 [E] or NULL;  out_bf16 bf16 [M, K] (overwritten)
 *   workspace    device scratch of at least moe_workspace_size(p) bytes, 256-B aligned. */
int moe_fused_experts(const moe_problem_t *p, const void *hidden_bf16, const moe_weight_t *w13,
                      const moe_weight_t *w2, const int32_t *topk_ids, const float *topk_weights,
                      const int32_t *expert_map, void *workspace, size_t ws_bytes, void *out_bf16,
                      void *stream);

/* The batched expert-parallel input format: the experts' rows arrive already
 * grouped per local expert, each with a device-side count of valid rows, as
 * AiterExperts.apply hands rocm_aiter_fused_experts the per-expert token
 * counts of expert_tokens_meta (expert_num_tokens) under num_local_tokens
 * (page "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe").
 * There is no routing and no sort: the padded blocks follow from a prefix sum
 * of the counts on the device.
 *   hidden_bf16        bf16 [E_l, max_tokens, K]; rows [e, 0:count[e]) are
 *                      expert e's tokens, the rest padding (never read)
 *   expert_num_tokens  device int32 [E_l]: count[e], clamped to [0, max_tokens]
 *   out_bf16           bf16 [E_l, max_tokens, K] (overwritten):
 *                      out[e, i] = W2_e act(W13_e QDQ(x[e, i]) + b13_e) + b2_e
 *                      for i < count[e], 0 for the padding rows
 * No top-k weight is applied (the combine that follows the experts weighs and
 * sums a token's rows).  p gives K, N, num_local_experts, the formats, the
 * activation and the scales; p->M, topk and num_experts are not read.  Not
 * supported: router_weight_on_input, num_local_tokens, MOE_A_FP8_TENSOR_DYN.
 * The tcgen05 kernels run when E_l * max_tokens >= 2048 (p->path as for
 * moe_fused_experts, FP4 weights with their MOE_LAYOUT_TC records), else the
 * generic ones.  workspace: moe_batched_workspace_size bytes, 256-B aligned. */
size_t moe_batched_workspace_size(const moe_problem_t *p, int max_tokens);
int moe_batched_experts(const moe_problem_t *p, int max_tokens, const void *hidden_bf16,
                        const int32_t *expert_num_tokens, const moe_weight_t *w13,
                        const moe_weight_t *w2, void *workspace, size_t ws_bytes, void *out_bf16,
                        void *stream);

/* No-allocation variant of moe_fused_experts (the pages have no counterpart:
 * it exists for callers that cannot allocate device memory -- hosts that own
 * every allocation and give out no scratch buffer, runtimes that must not call
 * cudaMalloc on the call path).  Same inputs and output as moe_fused_experts,
 * no workspace: the scratch is a file-scope device array of
 * moe_noalloc_scratch_bytes() bytes (32 MiB) that each GPU loading the library
 * holds until exit.  Problems needing more (moe_workspace_size) return
 * MOE_ERR_WORKSPACE.  The first call on a device looks up the array's address
 * (cudaGetSymbolAddress) and should come before any stream capture; that
 * address is kept for the life of the process, so a process using this entry
 * point must not call cudaDeviceReset (the array would be loaded again
 * elsewhere).  All calls on a device share the array: calls that overlap on
 * the GPU race, so order them on one stream.  Allocates nothing. */
size_t moe_noalloc_scratch_bytes(void);
int moe_fused_experts_noalloc(const moe_problem_t *p, const void *hidden_bf16,
                              const moe_weight_t *w13, const moe_weight_t *w2,
                              const int32_t *topk_ids, const float *topk_weights,
                              const int32_t *expert_map, void *out_bf16, void *stream);

/* Per-stage timing of moe_fused_experts (a profiling aid).  While enabled,
 * every moe_fused_experts call records a CUDA event pair around each of its
 * kernel launches on the call's stream, waits for the last event before
 * returning (the call becomes synchronous), and adds each launch's elapsed
 * time to the accumulator of its stage; timed calls are serialised by one
 * process-wide lock.  While disabled (the default) calls take no lock.  moe_stage_timing(1) enables and
 * resets, moe_stage_timing(0) disables; moe_stage_times copies the
 * accumulated milliseconds [MOE_NUM_STAGES] and the number of timed calls.
 * Not for use inside stream capture. */
enum { MOE_STAGE_ALIGN = 0, MOE_STAGE_QUANT = 1, MOE_STAGE_W13 = 2, MOE_STAGE_REQUANT = 3,
       MOE_STAGE_W2 = 4, MOE_STAGE_FINALIZE = 5, MOE_NUM_STAGES = 6 };
int moe_stage_timing(int enable);
int moe_stage_times(double *ms_out, int *calls_out);

/* Device error word: first error recorded by a bounded device wait or a
 * device-side check since the last reset (0 = none).  Reads synchronously
 * (call after synchronising the streams that ran the kernels). */
int moe_get_device_error(int *err_out);
int moe_reset_device_error(void);

/* Self-test of the failure detection (no part of the computation): enqueues
 * on `stream` one CTA that waits on a shared-memory barrier nothing completes,
 * with the same bounded wait every pipeline of this library uses, for
 * limit_cycles SM clock cycles (1 <= limit_cycles < 2^40).  When the limit runs
 * out the kernel records MOE_ERR_TIMEOUT in the device error word and returns;
 * the context stays usable.  Returns MOE_ERR_INVALID_ARG (nothing launched)
 * for a limit out of range. */
int moe_selftest_bounded_wait(long long limit_cycles, void *stream);

/* Tensor-core rate probe (a measurement aid with no counterpart on the pages:
 * it gives the benchmark the dense rate of each tcgen05 operand kind on this
 * GPU).  Enqueues on `stream` one CTA per SM; each issues `iters` MMAs of
 * 128 x n x k into Tensor Memory with its operands already in shared memory
 * (no loads, no epilogue) and waits, bounded, for them to finish.
 *   kind 0: f16 x f16 (k = 16);  kind 1: e4m3 x e4m3 (k = 32);
 *   kind 2: e2m1 x e2m1 with ue4m3 scales per 16 (kind::mxf4nvf4, k = 64)
 *   n: 128 or 256;  1 <= iters <= 2^31
 * The work is sm_count * iters * 2 * 128 * n * k floating-point operations;
 * *sm_count_out (may be NULL) receives the SM count used.  The caller times
 * the launch (CUDA events on `stream`).  MOE_ERR_INVALID_ARG for arguments
 * out of range (nothing launched). */
int moe_mma_probe(int kind, int n, long long iters, int *sm_count_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_EXPERTS_H_ */
