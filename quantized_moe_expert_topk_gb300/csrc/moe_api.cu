// moe_api.cu -- the C ABI (include/moe_experts.h): host-side validation,
// workspace layout and the launch sequence of the fused experts.
//
// Contract: rocm_aiter_fused_experts / AiterExperts.apply on the page
// "vllm.model_executor.layers.fused_moe.experts.rocm_aiter_moe" (output (M, K)
// written into a caller-owned buffer; workspaces sized by a query, like
// AiterExperts.workspace_shapes; unsupported combinations rejected, like the
// leaves' _supports_quant_scheme / _supports_activation checks).  Shape rules
// follow GptOssMxfp4MoEMethod._setup_kernel's assertions on
// "vLLM/vllm/model_executor/layers/quantization/mxfp4.py" (K and N multiples of
// the 32-element MXFP4 block) and QuarkNvfp4MoEMethod (group of 16).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/moe_experts.h"
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
__device__ int g_device_error_word = 0;
__device__ int g_scale_range[2];  // e8m0 code range found by moe_prepare_weights
}

namespace {

using namespace moe;

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Stage-2 (intermediate) format implied by the weight / activation formats.
int stage2_afmt(const moe_problem_t *p) {
  switch (p->wfmt) {
    case W_FP8_TENSOR: return p->afmt;
    case W_FP8_CHANNEL: return A_FP8_TOKEN_DYN;
    case W_FP8_BLOCK128: return A_FP8_GROUP128_DYN;
    case W_NVFP4: return A_NVFP4_DYN;
    case W_MXFP4:  // w4a4 / w4a8: the intermediate in the activation's MX format
      return (p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN) ? p->afmt : A_BF16;
    default: return A_BF16;
  }
}

// MXFP4 weights with OCP MX activations (w4a4 / w4a8) on the f16 kernels: the
// dequantised activations are exact in f16 after a per-token power of two, and
// with the bounded SwiGLU-OAI (no router weight folded in) the dequantised
// intermediate fits f16 as it is.
bool mx_act_f16(const moe_problem_t *p) {
  return p->wfmt == W_MXFP4 && (p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN) &&
         p->act == ACT_SWIGLU_OAI && p->swiglu_limit > 0.f && p->swiglu_limit <= 64.f &&
         fabsf(p->swiglu_beta) <= 64.f && !p->router_weight_on_input;
}

bool pair_supported(int wfmt, int afmt) {
  switch (wfmt) {
    case W_BF16: return afmt == A_BF16;
    case W_FP8_TENSOR: return afmt == A_FP8_TENSOR_STATIC || afmt == A_FP8_TENSOR_DYN;
    case W_FP8_CHANNEL: return afmt == A_FP8_TOKEN_DYN;
    case W_FP8_BLOCK128: return afmt == A_FP8_GROUP128_DYN;
    case W_MXFP4: return afmt == A_BF16 || afmt == A_MXFP4_DYN || afmt == A_MXFP8_DYN;
    case W_NVFP4: return afmt == A_NVFP4_DYN;
    default: return false;
  }
}

size_t codes_bytes(int afmt, long rows, long cols) {
  if (afmt == A_BF16) return 0;
  return (afmt == A_NVFP4_DYN || afmt == A_MXFP4_DYN) ? (size_t)rows * cols / 2
                                                     : (size_t)rows * cols;
}

size_t scales_bytes_of(int afmt, long rows, long cols) {
  switch (afmt) {
    case A_FP8_TENSOR_STATIC:
    case A_FP8_TENSOR_DYN: return 4;
    case A_FP8_TOKEN_DYN: return (size_t)rows * 4;
    case A_FP8_GROUP128_DYN: return (size_t)rows * ceil_div(cols, 128) * 4;
    case A_NVFP4_DYN: return (size_t)rows * (cols / 16);
    case A_MXFP4_DYN:
    case A_MXFP8_DYN: return (size_t)rows * (cols / 32);
    default: return 0;
  }
}

int validate_problem(const moe_problem_t *p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->M < 0 || p->K <= 0 || p->N <= 0 || p->topk < 1 || p->num_experts < 1 ||
      p->num_local_experts < 1)
    return MOE_ERR_INVALID_ARG;
  if (p->wfmt < W_BF16 || p->wfmt > W_NVFP4 || p->afmt < A_BF16 || p->afmt > A_MXFP8_DYN ||
      p->act < ACT_SILU || p->act > ACT_SWIGLU_OAI || p->gate < GATE_SEPARATED ||
      p->gate > GATE_INTERLEAVED || p->path < MOE_PATH_AUTO || p->path > MOE_PATH_TC_STREAM)
    return MOE_ERR_INVALID_ARG;
  if (!pair_supported(p->wfmt, p->afmt)) return MOE_ERR_UNSUPPORTED;
  if (p->num_local_experts > 1024) return MOE_ERR_UNSUPPORTED;
  // the router weight on the stage-1 output is defined for one slot per token
  if (p->router_weight_on_input && p->topk != 1) return MOE_ERR_UNSUPPORTED;
  // a per-tensor dynamic scale would span the padding rows beyond the valid tokens
  if (p->num_local_tokens && p->afmt == A_FP8_TENSOR_DYN) return MOE_ERR_UNSUPPORTED;
  // 32-element reduction tiles (and the 32-element MXFP4 / 16-element NVFP4 groups)
  if (p->K % 32 != 0 || p->N % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if ((long)p->M * p->topk > (1L << 30)) return MOE_ERR_UNSUPPORTED;
  const int s2 = stage2_afmt(p);
  if ((p->afmt == A_FP8_TENSOR_STATIC || p->afmt == A_NVFP4_DYN) && !p->a1_scale)
    return MOE_ERR_INVALID_ARG;
  if ((s2 == A_FP8_TENSOR_STATIC || s2 == A_NVFP4_DYN) && !p->a2_scale) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int validate_weight(const moe_problem_t *p, const moe_weight_t *w) {
  if (!w || !w->codes || !aligned16(w->codes)) return MOE_ERR_INVALID_ARG;
  if (p->wfmt != W_BF16 && !w->scales) return MOE_ERR_INVALID_ARG;
  if (p->wfmt == W_NVFP4 && !w->global_scale) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// ---- execution path (moe_problem_t.path)
constexpr long kTcMinSlots = 2048;  // slots from which the tcgen05 path is used

// The tcgen05 prefill path handles this problem (workspace sized for it).
bool tc_applies(const moe_problem_t *p) {
  if (p->path == MOE_PATH_TC) return true;
  return p->path == MOE_PATH_AUTO && (long)p->M * p->topk >= kTcMinSlots;
}

bool tc_mx_direct(const moe_problem_t *p);

// Band of slots per local expert (on average) in which MXFP4 w4a16 problems
// take the tcgen05 weight-streaming kernels.  Measured on the GPT-OSS-120B
// shape (96 local experts, ms per step): up to 64 per expert the mma.sync
// streaming kernels are faster (M = 1024, 43 per expert: 0.65 against 0.71);
// at 85 per expert these kernels win (M = 2048: 0.72 against 0.94 on the
// 128-row tcgen05 kernels); at 171 per expert the 128-row kernels win again
// (M = 4096: 1.36 against 1.49).
constexpr long kTcStreamMinPerExpert = 64, kTcStreamMaxPerExpert = 128;

// The tcgen05 weight-streaming kernels can run this problem: MXFP4 weights
// with bf16 activations and the bounded SwiGLU-OAI (an f16 intermediate with
// no rescale), K and N multiples of 64 (needs MOE_LAYOUT_TC weights too).
bool tcs_supported(const moe_problem_t *p) {
  return p->wfmt == W_MXFP4 && p->afmt == A_BF16 && tc_mx_direct(p) && p->K % 64 == 0 &&
         p->N % 64 == 0 && p->num_local_experts <= 1024;
}
// MXFP4 prefill batches above kTcStreamMaxPerExpert slots per local expert
// take the tcgen05 kernels that decode each weight stage once for two
// 128-slot blocks (moe_tcd.cu) instead of once per block: bf16 activations
// with the bounded SwiGLU-OAI straight to f16 (w4a16), or OCP MX activations
// under the same bounds (w4a4 / w4a8: the intermediate quantised and
// dequantised per 32-output block in the W13 epilogue).
bool tcd_applies(const moe_problem_t *p) {
  const bool formats = p->wfmt == W_MXFP4 && p->K % 64 == 0 && p->N % 64 == 0 &&
                       (tcs_supported(p) || mx_act_f16(p));
  return p->path == MOE_PATH_AUTO && tc_applies(p) && formats &&
         tcd_supported(p->num_local_experts) &&
         (long)p->M * p->topk > kTcStreamMaxPerExpert * p->num_local_experts;
}

// Sort block of the tcgen05 weight-streaming kernels: their passes start
// anywhere in an expert's rows, so 16-row blocks (fewer padding rows to
// gather) instead of the 128 of the other tcgen05 kernels.
constexpr int kTcsBlockM = 16;

// ... and runs it (workspace sized for it).
bool tcs_applies(const moe_problem_t *p) {
  if (!tcs_supported(p)) return false;
  if (p->path == MOE_PATH_TC_STREAM) return true;
  const long slots = (long)p->M * p->topk;
  return p->path == MOE_PATH_AUTO && slots > kTcStreamMinPerExpert * p->num_local_experts &&
         slots <= kTcStreamMaxPerExpert * p->num_local_experts;
}

// Workspace layout of the tcgen05 path (sort blocks of 128 rows).
struct TcLayout {
  long cap, blocks;
  size_t sorted, expert_ids, ntp, counts, offsets, active, n_active, align_scr, x16, x_inv,
      a1_codes, a1_scales, scratch, inter, i_scales, acc, total;
  bool f16_x;  // x converted to f16 once per token by the sort (MXFP4 weights)
};

// Workspace layout of moe_fused_experts.
struct Layout {
  long cap, blocks;
  size_t sorted, expert_ids, ntp, counts, offsets, active, n_active, counters, align_scr, x16,
      x_inv, a1_codes, a1_scales, inter, inter_scales, staging, acc, hpart, fixcnt, done13, total;
  int w13_ksplit;  // k-split of the streaming W13 units (1: none)
  long fixcnt_n;   // counters of the split W13 units
};

// SM count the split decisions assume (GB300); the grids use the real count.
constexpr int kNominalSms = 152;
// Slots per local expert (on average) above which the fused streaming grid
// runs 32-token passes (three CTAs per SM).  A second 16-token pass finds the
// unit's weight records in L2, so the narrow passes cost decode and MMA work,
// not HBM traffic: measured on the GPT-OSS-120B shape, 21 slots per expert
// (M = 512) run 0.366 ms narrow against 0.379 wide, 43 (M = 1024) 0.649
// against 0.630.
constexpr long kStreamWideMinPerExpert = 32;

Layout make_layout(const moe_problem_t *p) {
  Layout L;
  const int BM = kGenericBlockM;
  L.cap = moe_align_capacity(p->M, p->topk, p->num_local_experts, BM);
  L.blocks = L.cap / BM;
  const int s2 = stage2_afmt(p);
  size_t o = 0;
  L.sorted = o; o = align_up(o + (size_t)L.cap * 4);
  L.expert_ids = o; o = align_up(o + (size_t)L.blocks * 4);
  L.ntp = o; o = align_up(o + 4);
  L.counts = o; o = align_up(o + (size_t)p->num_local_experts * 4);
  L.offsets = o; o = align_up(o + (size_t)p->num_local_experts * 4);
  L.active = o; o = align_up(o + (size_t)p->num_local_experts * 4);
  L.n_active = o; o = align_up(o + 4);
  L.counters = o; o = align_up(o + 8);
  L.align_scr = o; o = align_up(o + align_scratch_bytes((long)p->M * p->topk, p->num_local_experts));
  const bool f16_x = p->wfmt == W_MXFP4 && (p->afmt == A_BF16 || mx_act_f16(p));
  if (f16_x) {  // f16 copy of x for the streaming kernels
    L.x16 = o; o = align_up(o + (size_t)p->M * p->K * 2);
    L.x_inv = o; o = align_up(o + (size_t)p->M * 4);
  } else {
    L.x16 = L.x_inv = o;
  }
  L.a1_codes = o; o = align_up(o + codes_bytes(p->afmt, p->M, p->K));
  L.a1_scales = o; o = align_up(o + scales_bytes_of(p->afmt, p->M, p->K));
  if (s2 == A_BF16) {
    L.inter = o; o = align_up(o + (size_t)L.cap * p->N * 2);
    L.inter_scales = o;
    L.staging = o;
  } else {
    // codes, or (MX on the streaming kernels) the f16 of the dequantised rows
    size_t ib = codes_bytes(s2, L.cap, p->N);
    if (f16_x && ib < (size_t)L.cap * p->N * 2) ib = (size_t)L.cap * p->N * 2;
    L.inter = o; o = align_up(o + ib);
    L.inter_scales = o; o = align_up(o + scales_bytes_of(s2, L.cap, p->N));
    L.staging = o; o = align_up(o + (size_t)L.cap * p->N * 4);
  }
  L.acc = o; o = align_up(o + (size_t)p->M * p->K * 4);
  // split-K W13 of the streaming path (very small batches): fp32 partials per
  // k-range and slot, and one counter per (pass, unit, consumer warp)
  L.w13_ksplit = f16_x
                     ? stream_w13_ksplit(p->M, p->topk, p->num_local_experts, p->N, p->K, kNominalSms)
                     : 1;
  L.fixcnt_n = 0;
  // completion counts per local expert of the fused W13 + W2 streaming grid,
  // then the split W13 units' counters: one range for the sort to zero
  L.done13 = o; o = align_up(o + (size_t)p->num_local_experts * 4);
  L.hpart = L.fixcnt = o;
  if (L.w13_ksplit > 1) {
    L.fixcnt_n = stream_w13_fixups(L.cap, p->N);
    L.fixcnt = o; o = align_up(o + (size_t)L.fixcnt_n * 4);
    L.hpart = o; o = align_up(o + (size_t)L.w13_ksplit * p->M * p->topk * p->N * 8);
  }
  L.total = o;
  return L;
}

// MXFP4 w4a16 with SwiGLU-OAI: |z| <= limit * (limit + |beta|) <= 8192 fits f16
// as it is (no per-row rescale pass); the router weight could scale it further.
bool tc_mx_direct(const moe_problem_t *p) {
  return p->wfmt == W_MXFP4 && stage2_afmt(p) == A_BF16 && p->act == ACT_SWIGLU_OAI &&
         p->swiglu_limit > 0.f && p->swiglu_limit <= 64.f && fabsf(p->swiglu_beta) <= 64.f &&
         !p->router_weight_on_input;
}

// Scratch of the tcgen05 stage 1 (the gathered A rows and their scales, fp32
// staging of an intermediate that a separate pass requantises / rescales),
// as offsets from its start; and the intermediate in the form stage 2 reads.
struct TcScratch {
  size_t a_sorted, a_rowscale, a_groupscale, a_sf, staging, total;
};
TcScratch tc_scratch_layout(const moe_problem_t *p, long cap) {
  TcScratch L;
  const int s2 = stage2_afmt(p);
  const bool mx = p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN;
  const bool fp8 = p->wfmt == W_FP8_TENSOR || p->wfmt == W_FP8_CHANNEL ||
                   p->wfmt == W_FP8_BLOCK128;
  const bool bs = p->wfmt == W_NVFP4;
  const long blocks = cap / kTcBlockM;
  size_t o = 0;
  L.a_sorted = o;
  o = align_up(o + (bs ? (size_t)cap * p->K / 2 : (size_t)cap * p->K * (fp8 ? 1 : 2)));
  L.a_rowscale = o; o = align_up(o + (size_t)cap * 4);
  L.a_groupscale = o; o = align_up(o + (fp8 ? (size_t)cap * ceil_div(p->K, 128) * 4 : 0));
  L.a_sf = o; o = align_up(o + (bs ? (size_t)blocks * ceil_div(p->K, kTcBsStage) * kBsSfaRecBytes : 0));
  const bool staged = !bs && !mx && p->wfmt != W_FP8_BLOCK128 &&
                      (s2 != A_BF16 || (p->wfmt == W_MXFP4 && !tc_mx_direct(p)));
  L.staging = o; o = align_up(o + (staged ? (size_t)cap * p->N * 4 : 0));
  L.total = o;
  return L;
}
void tc_inter_sizes(const moe_problem_t *p, long cap, size_t *inter, size_t *scales) {
  const int s2 = stage2_afmt(p);
  const bool mx = p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN;
  if (p->wfmt == W_NVFP4) {  // e2m1 codes + scale-factor records
    *inter = (size_t)cap * p->N / 2;
    *scales = (size_t)(cap / kTcBlockM) * ceil_div(p->N, kTcBsStage) * kBsSfaRecBytes;
  } else if (p->wfmt == W_MXFP4) {  // f16 values (MX: their QDQ), row scales unless direct
    *inter = (size_t)cap * p->N * 2;
    *scales = (mx || tc_mx_direct(p)) ? 0 : (size_t)cap * 4;
  } else if (s2 == A_BF16) {
    *inter = (size_t)cap * p->N * 2;
    *scales = 0;
  } else {  // e4m3 codes + the stage-2 scales, as the generic path writes them
    *inter = codes_bytes(s2, cap, p->N);
    *scales = scales_bytes_of(s2, cap, p->N);
  }
}

TcLayout make_tc_layout(const moe_problem_t *p, bool tcs = false) {
  TcLayout L;
  const int BM = tcs ? kTcsBlockM : kTcBlockM;
  L.cap = moe_align_capacity(p->M, p->topk, p->num_local_experts, BM);
  L.blocks = L.cap / BM;
  size_t o = 0;
  L.sorted = o; o = align_up(o + (size_t)L.cap * 4);
  L.expert_ids = o; o = align_up(o + (size_t)L.blocks * 4);
  L.ntp = o; o = align_up(o + 4);
  L.counts = o; o = align_up(o + (size_t)p->num_local_experts * 4);
  L.offsets = o; o = align_up(o + (size_t)p->num_local_experts * 4);
  L.active = o; o = align_up(o + (size_t)p->num_local_experts * 4);
  L.n_active = o; o = align_up(o + 4);
  L.align_scr = o; o = align_up(o + align_scratch_bytes((long)p->M * p->topk, p->num_local_experts));
  L.f16_x = p->wfmt == W_MXFP4 && (p->afmt == A_BF16 || mx_act_f16(p));
  L.x16 = L.x_inv = o;
  if (L.f16_x) {
    L.x16 = o; o = align_up(o + (size_t)p->M * p->K * 2);
    L.x_inv = o; o = align_up(o + (size_t)p->M * 4);
  }
  L.a1_codes = o; o = align_up(o + codes_bytes(p->afmt, p->M, p->K));
  L.a1_scales = o; o = align_up(o + scales_bytes_of(p->afmt, p->M, p->K));
  L.scratch = o; o = align_up(o + tc_scratch_layout(p, L.cap).total);
  size_t ib = 0, sb = 0;
  tc_inter_sizes(p, L.cap, &ib, &sb);
  L.inter = o; o = align_up(o + ib);
  L.i_scales = o; o = align_up(o + sb);
  L.acc = o; o = align_up(o + (size_t)p->M * p->K * 4);
  L.total = o;
  return L;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Per-device constants looked up once: SM count and the device error word.
struct DeviceInfo {
  int sm_count = 0;
  int *err = nullptr;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

int device_info(DeviceInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo &d = g_dev[dev];
  if (d.sm_count == 0) {
    int sms = 0;
    void *err = nullptr;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaGetSymbolAddress(&err, moe::g_device_error_word) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.sm_count = sms;
    d.err = static_cast<int *>(err);
  }
  *out = d;
  return MOE_OK;
}

// ---- per-stage timing (moe_stage_timing): events around each launch
// Stage timing is a profiling aid: while it is on, calls take g_timing_mu for
// their whole duration (their events and accumulators are shared).  While it
// is off, no call touches the lock or the shared state, so host threads that
// feed different streams run concurrently.
struct StageTiming {
  bool on = false;
  int device = -1;
  cudaEvent_t ev[MOE_NUM_STAGES][2] = {};
  double ms[MOE_NUM_STAGES] = {};
  int calls = 0;
  bool used[MOE_NUM_STAGES] = {};
};
std::mutex g_timing_mu;
StageTiming g_timing;
std::atomic<bool> g_timing_on{false};
thread_local bool t_timing = false;  // this thread's call is being timed

// Adds the elapsed time of every stage launched by the finished call.
void timing_collect() {
  for (int s = 0; s < MOE_NUM_STAGES; ++s) {
    if (!g_timing.used[s]) continue;
    float ms = 0.f;
    if (cudaEventSynchronize(g_timing.ev[s][1]) == cudaSuccess &&
        cudaEventElapsedTime(&ms, g_timing.ev[s][0], g_timing.ev[s][1]) == cudaSuccess)
      g_timing.ms[s] += ms;
    g_timing.used[s] = false;
  }
  g_timing.calls += 1;
}

// One timed call: holds the timing lock (only while timing is on) from the
// first launch to the collection of its events.
struct TimedCall {
  std::unique_lock<std::mutex> lk;
  bool active = false;
  TimedCall() {
    if (g_timing_on.load(std::memory_order_acquire)) {
      lk = std::unique_lock<std::mutex>(g_timing_mu);
      active = g_timing.on;
    }
    t_timing = active;
  }
  ~TimedCall() {
    if (active) timing_collect();
    t_timing = false;
  }
};

struct StageScope {  // records the start event now and the stop event on done()
  cudaStream_t st;
  int stage;
  bool on;
  StageScope(int stage_, cudaStream_t st_) : st(st_), stage(stage_), on(t_timing) {
    if (on) {
      cudaEventRecord(g_timing.ev[stage][0], st);
      g_timing.used[stage] = true;
    }
  }
  void done() {
    if (on) cudaEventRecord(g_timing.ev[stage][1], st);
  }
};

// The weight-streaming decode path applies (see moe_prepare_weights in the header).
bool stream_path(const moe_problem_t *p, const moe_weight_t *w13, const moe_weight_t *w2) {
  return p->wfmt == W_MXFP4 && (p->afmt == A_BF16 || mx_act_f16(p)) && w13->packed && w2->packed &&
         p->act == ACT_SWIGLU_OAI && p->swiglu_limit > 0.f && p->swiglu_limit <= 64.f &&
         fabsf(p->swiglu_beta) <= 64.f && p->K % 64 == 0 && p->N % 64 == 0 &&
         !(w13->bias && w13->bias_is_f32) && !(w2->bias && w2->bias_is_f32) &&
         aligned16(w13->packed) && aligned16(w2->packed) &&
         // up to 64 slots per local expert (measured on the GPT-OSS-120B shape:
         // 43 per expert streams in 650 us against 957 us on the tcgen05
         // kernels; at 85 per expert the tcgen05 kernels win, 972 against 1179)
         (long)p->M * p->topk <= 64L * p->num_local_experts;
}

GemmArgs gemm_args(const moe_problem_t *p, int BM) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.M = p->M; g.K = p->K; g.N = p->N; g.T = p->topk; g.El = p->num_local_experts; g.BM = BM;
  g.wfmt = p->wfmt; g.act = p->act; g.gate = p->gate;
  g.alpha = p->swiglu_alpha; g.beta = p->swiglu_beta; g.limit = p->swiglu_limit;
  g.S = p->M * p->topk;
  g.w_stage1 = p->router_weight_on_input ? 1 : 0;
  return g;
}

// Stage-1 GEMM (+ requantisation).  `staging` is the fp32 scratch when the
// intermediate is requantised.
int run_w13(const moe_problem_t *p, const void *a_codes, const void *a_scales,
            const moe_weight_t *w13, const float *topk_weights, const int32_t *sorted,
            const int32_t *eids, const int32_t *ntp, void *inter, void *inter_scales,
            void *staging, long cap, cudaStream_t st) {
  const int s2 = stage2_afmt(p);
  GemmArgs g = gemm_args(p, kGenericBlockM);
  g.topk_weights = topk_weights;  // read only with the router weight on the stage-1 output
  g.afmt = p->afmt;
  g.a_codes = a_codes; g.a_scales = a_scales; g.a_global = p->a1_scale;
  g.w_codes = w13->codes; g.w_scales = w13->scales; g.w_global = w13->global_scale;
  g.w_bias = w13->bias; g.bias_f32 = w13->bias_is_f32;
  g.sorted_ids = sorted; g.expert_ids = eids; g.num_post_pad = ntp;
  g.out = s2 == A_BF16 ? inter : staging;
  g.out_f32 = s2 != A_BF16;
  StageScope sc13(MOE_STAGE_W13, st);
  int rc = cuda_status(launch_gemm_w13(g, cap, st));
  sc13.done();
  if (rc != MOE_OK || s2 == A_BF16) return rc;
  QuantArgs q{};
  q.x = staging; q.x_is_f32 = 1; q.rows = cap; q.cols = p->N; q.afmt = s2;
  q.param = p->a2_scale; q.sorted_ids = sorted; q.expert_ids = eids; q.num_post_pad = ntp;
  q.S = p->M * p->topk; q.BM = kGenericBlockM; q.codes = inter; q.scales = inter_scales;
  StageScope scq(MOE_STAGE_REQUANT, st);
  rc = cuda_status(launch_quant(q, st));
  scq.done();
  return rc;
}

int run_w2(const moe_problem_t *p, const void *inter, const void *inter_scales,
           const moe_weight_t *w2, const float *topk_weights, const int32_t *sorted,
           const int32_t *eids, const int32_t *ntp, float *acc, void *out, long cap,
           cudaStream_t st) {
  GemmArgs g = gemm_args(p, kGenericBlockM);
  g.afmt = stage2_afmt(p);
  g.a_codes = inter; g.a_scales = inter_scales; g.a_global = p->a2_scale;
  g.w_codes = w2->codes; g.w_scales = w2->scales; g.w_global = w2->global_scale;
  g.w_bias = w2->bias; g.bias_f32 = w2->bias_is_f32;
  g.sorted_ids = sorted; g.expert_ids = eids; g.num_post_pad = ntp;
  g.acc = acc; g.topk_weights = topk_weights;
  StageScope sc2(MOE_STAGE_W2, st);
  int rc = cuda_status(launch_gemm_w2(g, cap, st));
  sc2.done();
  if (rc != MOE_OK) return rc;
  StageScope scf(MOE_STAGE_FINALIZE, st);
  rc = cuda_status(launch_finalize(acc, (long)p->M * p->K, out, st, true));
  scf.done();
  return rc;
}

// The tcgen05 prefill path: sort with 128-row blocks, stage-1 quantisation,
// gather into sorted bf16 rows, tcgen05 w13 (+ requantisation to exact bf16 +
// scales), tcgen05 w2 + reduce, bf16 output.
int run_tc_path(const moe_problem_t *p, const void *hidden, const moe_weight_t *w13,
                const moe_weight_t *w2, const int32_t *topk_ids, const float *topk_weights,
                const int32_t *expert_map, char *ws, void *out, cudaStream_t st, bool tcs,
                bool pair);
// The sort's per-expert tables that the tcgen05 weight-streaming kernels read.
struct TcsRefs {
  const int32_t *offsets, *counts, *active, *n_active;
  bool pair;  // the block-pair kernels (moe_tcd.cu) instead of the weight-streaming ones
};
int tc_stage1(const moe_problem_t *p, const void *a_codes, const void *a_scales, const void *x16,
              const float *x_inv, const moe_weight_t *w13, const float *topk_weights,
              const int32_t *sorted, const int32_t *eids, const int32_t *ntp, long cap,
              char *scratch, void *inter, void *i_scales, const DeviceInfo &dinfo,
              cudaStream_t st, const TcsRefs *tcs = nullptr);
int tc_stage2(const moe_problem_t *p, const void *inter, const void *i_scales,
              const moe_weight_t *w2, const float *topk_weights, const int32_t *sorted,
              const int32_t *eids, const int32_t *ntp, long cap, float *acc,
              const DeviceInfo &dinfo, cudaStream_t st, const TcsRefs *tcs = nullptr);

// The batched expert-parallel input as a problem of E_l * max_tokens tokens
// with one slot each (the slot of row i of expert e is its local expert e,
// weight 1).  The router weight on the stage-1 output and a valid-token count
// do not apply; a per-tensor dynamic fp8 scale would span the padding rows.
int batched_problem(const moe_problem_t *p, int max_tokens, moe_problem_t *q) {
  if (!p || max_tokens < 1 || p->num_local_experts < 1) return MOE_ERR_INVALID_ARG;
  if ((long)p->num_local_experts * max_tokens > (1L << 30)) return MOE_ERR_UNSUPPORTED;
  if (p->router_weight_on_input || p->num_local_tokens || p->afmt == A_FP8_TENSOR_DYN)
    return MOE_ERR_UNSUPPORTED;
  *q = *p;
  q->M = p->num_local_experts * max_tokens;
  q->topk = 1;
  q->num_experts = p->num_local_experts;
  return validate_problem(q);
}

// The batched call runs the tcgen05 kernels under the same conditions as
// moe_fused_experts, else the generic ones.
bool batched_tc(const moe_problem_t *q, const moe_weight_t *w13, const moe_weight_t *w2) {
  const bool fp4 = q->wfmt == W_MXFP4 || q->wfmt == W_NVFP4;
  const bool mx_generic = (q->afmt == A_MXFP4_DYN || q->afmt == A_MXFP8_DYN) && !mx_act_f16(q);
  return !mx_generic && tc_applies(q) &&
         (!fp4 || (w13 && w2 && w13->packed_tc && w2->packed_tc && aligned16(w13->packed_tc) &&
                   aligned16(w2->packed_tc)));
}

size_t batched_body_bytes(const moe_problem_t *q) {
  size_t n = make_layout(q).total;
  if (tc_applies(q)) {
    const size_t t = make_tc_layout(q).total;
    if (t > n) n = t;
  }
  return align_up(n);
}

// The step entry points with block_m = 128 run the tcgen05 kernels: every
// weight format, with bf16 / fp8 / NVFP4 activations (FP4 weights need their
// MOE_LAYOUT_TC records).
int tc_steps_supported(const moe_problem_t *p, const moe_weight_t *w) {
  if (p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN) return MOE_ERR_UNSUPPORTED;
  if ((p->wfmt == W_MXFP4 || p->wfmt == W_NVFP4) && (!w->packed_tc || !aligned16(w->packed_tc)))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_status_str(int s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported combination";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

long moe_align_capacity(int M, int topk, int num_local_experts, int block_m) {
  if (M < 0 || topk < 1 || num_local_experts < 1 || block_m < 1) return 0;
  const long S = (long)M * topk;
  const long nonempty = S < num_local_experts ? S : num_local_experts;
  return ceil_div(S + nonempty * (block_m - 1), block_m) * block_m;
}

size_t moe_workspace_size(const moe_problem_t *p) {
  if (validate_problem(p) != MOE_OK) return 0;
  size_t n = make_layout(p).total;
  if (tc_applies(p)) n = std::max(n, make_tc_layout(p).total);
  if (tcs_applies(p)) n = std::max(n, make_tc_layout(p, true).total);
  return n;
}

size_t moe_align_scratch_bytes(int M, int topk, int num_local_experts) {
  if (M < 0 || topk < 1 || num_local_experts < 1 || num_local_experts > 1024) return 0;
  return align_scratch_bytes((long)M * topk, num_local_experts);
}

int moe_align_block_size_scratch(const int32_t *topk_ids, int M, int topk,
                                 const int32_t *expert_map, int num_experts, int num_local_experts,
                                 int block_m, int32_t *sorted_ids, int32_t *expert_ids,
                                 int32_t *num_post_pad, int32_t *expert_counts, void *scratch,
                                 size_t scratch_bytes, void *stream) {
  if (M < 0 || topk < 1 || num_experts < 1 || num_local_experts < 1 ||
      num_local_experts > 1024 || block_m < 1 || block_m > 1024)
    return MOE_ERR_INVALID_ARG;
  if ((M > 0 && !topk_ids) || !sorted_ids || !expert_ids || !num_post_pad)
    return MOE_ERR_INVALID_ARG;
  if (scratch && (reinterpret_cast<uintptr_t>(scratch) % 16) != 0) return MOE_ERR_INVALID_ARG;
  if ((long)M * topk > (1L << 30)) return MOE_ERR_UNSUPPORTED;
  const long cap = moe_align_capacity(M, topk, num_local_experts, block_m);
  AlignExtras ex;
  ex.scratch = static_cast<int32_t *>(scratch);
  ex.scratch_bytes = scratch ? scratch_bytes : 0;
  return cuda_status(launch_align(topk_ids, M, topk, expert_map, num_experts, num_local_experts,
                                  block_m, sorted_ids, expert_ids, num_post_pad, expert_counts,
                                  cap, ex, static_cast<cudaStream_t>(stream)));
}

int moe_align_block_size(const int32_t *topk_ids, int M, int topk, const int32_t *expert_map,
                         int num_experts, int num_local_experts, int block_m,
                         int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_post_pad,
                         int32_t *expert_counts, void *stream) {
  return moe_align_block_size_scratch(topk_ids, M, topk, expert_map, num_experts,
                                      num_local_experts, block_m, sorted_ids, expert_ids,
                                      num_post_pad, expert_counts, nullptr, 0, stream);
}

int moe_route_topk(const void *logits, int logits_bf16, int M, int num_experts, int topk,
                   int scoring, int renorm, int num_groups, int topk_group, const float *bias,
                   float routed_scaling_factor, int32_t *topk_ids, float *topk_weights,
                   void *stream) {
  const int E = num_experts;
  if (M < 0 || E < 1 || E > 1024 || topk < 1 || topk > 32 || topk > E) return MOE_ERR_INVALID_ARG;
  if (scoring != MOE_SCORE_SOFTMAX && scoring != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (num_groups < 0 || num_groups > 32) return MOE_ERR_INVALID_ARG;
  if (num_groups > 1) {
    if (E % num_groups != 0 || topk_group < 1 || topk_group > num_groups) return MOE_ERR_INVALID_ARG;
    if ((long)topk_group * (E / num_groups) < topk) return MOE_ERR_INVALID_ARG;
  }
  if (!(routed_scaling_factor == routed_scaling_factor)) return MOE_ERR_INVALID_ARG;  // NaN
  if (M == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_weights) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_route(logits, logits_bf16 ? 1 : 0, M, E, topk, scoring, renorm ? 1 : 0,
                                  num_groups > 1 ? num_groups : 1, topk_group, bias,
                                  routed_scaling_factor, topk_ids, topk_weights,
                                  static_cast<cudaStream_t>(stream)));
}

int moe_quant_act(const void *x_bf16, int rows, int cols, int afmt, const float *scale_in,
                  void *codes, void *scales, void *stream) {
  if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
  if (afmt <= A_BF16 || afmt > A_MXFP8_DYN) return MOE_ERR_INVALID_ARG;
  if (afmt == A_NVFP4_DYN && cols % 16 != 0) return MOE_ERR_UNSUPPORTED;
  if ((afmt == A_MXFP4_DYN || afmt == A_MXFP8_DYN) && cols % 32 != 0) return MOE_ERR_UNSUPPORTED;
  if ((afmt == A_FP8_TENSOR_STATIC || afmt == A_NVFP4_DYN) && !scale_in) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x_bf16 || !aligned16(x_bf16) || !codes || !scales || !aligned16(codes) || !aligned16(scales))
    return MOE_ERR_INVALID_ARG;
  QuantArgs q{};  // every field zero / its default
  q.x = x_bf16; q.x_is_f32 = 0; q.rows = rows; q.cols = cols; q.afmt = afmt; q.param = scale_in;
  q.codes = codes; q.scales = scales; q.BM = 1;
  return cuda_status(launch_quant(q, static_cast<cudaStream_t>(stream)));
}

int moe_intermediate_size(const moe_problem_t *p, int block_m, size_t *inter_bytes,
                          size_t *scales_bytes) {
  if (!inter_bytes || !scales_bytes) return MOE_ERR_INVALID_ARG;
  int rc = validate_problem(p);
  if (rc != MOE_OK) return rc;
  if (block_m != kGenericBlockM && block_m != kTcBlockM) return MOE_ERR_UNSUPPORTED;
  const long cap = moe_align_capacity(p->M, p->topk, p->num_local_experts, block_m);
  if (block_m == kTcBlockM) {
    tc_inter_sizes(p, cap, inter_bytes, scales_bytes);
  } else {
    const int s2 = stage2_afmt(p);
    *inter_bytes = s2 == A_BF16 ? (size_t)cap * p->N * 2 : codes_bytes(s2, cap, p->N);
    *scales_bytes = scales_bytes_of(s2, cap, p->N);
  }
  return MOE_OK;
}

size_t moe_w13_workspace_size(const moe_problem_t *p, int block_m) {
  if (validate_problem(p) != MOE_OK) return 0;
  const long cap = moe_align_capacity(p->M, p->topk, p->num_local_experts, block_m);
  if (block_m == kTcBlockM) return tc_scratch_layout(p, cap).total;
  if (block_m != kGenericBlockM || stage2_afmt(p) == A_BF16) return 0;
  return (size_t)cap * p->N * 4;
}

int moe_grouped_gemm_w13_act(const moe_problem_t *p, const void *a_codes, const void *a_scales,
                             const moe_weight_t *w13, const int32_t *sorted_ids,
                             const int32_t *expert_ids, const int32_t *num_post_pad, int block_m,
                             void *inter, void *inter_scales, void *workspace, size_t ws_bytes,
                             void *stream) {
  int rc = validate_problem(p);
  if (rc != MOE_OK) return rc;
  if ((block_m != kGenericBlockM && block_m != kTcBlockM) || p->router_weight_on_input)
    return MOE_ERR_UNSUPPORTED;
  if ((rc = validate_weight(p, w13)) != MOE_OK) return rc;
  if (block_m == kTcBlockM && (rc = tc_steps_supported(p, w13)) != MOE_OK) return rc;
  if (p->M == 0) return MOE_OK;
  if (!a_codes || !aligned16(a_codes) || !sorted_ids || !expert_ids || !num_post_pad || !inter ||
      !aligned16(inter))
    return MOE_ERR_INVALID_ARG;
  if (p->afmt != A_BF16 && !a_scales) return MOE_ERR_INVALID_ARG;
  size_t ib = 0, sb = 0;
  moe_intermediate_size(p, block_m, &ib, &sb);
  if (sb > 0 && (!inter_scales || !aligned16(inter_scales))) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_w13_workspace_size(p, block_m);
  if (need > 0 && (!workspace || !aligned16(workspace) || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long cap = moe_align_capacity(p->M, p->topk, p->num_local_experts, block_m);
  if (block_m == kTcBlockM) {
    DeviceInfo dinfo;
    if ((rc = device_info(&dinfo)) != MOE_OK) return rc;
    return tc_stage1(p, a_codes, a_scales, nullptr, nullptr, w13, nullptr, sorted_ids, expert_ids,
                     num_post_pad, cap, static_cast<char *>(workspace), inter, inter_scales, dinfo,
                     st);
  }
  return run_w13(p, a_codes, a_scales, w13, nullptr, sorted_ids, expert_ids, num_post_pad, inter,
                 inter_scales, workspace, cap, st);
}

int moe_grouped_gemm_w2_reduce(const moe_problem_t *p, const void *inter, const void *inter_scales,
                               const moe_weight_t *w2, const float *topk_weights,
                               const int32_t *sorted_ids, const int32_t *expert_ids,
                               const int32_t *num_post_pad, int block_m, float *acc_f32,
                               void *out_bf16, void *stream) {
  int rc = validate_problem(p);
  if (rc != MOE_OK) return rc;
  if ((block_m != kGenericBlockM && block_m != kTcBlockM) || p->router_weight_on_input)
    return MOE_ERR_UNSUPPORTED;
  if ((rc = validate_weight(p, w2)) != MOE_OK) return rc;
  if (block_m == kTcBlockM && (rc = tc_steps_supported(p, w2)) != MOE_OK) return rc;
  if (p->M == 0) return MOE_OK;
  if (!inter || !aligned16(inter) || !topk_weights || !sorted_ids || !expert_ids ||
      !num_post_pad || !acc_f32 || !aligned16(acc_f32) || !out_bf16 || !aligned16(out_bf16))
    return MOE_ERR_INVALID_ARG;
  size_t ib = 0, sb = 0;
  moe_intermediate_size(p, block_m, &ib, &sb);
  if (sb > 0 && !inter_scales) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long cap = moe_align_capacity(p->M, p->topk, p->num_local_experts, block_m);
  if ((rc = cuda_status(launch_zero(acc_f32, (long)p->M * p->K, st))) != MOE_OK) return rc;
  if (block_m == kTcBlockM) {
    DeviceInfo dinfo;
    if ((rc = device_info(&dinfo)) != MOE_OK) return rc;
    if ((rc = tc_stage2(p, inter, inter_scales, w2, topk_weights, sorted_ids, expert_ids,
                        num_post_pad, cap, acc_f32, dinfo, st)) != MOE_OK)
      return rc;
    return cuda_status(launch_finalize(acc_f32, (long)p->M * p->K, out_bf16, st));
  }
  return run_w2(p, inter, inter_scales, w2, topk_weights, sorted_ids, expert_ids, num_post_pad,
                acc_f32, out_bf16, cap, st);
}

int moe_fused_experts(const moe_problem_t *p, const void *hidden_bf16, const moe_weight_t *w13,
                      const moe_weight_t *w2, const int32_t *topk_ids, const float *topk_weights,
                      const int32_t *expert_map, void *workspace, size_t ws_bytes, void *out_bf16,
                      void *stream) {
  int rc = validate_problem(p);
  if (rc != MOE_OK) return rc;
  if ((rc = validate_weight(p, w13)) != MOE_OK) return rc;
  if ((rc = validate_weight(p, w2)) != MOE_OK) return rc;
  if (p->M == 0) return MOE_OK;
  if (!hidden_bf16 || !aligned16(hidden_bf16) || !topk_ids || !topk_weights || !out_bf16 ||
      !aligned16(out_bf16))
    return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(p);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 || ws_bytes < L.total)
    return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  const bool tc_records = w13->packed_tc && w2->packed_tc && aligned16(w13->packed_tc) &&
                          aligned16(w2->packed_tc);
  const bool tcs = tc_records && tcs_applies(p);
  const bool streaming = !tcs && (p->path == MOE_PATH_AUTO || p->path == MOE_PATH_STREAM) &&
                         stream_path(p, w13, w2);
  const bool fp4 = p->wfmt == W_MXFP4 || p->wfmt == W_NVFP4;
  // MX activations run on the f16 kernels when bounded, else on the generic ones
  const bool mx_generic =
      (p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN) && !mx_act_f16(p);
  if (tcs || (!streaming && !mx_generic && tc_applies(p) && (!fp4 || tc_records))) {
    if (ws_bytes < make_tc_layout(p, tcs).total) return MOE_ERR_WORKSPACE;
    TimedCall timed;
    const bool pair = !tcs && tc_records && tcd_applies(p);
    return run_tc_path(p, hidden_bf16, w13, w2, topk_ids, topk_weights, expert_map, ws, out_bf16,
                       st, tcs, pair);
  }
  int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
  int32_t *eids = reinterpret_cast<int32_t *>(ws + L.expert_ids);
  int32_t *ntp = reinterpret_cast<int32_t *>(ws + L.ntp);
  int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
  float *acc = reinterpret_cast<float *>(ws + L.acc);
  const long MK = (long)p->M * p->K;

  DeviceInfo dinfo;
  if (streaming && (rc = device_info(&dinfo)) != MOE_OK) return rc;

  // 1. sort / pad (+ zero the stage-2 accumulator; for the streaming path also
  //    the expert offsets, the active-expert list and the f16 copy of x)
  AlignExtras ex;
  ex.zero_buf = acc;
  ex.zero_n = MK;
  ex.scratch = reinterpret_cast<int32_t *>(ws + L.align_scr);
  ex.scratch_bytes = align_scratch_bytes((long)p->M * p->topk, p->num_local_experts);
  if (streaming) {
    ex.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    ex.active = reinterpret_cast<int32_t *>(ws + L.active);
    ex.n_active = reinterpret_cast<int32_t *>(ws + L.n_active);
    ex.counters = reinterpret_cast<int32_t *>(ws + L.counters);
    ex.x = static_cast<const uint16_t *>(hidden_bf16);
    ex.x16 = ws + L.x16;
    ex.x_inv = reinterpret_cast<float *>(ws + L.x_inv);
    ex.xM = p->M;
    ex.xK = p->K;
    ex.x_mx = p->afmt == A_MXFP4_DYN ? 1 : p->afmt == A_MXFP8_DYN ? 2 : 0;
  }
  ex.num_valid_tokens = p->num_local_tokens;
  // W13 and W2 run as one streaming grid, except for MX activations with W13
  // split along K (the MX epilogue needs a whole block in one CTA)
  const bool fused_stream = streaming && (L.w13_ksplit == 1 || ex.x_mx == 0);
  if (streaming) {  // the completion counts and the split counters, one range
    ex.zero_ints = reinterpret_cast<int32_t *>(ws + L.done13);
    ex.zero_ints_n = (long)((L.fixcnt - L.done13) / 4) + L.fixcnt_n;
  }
  TimedCall timed;
  {
    StageScope sc(MOE_STAGE_ALIGN, st);
    rc = cuda_status(launch_align(topk_ids, p->M, p->topk, expert_map, p->num_experts,
                                  p->num_local_experts, kGenericBlockM, sorted, eids, ntp, counts,
                                  L.cap, ex, st));
    sc.done();
    if (rc != MOE_OK) return rc;
  }
  if (streaming) {
    StreamArgs sa;
    memset(&sa, 0, sizeof(sa));
    sa.M = p->M; sa.K = p->K; sa.N = p->N; sa.T = p->topk;
    sa.max_active = p->num_local_experts;
    sa.act = p->act; sa.gate = p->gate;
    sa.alpha = p->swiglu_alpha; sa.beta = p->swiglu_beta; sa.limit = p->swiglu_limit;
    sa.sorted_ids = sorted; sa.offsets = ex.offsets; sa.counts = counts;
    sa.active = ex.active; sa.n_active = ex.n_active;
    sa.err = dinfo.err;
    sa.w_stage1 = p->router_weight_on_input ? 1 : 0;
    // 2. gate/up: x16 x packed w13 -> f16 intermediate (+ bias, x-scale, SwiGLU-OAI)
    StreamArgs s13 = sa;
    s13.C = p->K;
    s13.units_per_expert = stream_units_per_expert(1, p->N, p->K);
    s13.ksplit = L.w13_ksplit;
    s13.kblocks = p->K / 64;
    s13.hpart = reinterpret_cast<float *>(ws + L.hpart);
    s13.fix_cnt = reinterpret_cast<int *>(ws + L.fixcnt);
    s13.S = p->M * p->topk;
    s13.packed = w13->packed; s13.bias = w13->bias;
    s13.x16 = ex.x16; s13.x_inv = ex.x_inv;
    s13.topk_weights = topk_weights;  // read only with the router weight on the stage-1 output
    // MX intermediate: quantised and dequantised in the fused grid's W13
    // epilogue, else fp32 rows and a pass of its own
    const bool mx = ex.x_mx != 0 && !fused_stream;
    s13.out = mx ? ws + L.staging : ws + L.inter;
    s13.out_f32 = mx ? 1 : 0;
    s13.out_mx = fused_stream ? ex.x_mx : 0;
    s13.work_counter = ex.counters;
    s13.done13 = fused_stream ? reinterpret_cast<int *>(ws + L.done13) : nullptr;
    // 3. down: intermediate x packed w2 -> fp32 accumulator (+ bias, router weight)
    StreamArgs s2 = sa;
    s2.C = p->N;
    s2.units_per_expert = stream_units_per_expert(0, p->N, p->K);
    s2.kblocks = p->N / 64;
    // split the reduction so that the units keep every CTA busy when few
    // experts are active (about two units per CTA), at least 8 k64 blocks each;
    // in the fused grid, W2 units that already give every CTA two of them
    // stay whole (fewer partial sums to add; measured 1-2% faster there)
    // 32-token passes when the experts hold more than 16 slots on average
    // (16-token passes would stream those experts' weights twice or more)
    const bool wide = fused_stream && !ex.x_mx && s13.ksplit == 1 &&
                      (long)p->M * p->topk > kStreamWideMinPerExpert * p->num_local_experts;
    const int ctas = wide ? 3 : 4;  // CTAs per SM of the grid
    if (wide) s13.tok_pass = s2.tok_pass = 32;
    {
      const long act = (long)p->M * p->topk < p->num_local_experts ? (long)p->M * p->topk
                                                                   : p->num_local_experts;
      const long units = act * s2.units_per_expert;
      const long want = ceil_div(2L * ctas * kNominalSms, units > 0 ? units : 1);
      const long cap_split = s2.kblocks / 8 > 1 ? s2.kblocks / 8 : 1;
      s2.ksplit = (int)(want < 2 ? (cap_split >= 2 ? 2 : 1) : (want < cap_split ? want : cap_split));
      if (fused_stream && units >= 2L * ctas * kNominalSms) s2.ksplit = 1;
    }
    s2.packed = w2->packed; s2.bias = w2->bias;
    s2.x16 = ws + L.inter;
    s2.acc = acc; s2.topk_weights = topk_weights;
    s2.work_counter = ex.counters + 1;
    if (fused_stream) {  // 2 + 3 in one grid, one work queue
      StageScope sc(MOE_STAGE_W13, st);
      rc = cuda_status(launch_stream_fused(s13, s2, dinfo.sm_count, st));
      sc.done();
      if (rc != MOE_OK) return rc;
    } else {
      StageScope sc(MOE_STAGE_W13, st);
      rc = cuda_status(launch_stream(s13, 1, dinfo.sm_count, st));
      sc.done();
      if (rc != MOE_OK) return rc;
    }
    if (mx) {
      StageScope sc(MOE_STAGE_REQUANT, st);
      rc = cuda_status(launch_mx_qdq_rows(reinterpret_cast<const float *>(ws + L.staging), L.cap,
                                          p->N, sorted, ntp, p->M * p->topk, ws + L.inter,
                                          ex.x_mx == 1, 0, st, true));
      sc.done();
      if (rc != MOE_OK) return rc;
    }
    if (!fused_stream) {
      StageScope sc(MOE_STAGE_W2, st);
      rc = cuda_status(launch_stream(s2, 0, dinfo.sm_count, st));
      sc.done();
      if (rc != MOE_OK) return rc;
    }
    // 4. bf16 output
    {
      StageScope sc(MOE_STAGE_FINALIZE, st);
      rc = cuda_status(launch_finalize(acc, MK, out_bf16, st, true));
      sc.done();
    }
    return rc;
  }
  // 2. stage-1 activation quantisation
  const void *a_codes = hidden_bf16;
  const void *a_scales = nullptr;
  if (p->afmt != A_BF16) {
    QuantArgs q{};  // every field zero / its default
    q.x = hidden_bf16; q.rows = p->M; q.cols = p->K; q.afmt = p->afmt; q.param = p->a1_scale;
    q.codes = ws + L.a1_codes; q.scales = ws + L.a1_scales; q.BM = 1;
    StageScope sc(MOE_STAGE_QUANT, st);
    rc = cuda_status(launch_quant(q, st));
    sc.done();
    if (rc != MOE_OK) return rc;
    a_codes = ws + L.a1_codes;
    a_scales = ws + L.a1_scales;
  }
  // 3. gate/up GEMM + activation (+ requantisation)
  if ((rc = run_w13(p, a_codes, a_scales, w13, topk_weights, sorted, eids, ntp, ws + L.inter,
                    ws + L.inter_scales, ws + L.staging, L.cap, st)) != MOE_OK)
    return rc;
  // 4. down GEMM + weighted reduce + bf16 output
  return run_w2(p, ws + L.inter, ws + L.inter_scales, w2, topk_weights, sorted, eids, ntp, acc,
                out_bf16, L.cap, st);
}

size_t moe_batched_workspace_size(const moe_problem_t *p, int max_tokens) {
  moe_problem_t q;
  if (batched_problem(p, max_tokens, &q) != MOE_OK) return 0;
  return batched_body_bytes(&q) + align_up((size_t)q.M * 4);
}

int moe_batched_experts(const moe_problem_t *p, int max_tokens, const void *hidden_bf16,
                        const int32_t *expert_num_tokens, const moe_weight_t *w13,
                        const moe_weight_t *w2, void *workspace, size_t ws_bytes, void *out_bf16,
                        void *stream) {
  moe_problem_t q;
  int rc = batched_problem(p, max_tokens, &q);
  if (rc != MOE_OK) return rc;
  if ((rc = validate_weight(&q, w13)) != MOE_OK) return rc;
  if ((rc = validate_weight(&q, w2)) != MOE_OK) return rc;
  if (!hidden_bf16 || !aligned16(hidden_bf16) || !expert_num_tokens || !out_bf16 ||
      !aligned16(out_bf16))
    return MOE_ERR_INVALID_ARG;
  const size_t body = batched_body_bytes(&q);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      ws_bytes < body + align_up((size_t)q.M * 4))
    return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  float *ones = reinterpret_cast<float *>(ws + body);
  DeviceInfo dinfo;
  if ((rc = device_info(&dinfo)) != MOE_OK) return rc;
  const bool mx = q.afmt == A_MXFP4_DYN || q.afmt == A_MXFP8_DYN;
  const long MK = (long)q.M * q.K;
  TimedCall timed;
  if (batched_tc(&q, w13, w2)) {
    const TcLayout L = make_tc_layout(&q);
    int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    int32_t *eids = reinterpret_cast<int32_t *>(ws + L.expert_ids);
    int32_t *ntp = reinterpret_cast<int32_t *>(ws + L.ntp);
    float *acc = reinterpret_cast<float *>(ws + L.acc);
    {
      StageScope sc(MOE_STAGE_ALIGN, st);
      rc = cuda_status(launch_batched_align(expert_num_tokens, q.num_local_experts, max_tokens,
                                            kTcBlockM, sorted, eids, ntp, L.cap, acc, MK, ones, st));
      sc.done();
      if (rc != MOE_OK) return rc;
    }
    const void *codes = hidden_bf16;
    const void *scales = nullptr;
    if (q.afmt != A_BF16 && !mx) {  // MX activations: quantised by the gather
      QuantArgs qa{};
      qa.x = hidden_bf16; qa.rows = q.M; qa.cols = q.K; qa.afmt = q.afmt; qa.param = q.a1_scale;
      qa.codes = ws + L.a1_codes; qa.scales = ws + L.a1_scales; qa.BM = 1;
      StageScope sc(MOE_STAGE_QUANT, st);
      rc = cuda_status(launch_quant(qa, st));
      sc.done();
      if (rc != MOE_OK) return rc;
      codes = ws + L.a1_codes;
      scales = ws + L.a1_scales;
    }
    if ((rc = tc_stage1(&q, codes, scales, nullptr, nullptr, w13, ones, sorted, eids, ntp, L.cap,
                        ws + L.scratch, ws + L.inter, ws + L.i_scales, dinfo, st)) != MOE_OK)
      return rc;
    if ((rc = tc_stage2(&q, ws + L.inter, ws + L.i_scales, w2, ones, sorted, eids, ntp, L.cap, acc,
                        dinfo, st)) != MOE_OK)
      return rc;
    StageScope sc(MOE_STAGE_FINALIZE, st);
    rc = cuda_status(launch_finalize(acc, MK, out_bf16, st));
    sc.done();
    return rc;
  }
  const Layout L = make_layout(&q);
  int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
  int32_t *eids = reinterpret_cast<int32_t *>(ws + L.expert_ids);
  int32_t *ntp = reinterpret_cast<int32_t *>(ws + L.ntp);
  float *acc = reinterpret_cast<float *>(ws + L.acc);
  {
    StageScope sc(MOE_STAGE_ALIGN, st);
    rc = cuda_status(launch_batched_align(expert_num_tokens, q.num_local_experts, max_tokens,
                                          kGenericBlockM, sorted, eids, ntp, L.cap, acc, MK, ones,
                                          st));
    sc.done();
    if (rc != MOE_OK) return rc;
  }
  const void *codes = hidden_bf16;
  const void *scales = nullptr;
  if (q.afmt != A_BF16) {
    QuantArgs qa{};
    qa.x = hidden_bf16; qa.rows = q.M; qa.cols = q.K; qa.afmt = q.afmt; qa.param = q.a1_scale;
    qa.codes = ws + L.a1_codes; qa.scales = ws + L.a1_scales; qa.BM = 1;
    StageScope sc(MOE_STAGE_QUANT, st);
    rc = cuda_status(launch_quant(qa, st));
    sc.done();
    if (rc != MOE_OK) return rc;
    codes = ws + L.a1_codes;
    scales = ws + L.a1_scales;
  }
  if ((rc = run_w13(&q, codes, scales, w13, ones, sorted, eids, ntp, ws + L.inter,
                    ws + L.inter_scales, ws + L.staging, L.cap, st)) != MOE_OK)
    return rc;
  return run_w2(&q, ws + L.inter, ws + L.inter_scales, w2, ones, sorted, eids, ntp, acc, out_bf16,
                L.cap, st);
}

size_t moe_packed_weight_bytes(const moe_problem_t *p, int which, int layout) {
  if (validate_problem(p) != MOE_OK || (which != 0 && which != 1)) return 0;
  if (layout == MOE_LAYOUT_STREAM) {
    if (p->wfmt != W_MXFP4 || p->K % 64 != 0 || p->N % 64 != 0) return 0;
    return stream_packed_bytes(which == 0, p->N, p->K, p->num_local_experts);
  }
  if (layout == MOE_LAYOUT_TC) {
    if (p->wfmt != W_MXFP4 && p->wfmt != W_NVFP4) return 0;
    return tc_packed_bytes(which == 0, p->wfmt == W_NVFP4, p->N, p->K, p->num_local_experts);
  }
  return 0;
}

int moe_prepare_weights(const moe_problem_t *p, int which, int layout, const moe_weight_t *w,
                        void *packed, void *stream) {
  int rc = validate_problem(p);
  if (rc != MOE_OK) return rc;
  if ((which != 0 && which != 1) || (layout != MOE_LAYOUT_STREAM && layout != MOE_LAYOUT_TC))
    return MOE_ERR_INVALID_ARG;
  if (moe_packed_weight_bytes(p, which, layout) == 0) return MOE_ERR_UNSUPPORTED;
  if ((rc = validate_weight(p, w)) != MOE_OK) return rc;
  if (!packed || !aligned16(packed)) return MOE_ERR_INVALID_ARG;
  const int w13 = which == 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (layout == MOE_LAYOUT_STREAM) {
    PackArgs a;
    a.codes = static_cast<const unsigned char *>(w->codes);
    a.scales = static_cast<const unsigned char *>(w->scales);
    a.out = static_cast<unsigned char *>(packed);
    a.total = (long)stream_packed_bytes(w13, p->N, p->K, p->num_local_experts);
    a.units = stream_units_per_expert(w13, p->N, p->K);
    a.w13 = w13;
    a.N = p->N;
    a.R = w13 ? 2 * p->N : p->K;
    a.C = w13 ? p->K : p->N;
    a.kblocks = a.C / 64;
    a.gate = p->gate;
    return cuda_status(launch_pack_mxfp4(a, st));
  }
  if (p->wfmt == W_MXFP4) {
    // The tcgen05 kernels decode MXFP4 into f16: every e2m1 * 2^(c-127) is an
    // exact f16 value when the exponent c-127 lies in [-21, 13].  Check the
    // codes once at load time (this synchronises `stream`).
    void *rng = nullptr;
    if (cudaGetSymbolAddress(&rng, moe::g_scale_range) != cudaSuccess) return MOE_ERR_CUDA;
    const long n = (long)p->num_local_experts * (w13 ? 2L * p->N : p->K) * ((w13 ? p->K : p->N) / 32);
    int host[2] = {0, 0};
    if (launch_scale_range(static_cast<const uint8_t *>(w->scales), n, static_cast<int *>(rng), st) !=
            cudaSuccess ||
        cudaMemcpyAsync(host, rng, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (host[0] < 127 - 21 || host[1] > 127 + 13) return MOE_ERR_UNSUPPORTED;
  }
  TcPackArgs a;
  a.codes = static_cast<const unsigned char *>(w->codes);
  a.scales = static_cast<const unsigned char *>(w->scales);
  a.out = static_cast<unsigned char *>(packed);
  a.nvfp4 = p->wfmt == W_NVFP4;
  a.total = (long)tc_packed_bytes(w13, a.nvfp4, p->N, p->K, p->num_local_experts);
  a.rec_bytes = 4096 + 128 * 2;
  a.w13 = w13;
  a.N = p->N;
  a.R = w13 ? 2 * p->N : p->K;
  a.C = w13 ? p->K : p->N;
  a.kstages = (int)ceil_div(a.C, a.nvfp4 ? kTcBsStage : 64);
  a.ntiles = a.nvfp4 ? bs_ntiles(w13, p->N, p->K) : tc_ntiles(w13, p->N, p->K);
  a.gate = p->gate;
  return cuda_status(launch_pack_tc_fp4(a, st));
}

int moe_stage_timing(int enable) {
  std::lock_guard<std::mutex> lock(g_timing_mu);
  if (enable) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (g_timing.device != dev) {
      for (int s = 0; s < MOE_NUM_STAGES; ++s)
        for (int k = 0; k < 2; ++k)
          if (cudaEventCreate(&g_timing.ev[s][k]) != cudaSuccess) return MOE_ERR_CUDA;
      g_timing.device = dev;
    }
    for (int s = 0; s < MOE_NUM_STAGES; ++s) {
      g_timing.ms[s] = 0.0;
      g_timing.used[s] = false;
    }
    g_timing.calls = 0;
  }
  g_timing.on = enable != 0;
  g_timing_on.store(g_timing.on, std::memory_order_release);
  return MOE_OK;
}

int moe_stage_times(double *ms_out, int *calls_out) {
  if (!ms_out) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  for (int s = 0; s < MOE_NUM_STAGES; ++s) ms_out[s] = g_timing.ms[s];
  if (calls_out) *calls_out = g_timing.calls;
  return MOE_OK;
}

int moe_get_device_error(int *err_out) {
  if (!err_out) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemcpyFromSymbol(err_out, moe::g_device_error_word, sizeof(int)));
}

int moe_reset_device_error(void) {
  const int zero = 0;
  return cuda_status(cudaMemcpyToSymbol(moe::g_device_error_word, &zero, sizeof(int)));
}

int moe_mma_probe(int kind, int n, long long iters, int *sm_count_out, void *stream) {
  if (kind < 0 || kind > 2 || (n != 128 && n != 256) || iters < 1 || iters > (1LL << 31))
    return MOE_ERR_INVALID_ARG;
  DeviceInfo dinfo;
  int rc = device_info(&dinfo);
  if (rc != MOE_OK) return rc;
  if (sm_count_out) *sm_count_out = dinfo.sm_count;
  return cuda_status(launch_mma_probe(kind, n, (long)iters, dinfo.sm_count, dinfo.err,
                                      static_cast<cudaStream_t>(stream)));
}

int moe_selftest_bounded_wait(long long limit_cycles, void *stream) {
  if (limit_cycles < 1 || limit_cycles >= (1LL << 40)) return MOE_ERR_INVALID_ARG;
  DeviceInfo dinfo;
  int rc = device_info(&dinfo);
  if (rc != MOE_OK) return rc;
  return cuda_status(launch_selftest_wait(dinfo.err, limit_cycles, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Stage 1 of the tcgen05 path: the stage-1 rows gathered into sort order
// (a_codes / a_scales: bf16 x or moe_quant_act's output; x16 / x_inv: the
// sort's per-token f16 copy of x, when made), the W13 GEMM + activation, and
// the intermediate in the form stage 2 reads (inter / i_scales, see
// tc_inter_sizes).  `scratch` holds tc_scratch_layout(p, cap).total bytes.
int tc_stage1(const moe_problem_t *p, const void *a_codes, const void *a_scales, const void *x16,
              const float *x_inv, const moe_weight_t *w13, const float *topk_weights,
              const int32_t *sorted, const int32_t *eids, const int32_t *ntp, long cap,
              char *scratch, void *inter, void *i_scales, const DeviceInfo &dinfo,
              cudaStream_t st, const TcsRefs *tcs) {
  const TcScratch L = tc_scratch_layout(p, cap);
  const int S = p->M * p->topk;
  const int s2 = stage2_afmt(p);
  const bool mx = p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN;
  const bool bs = p->wfmt == W_NVFP4;
  const bool mx_direct = tc_mx_direct(p);
  int rc;
  // gather: sorted rows (codes as they are, or exact f16 / bf16 values) +
  // per-row / per-group scales, or (NVFP4) codes + scale-factor records
  {
    GatherArgs g;
    g.sorted_ids = sorted; g.num_post_pad = ntp; g.S = S; g.T = p->topk; g.K = p->K;
    g.afmt = p->afmt; g.codes = a_codes; g.scales = a_scales;
    g.to_f16 = p->wfmt == W_MXFP4;
    g.x16 = x16;
    g.x_inv = x_inv;
    g.out = scratch + L.a_sorted;
    g.rowscale = reinterpret_cast<float *>(scratch + L.a_rowscale);
    g.groupscale = reinterpret_cast<float *>(scratch + L.a_groupscale);
    if (bs) g.sf_out = scratch + L.a_sf;
    if (bs && !a_scales) {  // NVFP4 rows quantised by the gather itself (bf16 x in a_codes)
      g.x_nvfp4 = static_cast<const uint16_t *>(a_codes);
      g.nv_global = p->a1_scale;
    }
    StageScope sc(MOE_STAGE_QUANT, st);
    rc = cuda_status(launch_gather_rows(g, cap, st));
    sc.done();
    if (rc != MOE_OK) return rc;
  }
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.M = p->M; a.K = p->K; a.N = p->N; a.T = p->topk; a.El = p->num_local_experts;
  a.wfmt = p->wfmt; a.act = p->act; a.gate = p->gate;
  a.alpha = p->swiglu_alpha; a.beta = p->swiglu_beta; a.limit = p->swiglu_limit;
  a.sorted_ids = sorted; a.expert_ids = eids; a.num_post_pad = ntp; a.S = S;
  a.err = dinfo.err;
  a.w_stage1 = p->router_weight_on_input ? 1 : 0;
  a.topk_weights = topk_weights;
  a.R = 2 * p->N; a.C = p->K;
  switch (p->afmt) {
    case A_FP8_TENSOR_STATIC:
    case A_FP8_TENSOR_DYN: a.a_scalar = static_cast<const float *>(a_scales); break;
    case A_FP8_TOKEN_DYN: a.a_rowscale = reinterpret_cast<const float *>(scratch + L.a_rowscale); break;
    case A_FP8_GROUP128_DYN:
      a.a_groupscale = reinterpret_cast<const float *>(scratch + L.a_groupscale);
      a.a_groups = (int)ceil_div(p->K, 128);
      break;
    case A_NVFP4_DYN: a.a_scalar = p->a1_scale; break;
    default:
      if (p->wfmt == W_MXFP4) a.a_rowscale = reinterpret_cast<const float *>(scratch + L.a_rowscale);
      break;
  }
  a.w_codes = w13->codes; a.w_scales = w13->scales; a.w_global = w13->global_scale;
  a.w_bias = w13->bias; a.bias_f32 = w13->bias_is_f32; a.w_packed = w13->packed_tc;
  a.out = inter;
  const bool fp8b = p->wfmt == W_FP8_BLOCK128;
  if (bs) {                       // block-scaled: codes + scale-factor records
    a.a_sf = scratch + L.a_sf;
    a.out_sf = i_scales;
    a.out_global = p->a2_scale;
  } else if (fp8b) {              // e4m3 codes + 1 x 128 scales from the epilogue
    a.out_scales = static_cast<float *>(i_scales);
  } else if (mx) {                // OCP MX quantise-dequantise inside the epilogue
    a.out_mode = s2 == A_MXFP4_DYN ? TC_OUT_MX4_F16 : TC_OUT_MX8_F16;
  } else if (mx_direct) {         // bounded SwiGLU-OAI intermediate straight to f16
    a.out_mode = TC_OUT_F16;
  } else if (s2 != A_BF16 || p->wfmt == W_MXFP4) {
    a.out = scratch + L.staging;  // fp32 staging, then a requantiser / row rescale
    a.out_mode = TC_OUT_F32;
  } else {
    a.out_mode = TC_OUT_BF16;
  }
  {
    StageScope sc(MOE_STAGE_W13, st);
    if (tcs) {  // weight-streaming kernels: f16 intermediate (bounded SwiGLU-OAI)
      a.offsets = tcs->offsets; a.counts = tcs->counts;
      a.active = tcs->active; a.n_active = tcs->n_active;
    }
    rc = cuda_status(tcs && tcs->pair
                         ? launch_tcd_gemm(a, scratch + L.a_sorted, cap, 1, dinfo.sm_count, st)
                     : tcs  ? launch_tcs_gemm(a, scratch + L.a_sorted, cap, 1, dinfo.sm_count, st)
                     : bs   ? launch_bs_gemm(a, scratch + L.a_sorted, cap, 1, dinfo.sm_count, st)
                     : fp8b ? launch_fp8b_gemm(a, scratch + L.a_sorted, cap, 1, dinfo.sm_count, st)
                            : launch_tc_gemm(a, scratch + L.a_sorted, cap, 1, st));
    sc.done();
    if (rc != MOE_OK) return rc;
  }
  if (s2 == A_BF16 && p->wfmt == W_MXFP4 && !mx_direct) {  // f16 intermediate with row scales
    StageScope sc(MOE_STAGE_REQUANT, st);
    rc = cuda_status(launch_rescale_rows(reinterpret_cast<const float *>(scratch + L.staging), cap,
                                         p->N, sorted, ntp, S, inter,
                                         static_cast<float *>(i_scales), st));
    sc.done();
    return rc;
  }
  // stage-2 requantisation of the per-tensor / per-token fp8 formats into
  // e4m3 codes + scales (NVFP4, FP8 block and OCP MX were quantised in the W13
  // epilogue)
  if (s2 != A_BF16 && !bs && !mx && !fp8b) {
    QuantArgs q{};  // every field zero / its default
    q.x = scratch + L.staging; q.x_is_f32 = 1; q.rows = cap; q.cols = p->N; q.afmt = s2;
    q.param = p->a2_scale; q.sorted_ids = sorted; q.expert_ids = eids; q.num_post_pad = ntp;
    q.S = S; q.BM = kTcBlockM; q.scales = i_scales; q.codes = inter;
    StageScope sc(MOE_STAGE_REQUANT, st);
    rc = cuda_status(launch_quant(q, st));
    sc.done();
  }
  return rc;
}

// Stage 2 of the tcgen05 path: the W2 GEMM + router weight + fp32 reduce into
// acc (zeroed by the caller) from the intermediate stage 1 wrote.
int tc_stage2(const moe_problem_t *p, const void *inter, const void *i_scales,
              const moe_weight_t *w2, const float *topk_weights, const int32_t *sorted,
              const int32_t *eids, const int32_t *ntp, long cap, float *acc,
              const DeviceInfo &dinfo, cudaStream_t st, const TcsRefs *tcs) {
  const int s2 = stage2_afmt(p);
  const bool mx = p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN;
  const bool bs = p->wfmt == W_NVFP4;
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.M = p->M; a.K = p->K; a.N = p->N; a.T = p->topk; a.El = p->num_local_experts;
  a.wfmt = p->wfmt; a.act = p->act; a.gate = p->gate;
  a.alpha = p->swiglu_alpha; a.beta = p->swiglu_beta; a.limit = p->swiglu_limit;
  a.sorted_ids = sorted; a.expert_ids = eids; a.num_post_pad = ntp; a.S = p->M * p->topk;
  a.err = dinfo.err;
  a.w_stage1 = p->router_weight_on_input ? 1 : 0;
  a.R = p->K; a.C = p->N;
  switch (s2) {
    case A_FP8_TENSOR_STATIC:
    case A_FP8_TENSOR_DYN: a.a_scalar = static_cast<const float *>(i_scales); break;
    case A_FP8_TOKEN_DYN: a.a_rowscale = static_cast<const float *>(i_scales); break;
    case A_FP8_GROUP128_DYN:
      a.a_groupscale = static_cast<const float *>(i_scales);
      a.a_groups = (int)ceil_div(p->N, 128);
      break;
    case A_NVFP4_DYN: a.a_expertscale = p->a2_scale; break;
    default:
      if (p->wfmt == W_MXFP4 && !tc_mx_direct(p) && !mx)
        a.a_rowscale = static_cast<const float *>(i_scales);
      break;
  }
  a.w_codes = w2->codes; a.w_scales = w2->scales; a.w_global = w2->global_scale;
  a.w_bias = w2->bias; a.bias_f32 = w2->bias_is_f32; a.w_packed = w2->packed_tc;
  a.acc = acc; a.topk_weights = topk_weights;
  if (bs) a.a_sf = i_scales;
  if (tcs) {
    a.offsets = tcs->offsets; a.counts = tcs->counts;
    a.active = tcs->active; a.n_active = tcs->n_active;
  }
  StageScope sc(MOE_STAGE_W2, st);
  const int rc = cuda_status(tcs && tcs->pair ? launch_tcd_gemm(a, inter, cap, 0, dinfo.sm_count, st)
                             : tcs  ? launch_tcs_gemm(a, inter, cap, 0, dinfo.sm_count, st)
                             : bs ? launch_bs_gemm(a, inter, cap, 0, dinfo.sm_count, st)
                             : p->wfmt == W_FP8_BLOCK128
                                 ? launch_fp8b_gemm(a, inter, cap, 0, dinfo.sm_count, st)
                                 : launch_tc_gemm(a, inter, cap, 0, st));
  sc.done();
  return rc;
}

// The tcgen05 prefill path: sort with 128-row blocks (+ zero the accumulator;
// MXFP4 weights: + the f16 copy of x), stage-1 quantisation, stage 1, stage 2,
// bf16 output.
// tcs: the weight-streaming kernels (16-row sort blocks); pair: the
// block-pair kernels (128-row blocks); both read the sort's per-expert tables.
int run_tc_path(const moe_problem_t *p, const void *hidden, const moe_weight_t *w13,
                const moe_weight_t *w2, const int32_t *topk_ids, const float *topk_weights,
                const int32_t *expert_map, char *ws, void *out, cudaStream_t st, bool tcs,
                bool pair) {
  const TcLayout L = make_tc_layout(p, tcs);
  DeviceInfo dinfo;
  int rc = device_info(&dinfo);
  if (rc != MOE_OK) return rc;
  int32_t *sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
  int32_t *eids = reinterpret_cast<int32_t *>(ws + L.expert_ids);
  int32_t *ntp = reinterpret_cast<int32_t *>(ws + L.ntp);
  int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
  float *acc = reinterpret_cast<float *>(ws + L.acc);
  const long MK = (long)p->M * p->K;
  {
    AlignExtras ex;
    ex.zero_buf = acc;
    ex.zero_n = MK;
    ex.num_valid_tokens = p->num_local_tokens;
    ex.scratch = reinterpret_cast<int32_t *>(ws + L.align_scr);
    ex.scratch_bytes = align_scratch_bytes((long)p->M * p->topk, p->num_local_experts);
    if (tcs || pair) {  // per-expert tables of the weight-streaming / block-pair kernels
      ex.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
      ex.active = reinterpret_cast<int32_t *>(ws + L.active);
      ex.n_active = reinterpret_cast<int32_t *>(ws + L.n_active);
    }
    if (L.f16_x) {
      ex.x = static_cast<const uint16_t *>(hidden);
      ex.x16 = ws + L.x16;
      ex.x_inv = reinterpret_cast<float *>(ws + L.x_inv);
      ex.xM = p->M;
      ex.xK = p->K;
      ex.x_mx = p->afmt == A_MXFP4_DYN ? 1 : p->afmt == A_MXFP8_DYN ? 2 : 0;
    }
    StageScope sc(MOE_STAGE_ALIGN, st);
    rc = cuda_status(launch_align(topk_ids, p->M, p->topk, expert_map, p->num_experts,
                                  p->num_local_experts, tcs ? kTcsBlockM : kTcBlockM, sorted, eids,
                                  ntp, counts, L.cap, ex, st));
    sc.done();
    if (rc != MOE_OK) return rc;
  }
  // stage-1 quantisation of x (once per token); OCP MX activations are
  // quantised and dequantised by the sort's conversion CTAs
  const bool mx = p->afmt == A_MXFP4_DYN || p->afmt == A_MXFP8_DYN;
  const void *codes = hidden;
  const void *scales = nullptr;
  // NVFP4 weights and activations: the gather quantises the rows it writes
  // (tc_stage1 sees bf16 x and no scales)
  const bool nvfp4_in_gather = p->wfmt == W_NVFP4 && p->afmt == A_NVFP4_DYN;
  if (p->afmt != A_BF16 && !mx && !nvfp4_in_gather) {
    QuantArgs q{};  // every field zero / its default
    q.x = hidden; q.rows = p->M; q.cols = p->K; q.afmt = p->afmt; q.param = p->a1_scale;
    q.codes = ws + L.a1_codes; q.scales = ws + L.a1_scales; q.BM = 1;
    StageScope sc(MOE_STAGE_QUANT, st);
    rc = cuda_status(launch_quant(q, st));
    sc.done();
    if (rc != MOE_OK) return rc;
    codes = ws + L.a1_codes;
    scales = ws + L.a1_scales;
  }
  TcsRefs tr{};
  tr.pair = pair;
  if (tcs || pair) {
    tr.counts = counts;
    tr.offsets = reinterpret_cast<const int32_t *>(ws + L.offsets);
    tr.active = reinterpret_cast<const int32_t *>(ws + L.active);
    tr.n_active = reinterpret_cast<const int32_t *>(ws + L.n_active);
  }
  if ((rc = tc_stage1(p, codes, scales, L.f16_x ? ws + L.x16 : nullptr,
                      L.f16_x ? reinterpret_cast<const float *>(ws + L.x_inv) : nullptr, w13,
                      topk_weights, sorted, eids, ntp, L.cap, ws + L.scratch, ws + L.inter,
                      ws + L.i_scales, dinfo, st, (tcs || pair) ? &tr : nullptr)) != MOE_OK)
    return rc;
  if ((rc = tc_stage2(p, ws + L.inter, ws + L.i_scales, w2, topk_weights, sorted, eids, ntp,
                      L.cap, acc, dinfo, st, (tcs || pair) ? &tr : nullptr)) != MOE_OK)
    return rc;
  StageScope sc(MOE_STAGE_FINALIZE, st);
  rc = cuda_status(launch_finalize(acc, MK, out, st));
  sc.done();
  return rc;
}

}  // namespace
