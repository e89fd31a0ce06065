// moe_noalloc.cu -- moe_fused_experts_noalloc: the whole fused-experts call
// for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code running
// inside a host framework or plugin slot that owns every device allocation
// and exposes no scratch buffer, memory-planned inference runtimes that must
// not call cudaMalloc after start-up (a cudaMalloc can synchronise the device
// and breaks their fixed memory budget), and latency-critical loops where an
// allocation on the call path is not acceptable.  For them this entry point
// takes the same inputs and output as moe_fused_experts but no workspace: its
// scratch is a file-scope __device__ array of kNoAllocScratchBytes that every
// GPU which loads the library holds until the process exits.
//
// Rules of use:
//  - Problems whose workspace (moe_workspace_size) exceeds the array are
//    rejected with MOE_ERR_WORKSPACE before anything is launched.
//  - The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current) and caches it; make that
//    first call before any stream capture on the device.  The cached address
//    belongs to the device's primary context: do not call cudaDeviceReset (or
//    otherwise tear that context down) in a process that uses this entry
//    point, since the array would be loaded again at another address.
//  - Every call on a device shares the one array and it keeps the last
//    call's contents.  Calls that overlap on the GPU (different streams, no
//    ordering between them) race on it; serialise them.  What must start at
//    zero (the fp32 reduce accumulator) is cleared inside each call.
//  - No cudaMalloc, cudaFree or allocating library routine is called.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe_experts.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up once).
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int moe_fused_experts_noalloc(const moe_problem_t *p, const void *hidden_bf16,
                              const moe_weight_t *w13, const moe_weight_t *w2,
                              const int32_t *topk_ids, const float *topk_weights,
                              const int32_t *expert_map, void *out_bf16, void *stream) {
  const size_t need = moe_workspace_size(p);
  if (need == 0)  // invalid problem: report the same status moe_fused_experts gives
    return moe_fused_experts(p, hidden_bf16, w13, w2, topk_ids, topk_weights, expert_map,
                             nullptr, 0, out_bf16, stream);
  if (need > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE;
  void *scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  return moe_fused_experts(p, hidden_bf16, w13, w2, topk_ids, topk_weights, expert_map, scratch,
                           kNoAllocScratchBytes, out_bf16, stream);
}

}  // extern "C"
