// moe_probe.cu -- tensor-core rate probe: the dense tcgen05 MMA rate of this
// GPU for the operand kinds the fused experts use, measured with operands
// already resident in shared memory (no loads, no epilogue).  It is the
// denominator the benchmark reports beside the recipe's nominal ratios for the
// FP8 and FP4 kinds, whose dense rates the measured-peaks file does not hold.
//
// One CTA per SM; lane 0 of warp 0 issues `iters` MMAs of 128 x n x k_kind
// (k = 16 for f16 / bf16, 32 for e4m3, 64 for e2m1 with ue4m3 scales) back to
// back into one Tensor Memory accumulator, then waits (bounded) for them to
// complete.  Operands are zeros: the rate does not depend on the values.
#include <cuda_runtime.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int kThreads = 128;
constexpr long long kWaitCycles = 4000000000LL;
constexpr int kErrTimeout = 5;

struct ProbeSmem {
  unsigned char a[128 * 128];   // 128 rows x 128 B, 128-byte swizzle
  unsigned char b[256 * 128];   // up to 256 rows
  unsigned char sf[3 * 512];    // scale-factor chunks (A, B rows 0-127, B rows 128-255)
  uint64_t done;
  uint32_t tmem_base;
};

__global__ void __launch_bounds__(kThreads, 1)
mma_probe_kernel(int kind, int n, long iters, int *err) {
  extern __shared__ unsigned char smem_raw[];
  ProbeSmem &sm = *reinterpret_cast<ProbeSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                 ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (int)sizeof(sm.a) / 16; i += kThreads)
    reinterpret_cast<uint4 *>(sm.a)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < (int)sizeof(sm.b) / 16; i += kThreads)
    reinterpret_cast<uint4 *>(sm.b)[i] = make_uint4(0, 0, 0, 0);
  for (int i = threadIdx.x; i < (int)sizeof(sm.sf) / 16; i += kThreads)
    reinterpret_cast<uint4 *>(sm.sf)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(&sm.done, 1);
    mbar_fence_init();
  }
  fence_proxy_async_smem();  // the zeros are read by the tensor cores
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (warp == 0 && lane == 0) {
    const uint64_t ad = umma_desc_sw128(smem_addr(sm.a));
    const uint64_t bd = umma_desc_sw128(smem_addr(sm.b));
    const uint32_t sf = tmem + 256;  // A scale factors at +0, B at +4
    if (kind == 2) {
      const uint32_t s0 = smem_addr(sm.sf);
      tc_cp_32x128b_x4(sf, sf_smem_desc(s0));
      tc_cp_32x128b_x4(sf + 4, sf_smem_desc(s0 + 512));
      tc_cp_32x128b_x4(sf + 8, sf_smem_desc(s0 + 1024));
    }
    const uint32_t id16 = umma_idesc_f16(128, n), id8 = umma_idesc_e4m3(128, n),
                   id4 = umma_idesc_nvf4(128, n);
    for (long i = 0; i < iters; ++i) {
      const uint32_t acc = i == 0 ? 0u : 1u;
      if (kind == 0) umma_f16(tmem, ad, bd, id16, acc);
      else if (kind == 1) umma_f8(tmem, ad, bd, id8, acc);
      else umma_nvf4(tmem, ad, bd, id4, sf, sf + 4, acc);
    }
    umma_commit(&sm.done);
    if (!mbar_wait_bounded(&sm.done, 0, kWaitCycles)) record_device_error(err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_mma_probe(int kind, int n, long iters, int sm_count, int *err,
                             cudaStream_t st) {
  // more shared memory than two CTAs of this size fit in, so that every SM
  // runs exactly one of them (each holds all 512 Tensor Memory columns)
  const size_t smem = sizeof(ProbeSmem) + 1024 > 120 * 1024 ? sizeof(ProbeSmem) + 1024 : 120 * 1024;
  static int attr_dev[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_dev[dev]) {
    cudaError_t e = cudaFuncSetAttribute(mma_probe_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_dev[dev] = 1;
  }
  mma_probe_kernel<<<(unsigned)sm_count, kThreads, smem, st>>>(kind, n, iters, err);
  return cudaGetLastError();
}

}  // namespace moe
