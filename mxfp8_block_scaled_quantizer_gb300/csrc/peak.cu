// Rate of the tensor pipe on block-scaled MXFP8 MMAs (lpfa_mma_peak).
//
// The dense MX MMA peak of this GPU, measured in the same run as the
// attention kernels so that their fraction of it can be stated ("Low
// Precision Flash Attention 4 ...", paragraph 2: tcgen05.mma.block_scale on
// MXFP8 operands).  One CTA per SM keeps its operands resident in shared
// memory and issues M128 N256 K32 block-scaled MMAs back to back into one
// TMEM accumulator, so nothing but the tensor pipe bounds it: no global
// traffic, no epilogue.  The operand bytes are arbitrary finite E4M3 values
// with scale 1 (the pipe's rate does not depend on them).
#include <cuda_runtime.h>

#include "lpfa_device.cuh"
#include "lpfa_internal.h"

namespace lpfa {
namespace {

constexpr int kPM = 128, kPN = 256, kPK = 128;    // one 128-byte K row per operand row
constexpr int kPA = kPM * kPK;                    // 16 KB
constexpr int kPB = kPN * kPK;                    // 32 KB
constexpr int kPSf = 3 * 512;                     // A, B(0..127), B(128..255) scale tiles
constexpr int kPSmem = kPA + kPB + kPSf;
constexpr int kPThreads = 128;
constexpr uint32_t kPColSfA = 256, kPColSfB = 260;

// error word of the last launch on this device (ERR_* bits)
__device__ uint32_t g_peak_err[4];

__global__ void __launch_bounds__(kPThreads, 1) mma_peak_kernel(int iters) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5;

  // operands: finite E4M3 bytes (exponent field <= 14), scale codes 127
  for (int i = threadIdx.x; i < kPA + kPB; i += kPThreads)
    sm[i] = static_cast<uint8_t>(((static_cast<uint32_t>(i) * 2654435761u) >> 24) & 0x77u);
  for (int i = threadIdx.x; i < kPSf; i += kPThreads) sm[kPA + kPB + i] = 127;
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    const uint32_t idesc = idesc_mxf8(kPM, kPN, 0, 0);
    const uint64_t da = make_sdesc(smem_u32(sm), 16, 1024, 2);
    const uint64_t db = make_sdesc(smem_u32(sm + kPA), 16, 1024, 2);
    const uint64_t dsf = sf_tile_desc(smem_u32(sm + kPA + kPB));
    tc_cp_32x128b_warpx4_elect(tmem + kPColSfA, dsf);
    tc_cp_32x128b_warpx4_elect(tmem + kPColSfB, dsf + (512 >> 4));
    tc_cp_32x128b_warpx4_elect(tmem + kPColSfB + 4, dsf + (1024 >> 4));
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kb = 0; kb < kPK / 32; ++kb)
        mma_mxf8_ss_elect(tmem, da + 2 * kb, db + 2 * kb, idesc_sf_ids(idesc, kb, kb),
                          tmem + kPColSfA, tmem + kPColSfB, (it | kb) != 0);
    }
    tc_commit_elect(&done);
    if (!mbar_wait_sleep(&done, 0, g_peak_err, nullptr, 90)) {
      // the MMAs did not finish within the bound: wait again before the
      // tensor memory they write is released
      mbar_wait_sleep(&done, 0, nullptr, nullptr, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace
}  // namespace lpfa

using namespace lpfa;

extern "C" lpfa_status lpfa_mma_peak(double* flops_per_s, void* stream) {
  LPFA_CHECK_ARG(flops_per_s != nullptr);
  *flops_per_s = 0.0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int nsm = num_sms();
  // more than half of an SM's shared memory: one CTA per SM, so no two CTAs
  // queue for the 512 TMEM columns of one SM
  const int smem = 120 * 1024;
  static_assert(kPSmem + 1024 <= 120 * 1024, "operands fit");
  lpfa_status st = set_max_dynamic_smem(reinterpret_cast<const void*>(&mma_peak_kernel), smem);
  if (st != LPFA_OK) return st;
  const uint32_t zero[4] = {0, 0, 0, 0};
  LPFA_CHECK_CUDA(cudaMemcpyToSymbolAsync(g_peak_err, zero, sizeof(zero), 0,
                                          cudaMemcpyHostToDevice, cs));
  constexpr int kWarm = 4096, kIters = 65536;      // ~17 ms timed at 2 GHz
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  LPFA_CHECK_CUDA(cudaEventCreate(&e0));
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return LPFA_ERR_CUDA;
  }
  float ms = 0.f;
  cudaError_t e = cudaSuccess;
  mma_peak_kernel<<<nsm, kPThreads, smem, cs>>>(kWarm);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaEventRecord(e0, cs);
  if (e == cudaSuccess) {
    mma_peak_kernel<<<nsm, kPThreads, smem, cs>>>(kIters);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventRecord(e1, cs);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  LPFA_CHECK_CUDA(e);
  uint32_t err[4] = {0, 0, 0, 0};
  LPFA_CHECK_CUDA(cudaMemcpyFromSymbol(err, g_peak_err, sizeof(err)));
  if (err[0] != 0) return LPFA_ERR_TIMEOUT;
  LPFA_CHECK_ARG(ms > 0.f);
  const double flops = 2.0 * kPM * kPN * kPK * static_cast<double>(kIters) * nsm;
  *flops_per_s = flops / (static_cast<double>(ms) * 1e-3);
  return LPFA_OK;
}
