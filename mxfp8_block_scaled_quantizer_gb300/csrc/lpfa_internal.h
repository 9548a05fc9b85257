// Host-side helpers shared by the lpfa translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "../../include/lpfa.h"

namespace lpfa {

#define LPFA_CHECK_ARG(cond)                                             \
  do {                                                                   \
    if (!(cond)) {                                                       \
      if (::lpfa::debug_enabled())                                       \
        std::fprintf(stderr, "lpfa: invalid argument: %s (%s:%d)\n",     \
                     #cond, __FILE__, __LINE__);                         \
      return LPFA_ERR_INVALID_ARG;                                       \
    }                                                                    \
  } while (0)

#define LPFA_CHECK_CUDA(expr)                                            \
  do {                                                                   \
    cudaError_t e_ = (expr);                                             \
    if (e_ != cudaSuccess) {                                             \
      if (::lpfa::debug_enabled())                                       \
        std::fprintf(stderr, "lpfa: CUDA error %s at %s:%d\n",           \
                     cudaGetErrorString(e_), __FILE__, __LINE__);        \
      return LPFA_ERR_CUDA;                                              \
    }                                                                    \
  } while (0)

bool debug_enabled();

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Device view of lpfa_seqs (plain values; the kernels look sequences up).
struct SeqView {
  const int32_t* cu_seqlens;  // nullptr: dense
  const int32_t* cu_sf_rows;
  int32_t nseq;
  int32_t seqlen;       // dense length (or max length)
  int32_t pad_seqlen;   // dense: ceil(seqlen/128)*128
  int64_t total_tokens;
  int64_t total_sf_rows;
};

lpfa_status make_seq_view(const lpfa_seqs* s, SeqView* out);

// Validates an attention descriptor and builds its sequence view.
lpfa_status validate_attn(const lpfa_attn_desc* desc, SeqView* sv);
// The bf16 forward with two query tiles in flight (fwd_pair.cu), called by
// lpfa_fwd_bf16 after validation; err is the workspace's error word.
lpfa_status launch_fwd_pair_bf16(const lpfa_attn_desc* desc, const SeqView& sv,
                                 const void* q, const void* k, const void* v, void* o,
                                 float* lse, uint32_t* err, cudaStream_t cs);

// Number of SMs of the current device (cached per device).
int num_sms();

// cudaFuncAttributeMaxDynamicSharedMemorySize for a kernel on the current
// device, set once per (kernel, device).
lpfa_status set_max_dynamic_smem(const void* func, int bytes);

// Clusters of `func` (compile-time cluster dimensions) resident at once on
// the current device with this block size and dynamic shared memory; 0 if
// the query fails.  Cached per (kernel, device).
int max_active_clusters(const void* func, int threads, int smem_bytes);

// cuTensorMapEncodeTiled through the driver entry point.
lpfa_status encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype,
                        uint32_t rank, const void* base, const uint64_t* dims,
                        const uint64_t* strides_bytes, const uint32_t* box,
                        CUtensorMapSwizzle swizzle);

}  // namespace lpfa
