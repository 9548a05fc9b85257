// Device-side sequence lookup shared by the kernels.
#pragma once

#include "lpfa_internal.h"

namespace lpfa {

struct SeqInfo {
  int64_t start;     // first token
  int32_t len;       // tokens
  int64_t sf_start;  // first padded scale row (multiple of 128)
};

__device__ __forceinline__ SeqInfo seq_info(const SeqView& v, int s) {
  SeqInfo r;
  if (v.cu_seqlens == nullptr) {
    r.start = static_cast<int64_t>(s) * v.seqlen;
    r.len = v.seqlen;
    r.sf_start = static_cast<int64_t>(s) * v.pad_seqlen;
  } else {
    int32_t a = __ldg(v.cu_seqlens + s);
    r.start = a;
    r.len = __ldg(v.cu_seqlens + s + 1) - a;
    r.sf_start = __ldg(v.cu_sf_rows + s);
  }
  return r;
}

// Sequence owning padded scale row `pr` (largest s with sf_start[s] <= pr).
__device__ __forceinline__ int seq_of_sf_row(const SeqView& v, int64_t pr) {
  if (v.cu_seqlens == nullptr) return static_cast<int>(pr / v.pad_seqlen);
  int lo = 0, hi = v.nseq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(v.cu_sf_rows + mid) <= pr) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace lpfa
