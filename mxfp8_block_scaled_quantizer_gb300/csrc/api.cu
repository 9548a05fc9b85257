// Library-wide entry points: status strings, device gate, varlen scale-row
// offsets, error-word check, and host helpers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>
#include <tuple>
#include <vector>

#include "lpfa_internal.h"

namespace lpfa {

bool debug_enabled() {
  static int v = [] {
    const char* e = std::getenv("LPFA_DEBUG");
    return (e != nullptr && e[0] != '0') ? 1 : 0;
  }();
  return v != 0;
}

namespace {
std::mutex g_device_cache_mutex;
}  // namespace

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(g_device_cache_mutex);
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

// A kernel's dynamic shared-memory opt-in belongs to the device that is
// current when it is set, so it is recorded per (kernel, device, size).
lpfa_status set_max_dynamic_smem(const void* func, int bytes) {
  static std::vector<std::tuple<const void*, int, int>> done;
  int dev = 0;
  LPFA_CHECK_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_device_cache_mutex);
  for (const auto& t : done)
    if (std::get<0>(t) == func && std::get<1>(t) == dev && std::get<2>(t) >= bytes)
      return LPFA_OK;
  LPFA_CHECK_CUDA(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  done.emplace_back(func, dev, bytes);
  return LPFA_OK;
}

// Clusters of a kernel with compile-time cluster dimensions that can be
// resident at once on the current device, recorded per (kernel, device).
int max_active_clusters(const void* func, int threads, int smem_bytes) {
  static std::vector<std::tuple<const void*, int, int>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_device_cache_mutex);
  for (const auto& t : done)
    if (std::get<0>(t) == func && std::get<1>(t) == dev) return std::get<2>(t);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  done.emplace_back(func, dev, n);
  return n;
}

lpfa_status make_seq_view(const lpfa_seqs* s, SeqView* out) {
  LPFA_CHECK_ARG(s != nullptr && out != nullptr);
  LPFA_CHECK_ARG(s->nseq >= 1 && s->nseq <= (1 << 20));
  LPFA_CHECK_ARG(s->seqlen >= 0 && s->seqlen <= (1 << 24));
  LPFA_CHECK_ARG((s->cu_seqlens == nullptr) == (s->cu_sf_rows == nullptr));
  LPFA_CHECK_ARG(s->total_tokens >= 0 && s->total_tokens < (1ll << 31));
  out->cu_seqlens = s->cu_seqlens;
  out->cu_sf_rows = s->cu_sf_rows;
  out->nseq = static_cast<int32_t>(s->nseq);
  out->seqlen = static_cast<int32_t>(s->seqlen);
  out->pad_seqlen = static_cast<int32_t>(ceil_div(s->seqlen, 128) * 128);
  out->total_tokens = s->total_tokens;
  out->total_sf_rows = s->total_sf_rows;
  if (s->cu_seqlens == nullptr) {
    LPFA_CHECK_ARG(s->seqlen >= 1);
    LPFA_CHECK_ARG(s->total_tokens == s->nseq * s->seqlen);
    LPFA_CHECK_ARG(s->total_sf_rows == s->nseq * out->pad_seqlen);
  } else {
    LPFA_CHECK_ARG(s->total_sf_rows % 128 == 0);
    LPFA_CHECK_ARG(s->total_sf_rows >= s->total_tokens);
  }
  return LPFA_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

// The driver function is fetched through the runtime, so the library has no
// link-time dependency on libcuda (it loads on machines without a driver).
static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

lpfa_status encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype,
                        uint32_t rank, const void* base, const uint64_t* dims,
                        const uint64_t* strides_bytes, const uint32_t* box,
                        CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return LPFA_ERR_CUDA;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (uint32_t i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dtype, rank, const_cast<void*>(base), gdim, gstride,
                  bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (debug_enabled()) std::fprintf(stderr, "lpfa: tensor map encode %d\n", (int)r);
    return LPFA_ERR_INVALID_ARG;
  }
  return LPFA_OK;
}

// cu_sf_rows[s] = sum_{t<s} ceil(L_t/128)*128, one block, chunked scan.
__global__ void varlen_sf_rows_kernel(const int32_t* __restrict__ cu,
                                      int32_t nseq, int32_t* __restrict__ out) {
  __shared__ int32_t buf[1024];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) {
    carry = 0;
    out[0] = 0;
  }
  __syncthreads();
  for (int32_t base = 0; base < nseq; base += 1024) {
    int32_t i = base + static_cast<int32_t>(threadIdx.x);
    int32_t v = 0;
    if (i < nseq) {
      int32_t len = cu[i + 1] - cu[i];
      v = ((len + 127) / 128) * 128;
    }
    buf[threadIdx.x] = v;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      int32_t add = threadIdx.x >= static_cast<unsigned>(off) ? buf[threadIdx.x - off] : 0;
      __syncthreads();
      buf[threadIdx.x] += add;
      __syncthreads();
    }
    if (i < nseq) out[i + 1] = carry + buf[threadIdx.x];
    __syncthreads();
    if (threadIdx.x == 1023) carry += buf[1023];
    __syncthreads();
  }
}

}  // namespace lpfa

using namespace lpfa;

extern "C" const char* lpfa_status_string(lpfa_status s) {
  switch (s) {
    case LPFA_OK: return "LPFA_OK";
    case LPFA_ERR_INVALID_ARG: return "LPFA_ERR_INVALID_ARG";
    case LPFA_ERR_UNSUPPORTED: return "LPFA_ERR_UNSUPPORTED";
    case LPFA_ERR_CUDA: return "LPFA_ERR_CUDA";
    case LPFA_ERR_TIMEOUT: return "LPFA_ERR_TIMEOUT";
  }
  return "LPFA_ERR_UNKNOWN";
}

extern "C" int lpfa_version(void) { return LPFA_VERSION; }

extern "C" lpfa_status lpfa_device_supported(void) {
  int dev = 0, major = 0;
  LPFA_CHECK_CUDA(cudaGetDevice(&dev));
  LPFA_CHECK_CUDA(
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  return major == 10 ? LPFA_OK : LPFA_ERR_UNSUPPORTED;
}

extern "C" lpfa_status lpfa_varlen_sf_rows(const int32_t* cu_seqlens,
                                           int64_t nseq, int32_t* cu_sf_rows,
                                           void* stream) {
  LPFA_CHECK_ARG(cu_seqlens != nullptr && cu_sf_rows != nullptr);
  LPFA_CHECK_ARG(nseq >= 1 && nseq <= (1 << 20));
  varlen_sf_rows_kernel<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(
      cu_seqlens, static_cast<int32_t>(nseq), cu_sf_rows);
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}

extern "C" lpfa_status lpfa_check(const void* workspace, void* stream) {
  LPFA_CHECK_ARG(workspace != nullptr);
  uint32_t word[4] = {0, 0, 0, 0};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LPFA_CHECK_CUDA(cudaStreamSynchronize(st));
  LPFA_CHECK_CUDA(cudaMemcpy(word, workspace, sizeof(word),
                             cudaMemcpyDeviceToHost));
  if (word[0] != 0) {
    if (debug_enabled())
      std::fprintf(stderr, "lpfa: kernel error bits 0x%x site %u block %u\n",
                   word[0], word[1], word[2]);
    return LPFA_ERR_TIMEOUT;
  }
  return LPFA_OK;
}
