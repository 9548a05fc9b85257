// Jagged GEMM-Norm backward pieces: 32x32 MX quantization with the payload in
// both physical orientations, and the same fused behind the RMSNorm backward.
//
// "Low Precision Flash Attention 4: End-to-End Block-Scaled Attention for
// Blackwell", paragraph 4 (a jagged GEMM-Norm backward, reported for
// throughput only) and paragraph 2 (fused RMSNorm + Quantize producers with
// dual scale layouts in one pass; jagged inputs keep FP8 data unpadded and pad
// only the scale tiles).  The operation (a reading): over T tokens,
// Y = X W^T, Z = Y r gamma with r = rsqrt(mean(Y^2) + eps); backward
// dY = r (gamma dZ - Y r^2 c), c = mean_n(gamma_n dZ_n Y_n),
// dgamma = sum_t dZ Y r, dX = dY W, dW = dY^T X.  dY, X and W are quantized
// in square 32x32 blocks: the payload is transpose-invariant, so one
// quantization feeds the GEMM over N (dX, payload [T, N]) and the GEMM over T
// (dW, payload [N, T]), each with its own scale arrangement.
//
// Kernel: one CTA per 32-row block, 8 warps; a warp takes 32-column blocks
// in turn with one lane per row.  Per block: the 32x32 maximum by redux.sync,
// E4M3 payloads written row-major (a lane's 32 bytes) and transposed through
// a 1 KB shared tile (a lane writes one column's 32 bytes), the scale code
// into the compact grid and both tensor-core arrangements.  The norm variant
// first forms each row's c_t (4 rows per warp, 16-byte loads, butterfly) and
// writes the per-block column partials of dgamma, which a second kernel sums
// in a fixed order.
#include <cuda_runtime.h>

#include "lpfa_device.cuh"
#include "lpfa_internal.h"

namespace lpfa {
namespace {

struct QuantTArgs {
  const __nv_bfloat16* x;     // plain: [R, C]; norm: Y [R, C]
  const __nv_bfloat16* dz;    // norm: dZ [R, C]
  const __nv_bfloat16* gamma; // norm: [C]
  const float* rstd;          // norm: [R]
  int64_t R, C, Rp;           // Rp = R rounded up to 128
  uint8_t* out;               // [R, C]
  uint8_t* out_t;             // [C, Rp]
  uint8_t* sf;                // [Rp/32, C/32] or null
  uint8_t* sf_mma;            // [Rp/128][C/128][512] rows = R, or null
  uint8_t* sf_mma_t;          // [C/128][Rp/128][512] rows = C, or null
  float* dgamma_part;         // norm: [Rp/32, C]
};

template <bool kNorm>
__global__ void __launch_bounds__(256) quant_t_kernel(const QuantTArgs a) {
  __shared__ float cs[32];                 // norm: c_t of the block's rows
  __shared__ uint8_t tile[8][32][36];      // per warp: transpose staging
  __shared__ float part[8][32][33];        // per warp: dgamma column partials
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rb = blockIdx.x;
  const int64_t r0 = rb * 32;
  const int64_t row = r0 + lane;
  const bool rin = row < a.R;
  float rt = 0.f;
  if constexpr (kNorm) {
    // c_t = (1/C) sum_n gamma_n dZ_tn Y_tn, four rows per warp
    for (int k = 0; k < 4; ++k) {
      const int lr = warp * 4 + k;
      const int64_t t = r0 + lr;
      float acc = 0.f;
      if (t < a.R) {
        for (int64_t c = 8 * lane; c < a.C; c += 256) {
          const uint4 yv = *reinterpret_cast<const uint4*>(a.x + t * a.C + c);
          const uint4 dv = *reinterpret_cast<const uint4*>(a.dz + t * a.C + c);
          const uint4 gv = *reinterpret_cast<const uint4*>(a.gamma + c);
          const __nv_bfloat162* y2 = reinterpret_cast<const __nv_bfloat162*>(&yv);
          const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
          const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 y = __bfloat1622float2(y2[i]), d = __bfloat1622float2(d2[i]),
                         g = __bfloat1622float2(g2[i]);
            acc = fmaf(g.x * d.x, y.x, acc);
            acc = fmaf(g.y * d.y, y.y, acc);
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
      if (lane == 0) cs[lr] = acc / static_cast<float>(a.C);
    }
    __syncthreads();
    rt = rin ? a.rstd[row] : 0.f;
  }
  const float ct = kNorm ? cs[lane] : 0.f;
  const float k2 = rt * rt * ct;
  const int64_t ncb = a.C / 32;
  for (int64_t cb = warp; cb < ncb; cb += 8) {
    const int64_t c0 = cb * 32;
    float v[32];
    float pg[32];
    if (rin) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x + row * a.C + c0);
      if constexpr (kNorm) {
        const uint4* dsrc = reinterpret_cast<const uint4*>(a.dz + row * a.C + c0);
        const uint4* gsrc = reinterpret_cast<const uint4*>(a.gamma + c0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 yv = src[q], dv = dsrc[q], gv = gsrc[q];
          const __nv_bfloat162* y2 = reinterpret_cast<const __nv_bfloat162*>(&yv);
          const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
          const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 y = __bfloat1622float2(y2[i]), d = __bfloat1622float2(d2[i]),
                         g = __bfloat1622float2(g2[i]);
            // dY = r (gamma dZ - Y r^2 c); dgamma term dZ Y r
            v[8 * q + 2 * i] = rt * (g.x * d.x - y.x * k2);
            v[8 * q + 2 * i + 1] = rt * (g.y * d.y - y.y * k2);
            pg[8 * q + 2 * i] = d.x * y.x * rt;
            pg[8 * q + 2 * i + 1] = d.y * y.y * rt;
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 xv = src[q];
          const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 x = __bfloat1622float2(x2[i]);
            v[8 * q + 2 * i] = x.x;
            v[8 * q + 2 * i + 1] = x.y;
          }
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = 0.f;
        pg[i] = 0.f;
      }
    }
    if constexpr (kNorm) {
      // column partials of dgamma over the block's 32 rows, fixed order
#pragma unroll
      for (int i = 0; i < 32; ++i) part[warp][lane][i] = pg[i];
      __syncwarp();
      float s = 0.f;
#pragma unroll 8
      for (int rr = 0; rr < 32; ++rr) s += part[warp][rr][lane];
      a.dgamma_part[rb * a.C + c0 + lane] = s;
      __syncwarp();
    }
    // the 32x32 block's maximum (NaN above Inf as bits), code, payload
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = max(m, __float_as_uint(v[i]) & 0x7FFFFFFFu);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const uint32_t code = e8m0_code_from_amax_bits(m);
    const float inv = inv_scale_from_code(code);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      w[j] = cvt_e4m3x4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv, v[4 * j + 3] * inv);
    if (code == 0xFFu) {
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = 0x7F7F7F7Fu;
    }
    if (rin) {
      uint4* dst = reinterpret_cast<uint4*>(a.out + row * a.C + c0);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    // transposed payload: column c0 + lane, rows r0 .. r0 + 31 (zero past R)
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint32_t*>(&tile[warp][lane][4 * j]) = rin ? w[j] : 0u;
    __syncwarp();
    uint32_t t4[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      t4[j] = static_cast<uint32_t>(tile[warp][4 * j][lane]) |
              (static_cast<uint32_t>(tile[warp][4 * j + 1][lane]) << 8) |
              (static_cast<uint32_t>(tile[warp][4 * j + 2][lane]) << 16) |
              (static_cast<uint32_t>(tile[warp][4 * j + 3][lane]) << 24);
    }
    uint4* tdst = reinterpret_cast<uint4*>(a.out_t + (c0 + lane) * a.Rp + r0);
    tdst[0] = make_uint4(t4[0], t4[1], t4[2], t4[3]);
    tdst[1] = make_uint4(t4[4], t4[5], t4[6], t4[7]);
    __syncwarp();
    // scales: compact; rows = R arrangement (row r0 + lane, block cb); rows =
    // C arrangement (row c0 + lane, block rb)
    const uint8_t c8 = static_cast<uint8_t>(code);
    if (a.sf != nullptr && lane == 0) a.sf[rb * ncb + cb] = c8;
    if (a.sf_mma != nullptr) {
      const int64_t rr = row % 128;
      a.sf_mma[((row / 128) * (a.C / 128) + cb / 4) * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cb % 4] = c8;
    }
    if (a.sf_mma_t != nullptr) {
      const int64_t c = c0 + lane, cc = c % 128;
      a.sf_mma_t[((c / 128) * (a.Rp / 128) + rb / 4) * 512 + (cc % 32) * 16 + (cc / 32) * 4 + rb % 4] = c8;
    }
  }
}

// dgamma[n] = sum over row blocks of the partials, in block order.
__global__ void dgamma_reduce_kernel(const float* __restrict__ part, int64_t nblk, int64_t C,
                                     float* __restrict__ dgamma) {
  const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (n >= C) return;
  float s = 0.f;
  for (int64_t b = 0; b < nblk; ++b) s += part[b * C + n];
  dgamma[n] = s;
}

lpfa_status check_quant_t(const void* x, int64_t rows, int64_t cols, const void* out,
                          const void* out_t, const void* sf_mma, const void* sf_mma_t) {
  LPFA_CHECK_ARG(x != nullptr && out != nullptr && out_t != nullptr);
  LPFA_CHECK_ARG(aligned16(x) && aligned16(out) && aligned16(out_t));
  LPFA_CHECK_ARG(rows >= 0 && rows < (1ll << 31) && cols > 0 && cols % 128 == 0);
  (void)sf_mma;
  (void)sf_mma_t;
  return LPFA_OK;
}

}  // namespace
}  // namespace lpfa

using namespace lpfa;

extern "C" lpfa_status lpfa_mx_quantize_t(const void* x, int64_t rows, int64_t cols, void* out,
                                          void* out_t, void* out_sf, void* out_sf_mma,
                                          void* out_sf_mma_t, void* stream) {
  lpfa_status st = check_quant_t(x, rows, cols, out, out_t, out_sf_mma, out_sf_mma_t);
  if (st != LPFA_OK) return st;
  if (rows == 0) return LPFA_OK;
  QuantTArgs a{};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.R = rows;
  a.C = cols;
  a.Rp = ceil_div(rows, 128) * 128;
  a.out = static_cast<uint8_t*>(out);
  a.out_t = static_cast<uint8_t*>(out_t);
  a.sf = static_cast<uint8_t*>(out_sf);
  a.sf_mma = static_cast<uint8_t*>(out_sf_mma);
  a.sf_mma_t = static_cast<uint8_t*>(out_sf_mma_t);
  quant_t_kernel<false><<<static_cast<unsigned>(a.Rp / 32), 256, 0,
                          static_cast<cudaStream_t>(stream)>>>(a);
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}

extern "C" lpfa_status lpfa_rmsnorm_bwd_mx_quantize(const void* y, const void* dz,
                                                    const void* gamma, const float* rstd,
                                                    int64_t rows, int64_t cols, void* out,
                                                    void* out_t, void* out_sf, void* out_sf_mma,
                                                    void* out_sf_mma_t, float* dgamma_part,
                                                    float* dgamma, void* stream) {
  lpfa_status st = check_quant_t(y, rows, cols, out, out_t, out_sf_mma, out_sf_mma_t);
  if (st != LPFA_OK) return st;
  LPFA_CHECK_ARG(dz != nullptr && gamma != nullptr && rstd != nullptr && aligned16(dz) &&
                 aligned16(gamma) && dgamma_part != nullptr && dgamma != nullptr);
  if (rows == 0) return LPFA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  QuantTArgs a{};
  a.x = static_cast<const __nv_bfloat16*>(y);
  a.dz = static_cast<const __nv_bfloat16*>(dz);
  a.gamma = static_cast<const __nv_bfloat16*>(gamma);
  a.rstd = rstd;
  a.R = rows;
  a.C = cols;
  a.Rp = ceil_div(rows, 128) * 128;
  a.out = static_cast<uint8_t*>(out);
  a.out_t = static_cast<uint8_t*>(out_t);
  a.sf = static_cast<uint8_t*>(out_sf);
  a.sf_mma = static_cast<uint8_t*>(out_sf_mma);
  a.sf_mma_t = static_cast<uint8_t*>(out_sf_mma_t);
  a.dgamma_part = dgamma_part;
  quant_t_kernel<true><<<static_cast<unsigned>(a.Rp / 32), 256, 0, cs>>>(a);
  LPFA_CHECK_CUDA(cudaGetLastError());
  dgamma_reduce_kernel<<<static_cast<unsigned>(ceil_div(cols, 256)), 256, 0, cs>>>(
      dgamma_part, a.Rp / 32, cols, dgamma);
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}
