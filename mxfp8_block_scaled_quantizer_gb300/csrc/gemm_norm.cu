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
// Kernels: the quantizer takes 32-row x 64-column chunks per warp with
// coalesced 16-byte loads (emit_chunk below); the RMSNorm backward first
// forms c_t per row (a warp per row), then computes dY in the quantizer's
// chunk layout together with the per-block column partials of dgamma, which
// a third kernel sums in a fixed order.
#include <cuda_runtime.h>

#include "lpfa_device.cuh"
#include "lpfa_internal.h"

namespace lpfa {
namespace {

// ---------------------------------------------------------------------------
// Coalesced form.  A warp takes a 32-row x 64-column chunk (two 32x32
// blocks): lane l holds v[i][k] = element (row r0 + 4i + l/8, column
// c0 + 8(l%8) + k), so each load instruction reads four whole 128-byte row
// segments.  The block maximum is a 4-step butterfly over the block's 8
// lanes; the transposed payload goes through a 32 x 68-byte shared tile,
// read back as 32-bit words and transposed 4x4 bytes at a time in registers
// (a lane writes 16 rows of 4 columns as four 16-byte stores).
struct QtOut {
  uint8_t* out;       // [R, C]
  uint8_t* out_t;     // [C, Rp]
  uint8_t* sf;        // [Rp/32, C/32] or null
  uint8_t* sf_mma;    // rows = R: [Rp/128][C/128][512] or null
  uint8_t* sf_mma_t;  // rows = C: [C/128][Rp/128][512] or null
  int64_t R, C, Rp;
};

constexpr int kTileRow = 68;   // bytes per row of the transpose tile

__device__ __forceinline__ void emit_chunk(const QtOut& o, const float (&v)[8][8], int64_t r0,
                                           int64_t c0, int lane, uint8_t* tile) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < 8; ++k) m = max(m, __float_as_uint(v[i][k]) & 0x7FFFFFFFu);
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
  const uint32_t code = e8m0_code_from_amax_bits(m);
  const float inv = inv_scale_from_code(code);
  const int g = lane & 7, rs = lane >> 3;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t w0 = cvt_e4m3x4(v[i][0] * inv, v[i][1] * inv, v[i][2] * inv, v[i][3] * inv);
    uint32_t w1 = cvt_e4m3x4(v[i][4] * inv, v[i][5] * inv, v[i][6] * inv, v[i][7] * inv);
    if (code == 0xFFu) w0 = w1 = 0x7F7F7F7Fu;
    const int rl = 4 * i + rs;
    const int64_t row = r0 + rl;
    if (row < o.R) *reinterpret_cast<uint2*>(o.out + row * o.C + c0 + 8 * g) = make_uint2(w0, w1);
    uint32_t* tw = reinterpret_cast<uint32_t*>(tile + rl * kTileRow + 8 * g);
    tw[0] = w0;
    tw[1] = w1;
  }
  __syncwarp();
  // transposed payload: lane -> columns 4 cq .. 4 cq + 3, rows 16 rh ..
  const int cq = lane & 15, rh = lane >> 4;
  uint32_t wr[16];
#pragma unroll
  for (int j = 0; j < 16; ++j)
    wr[j] = *reinterpret_cast<const uint32_t*>(tile + (16 * rh + j) * kTileRow + 4 * cq);
  uint32_t col[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const uint32_t t0 = __byte_perm(wr[4 * a], wr[4 * a + 1], 0x5140);
    const uint32_t t1 = __byte_perm(wr[4 * a + 2], wr[4 * a + 3], 0x5140);
    const uint32_t t2 = __byte_perm(wr[4 * a], wr[4 * a + 1], 0x7362);
    const uint32_t t3 = __byte_perm(wr[4 * a + 2], wr[4 * a + 3], 0x7362);
    col[0][a] = __byte_perm(t0, t1, 0x5410);
    col[1][a] = __byte_perm(t0, t1, 0x7632);
    col[2][a] = __byte_perm(t2, t3, 0x5410);
    col[3][a] = __byte_perm(t2, t3, 0x7632);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(o.out_t + (c0 + 4 * cq + k) * o.Rp + r0 + 16 * rh) =
        make_uint4(col[k][0], col[k][1], col[k][2], col[k][3]);
  __syncwarp();
  // scales of the two blocks
  const uint32_t code0 = __shfl_sync(0xFFFFFFFFu, code, 0);
  const uint32_t code1 = __shfl_sync(0xFFFFFFFFu, code, 4);
  const int64_t rb = r0 / 32, cb0 = c0 / 32;
  if (o.sf != nullptr && lane < 2) o.sf[rb * (o.C / 32) + cb0 + lane] = lane ? code1 : code0;
  if (o.sf_mma != nullptr) {
    const int64_t row = r0 + lane, rr = row % 128;
    // cb0 is even: the two blocks' bytes are adjacent
    *reinterpret_cast<uint16_t*>(o.sf_mma + ((row / 128) * (o.C / 128) + cb0 / 4) * 512 +
                                 (rr % 32) * 16 + (rr / 32) * 4 + cb0 % 4) =
        static_cast<uint16_t>(code0 | code1 << 8);
  }
  if (o.sf_mma_t != nullptr) {
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      const int64_t c = c0 + 32 * bb + lane, cc = c % 128;
      o.sf_mma_t[((c / 128) * (o.Rp / 128) + rb / 4) * 512 + (cc % 32) * 16 + (cc / 32) * 4 + rb % 4] =
          static_cast<uint8_t>(bb ? code1 : code0);
    }
  }
}

__device__ __forceinline__ void unpack8(const uint4 p, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&p);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __bfloat1622float2(h[j]);
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}

// Plain quantization: CTA = 4 warps over one 32-row block and 256 columns.
__global__ void __launch_bounds__(128) quant_t64_kernel(const __nv_bfloat16* __restrict__ x,
                                                        const QtOut o) {
  __shared__ __align__(16) uint8_t tiles[4][32 * kTileRow];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.y) * 4 + warp) * 64;
  if (c0 >= o.C) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32;
  float v[8][8];
  uint4 raw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = r0 + 4 * i + (lane >> 3);
    raw[i] = row < o.R ? *reinterpret_cast<const uint4*>(x + row * o.C + c0 + 8 * (lane & 7))
                       : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) unpack8(raw[i], v[i]);
  emit_chunk(o, v, r0, c0, lane, tiles[warp]);
}

// c_t = (1/C) sum_n gamma_n dZ_tn Y_tn, one warp per row: lane l takes the
// 8-element chunks at 8 l + 256 j (fused multiply-adds in j order), then a
// 5-level butterfly.
__global__ void __launch_bounds__(256) norm_ct_kernel(const __nv_bfloat16* __restrict__ y,
                                                      const __nv_bfloat16* __restrict__ dz,
                                                      const __nv_bfloat16* __restrict__ gamma,
                                                      int64_t R, int64_t C, float* __restrict__ ct) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (row >= R) return;
  float acc = 0.f;
#pragma unroll 4
  for (int64_t c = 8 * lane; c < C; c += 256) {
    float yv[8], dv[8], gv[8];
    unpack8(*reinterpret_cast<const uint4*>(y + row * C + c), yv);
    unpack8(*reinterpret_cast<const uint4*>(dz + row * C + c), dv);
    unpack8(*reinterpret_cast<const uint4*>(gamma + c), gv);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = fmaf(gv[j] * dv[j], yv[j], acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (lane == 0) ct[row] = acc / static_cast<float>(C);
}

// dY = r (gamma dZ - Y r^2 c) in the quantizer's chunk layout (CTA = 4 warps
// over one 32-row block and 256 columns), the block's dgamma column partials
// (8 rows per lane, then the four row groups: a fixed order) and the 32x32
// quantization of dY.
__global__ void __launch_bounds__(128) norm_quant_kernel(const __nv_bfloat16* __restrict__ y,
                                                         const __nv_bfloat16* __restrict__ dz,
                                                         const __nv_bfloat16* __restrict__ gamma,
                                                         const float* __restrict__ rstd,
                                                         const float* __restrict__ ct,
                                                         float* __restrict__ dgamma_part,
                                                         const QtOut o) {
  __shared__ __align__(16) uint8_t tiles[4][32 * kTileRow];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.y) * 4 + warp) * 64;
  if (c0 >= o.C) return;
  const int64_t rb = blockIdx.x, r0 = rb * 32;
  const int cl = 8 * (lane & 7);
  float gv[8];
  unpack8(*reinterpret_cast<const uint4*>(gamma + c0 + cl), gv);
  uint4 ry[8], rd[8];
  float rt[8], k2[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = r0 + 4 * i + (lane >> 3);
    const bool in = row < o.R;
    ry[i] = in ? *reinterpret_cast<const uint4*>(y + row * o.C + c0 + cl) : make_uint4(0u, 0u, 0u, 0u);
    rd[i] = in ? *reinterpret_cast<const uint4*>(dz + row * o.C + c0 + cl) : make_uint4(0u, 0u, 0u, 0u);
    rt[i] = in ? rstd[row] : 0.f;
    k2[i] = in ? rt[i] * rt[i] * ct[row] : 0.f;
  }
  float v[8][8];
  float pg[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float yv[8], dv[8];
    unpack8(ry[i], yv);
    unpack8(rd[i], dv);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      // dY = r (gamma dZ - Y r^2 c); dgamma term dZ Y r
      v[i][k] = rt[i] * (gv[k] * dv[k] - yv[k] * k2[i]);
      pg[k] += dv[k] * yv[k] * rt[i];
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    pg[k] += __shfl_xor_sync(0xFFFFFFFFu, pg[k], 8);
    pg[k] += __shfl_xor_sync(0xFFFFFFFFu, pg[k], 16);
  }
  if (lane < 8) {
    float4* dst = reinterpret_cast<float4*>(dgamma_part + rb * o.C + c0 + cl);
    dst[0] = make_float4(pg[0], pg[1], pg[2], pg[3]);
    dst[1] = make_float4(pg[4], pg[5], pg[6], pg[7]);
  }
  emit_chunk(o, v, r0, c0, lane, tiles[warp]);
}

// dgamma[n] = sum over row blocks of the partials: CTA per 32 columns, warp
// w sums blocks w, w + 8, ... (8 loads in flight per lane), then the eight
// warp sums are added in warp order (a fixed order).
__global__ void __launch_bounds__(256) dgamma_reduce_kernel(const float* __restrict__ part,
                                                            int64_t nblk, int64_t C,
                                                            float* __restrict__ dgamma) {
  __shared__ float ws[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  float s = 0.f;
  int64_t b = warp;
  for (; b + 56 < nblk; b += 64) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = part[(b + 8 * j) * C + n];
#pragma unroll
    for (int j = 0; j < 8; ++j) s += v[j];
  }
  for (; b < nblk; b += 8) s += part[b * C + n];
  ws[warp][lane] = s;
  __syncthreads();
  if (warp == 0) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += ws[w][lane];
    dgamma[n] = t;
  }
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
  const int64_t Rp = ceil_div(rows, 128) * 128;
  const QtOut o{static_cast<uint8_t*>(out),        static_cast<uint8_t*>(out_t),
                static_cast<uint8_t*>(out_sf),     static_cast<uint8_t*>(out_sf_mma),
                static_cast<uint8_t*>(out_sf_mma_t), rows, cols, Rp};
  const dim3 grid(static_cast<unsigned>(Rp / 32), static_cast<unsigned>(ceil_div(cols, 256)));
  quant_t64_kernel<<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), o);
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
                 aligned16(gamma) && aligned16(dgamma_part) && dgamma != nullptr);
  if (rows == 0) return LPFA_OK;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int64_t Rp = ceil_div(rows, 128) * 128;
  const auto* y16 = static_cast<const __nv_bfloat16*>(y);
  const auto* dz16 = static_cast<const __nv_bfloat16*>(dz);
  const auto* g16 = static_cast<const __nv_bfloat16*>(gamma);
  // scratch: the dgamma partials [Rp/32, C], then c_t [Rp]
  float* ct = dgamma_part + (Rp / 32) * cols;
  norm_ct_kernel<<<static_cast<unsigned>(ceil_div(rows, 8)), 256, 0, cs>>>(y16, dz16, g16, rows,
                                                                          cols, ct);
  LPFA_CHECK_CUDA(cudaGetLastError());
  const QtOut o{static_cast<uint8_t*>(out),        static_cast<uint8_t*>(out_t),
                static_cast<uint8_t*>(out_sf),     static_cast<uint8_t*>(out_sf_mma),
                static_cast<uint8_t*>(out_sf_mma_t), rows, cols, Rp};
  const dim3 grid(static_cast<unsigned>(Rp / 32), static_cast<unsigned>(ceil_div(cols, 256)));
  norm_quant_kernel<<<grid, 128, 0, cs>>>(y16, dz16, g16, rstd, ct, dgamma_part, o);
  LPFA_CHECK_CUDA(cudaGetLastError());
  dgamma_reduce_kernel<<<static_cast<unsigned>(cols / 32), 256, 0, cs>>>(dgamma_part, Rp / 32,
                                                                         cols, dgamma);
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}
