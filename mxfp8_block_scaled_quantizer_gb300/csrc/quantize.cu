// MX quantizer: bf16 -> E4M3 payload + E8M0 scales (compact and tensor-core
// layouts).
//
// Rule ("Low-Precision FlashAttention-4 ...", "Understanding OCP MXFP8
// Microscaling on Blackwell"; block shapes from "Low Precision Flash
// Attention 4 ...", paragraphs 2-3): per block, amax = max|x|, scale code =
// floor(log2 amax) - 8 + 127 clamped at 0 (taken from amax's exponent bits),
// payload = RNE-satfinite E4M3 of x * 2^-e.
//
// One warp owns a 32-token x head_dim block of one head; head_dim/32 lanes
// share each token row.  The block shape only changes how amax is grouped:
// per lane row (1x32), per channel across the block's tokens (32x1), or the
// whole 32x32 tile (32x32).  The kernel is a single pass over HBM: 2 bytes read and
// 1 + 1/32 (+1/32 per extra scale layout) bytes written per element.
#include <cuda_runtime.h>

#include "lpfa_device.cuh"
#include "lpfa_internal.h"
#include "lpfa_seq.cuh"

namespace lpfa {
namespace {

struct QuantArgs {
  SeqView seqs;
  const __nv_bfloat16* x;
  uint8_t* out;
  uint8_t* sf;        // compact
  uint8_t* sf_mma;    // K-major tensor-core layout (32X1: contraction over tokens)
  uint8_t* sf_mma_t;  // 32X32 only: contraction over tokens
  int32_t H;
  int32_t D;
  int64_t ntiles;     // (Tp/32) * H * (D/32)
};

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ uint32_t abs_bits(float f) {
  return __float_as_uint(f) & 0x7FFFFFFFu;
}

// Quantize 32 floats with their scale codes into 32 element bytes (8 words).
template <int kFmt = kFmtE4M3>
__device__ __forceinline__ void quant_row(const float (&f)[32],
                                          const uint32_t (&code)[32],
                                          uint32_t (&w)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a = f[4 * j + 0] * inv_scale_from_code(code[4 * j + 0]);
    float b = f[4 * j + 1] * inv_scale_from_code(code[4 * j + 1]);
    float c = f[4 * j + 2] * inv_scale_from_code(code[4 * j + 2]);
    float d = f[4 * j + 3] * inv_scale_from_code(code[4 * j + 3]);
    w[j] = cvt_x4<kFmt>(a, b, c, d);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (code[4 * j + q] == 0xFFu)
        w[j] = (w[j] & ~(0xFFu << (8 * q))) | (fmt_nan_byte<kFmt>() << (8 * q));
  }
}

// As quant_row with the codes of the 32 values packed four to a word
// (element 4i + q takes byte q of cw[i]).
template <int kFmt = kFmtE4M3>
__device__ __forceinline__ void quant_row_packed(const float (&f)[32], const uint32_t (&cw)[8],
                                                 uint32_t (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float x[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) x[q] = f[4 * i + q] * inv_scale_from_code((cw[i] >> (8 * q)) & 0xFFu);
    w[i] = cvt_x4<kFmt>(x[0], x[1], x[2], x[3]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (((cw[i] >> (8 * q)) & 0xFFu) == 0xFFu)
        w[i] = (w[i] & ~(0xFFu << (8 * q))) | (fmt_nan_byte<kFmt>() << (8 * q));
  }
}

// bf16 pair -> two floats
__device__ __forceinline__ void unpack_row(const uint4 (&v)[4], float (&f)[32]) {
  const uint32_t* u = reinterpret_cast<const uint32_t*>(v);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    f[2 * i + 0] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// One warp per (32-row padded block rb, head h).  kNcb = head_dim / 32
// consecutive lanes share a token row (lane = t * kNcb + cb: channel block
// cb of token t), so one load instruction of the warp reads whole 2*head_dim
// byte head rows of 32 / kNcb tokens; kNcb loads cover the 32 tokens.
// (Token-per-lane loads, 64 bytes at the token stride, reach ~2/3 of the
// bandwidth of these.)  Block maxima over tokens reduce across the lanes
// that share cb.
template <int kMode, int kNcb, int kFmt>  // mode 0: 1x32, 1: 32x1, 2: 32x32
__global__ void __launch_bounds__(kWarpsPerBlock * 32, 2)   // >= 16 warps per SM
    mx_quantize_kernel(const QuantArgs a) {
  constexpr int kTpl = 32 / kNcb;                  // tokens per load
  const int lane = threadIdx.x & 31;
  const int cb = lane % kNcb, t = lane / kNcb;
  const int64_t task = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t ntasks = (a.seqs.total_sf_rows / 32) * a.H;
  if (task >= ntasks) return;
  const int h = static_cast<int>(task % a.H);
  const int64_t rb = task / a.H;
  const int64_t pr0 = rb * 32;                     // first padded row of the block
  const int sq = seq_of_sf_row(a.seqs, pr0);
  const SeqInfo si = seq_info(a.seqs, sq);
  const int64_t off = pr0 - si.sf_start;           // token offset in sequence
  const int64_t nvalid64 = static_cast<int64_t>(si.len) - off;
  const int nvalid = nvalid64 < 0 ? 0 : (nvalid64 > 32 ? 32 : static_cast<int>(nvalid64));
  const int64_t tile_base = ((rb >> 2) * a.H + h) * 512;   // 512-byte scale tile
  const int kb_row = static_cast<int>(rb & 3);     // token block within the tile

  // ---- all rows of this lane in flight at once
  uint4 v[kNcb][4];
#pragma unroll
  for (int r = 0; r < kNcb; ++r) {
    const int row = r * kTpl + t;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[r][i] = make_uint4(0, 0, 0, 0);
    if (row < nvalid) {
      const uint4* src = reinterpret_cast<const uint4*>(
          a.x + ((si.start + off + row) * a.H + h) * a.D + 32 * cb);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[r][i] = __ldcs(src + i);
    }
  }

  uint32_t bcode = 0;                              // 32x32: the block's code
  uint32_t cw[8];                                  // 32x1: codes of cb's 32 channels, 4 per word
  if (kMode == 2) {
    // maximum over this lane's rows, then over the lanes sharing cb
    uint32_t m = 0;
#pragma unroll
    for (int r = 0; r < kNcb; ++r) {
      const uint32_t* u = reinterpret_cast<const uint32_t*>(v[r]);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        m = max(m, max((u[i] << 16) & 0x7FFFFFFFu, u[i] & 0x7FFF0000u));
    }
#pragma unroll
    for (int x = kNcb; x < 32; x <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, x));
    bcode = scale_code_from_amax_bits<kFmt>(m);
  } else if (kMode == 1) {
    // per channel: maximum over this lane's rows, then over the lanes
    // sharing cb; four channels at a time keeps the live state small
#pragma unroll
    for (int g4 = 0; g4 < 8; ++g4) {
      uint32_t q[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int r = 0; r < kNcb; ++r) {
        const uint32_t* u = reinterpret_cast<const uint32_t*>(v[r]);
        const uint32_t lo = u[2 * g4], hi = u[2 * g4 + 1];   // channels 4 g4 .. 4 g4 + 3
        q[0] = max(q[0], (lo << 16) & 0x7FFFFFFFu);
        q[1] = max(q[1], lo & 0x7FFF0000u);
        q[2] = max(q[2], (hi << 16) & 0x7FFFFFFFu);
        q[3] = max(q[3], hi & 0x7FFF0000u);
      }
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t qq = q[k];
#pragma unroll
        for (int x = kNcb; x < 32; x <<= 1) qq = max(qq, __shfl_xor_sync(0xFFFFFFFFu, qq, x));
        word |= scale_code_from_amax_bits<kFmt>(qq) << (8 * k);
      }
      cw[g4] = word;
    }
  }

  // ---- payload and per-row scales
#pragma unroll
  for (int r = 0; r < kNcb; ++r) {
    const int row = r * kTpl + t;                  // token row within the block
    const bool valid = row < nvalid;
    const int64_t tok = si.start + off + row;
    float f[32];
    unpack_row(v[r], f);
    uint32_t code[32];
    if (kMode == 0) {
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) m = max(m, abs_bits(f[j]));
      const uint32_t c = scale_code_from_amax_bits<kFmt>(m);
#pragma unroll
      for (int j = 0; j < 32; ++j) code[j] = c;
    } else if (kMode == 2) {
#pragma unroll
      for (int j = 0; j < 32; ++j) code[j] = bcode;
    }
    if (valid) {
      uint32_t w[8];
      if (kMode == 1) quant_row_packed<kFmt>(f, cw, w);
      else quant_row<kFmt>(f, code, w);
      uint4* dst = reinterpret_cast<uint4*>(a.out + (tok * a.H + h) * a.D + 32 * cb);
      __stcs(dst + 0, make_uint4(w[0], w[1], w[2], w[3]));
      __stcs(dst + 1, make_uint4(w[4], w[5], w[6], w[7]));
    }
    if (kMode != 1) {
      // this row's kNcb codes gathered into one word by the cb = 0 lane:
      // compact [tok][h][cb] bytes and tensor-core bytes
      // row * 16 + kb_row * 4 + cb are both contiguous in cb
      const uint32_t c = (kMode == 0 && !valid) ? 0u : code[0];
      uint32_t word = c;
#pragma unroll
      for (int k = 1; k < kNcb; ++k)
        word |= __shfl_down_sync(0xFFFFFFFFu, c, k) << (8 * k);
      if (cb == 0) {
        if (a.sf_mma != nullptr) {
          const uint32_t wm = (kMode == 2 && !valid) ? 0u : word;
          uint8_t* d = a.sf_mma + tile_base + row * 16 + kb_row * 4;
          if (kNcb == 4) *reinterpret_cast<uint32_t*>(d) = wm;
          else *reinterpret_cast<uint16_t*>(d) = static_cast<uint16_t>(wm);
        }
        if (kMode == 0 && a.sf != nullptr && valid) {
          uint8_t* d = a.sf + (tok * a.H + h) * kNcb;
          if (kNcb == 4) *reinterpret_cast<uint32_t*>(d) = word;
          else *reinterpret_cast<uint16_t*>(d) = static_cast<uint16_t>(word);
        }
      }
      if (kMode == 2 && a.sf_mma_t != nullptr)
        a.sf_mma_t[tile_base + row * 16 + cb * 4 + kb_row] = static_cast<uint8_t>(bcode);
    }
  }

  // ---- block-level scales
  if (kMode == 2 && a.sf != nullptr && t == 0)
    a.sf[(rb * a.H + h) * kNcb + cb] = static_cast<uint8_t>(bcode);
  if (kMode == 1) {
    // channel 32 cb + j of the block: the kTpl lanes of cb each write 32 /
    // kTpl consecutive channels
    constexpr int kPer = 32 / kTpl;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int j = t * kPer + k;
      uint32_t word = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) word = (q == (j >> 2)) ? cw[q] : word;
      const uint32_t cj = (word >> (8 * (j & 3))) & 0xFFu;
      if (a.sf != nullptr) a.sf[(rb * a.H + h) * a.D + 32 * cb + j] = static_cast<uint8_t>(cj);
      if (a.sf_mma != nullptr)
        a.sf_mma[tile_base + j * 16 + cb * 4 + kb_row] = static_cast<uint8_t>(cj);
    }
  }
}

// ---------------------------------------------------------------------------
// 32 consecutive tokens per channel (the forward's V), E4M3: a warp takes 32
// tokens x 64 channels of the token-major [T, H*D] view, lane l on tokens
// 4i + l/8 (i < 8) and channels 8(l%8)..+7, so each load instruction reads
// four whole 128-byte row segments.  A channel's block maximum is the
// maximum over the lane's 8 tokens, then over the 4 lanes holding the same
// channels (lane distance 8, 16).
__global__ void __launch_bounds__(128) mx_quantize_32x1_e4m3_kernel(const QuantArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t HD = static_cast<int64_t>(a.H) * a.D;
  const int64_t c0 = (static_cast<int64_t>(blockIdx.y) * 4 + warp) * 64;
  if (c0 >= HD) return;
  const int64_t rb = blockIdx.x, pr0 = rb * 32;
  const int sq = seq_of_sf_row(a.seqs, pr0);
  const SeqInfo si = seq_info(a.seqs, sq);
  const int64_t off = pr0 - si.sf_start;            // token offset in sequence
  const int64_t nv64 = static_cast<int64_t>(si.len) - off;
  const int nvalid = nv64 < 0 ? 0 : (nv64 > 32 ? 32 : static_cast<int>(nv64));
  const int g = lane & 7, rs = lane >> 3;
  const int64_t col = c0 + 8 * g;
  uint4 raw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + rs;
    raw[i] = r < nvalid ? __ldcs(reinterpret_cast<const uint4*>(a.x + (si.start + off + r) * HD + col))
                        : make_uint4(0u, 0u, 0u, 0u);
  }
  uint32_t cm[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t* u = reinterpret_cast<const uint32_t*>(&raw[i]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cm[2 * k] = max(cm[2 * k], (u[k] << 16) & 0x7FFFFFFFu);
      cm[2 * k + 1] = max(cm[2 * k + 1], u[k] & 0x7FFF0000u);
    }
  }
  uint32_t code[8];
  float inv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    cm[k] = max(cm[k], __shfl_xor_sync(0xFFFFFFFFu, cm[k], 8));
    cm[k] = max(cm[k], __shfl_xor_sync(0xFFFFFFFFu, cm[k], 16));
    code[k] = e8m0_code_from_amax_bits(cm[k]);
    inv[k] = inv_scale_from_code(code[k]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + rs;
    if (r < nvalid) {
      const uint32_t* u = reinterpret_cast<const uint32_t*>(&raw[i]);
      float f[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(u[k] << 16);
        f[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
      }
      uint32_t w[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        w[h] = cvt_e4m3x4(f[4 * h] * inv[4 * h], f[4 * h + 1] * inv[4 * h + 1],
                          f[4 * h + 2] * inv[4 * h + 2], f[4 * h + 3] * inv[4 * h + 3]);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (code[4 * h + q] == 0xFFu) w[h] = (w[h] & ~(0xFFu << (8 * q))) | (0x7Fu << (8 * q));
      }
      __stcs(reinterpret_cast<uint2*>(a.out + (si.start + off + r) * HD + col), make_uint2(w[0], w[1]));
    }
  }
  if (rs == 0) {
    if (a.sf != nullptr)
      *reinterpret_cast<uint2*>(a.sf + rb * HD + col) =
          make_uint2(code[0] | code[1] << 8 | code[2] << 16 | code[3] << 24,
                     code[4] | code[5] << 8 | code[6] << 16 | code[7] << 24);
    if (a.sf_mma != nullptr) {
      // operand rows = channels of a head, contraction blocks = token blocks
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t cc = col + k;
        const int64_t h = cc / a.D, d = cc % a.D;
        a.sf_mma[((rb >> 2) * a.H + h) * 512 + (d % 32) * 16 + (d / 32) * 4 + (rb & 3)] =
            static_cast<uint8_t>(code[k]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Fused RMSNorm + MX quantization ("Low Precision Flash Attention 4 ...",
// paragraph 2: fused RMSNorm+Quantize kernels producing FP8 output with dual
// scale factor layouts in one pass).  y = x / sqrt(mean(x^2) + eps) * w over
// each token's H * D values, then the quantizer's 1x32 or 32x32 blocks and
// scale layouts on y.  The codes are decided on fp32 y formed by a fixed
// sequence of correctly rounded operations (no contraction into FMA):
//   ss   = fp32 sum of the exact squares; lane l of a warp adds the row's
//          8-element chunks l, l + 32, ... element by element, then a
//          butterfly adds partner sums at lane distance 16, 8, 4, 2, 1;
//   rstd = 1 / sqrt(ss / N + eps);     y = (x * rstd) * w.
// CTA = one 32-row padded block, all heads.  Phase 1: the block's rstd (four
// rows per warp), phase 2: each warp quantizes whole heads of the block,
// reading x again (from L2: the CTA has just read it), so HBM sees x once.

struct NormArgs {
  const __nv_bfloat16* w;   // [H * D]
  float eps;
  float* rstd;              // [T] or null
};

// a 16-byte load the compiler may not merge with an earlier load of the
// same address
__device__ __forceinline__ uint4 ld_global_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// y for the 8 bf16 of one 16-byte chunk of x and of w
__device__ __forceinline__ void norm8(const uint4& xv, const uint4& wv, float rs, float* y) {
  const uint32_t* xu = reinterpret_cast<const uint32_t*>(&xv);
  const uint32_t* wu = reinterpret_cast<const uint32_t*>(&wv);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    y[2 * i] = __fmul_rn(__fmul_rn(__uint_as_float(xu[i] << 16), rs), __uint_as_float(wu[i] << 16));
    y[2 * i + 1] = __fmul_rn(__fmul_rn(__uint_as_float(xu[i] & 0xFFFF0000u), rs),
                             __uint_as_float(wu[i] & 0xFFFF0000u));
  }
}

// |y| for the same 8 values, formed from |x| and |w| (round to nearest is
// sign-symmetric, so these are the magnitudes of norm8's results bit for
// bit); a separate form keeps the compiler from holding norm8's results of
// the maxima pass live until the payload pass
__device__ __forceinline__ uint32_t norm8_amax_bits(const uint4& xv, const uint4& wv, float rs) {
  const uint32_t* xu = reinterpret_cast<const uint32_t*>(&xv);
  const uint32_t* wu = reinterpret_cast<const uint32_t*>(&wv);
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a0 = __uint_as_float((xu[i] << 16) & 0x7FFFFFFFu);
    const float a1 = __uint_as_float(xu[i] & 0x7FFF0000u);
    const float b0 = __uint_as_float((wu[i] << 16) & 0x7FFFFFFFu);
    const float b1 = __uint_as_float(wu[i] & 0x7FFF0000u);
    m = max(m, __float_as_uint(__fmul_rn(__fmul_rn(a0, rs), b0)));
    m = max(m, __float_as_uint(__fmul_rn(__fmul_rn(a1, rs), b1)));
  }
  return m;
}

// 8 values with one scale code -> 8 E4M3 bytes (two words)
__device__ __forceinline__ void quant8(const float* y, uint32_t code, uint32_t& w0, uint32_t& w1) {
  const float inv = inv_scale_from_code(code);
  w0 = cvt_e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv);
  w1 = cvt_e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv);
  if (code == 0xFFu) w0 = w1 = 0x7F7F7F7Fu;
}

template <int kMode, int kNcb>  // mode 0: 1x32, 2: 32x32
__global__ void __launch_bounds__(kWarpsPerBlock * 32, 2)
    rms_mx_quantize_kernel(const QuantArgs a, const NormArgs nrm) {
  static_assert(kMode == 0 || kMode == 2, "1x32 or 32x32 blocks");
  constexpr int kTpl = 32 / kNcb;                  // tokens per load
  __shared__ float s_rstd[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rb = blockIdx.x;
  const int64_t pr0 = rb * 32;                     // first padded row of the block
  const int sq = seq_of_sf_row(a.seqs, pr0);
  const SeqInfo si = seq_info(a.seqs, sq);
  const int64_t off = pr0 - si.sf_start;           // token offset in sequence
  const int64_t nvalid64 = static_cast<int64_t>(si.len) - off;
  const int nvalid = nvalid64 < 0 ? 0 : (nvalid64 > 32 ? 32 : static_cast<int>(nvalid64));
  const int n = a.H * a.D;
  const int nch = n / 8;                           // 16-byte chunks per row

  // ---- phase 1: rstd of rows warp*4 .. warp*4+3
#pragma unroll 1
  for (int rr = 0; rr < 4; ++rr) {
    const int row = warp * 4 + rr;
    float ss = 0.f;
    if (row < nvalid) {
      const uint4* src = reinterpret_cast<const uint4*>(a.x + (si.start + off + row) * static_cast<int64_t>(n));
#pragma unroll 1
      for (int c0 = lane; c0 < nch; c0 += 32 * 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = c0 + 32 * u;
          v[u] = c < nch ? src[c] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t* xu = reinterpret_cast<const uint32_t*>(&v[u]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(xu[i] << 16), hi = __uint_as_float(xu[i] & 0xFFFF0000u);
            ss = __fadd_rn(ss, __fmul_rn(lo, lo));   // exact squares; the zero
            ss = __fadd_rn(ss, __fmul_rn(hi, hi));   // chunks past the row add 0
          }
        }
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, d));
    if (lane == 0) {
      float r = 0.f;
      if (row < nvalid) {
        r = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(n)), nrm.eps)));
        if (nrm.rstd != nullptr) nrm.rstd[si.start + off + row] = r;
      }
      s_rstd[row] = r;
    }
  }
  __syncthreads();

  // ---- phase 2: one head of the block per warp at a time
  const int cb = lane % kNcb, t = lane / kNcb;
  const int64_t tile_row = (rb >> 2) * a.H;        // 512-byte scale tiles of the block
  const int kb_row = static_cast<int>(rb & 3);     // token block within the tile
#pragma unroll 1
  for (int h = warp; h < a.H; h += kWarpsPerBlock) {
    const int64_t tile_base = (tile_row + h) * 512;
    // this lane's 32 weights (L1-resident) and x rows: the maxima pass loads
    // every row of the lane at once; the payload pass loads each row again
    // (from L1) just before it is used, so that y never has to stay live
    const uint4* wsrc = reinterpret_cast<const uint4*>(nrm.w + h * a.D + 32 * cb);
    auto xrow = [&](int row) {
      return reinterpret_cast<const uint4*>(a.x + ((si.start + off + row) * a.H + h) * a.D + 32 * cb);
    };
    uint32_t rcode[kNcb];
    uint32_t m2 = 0;
    {
      uint4 v[kNcb][4];
#pragma unroll
      for (int r = 0; r < kNcb; ++r) {
        const int row = r * kTpl + t;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[r][i] = make_uint4(0, 0, 0, 0);
        if (row < nvalid) {
#pragma unroll
          for (int i = 0; i < 4; ++i) v[r][i] = xrow(row)[i];
        }
      }
      // block maxima: per row (1x32) or over the whole 32x32 tile
#pragma unroll
      for (int r = 0; r < kNcb; ++r) {
        const float rs = s_rstd[r * kTpl + t];
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) m = max(m, norm8_amax_bits(v[r][i], __ldg(wsrc + i), rs));
        rcode[r] = e8m0_code_from_amax_bits(m);
        m2 = max(m2, m);
      }
    }
    uint32_t bcode = 0;                            // 32x32: the block's code
    if (kMode == 2) {
#pragma unroll
      for (int x = kNcb; x < 32; x <<= 1) m2 = max(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, x));
      bcode = e8m0_code_from_amax_bits(m2);
    }
#pragma unroll
    for (int r = 0; r < kNcb; ++r) {
      const int row = r * kTpl + t;
      const bool valid = row < nvalid;
      const int64_t tok = si.start + off + row;
      const float rs = s_rstd[row];
      const uint32_t code = kMode == 0 ? rcode[r] : bcode;
      if (valid) {
        uint4 xv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = ld_global_v4(xrow(row) + i);
        uint32_t wq[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float y[8];
          norm8(xv[i], __ldg(wsrc + i), rs, y);
          quant8(y, code, wq[2 * i], wq[2 * i + 1]);
        }
        uint4* dst = reinterpret_cast<uint4*>(a.out + (tok * a.H + h) * a.D + 32 * cb);
        __stcs(dst + 0, make_uint4(wq[0], wq[1], wq[2], wq[3]));
        __stcs(dst + 1, make_uint4(wq[4], wq[5], wq[6], wq[7]));
      }
      // this row's kNcb codes gathered into one word by the cb = 0 lane
      const uint32_t c = (kMode == 0 && !valid) ? 0u : code;
      uint32_t word = c;
#pragma unroll
      for (int k = 1; k < kNcb; ++k) word |= __shfl_down_sync(0xFFFFFFFFu, c, k) << (8 * k);
      if (cb == 0) {
        if (a.sf_mma != nullptr) {
          const uint32_t wm = (kMode == 2 && !valid) ? 0u : word;
          uint8_t* d = a.sf_mma + tile_base + row * 16 + kb_row * 4;
          if (kNcb == 4) *reinterpret_cast<uint32_t*>(d) = wm;
          else *reinterpret_cast<uint16_t*>(d) = static_cast<uint16_t>(wm);
        }
        if (kMode == 0 && a.sf != nullptr && valid) {
          uint8_t* d = a.sf + (tok * a.H + h) * kNcb;
          if (kNcb == 4) *reinterpret_cast<uint32_t*>(d) = word;
          else *reinterpret_cast<uint16_t*>(d) = static_cast<uint16_t>(word);
        }
      }
      if (kMode == 2 && a.sf_mma_t != nullptr)
        a.sf_mma_t[tile_base + row * 16 + cb * 4 + kb_row] = static_cast<uint8_t>(bcode);
    }
    if (kMode == 2 && a.sf != nullptr && t == 0)
      a.sf[(rb * a.H + h) * kNcb + cb] = static_cast<uint8_t>(bcode);
  }
}

}  // namespace
}  // namespace lpfa

using namespace lpfa;

namespace {
template <int kFmt>
void launch_quantize(lpfa_block blk, bool d128, dim3 grid, dim3 block, cudaStream_t cs,
                     const QuantArgs& a) {
  switch (blk) {
    case LPFA_BLK_1X32:
      if (d128) mx_quantize_kernel<0, 4, kFmt><<<grid, block, 0, cs>>>(a);
      else mx_quantize_kernel<0, 2, kFmt><<<grid, block, 0, cs>>>(a);
      break;
    case LPFA_BLK_32X1:
      if constexpr (kFmt == kFmtE4M3) {
        const dim3 g2(static_cast<unsigned>(a.seqs.total_sf_rows / 32),
                      static_cast<unsigned>((static_cast<int64_t>(a.H) * a.D + 255) / 256));
        mx_quantize_32x1_e4m3_kernel<<<g2, 128, 0, cs>>>(a);
      } else if (d128) {
        mx_quantize_kernel<1, 4, kFmt><<<grid, block, 0, cs>>>(a);
      } else {
        mx_quantize_kernel<1, 2, kFmt><<<grid, block, 0, cs>>>(a);
      }
      break;
    case LPFA_BLK_32X32:
      if (d128) mx_quantize_kernel<2, 4, kFmt><<<grid, block, 0, cs>>>(a);
      else mx_quantize_kernel<2, 2, kFmt><<<grid, block, 0, cs>>>(a);
      break;
  }
}
}  // namespace

extern "C" lpfa_status lpfa_mx_quantize(const lpfa_seqs* seqs, const void* x,
                                        int64_t heads, int64_t head_dim,
                                        lpfa_block blk, void* out_e4m3,
                                        void* out_sf, void* out_sf_mma,
                                        void* out_sf_mma_t, void* stream) {
  return lpfa_mx_quantize_fmt(seqs, x, heads, head_dim, blk, LPFA_ELEM_E4M3, out_e4m3, out_sf,
                              out_sf_mma, out_sf_mma_t, stream);
}

extern "C" lpfa_status lpfa_mx_quantize_fmt(const lpfa_seqs* seqs, const void* x,
                                            int64_t heads, int64_t head_dim,
                                            lpfa_block blk, lpfa_elem fmt, void* out_e4m3,
                                            void* out_sf, void* out_sf_mma,
                                            void* out_sf_mma_t, void* stream) {
  SeqView sv;
  lpfa_status st = make_seq_view(seqs, &sv);
  if (st != LPFA_OK) return st;
  LPFA_CHECK_ARG(x != nullptr && out_e4m3 != nullptr);
  LPFA_CHECK_ARG(aligned16(x) && aligned16(out_e4m3));
  LPFA_CHECK_ARG(heads >= 1 && heads <= 4096);
  LPFA_CHECK_ARG(blk == LPFA_BLK_1X32 || blk == LPFA_BLK_32X1 ||
                 blk == LPFA_BLK_32X32);
  LPFA_CHECK_ARG(out_sf_mma_t == nullptr || blk == LPFA_BLK_32X32);
  LPFA_CHECK_ARG(fmt >= LPFA_ELEM_E4M3 && fmt <= LPFA_ELEM_E2M1);
  if (head_dim != 64 && head_dim != 128) return LPFA_ERR_UNSUPPORTED;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (sv.total_tokens == 0) return LPFA_OK;

  const int64_t Tp = sv.total_sf_rows;
  const int64_t mma_bytes = (Tp / 128) * heads * 512;
  // head_dim 64 leaves half of each tensor-core scale tile unused: zero it.
  if (head_dim < 128) {
    if (out_sf_mma != nullptr)
      LPFA_CHECK_CUDA(cudaMemsetAsync(out_sf_mma, 0, mma_bytes, cs));
    if (out_sf_mma_t != nullptr)
      LPFA_CHECK_CUDA(cudaMemsetAsync(out_sf_mma_t, 0, mma_bytes, cs));
  }

  QuantArgs a;
  a.seqs = sv;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.out = static_cast<uint8_t*>(out_e4m3);
  a.sf = static_cast<uint8_t*>(out_sf);
  a.sf_mma = static_cast<uint8_t*>(out_sf_mma);
  a.sf_mma_t = static_cast<uint8_t*>(out_sf_mma_t);
  a.H = static_cast<int32_t>(heads);
  a.D = static_cast<int32_t>(head_dim);
  a.ntiles = (Tp / 32) * heads * (head_dim / 32);
  const int64_t ntasks = (Tp / 32) * heads;        // one warp per (32-row block, head)
  const int64_t blocks = ceil_div(ntasks, kWarpsPerBlock);
  LPFA_CHECK_ARG(blocks < (1ll << 31));
  dim3 grid(static_cast<unsigned>(blocks)), block(kWarpsPerBlock * 32);
  const bool d128 = head_dim == 128;
  switch (fmt) {
    case LPFA_ELEM_E4M3: launch_quantize<kFmtE4M3>(blk, d128, grid, block, cs, a); break;
    case LPFA_ELEM_E5M2: launch_quantize<kFmtE5M2>(blk, d128, grid, block, cs, a); break;
    case LPFA_ELEM_E3M2: launch_quantize<kFmtE3M2>(blk, d128, grid, block, cs, a); break;
    case LPFA_ELEM_E2M3: launch_quantize<kFmtE2M3>(blk, d128, grid, block, cs, a); break;
    case LPFA_ELEM_E2M1: launch_quantize<kFmtE2M1>(blk, d128, grid, block, cs, a); break;
  }
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}

extern "C" lpfa_status lpfa_rmsnorm_mx_quantize(const lpfa_seqs* seqs, const void* x,
                                                const void* weight, int64_t heads,
                                                int64_t head_dim, float eps, lpfa_block blk,
                                                void* out_e4m3, void* out_sf, void* out_sf_mma,
                                                void* out_sf_mma_t, float* out_rstd,
                                                void* stream) {
  SeqView sv;
  lpfa_status st = make_seq_view(seqs, &sv);
  if (st != LPFA_OK) return st;
  LPFA_CHECK_ARG(x != nullptr && weight != nullptr && out_e4m3 != nullptr);
  LPFA_CHECK_ARG(aligned16(x) && aligned16(weight) && aligned16(out_e4m3));
  LPFA_CHECK_ARG(heads >= 1 && heads <= 4096);
  LPFA_CHECK_ARG(eps > 0.f && eps < 3.0e38f);
  LPFA_CHECK_ARG(out_sf_mma_t == nullptr || blk == LPFA_BLK_32X32);
  if (blk != LPFA_BLK_1X32 && blk != LPFA_BLK_32X32) return LPFA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return LPFA_ERR_UNSUPPORTED;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (sv.total_tokens == 0) return LPFA_OK;

  const int64_t Tp = sv.total_sf_rows;
  const int64_t mma_bytes = (Tp / 128) * heads * 512;
  if (head_dim < 128) {
    if (out_sf_mma != nullptr)
      LPFA_CHECK_CUDA(cudaMemsetAsync(out_sf_mma, 0, mma_bytes, cs));
    if (out_sf_mma_t != nullptr)
      LPFA_CHECK_CUDA(cudaMemsetAsync(out_sf_mma_t, 0, mma_bytes, cs));
  }
  QuantArgs a;
  a.seqs = sv;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.out = static_cast<uint8_t*>(out_e4m3);
  a.sf = static_cast<uint8_t*>(out_sf);
  a.sf_mma = static_cast<uint8_t*>(out_sf_mma);
  a.sf_mma_t = static_cast<uint8_t*>(out_sf_mma_t);
  a.H = static_cast<int32_t>(heads);
  a.D = static_cast<int32_t>(head_dim);
  a.ntiles = (Tp / 32) * heads * (head_dim / 32);
  NormArgs nrm;
  nrm.w = static_cast<const __nv_bfloat16*>(weight);
  nrm.eps = eps;
  nrm.rstd = out_rstd;
  const int64_t blocks = Tp / 32;                  // one CTA per 32-row block
  LPFA_CHECK_ARG(blocks < (1ll << 31));
  dim3 grid(static_cast<unsigned>(blocks)), block(kWarpsPerBlock * 32);
  const bool d128 = head_dim == 128;
  if (blk == LPFA_BLK_1X32) {
    if (d128) rms_mx_quantize_kernel<0, 4><<<grid, block, 0, cs>>>(a, nrm);
    else rms_mx_quantize_kernel<0, 2><<<grid, block, 0, cs>>>(a, nrm);
  } else {
    if (d128) rms_mx_quantize_kernel<2, 4><<<grid, block, 0, cs>>>(a, nrm);
    else rms_mx_quantize_kernel<2, 2><<<grid, block, 0, cs>>>(a, nrm);
  }
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}

// ---------------------------------------------------------------------------
// NVFP4 quantizer (lpfa_nvfp4_quantize): 16-element blocks along a row, E2M1
// elements, one E4M3 scale per block: s = E4M3(amax / 6), element =
// E2M1(x / s), both round to nearest even with saturation, both divisions
// single fp32 divisions.  One thread per block.
// ---------------------------------------------------------------------------
namespace lpfa {
namespace {
__global__ void nvfp4_quantize_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                      int64_t cols, uint8_t* __restrict__ out,
                                      uint8_t* __restrict__ sf, uint8_t* __restrict__ sf_mma) {
  const int64_t nb = cols / 16;
  const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (blk >= rows * nb) return;
  const int64_t r = blk / nb, b = blk % nb;
  const uint4* src = reinterpret_cast<const uint4*>(x + r * cols + b * 16);
  const uint4 v[2] = {src[0], src[1]};
  float f[16];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v[h]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 t = __bfloat1622float2(p2[k]);
      f[8 * h + 2 * k] = t.x;
      f[8 * h + 2 * k + 1] = t.y;
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const uint32_t code = cvt_e4m3x2(__fdiv_rn(amax, 6.0f), 0.f) & 0xFFu;
  // the scale's value: E4M3 -> f16 -> f32, exact (the code in both bytes, so
  // both halves of the result hold it)
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code | (code << 8))));
  const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
  uint32_t o[2] = {0u, 0u};
  if (s > 0.f) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      uint16_t pr;
      asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.u16.u8 %0, t;\n\t}"
          : "=h"(pr)
          : "f"(__fdiv_rn(f[i], s)), "f"(__fdiv_rn(f[i + 1], s)));
      o[i >> 3] |= static_cast<uint32_t>(pr & 0xFFu) << (8 * ((i >> 1) & 3));
    }
  }
  *reinterpret_cast<uint2*>(out + r * (cols / 2) + b * 8) = make_uint2(o[0], o[1]);
  const uint8_t c = s > 0.f ? static_cast<uint8_t>(code) : 0u;
  if (sf != nullptr) sf[r * nb + b] = c;
  if (sf_mma != nullptr) {
    const int64_t tile = (r / 128) * (nb / 4) + b / 4;
    const int64_t rr = r % 128;
    sf_mma[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (b % 4)] = c;
  }
}
}  // namespace
}  // namespace lpfa

extern "C" lpfa_status lpfa_nvfp4_quantize(const void* x, int64_t rows, int64_t cols,
                                           void* out, void* out_sf, void* out_sf_mma,
                                           void* stream) {
  using namespace lpfa;
  LPFA_CHECK_ARG(x != nullptr && out != nullptr && aligned16(x));
  LPFA_CHECK_ARG((reinterpret_cast<uintptr_t>(out) & 7u) == 0);
  LPFA_CHECK_ARG(rows >= 0 && cols >= 0 && cols % 16 == 0);
  LPFA_CHECK_ARG(out_sf_mma == nullptr || (rows % 128 == 0 && cols % 64 == 0));
  const int64_t n = rows * (cols / 16);
  if (n == 0) return LPFA_OK;
  LPFA_CHECK_ARG(ceil_div(n, 256) < (1ll << 31));
  nvfp4_quantize_kernel<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0,
                          static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), rows, cols, static_cast<uint8_t*>(out),
      static_cast<uint8_t*>(out_sf), static_cast<uint8_t*>(out_sf_mma));
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}
