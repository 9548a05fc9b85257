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

// Quantize 32 floats with one scale code into 32 bytes (8 words).
__device__ __forceinline__ void quant_row(const float (&f)[32],
                                          const uint32_t (&code)[32],
                                          uint32_t (&w)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a = f[4 * j + 0] * inv_scale_from_code(code[4 * j + 0]);
    float b = f[4 * j + 1] * inv_scale_from_code(code[4 * j + 1]);
    float c = f[4 * j + 2] * inv_scale_from_code(code[4 * j + 2]);
    float d = f[4 * j + 3] * inv_scale_from_code(code[4 * j + 3]);
    w[j] = cvt_e4m3x4(a, b, c, d);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (code[4 * j + q] == 0xFFu) w[j] = (w[j] & ~(0xFFu << (8 * q))) | (0x7Fu << (8 * q));
  }
}

// As quant_row with the codes of the 32 values packed four to a word
// (element 4i + q takes byte q of cw[i]).
__device__ __forceinline__ void quant_row_packed(const float (&f)[32], const uint32_t (&cw)[8],
                                                 uint32_t (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float x[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) x[q] = f[4 * i + q] * inv_scale_from_code((cw[i] >> (8 * q)) & 0xFFu);
    w[i] = cvt_e4m3x4(x[0], x[1], x[2], x[3]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (((cw[i] >> (8 * q)) & 0xFFu) == 0xFFu) w[i] = (w[i] & ~(0xFFu << (8 * q))) | (0x7Fu << (8 * q));
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
template <int kMode, int kNcb>  // mode 0: 1x32, 1: 32x1, 2: 32x32
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
    bcode = e8m0_code_from_amax_bits(m);
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
        word |= e8m0_code_from_amax_bits(qq) << (8 * k);
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
      const uint32_t c = e8m0_code_from_amax_bits(m);
#pragma unroll
      for (int j = 0; j < 32; ++j) code[j] = c;
    } else if (kMode == 2) {
#pragma unroll
      for (int j = 0; j < 32; ++j) code[j] = bcode;
    }
    if (valid) {
      uint32_t w[8];
      if (kMode == 1) quant_row_packed(f, cw, w);
      else quant_row(f, code, w);
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

}  // namespace
}  // namespace lpfa

using namespace lpfa;

extern "C" lpfa_status lpfa_mx_quantize(const lpfa_seqs* seqs, const void* x,
                                        int64_t heads, int64_t head_dim,
                                        lpfa_block blk, void* out_e4m3,
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
  switch (blk) {
    case LPFA_BLK_1X32:
      if (d128) mx_quantize_kernel<0, 4><<<grid, block, 0, cs>>>(a);
      else mx_quantize_kernel<0, 2><<<grid, block, 0, cs>>>(a);
      break;
    case LPFA_BLK_32X1:
      if (d128) mx_quantize_kernel<1, 4><<<grid, block, 0, cs>>>(a);
      else mx_quantize_kernel<1, 2><<<grid, block, 0, cs>>>(a);
      break;
    case LPFA_BLK_32X32:
      if (d128) mx_quantize_kernel<2, 4><<<grid, block, 0, cs>>>(a);
      else mx_quantize_kernel<2, 2><<<grid, block, 0, cs>>>(a);
      break;
  }
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}
