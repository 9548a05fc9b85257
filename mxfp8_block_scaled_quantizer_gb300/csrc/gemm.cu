// Block-scaled GEMM on tcgen05: D[M,N] (fp32) = A[M,K] * B[N,K]^T, MXFP8 and
// the other MX / NV element formats.
//
// Purpose: the dense MX MMA rate of this GPU, measured in the same run as the
// attention kernels ("Low Precision Flash Attention 4 ...", paragraph 2:
// tcgen05.mma.block_scale on MXFP8, MXFP6, MXFP4 and NVFP4 operands), the
// GEMM + Quantize producer of the same paragraph, and the two backward GEMMs
// of the GEMM-Norm backward (paragraph 4).
//
// Two kernels:
//   mx_gemm_pair_kernel   256x256 tiles on CTA pairs (cta_group::2; below),
//                         every kind, one or two problems per launch;
//   mx_gemm_kernel        128x256 tiles, one CTA each: the quantizing
//                         epilogue when M % 256 == 128.
// One-CTA design (persistent, one CTA per SM):
//   warp 0      TMA producer: A tile 128x128 B, B tile 256x128 B (128-byte
//               swizzle, K-major) + three 512-byte scale tiles per stage.
//   warp 1      TMEM allocator and MMA issuer: per stage copies the scale
//               tiles into TMEM (tcgen05.cp) and issues 4 MMAs of K = 32.
//   warps 2-9   epilogue: two warps per TMEM lane quarter, one per column
//               half; each reads its 32 rows x 128 columns in four loads and
//               one wait and releases the accumulator before its global
//               stores, so the next tile's main loop overlaps them.
//
// Quantizing epilogue (lpfa_mx_gemm_quantize): the fp32 tile is quantized in
// registers to E4M3 with E8M0 scales, in 1x32 blocks along N (a thread's 32
// columns of one row) or 32x32 blocks (a warp's 32 rows x 32 columns, maximum
// by redux.sync), with the scales written in the compact layout and as the
// next GEMM's operand: rows = M (contraction over N) and, for square blocks,
// rows = N (contraction over M).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "lpfa_device.cuh"
#include "lpfa_internal.h"

namespace lpfa {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 128;            // bytes = fp8 elements per stage
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK;  // 16 KB
constexpr int kBBytes = kBN * kBK;  // 32 KB
constexpr int kSfBytes = 512;
constexpr int kThreads = 320;      // producer, MMA issuer, 8 epilogue warps
constexpr int kEpiChunks = kBN / 64;  // 32-column chunks per epilogue warp
constexpr int kTmemCols = 512;
constexpr int kSfCol0 = 256;        // TMEM scale buffers after the accumulator

// MMA kind of the main loop.  A stage holds 128 bytes of K per operand row:
//   kKindF8F6F4  kind::mxf8f6f4 (1 byte per element slot), 4 MMAs of K = 32,
//                one 512-byte scale tile per 128 rows (four 32-element E8M0
//                blocks per row), scale byte sf_id = K-step;
//   kKindMxf4    kind::mxf4nvf4 scale_vec::2X: dense FP4 (two per byte), 4
//                MMAs of K = 64, two scale tiles per 128 rows (each four
//                32-element E8M0 blocks: two MMAs, scale bytes 0-1 / 2-3);
//   kKindNvf4    kind::mxf4nvf4 scale_vec::4X: dense FP4, 4 MMAs of K = 64,
//                four scale tiles per 128 rows (each the four 16-element E4M3
//                scales of one MMA).
enum : int { kKindF8F6F4 = 0, kKindMxf4 = 1, kKindNvf4 = 2 };

template <int kKind>
struct GemmCfg {
  static constexpr int kSfA = kKind == kKindNvf4 ? 4 : kKind == kKindMxf4 ? 2 : 1;  // tiles per 128 rows
  static constexpr int kSfTiles = 3 * kSfA;                                           // A + two B row tiles
  static constexpr int kStageTx = kABytes + kBBytes + kSfTiles * kSfBytes;            // bytes landed
  static constexpr int kStageBytes = (kStageTx + 1023) / 1024 * 1024;                 // 1024-aligned
  static constexpr int kSfColsPerStage = 4 * kSfTiles;
  static_assert(kSfCol0 + kStages * kSfColsPerStage <= 512, "TMEM columns");
};

struct GemmArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  float* d;             // fp32 result, or null (quantizing epilogue only)
  uint8_t* q;           // E4M3 [M, N]
  uint8_t* qsf;         // compact scales, or null
  uint8_t* qsf_mma;     // [M/128][N/128][512], or null
  uint8_t* qsf_mma_t;   // 32x32: [N/128][M/128][512], or null
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, kt;
  uint32_t idesc;       // instruction descriptor (element types of A and B)
  uint32_t* err;
};

struct __align__(8) GemmSmem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// 32 fp32 values with one scale code -> 32 E4M3 bytes (8 words)
__device__ __forceinline__ void quant32(const uint32_t (&r)[32], uint32_t code, uint32_t (&w)[8]) {
  const float inv = inv_scale_from_code(code);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    w[j] = cvt_e4m3x4(__uint_as_float(r[4 * j]) * inv, __uint_as_float(r[4 * j + 1]) * inv,
                      __uint_as_float(r[4 * j + 2]) * inv, __uint_as_float(r[4 * j + 3]) * inv);
  if (code == 0xFFu) {
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = 0x7F7F7F7Fu;
  }
}

// Epilogue of one 128 x 256 output tile, from the registers holding TMEM
// lane quarter q (rows 32q.. of 128-row M tile tm), column half h of N tile
// tn: fp32 stores and / or the quantizing epilogue.
template <int kQuant>
__device__ __forceinline__ void epilogue_store(const GemmArgs& g, const uint32_t (&r)[kEpiChunks][32],
                                               int tm, int tn, int q, int h, int lane) {
  const int row = tm * kBM + q * 32 + lane;
  const int col0 = tn * kBN + h * (kBN / 2);
  float* drow = g.d + static_cast<int64_t>(row) * g.N + col0;
  uint32_t codes[kEpiChunks];                // this row's (or block's) codes
#pragma unroll
  for (int c = 0; c < kEpiChunks; ++c) {
    if ((kQuant < 0 || g.d != nullptr) && row < g.M) {
      float4* dst = reinterpret_cast<float4*>(drow + c * 32);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = make_float4(__uint_as_float(r[c][4 * j]), __uint_as_float(r[c][4 * j + 1]),
                             __uint_as_float(r[c][4 * j + 2]), __uint_as_float(r[c][4 * j + 3]));
    }
    if (kQuant >= 0) {
      // block maximum of |d| as bits (NaN above Inf), then the code
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) m = max(m, r[c][j] & 0x7FFFFFFFu);
      if (kQuant == 2) m = __reduce_max_sync(0xFFFFFFFFu, m);
      const uint32_t code = e8m0_code_from_amax_bits(m);
      codes[c] = code;
      uint32_t w[8];
      quant32(r[c], code, w);
      uint4* qdst = reinterpret_cast<uint4*>(g.q + static_cast<int64_t>(row) * g.N + col0 + c * 32);
      qdst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      qdst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      // rows = N arrangement (square blocks): column n = col0 + 32c +
      // lane, i.e. 128-column N tile 2 tn + h, contraction block q of the
      // M tile
      if (kQuant == 2 && g.qsf_mma_t != nullptr) {
        const int64_t nt = static_cast<int64_t>(tn) * 2 + h;
        g.qsf_mma_t[(nt * g.tiles_m + tm) * 512 + lane * 16 + c * 4 + q] =
            static_cast<uint8_t>(code);
      }
    }
  }
  if (kQuant >= 0) {
    const int nb = g.N / 32;
    const uint32_t packed = codes[0] | codes[1] << 8 | codes[2] << 16 | codes[3] << 24;
    if (g.qsf != nullptr) {
      if (kQuant == 0) {
        *reinterpret_cast<uint32_t*>(g.qsf + static_cast<int64_t>(row) * nb + col0 / 32) = packed;
      } else if (lane == 0) {
        *reinterpret_cast<uint32_t*>(g.qsf + static_cast<int64_t>(tm * 4 + q) * nb + col0 / 32) =
            packed;
      }
    }
    if (g.qsf_mma != nullptr) {
      // rows = M arrangement: row (lane, quarter q) of the M tile, the
      // four contraction blocks of the 128-column N tile 2 tn + h
      const int64_t nt = static_cast<int64_t>(tn) * 2 + h;
      *reinterpret_cast<uint32_t*>(
          g.qsf_mma + (static_cast<int64_t>(tm) * (g.N / 128) + nt) * 512 + lane * 16 + q * 4) =
          packed;
    }
  }
}

template <int kQuant, int kKind>   // kQuant -1: fp32 only; 0: 1x32 along N; 2: 32x32
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                   const __grid_constant__ CUtensorMap tma_b,
                   const GemmArgs g) {
  using C = GemmCfg<kKind>;
  constexpr int kStageTx = C::kStageTx;
  constexpr int kStageBytes = C::kStageBytes;
  constexpr int kSfColsPerStage = C::kSfColsPerStage;
  constexpr int kSfA = C::kSfA;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // stage buffers start 1024-aligned (128-byte swizzle atoms)
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GemmSmem* sh = reinterpret_cast<GemmSmem*>(stage_base + kStages * kStageBytes);
  volatile int* abort = &sh->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ntiles = g.tiles_m * g.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->acc_full, 1);
    mbar_init(&sh->acc_empty, 8);
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int issued[kStages];     // parity of the last load issued per stage
      for (int s = 0; s < kStages; ++s) issued[s] = -1;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int tm = t % g.tiles_m, tn = t / g.tiles_m;
        for (int kt = 0; kt < g.kt && ok; ++kt) {
          ok = mbar_wait(&sh->empty[stage], phase ^ 1, g.err, abort, 1);
          if (!ok) break;
          uint8_t* buf = stage_base + stage * kStageBytes;
          uint64_t* bar = &sh->full[stage];
          mbar_arrive_expect_tx(bar, kStageTx);
          tma_load_2d(buf, &tma_a, kt * kBK, tm * kBM, bar);
          tma_load_2d(buf + kABytes, &tma_b, kt * kBK, tn * kBN, bar);
          // scale tiles: A's kSfA, then each B row tile's kSfA; a row tile's
          // tiles are consecutive along K in global memory
          uint8_t* sfbuf = buf + kABytes + kBBytes;
          const int64_t ktiles = static_cast<int64_t>(g.kt) * kSfA;
#pragma unroll
          for (int t = 0; t < kSfA; ++t) {
            bulk_load(sfbuf + t * kSfBytes,
                      g.sfa + (tm * ktiles + kt * kSfA + t) * kSfBytes, kSfBytes, bar);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              bulk_load(sfbuf + (kSfA * (1 + h) + t) * kSfBytes,
                        g.sfb + ((2 * tn + h) * ktiles + kt * kSfA + t) * kSfBytes, kSfBytes,
                        bar);
          }
          issued[stage] = static_cast<int>(phase);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      // on abort: wait (bounded) until every issued load has landed
      if (!ok) {
        for (int s = 0; s < kStages; ++s)
          if (issued[s] >= 0)
            mbar_wait(&sh->full[s], static_cast<uint32_t>(issued[s]), nullptr, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = g.idesc;
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int local = 0;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++local) {
        if (local > 0) {
          ok = mbar_wait(&sh->acc_empty, acc_phase ^ 1, g.err, abort, 2);
          if (!ok) break;
        }
        tc_fence_after();
        for (int kt = 0; kt < g.kt; ++kt) {
          ok = mbar_wait(&sh->full[stage], phase, g.err, abort, 3);
          if (!ok) break;
          tc_fence_after();
          uint8_t* buf = stage_base + stage * kStageBytes;
          const uint32_t a_addr = smem_u32(buf);
          const uint32_t b_addr = smem_u32(buf + kABytes);
          const uint32_t sf_addr = smem_u32(buf + kABytes + kBBytes);
          // TMEM: A scale tile t at sfa_t + 4t; B tile t at sfb_t + 8t
          // (rows 0-127) and + 4 (rows 128-255)
          const uint32_t sfa_t = tmem + kSfCol0 + stage * kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + 4 * kSfA;
#pragma unroll
          for (int t = 0; t < kSfA; ++t) {
            tc_cp_32x128b_warpx4(sfa_t + 4 * t, sf_tile_desc(sf_addr + t * kSfBytes));
            tc_cp_32x128b_warpx4(sfb_t + 8 * t, sf_tile_desc(sf_addr + (kSfA + t) * kSfBytes));
            tc_cp_32x128b_warpx4(sfb_t + 8 * t + 4,
                                 sf_tile_desc(sf_addr + (2 * kSfA + t) * kSfBytes));
          }
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint64_t ad = make_sdesc(a_addr + kb * 32, 16, 1024, 2);
            const uint64_t bd = make_sdesc(b_addr + kb * 32, 16, 1024, 2);
            const uint32_t acc = (kt | kb) != 0;
            if constexpr (kKind == kKindF8F6F4) {
              mma_mxf8_ss(tmem, ad, bd, idesc_sf_ids(idesc, kb, kb), sfa_t, sfb_t, acc);
            } else if constexpr (kKind == kKindMxf4) {
              const uint32_t t = kb >> 1, id = 2 * (kb & 1);
              mma_mxf4_ss(tmem, ad, bd, idesc_sf_ids(idesc, id, id), sfa_t + 4 * t,
                          sfb_t + 8 * t, acc);
            } else {
              mma_nvf4_ss(tmem, ad, bd, idesc, sfa_t + 4 * kb, sfb_t + 8 * kb, acc);
            }
          }
          tc_commit(&sh->empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&sh->acc_full);
        acc_phase ^= 1;
      }
      if (!ok) *abort = 1;
      // every issued MMA has completed before TMEM is released
      tc_commit(&sh->drain);
      mbar_wait(&sh->drain, 0, nullptr, nullptr, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warps 2-9: TMEM lane quarter q (a warp reaches only lanes 32 (warp % 4)
    // ..), column half h of the 256-column accumulator
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const int tm = t % g.tiles_m, tn = t / g.tiles_m;
      ok = mbar_wait(&sh->acc_full, acc_phase, g.err, abort, 4);
      if (!ok) break;
      acc_phase ^= 1;
      tc_fence_after();
      // the half-row in four loads and one wait; the accumulator is released
      // before any store so the next tile's MMAs overlap the stores
      uint32_t r[kEpiChunks][32];
#pragma unroll
      for (int c = 0; c < kEpiChunks; ++c)
        tmem_ld32(tmem_addr(tmem, q * 32, (h * kEpiChunks + c) * 32), r[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty);
      epilogue_store<kQuant>(g, r, tm, tn, q, h, lane);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ----------------------------------------------------------- CTA pairs
// The same GEMM on 256 x 256 output tiles, one per CTA pair (cluster of
// two): the even CTA issues tcgen05.mma.cta_group::2 with M = 256, each CTA
// holding 128 rows of A, 128 rows (N) of B and its 128 rows of D.  Per MMA
// each SM reads 8 KB of operands from its shared memory instead of 12 KB,
// and per stage receives 33 KB instead of 49 KB, for the same work.
//   producer (warp 0, both CTAs)  TMA of this CTA's A and B halves, its A
//     scale tile and both B scale tiles (every SM's tensor core needs the
//     scales of all 256 B rows), each signalling the even CTA's stage barrier
//     (cta_group::2 completion), whose expected bytes cover both CTAs;
//   MMA issuer (warp 1 of the even CTA)  scale copies and MMAs for the pair;
//     commits free the stage in both CTAs and hand the accumulator to both
//     epilogues;
//   epilogue (warps 2-9, both CTAs)  as above on this CTA's rows; the odd
//     CTA releases the accumulator by a remote arrive.
constexpr int kPairStageOut = 32 * 64;                          // epilogue slot per warp:
                                                                // 32 rows x 16 fp32
constexpr int kGroupM = 8;                                      // raster group (M tiles)

// Tile t of the persistent loop -> (M tile, N tile): groups of kGroupM M
// tiles walked along N, so the pairs resident at once share A and B tiles
// in L2.
__device__ __forceinline__ void pair_tile(int t, int tiles_m2, int tiles_n, int& tm, int& tn) {
  const int per_group = kGroupM * tiles_n;
  const int grp = t / per_group, first = grp * kGroupM;
  const int gm = min(kGroupM, tiles_m2 - first);
  const int w = t - grp * per_group;
  tm = first + w % gm;
  tn = w / gm;
}
constexpr int kPairBBytes = 128 * kBK;                          // B half, 16 KB

// Per-kind pair stage: A 128 rows, B 128 rows (one N half), the A scale
// tiles and the scale tiles of both B halves (kSfA tiles per 128 rows).
template <int kKind>
struct PairCfg {
  static constexpr int kSfA = GemmCfg<kKind>::kSfA;
  static constexpr int kTx = kABytes + kPairBBytes + 3 * kSfA * kSfBytes;   // per CTA
  static constexpr int kStageBytes = (kTx + 1023) / 1024 * 1024;
  static constexpr int kSfCols = 12 * kSfA;                                // TMEM, per stage
  // as many stages as shared memory holds (6 for one scale tile per 128
  // rows, 5 for FP4's two or four)
  static constexpr int kStages = kSfA == 1 ? 6 : 5;
  static constexpr int kSmem = kStages * kStageBytes + 8 * kPairStageOut + 256 + 1024;
  static_assert(kSfCol0 + kStages * kSfCols <= kTmemCols, "TMEM columns");
  static_assert(kSmem <= 232448, "shared memory");
};

// Up to two GEMMs of one kind in one persistent launch (a grouped GEMM:
// the two backward GEMMs of the GEMM-Norm backward).  Problem 1, the one
// with the longer contraction, goes first: its tiles round-robin over the
// pairs; then each pair takes a number of problem 0's tiles chosen so that
// every pair's total stage count is about the same (c_hi for the r pairs
// that took one more problem-1 tile, c_lo for the others, one more for pairs
// < extra).  Every role of both CTAs walks the same sequence.
struct PairMaps {
  CUtensorMap a, b, sfa, sfb, d;
};
struct PairProblem {
  GemmArgs g;
  int32_t tiles_m2;     // 256-row tiles
  int32_t ntiles;       // pair tiles
};
struct PairGroup {
  PairProblem p[2];
  int32_t nprob;
  int32_t r, c_hi, c_lo, extra;
};

// k-th tile of this pair's sequence -> (problem, M tile, N tile); false when
// the sequence is done.
__device__ __forceinline__ bool pair_walk(const PairGroup& G, int pair, int npairs, int k,
                                          int& prob, int& tm, int& tn) {
  if (G.nprob == 1) {
    const int t = pair + k * npairs;
    if (t >= G.p[0].ntiles) return false;
    prob = 0;
    pair_tile(t, G.p[0].tiles_m2, G.p[0].g.tiles_n, tm, tn);
    return true;
  }
  const int n1 = G.p[1].ntiles;
  const int cnt1 = n1 / npairs + (pair < n1 % npairs ? 1 : 0);
  if (k < cnt1) {
    prob = 1;
    pair_tile(pair + k * npairs, G.p[1].tiles_m2, G.p[1].g.tiles_n, tm, tn);
    return true;
  }
  // problem 0 in rounds, so that the pairs running at once work on
  // neighbouring tiles (shared A and B tiles in L2): first c_lo - c_hi rounds
  // over the pairs that took fewer problem-1 tiles (they start earlier), then
  // c_hi rounds over all pairs, then one tile for pairs < extra
  const int j = k - cnt1;
  const int cnt0 = (pair < G.r ? G.c_hi : G.c_lo) + (pair < G.extra ? 1 : 0);
  if (j >= cnt0) return false;
  const int nlo = npairs - G.r, dlo = G.c_lo - G.c_hi;
  int t;
  if (pair >= G.r && j < dlo) {
    t = j * nlo + (pair - G.r);
  } else {
    const int jb = pair >= G.r ? j - dlo : j;
    t = dlo * nlo + jb * npairs + pair;            // jb == c_hi: the extra tile
  }
  prob = 0;
  pair_tile(t, G.p[0].tiles_m2, G.p[0].g.tiles_n, tm, tn);
  return true;
}

template <int kQuant, int kKind>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mx_gemm_pair_kernel(const __grid_constant__ PairMaps m0, const __grid_constant__ PairMaps m1,
                        const PairGroup G) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  struct __align__(8) PairSmem {
    uint64_t full[PairCfg<kKind>::kStages];
    uint64_t empty[PairCfg<kKind>::kStages];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
  };
  using PC = PairCfg<kKind>;
  constexpr int kSfA = PC::kSfA;
  constexpr int kStageBytes = PC::kStageBytes;
  constexpr int kPairStages = PC::kStages;
  uint8_t* out_base = stage_base + kPairStages * kStageBytes;       // 8 epilogue slots
  PairSmem* sh = reinterpret_cast<PairSmem*>(out_base + 8 * kPairStageOut);
  volatile int* abort = &sh->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();           // 0: issues the MMAs
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  uint32_t* const err = G.p[0].g.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->acc_full, 1);
    mbar_init(&sh->acc_empty, 16);                   // 8 epilogue warps per CTA
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_barrier_init();
    for (int q = 0; q < G.nprob; ++q) {
      const PairMaps& m = q ? m1 : m0;
      tma_prefetch_desc(&m.a);
      tma_prefetch_desc(&m.b);
      tma_prefetch_desc(&m.sfa);
      tma_prefetch_desc(&m.sfb);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(&sh->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                    // peer barriers initialised
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // the whole warp runs the loop converged; lane 0 waits, the elected lane
    // issues the copies: A, B, the A scale tiles and both B halves' scale
    // tiles (one 3D box), four copies per stage
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int prob, tm, tn;
    for (int k = 0; ok && pair_walk(G, pair, npairs, k, prob, tm, tn); ++k) {
      const GemmArgs& g = G.p[prob].g;
      const PairMaps& m = prob ? m1 : m0;
      const int tm128 = 2 * tm + static_cast<int>(rank);
      for (int kt = 0; kt < g.kt && ok; ++kt) {
        if (lane == 0) ok = mbar_wait(&sh->empty[stage], phase ^ 1, err, abort, 11);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        uint8_t* buf = stage_base + stage * kStageBytes;
        const uint32_t bar = mapa_shared(smem_u32(&sh->full[stage]), 0);
        if (rank == 0) mbar_arrive_expect_tx_elect(&sh->full[stage], 2 * PC::kTx);
        tma_load_2d_pair_elect(buf, &m.a, kt * kBK, tm128 * kBM, bar);
        tma_load_2d_pair_elect(buf + kABytes, &m.b, kt * kBK,
                               (2 * tn + static_cast<int>(rank)) * 128, bar);
        // a row tile's scale tiles of one stage are consecutive in global
        // memory: A's kSfA as one box, both B halves' as one 3D box
        uint8_t* sf = buf + kABytes + kPairBBytes;
        tma_load_2d_pair_elect(sf, &m.sfa, 0, tm128 * g.kt * kSfA + kt * kSfA, bar);
        tma_load_3d_pair_elect(sf + kSfA * kSfBytes, &m.sfb, 0, kt * kSfA, 2 * tn, bar);
        if (++stage == kPairStages) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // the whole warp runs the loop converged; lane 0 waits, the elected lane
    // issues (fewer issue cycles per tcgen05 instruction than a lane branch)
    if (rank == 0) {
      const uint32_t idesc = G.p[0].g.idesc;
      // descriptors of stage 0; a stage adds kStageBytes >> 4, a K-step
      // 32 >> 4 (the 14-bit address field does not carry)
      const uint64_t ad0 = make_sdesc(smem_u32(stage_base), 16, 1024, 2);
      const uint64_t bd0 = make_sdesc(smem_u32(stage_base + kABytes), 16, 1024, 2);
      const uint64_t sd0 = sf_tile_desc(smem_u32(stage_base + kABytes + kPairBBytes));
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int local = 0;
      int prob, tm, tn;
      for (int k = 0; ok && pair_walk(G, pair, npairs, k, prob, tm, tn); ++k, ++local) {
        const int nkt = G.p[prob].g.kt;
        if (local > 0) {
          if (lane == 0) ok = mbar_wait_cluster(&sh->acc_empty, acc_phase ^ 1, err, abort, 12);
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) break;
        }
        tc_fence_after();
        for (int kt = 0; kt < nkt; ++kt) {
          if (lane == 0) ok = mbar_wait(&sh->full[stage], phase, err, abort, 13);
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) break;
          tc_fence_after();
          const uint64_t so = static_cast<uint64_t>(stage * (kStageBytes >> 4));
          // TMEM: A scale tile u at sfa_t + 4u; B tile u at sfb_t + 8u (N rows
          // 0-127) and + 4 (rows 128-255)
          const uint32_t sfa_t = tmem + kSfCol0 + stage * PC::kSfCols;
          const uint32_t sfb_t = sfa_t + 4 * kSfA;
#pragma unroll
          for (int u = 0; u < kSfA; ++u) {
            tc_cp_pair_32x128b_warpx4_elect(sfa_t + 4 * u, sd0 + so + ((u * kSfBytes) >> 4));
            tc_cp_pair_32x128b_warpx4_elect(sfb_t + 8 * u,
                                            sd0 + so + (((kSfA + u) * kSfBytes) >> 4));
            tc_cp_pair_32x128b_warpx4_elect(sfb_t + 8 * u + 4,
                                            sd0 + so + (((2 * kSfA + u) * kSfBytes) >> 4));
          }
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint64_t ad = ad0 + so + 2 * kb, bd = bd0 + so + 2 * kb;
            const uint32_t acc = (kt | kb) != 0;
            if constexpr (kKind == kKindF8F6F4) {
              mma_pair_mxf8_ss_elect(tmem, ad, bd, idesc_sf_ids(idesc, kb, kb), sfa_t, sfb_t, acc);
            } else if constexpr (kKind == kKindMxf4) {
              const uint32_t u = kb >> 1, id = 2 * (kb & 1);
              mma_pair_mxf4_ss_elect(tmem, ad, bd, idesc_sf_ids(idesc, id, id), sfa_t + 4 * u,
                                     sfb_t + 8 * u, acc);
            } else {
              mma_pair_nvf4_ss_elect(tmem, ad, bd, idesc, sfa_t + 4 * kb, sfb_t + 8 * kb, acc);
            }
          }
          tc_commit_pair_mc_elect(&sh->empty[stage], 0x3);
          if (++stage == kPairStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair_mc_elect(&sh->acc_full, 0x3);
        acc_phase ^= 1;
      }
      if (!ok && lane == 0) *abort = 1;
      tc_commit_pair_elect(&sh->drain);
      if (lane == 0) mbar_wait(&sh->drain, 0, nullptr, nullptr, 0);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&sh->acc_empty), 0);
    uint8_t* slot = out_base + (warp - 2) * kPairStageOut;
    uint32_t acc_phase = 0;
    bool ok = true;
    int prob, tm, tn;
    for (int k = 0; ok && pair_walk(G, pair, npairs, k, prob, tm, tn); ++k) {
      const GemmArgs& g = G.p[prob].g;
      ok = mbar_wait(&sh->acc_full, acc_phase, err, abort, 14);
      if (!ok) break;
      acc_phase ^= 1;
      tc_fence_after();
      uint32_t r[kEpiChunks][32];
#pragma unroll
      for (int c = 0; c < kEpiChunks; ++c)
        tmem_ld32(tmem_addr(tmem, q * 32, (h * kEpiChunks + c) * 32), r[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc_empty0);
      if constexpr (kQuant < 0) {
        // fp32 rows through this warp's 2 KB slot, 16 columns at a time
        // (64-byte swizzle: 16-byte chunk j of row r at j ^ ((r / 2) % 4)),
        // and a TMA store per 32x16 chunk
        const int row0 = (2 * tm + static_cast<int>(rank)) * kBM + q * 32;
        const int col0 = tn * kBN + h * (kBN / 2);
#pragma unroll
        for (int c = 0; c < 2 * kEpiChunks; ++c) {
          if (lane == 0) bulk_wait_read0();          // the slot's last store has read it
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t* v = &r[c >> 1][16 * (c & 1) + 4 * j];
            *reinterpret_cast<float4*>(slot + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                            __uint_as_float(v[3]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < g.M) {
            tma_store_2d(prob ? &m1.d : &m0.d, col0 + 16 * c, row0, slot);
            bulk_commit();
          }
        }
      } else {
        epilogue_store<kQuant>(g, r, 2 * tm + static_cast<int>(rank), tn, q, h, lane);
      }
    }
    if (kQuant < 0 && lane == 0) bulk_wait0();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();                                    // both CTAs done with TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  cluster_sync();
}

}  // namespace
}  // namespace lpfa

using namespace lpfa;

namespace {
// tcgen05 type code of an element format (kind::mxf8f6f4)
uint32_t mma_type_code(lpfa_elem f) {
  switch (f) {
    case LPFA_ELEM_E4M3: return 0;
    case LPFA_ELEM_E5M2: return 1;
    case LPFA_ELEM_E2M3: return 3;
    case LPFA_ELEM_E3M2: return 4;
    case LPFA_ELEM_E2M1: return 5;
  }
  return 0;
}

// One pair-kernel problem from the GEMM's arguments (g: M, N, K, tile counts
// and outputs already set): the tensor maps of A and B (128-row boxes), of
// the scale tiles (rows of 128 32-bit words; A rows past the last 128-row
// tile read as zeros) and of the fp32 D (32-row x 16-column boxes, 64-byte
// swizzle; rows past M are not written), and the M = 256 instruction
// descriptor.
lpfa_status pair_problem(const GemmArgs& g, const void* a8, const void* b8, const void* sfa_mma,
                         const void* sfb_mma, float* d, int quant, lpfa_elem a_fmt,
                         lpfa_elem b_fmt, int kind, PairProblem* pp, PairMaps* pm) {
  const int sfa_tiles = kind == kKindNvf4 ? 4 : kind == kKindMxf4 ? 2 : 1;
  const uint64_t M = static_cast<uint64_t>(g.M), N = static_cast<uint64_t>(g.N),
                 K = static_cast<uint64_t>(g.K);
  {
    uint64_t dims[2] = {K, M};
    uint64_t strides[1] = {K};
    uint32_t box[2] = {kBK, 128};
    lpfa_status st = encode_tmap(&pm->a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a8, dims, strides, box,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != LPFA_OK) return st;
  }
  {
    uint64_t dims[2] = {K, N};
    uint64_t strides[1] = {K};
    uint32_t box[2] = {kBK, 128};
    lpfa_status st = encode_tmap(&pm->b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b8, dims, strides, box,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != LPFA_OK) return st;
  }
  {
    uint64_t dims[2] = {128, static_cast<uint64_t>(g.tiles_m) * g.kt * sfa_tiles};
    uint64_t strides[1] = {512};
    uint32_t box[2] = {128, static_cast<uint32_t>(sfa_tiles)};
    lpfa_status st = encode_tmap(&pm->sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, sfa_mma, dims,
                                 strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != LPFA_OK) return st;
  }
  {
    // [N/128 row tiles][kt * sfa_tiles tiles][128 words]: both B halves of a
    // stage in one box
    const uint64_t tiles_k = static_cast<uint64_t>(g.kt) * sfa_tiles;
    uint64_t dims[3] = {128, tiles_k, N / 128};
    uint64_t strides[2] = {512, tiles_k * 512};
    uint32_t box[3] = {128, static_cast<uint32_t>(sfa_tiles), 2};
    lpfa_status st = encode_tmap(&pm->sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, sfb_mma, dims,
                                 strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != LPFA_OK) return st;
  }
  pm->d = pm->sfa;
  if (quant < 0) {
    uint64_t dims[2] = {N, M};
    uint64_t strides[1] = {N * 4};
    uint32_t box[2] = {16, 32};
    lpfa_status st = encode_tmap(&pm->d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, d, dims, strides, box,
                                 CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != LPFA_OK) return st;
  }
  pp->g = g;
  pp->g.idesc = kind == kKindF8F6F4
                    ? idesc_mx_types(2 * kBM, kBN, mma_type_code(a_fmt), mma_type_code(b_fmt))
                    : (idesc_mx_types(2 * kBM, kBN, 1, 1) & ~(1u << 23)) |
                          (kind == kKindMxf4 ? (1u << 23) : 0u);
  pp->tiles_m2 = static_cast<int32_t>((g.M + 255) / 256);
  pp->ntiles = pp->tiles_m2 * g.tiles_n;
  return LPFA_OK;
}

// Launches the pair kernel on one or two problems (two: fp32 output, one
// kind; the longer-contraction problem is put in slot 1 and the split of
// slot 0's tiles over the pairs balances the stage counts).
lpfa_status launch_pair(int kind, int quant, PairGroup& G, const PairMaps& m0,
                        const PairMaps& m1, cudaStream_t cs) {
  const size_t psmem = kind == kKindNvf4   ? PairCfg<kKindNvf4>::kSmem
                       : kind == kKindMxf4 ? PairCfg<kKindMxf4>::kSmem
                                           : PairCfg<kKindF8F6F4>::kSmem;
  auto go2 = [&](auto kernel) -> lpfa_status {
    lpfa_status st = set_max_dynamic_smem(reinterpret_cast<const void*>(kernel),
                                          static_cast<int>(psmem));
    if (st != LPFA_OK) return st;
    const int clusters = max_active_clusters(reinterpret_cast<const void*>(kernel), kThreads,
                                             static_cast<int>(psmem));
    if (clusters <= 0) return LPFA_ERR_UNSUPPORTED;
    int64_t ptiles = G.p[0].ntiles + (G.nprob > 1 ? G.p[1].ntiles : 0);
    const int np = static_cast<int>(ptiles < clusters ? ptiles : clusters);
    if (G.nprob > 1) {
      // closed-form balance of the stage counts
      const int64_t n0 = G.p[0].ntiles, n1 = G.p[1].ntiles;
      const double kt0 = G.p[0].g.kt, kt1 = G.p[1].g.kt;
      const double target = (n0 * kt0 + n1 * kt1) / np;
      const int64_t a1 = n1 / np;
      G.r = static_cast<int32_t>(n1 % np);
      G.c_hi = static_cast<int32_t>(std::max(0.0, std::floor((target - (a1 + 1) * kt1) / kt0)));
      G.c_lo = static_cast<int32_t>(std::max(0.0, std::floor((target - a1 * kt1) / kt0)));
      const int64_t extra = n0 - (static_cast<int64_t>(G.r) * G.c_hi +
                                  static_cast<int64_t>(np - G.r) * G.c_lo);
      if (extra >= 0 && extra <= np) {
        G.extra = static_cast<int32_t>(extra);
      } else {                                   // plain even split
        G.r = 0;
        G.c_hi = G.c_lo = static_cast<int32_t>(n0 / np);
        G.extra = static_cast<int32_t>(n0 % np);
      }
    }
    kernel<<<2 * np, kThreads, psmem, cs>>>(m0, m1, G);
    LPFA_CHECK_CUDA(cudaGetLastError());
    return LPFA_OK;
  };
  if (kind == kKindMxf4) return go2(mx_gemm_pair_kernel<-1, kKindMxf4>);
  if (kind == kKindNvf4) return go2(mx_gemm_pair_kernel<-1, kKindNvf4>);
  if (quant < 0) return go2(mx_gemm_pair_kernel<-1, kKindF8F6F4>);
  if (quant == 0) return go2(mx_gemm_pair_kernel<0, kKindF8F6F4>);
  return go2(mx_gemm_pair_kernel<2, kKindF8F6F4>);
}

lpfa_status launch_gemm(const void* a8, const void* sfa_mma, const void* b8,
                        const void* sfb_mma, float* d, int64_t M, int64_t N, int64_t K,
                        int quant, uint8_t* q, uint8_t* qsf, uint8_t* qsf_mma,
                        uint8_t* qsf_mma_t, void* stream,
                        lpfa_elem a_fmt = LPFA_ELEM_E4M3, lpfa_elem b_fmt = LPFA_ELEM_E4M3,
                        int kind = kKindF8F6F4) {
  LPFA_CHECK_ARG(a8 && sfa_mma && b8 && sfb_mma);
  LPFA_CHECK_ARG(aligned16(a8) && aligned16(b8) && aligned16(sfa_mma) &&
                 aligned16(sfb_mma) && aligned16(d));
  LPFA_CHECK_ARG(M > 0 && N > 0 && K > 0);
  // a ragged M (rows past it load as zeros and are not stored) only with the
  // fp32 output
  if ((quant >= 0 && M % kBM != 0) || N % kBN != 0 || K % kBK != 0) return LPFA_ERR_UNSUPPORTED;
  LPFA_CHECK_ARG(M < (1 << 20) && N < (1 << 20) && K < (1 << 20));
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  CUtensorMap ta, tb;
  {
    uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    uint64_t strides[1] = {static_cast<uint64_t>(K)};
    uint32_t box[2] = {kBK, kBM};
    lpfa_status st = encode_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a8, dims,
                                 strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != LPFA_OK) return st;
  }
  {
    uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N)};
    uint64_t strides[1] = {static_cast<uint64_t>(K)};
    uint32_t box[2] = {kBK, kBN};
    lpfa_status st = encode_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b8, dims,
                                 strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != LPFA_OK) return st;
  }
  GemmArgs g;
  g.sfa = static_cast<const uint8_t*>(sfa_mma);
  g.sfb = static_cast<const uint8_t*>(sfb_mma);
  g.d = d;
  g.q = q;
  g.qsf = qsf;
  g.qsf_mma = qsf_mma;
  g.qsf_mma_t = qsf_mma_t;
  g.M = static_cast<int32_t>(M);
  g.N = static_cast<int32_t>(N);
  g.K = static_cast<int32_t>(K);
  g.tiles_m = static_cast<int32_t>(ceil_div(M, kBM));
  g.tiles_n = static_cast<int32_t>(N / kBN);
  g.kt = static_cast<int32_t>(K / kBK);
  g.err = nullptr;
  // kind::mxf4nvf4: E2M1 is type 1; bit 23 selects UE8M0 (MXFP4) or UE4M3
  // (NVFP4) scales
  g.idesc = kind == kKindF8F6F4
                ? idesc_mx_types(kBM, kBN, mma_type_code(a_fmt), mma_type_code(b_fmt))
                : (idesc_mx_types(kBM, kBN, 1, 1) & ~(1u << 23)) |
                      (kind == kKindMxf4 ? (1u << 23) : 0u);

  // CTA pairs (every kind): any M with the fp32 output, M a multiple of 256
  // with the quantizing epilogue
  if (quant < 0 || M % 256 == 0) {
    PairGroup G{};
    PairMaps m0;
    lpfa_status st = pair_problem(g, a8, b8, sfa_mma, sfb_mma, d, quant, a_fmt, b_fmt, kind,
                                  &G.p[0], &m0);
    if (st != LPFA_OK) return st;
    G.nprob = 1;
    return launch_pair(kind, quant, G, m0, m0, cs);
  }

  const size_t smem = kStages * (kind == kKindNvf4   ? GemmCfg<kKindNvf4>::kStageBytes
                                 : kind == kKindMxf4 ? GemmCfg<kKindMxf4>::kStageBytes
                                                     : GemmCfg<kKindF8F6F4>::kStageBytes) +
                      sizeof(GemmSmem) + 1024;
  const int ntiles = g.tiles_m * g.tiles_n;
  const int grid = ntiles < num_sms() ? ntiles : num_sms();
  auto go = [&](auto kernel) -> lpfa_status {
    lpfa_status st = set_max_dynamic_smem(reinterpret_cast<const void*>(kernel),
                                          static_cast<int>(smem));
    if (st != LPFA_OK) return st;
    kernel<<<grid, kThreads, smem, cs>>>(ta, tb, g);
    LPFA_CHECK_CUDA(cudaGetLastError());
    return LPFA_OK;
  };
  // one CTA per 128x256 tile: the quantizing epilogue when M % 256 == 128
  if (quant == 0) return go(mx_gemm_kernel<0, kKindF8F6F4>);
  return go(mx_gemm_kernel<2, kKindF8F6F4>);
}
}  // namespace

extern "C" lpfa_status lpfa_mx_gemm_grouped(const lpfa_gemm_problem* problems, int32_t count,
                                            void* stream) {
  LPFA_CHECK_ARG(problems != nullptr && (count == 1 || count == 2));
  PairGroup G{};
  PairMaps m[2];
  for (int i = 0; i < count; ++i) {
    const lpfa_gemm_problem& pr = problems[i];
    LPFA_CHECK_ARG(pr.a && pr.sfa_mma && pr.b && pr.sfb_mma && pr.d);
    LPFA_CHECK_ARG(aligned16(pr.a) && aligned16(pr.b) && aligned16(pr.sfa_mma) &&
                   aligned16(pr.sfb_mma) && aligned16(pr.d));
    LPFA_CHECK_ARG(pr.M > 0 && pr.N > 0 && pr.K > 0);
    LPFA_CHECK_ARG(pr.M < (1 << 20) && pr.N < (1 << 20) && pr.K < (1 << 20));
    if (pr.N % kBN != 0 || pr.K % kBK != 0) return LPFA_ERR_UNSUPPORTED;
    GemmArgs g{};
    g.sfa = static_cast<const uint8_t*>(pr.sfa_mma);
    g.sfb = static_cast<const uint8_t*>(pr.sfb_mma);
    g.d = pr.d;
    g.M = static_cast<int32_t>(pr.M);
    g.N = static_cast<int32_t>(pr.N);
    g.K = static_cast<int32_t>(pr.K);
    g.tiles_m = static_cast<int32_t>(ceil_div(pr.M, kBM));
    g.tiles_n = static_cast<int32_t>(pr.N / kBN);
    g.kt = static_cast<int32_t>(pr.K / kBK);
    lpfa_status st = pair_problem(g, pr.a, pr.b, pr.sfa_mma, pr.sfb_mma, pr.d, -1, LPFA_ELEM_E4M3,
                                  LPFA_ELEM_E4M3, kKindF8F6F4, &G.p[i], &m[i]);
    if (st != LPFA_OK) return st;
  }
  G.nprob = count;
  if (count == 2 && G.p[0].g.kt > G.p[1].g.kt) {   // slot 1: the longer contraction
    std::swap(G.p[0], G.p[1]);
    std::swap(m[0], m[1]);
  }
  return launch_pair(kKindF8F6F4, -1, G, m[0], m[count - 1], static_cast<cudaStream_t>(stream));
}

extern "C" lpfa_status lpfa_mx_gemm(const void* a8, const void* sfa_mma,
                                    const void* b8, const void* sfb_mma,
                                    float* d, int64_t M, int64_t N, int64_t K,
                                    void* stream) {
  LPFA_CHECK_ARG(d != nullptr);
  return launch_gemm(a8, sfa_mma, b8, sfb_mma, d, M, N, K, -1, nullptr, nullptr, nullptr,
                     nullptr, stream);
}

namespace lpfa {
namespace {
// One thread per 16-element group: one-per-byte codes -> the tensor core's
// operand bytes (FP6: a little-endian 96-bit stream of 6-bit codes, then 4
// zero bytes; FP4: 8 bytes of nibbles, element 2i low, then 8 zero bytes).
template <int kBits>
__global__ void pack_operand_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                    int64_t groups) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= groups) return;
  const uint4 v = in[i];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint64_t lo = 0, hi = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint64_t c = (w[e >> 2] >> (8 * (e & 3))) & ((1u << kBits) - 1u);
    const int pos = kBits * e;
    if (pos < 64) {
      lo |= c << pos;
      if (pos + kBits > 64) hi |= c >> (64 - pos);
    } else {
      hi |= c << (pos - 64);
    }
  }
  out[i] = make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32),
                      static_cast<uint32_t>(hi), 0u);
}
// One thread per 16 codes: one-per-byte E2M1 codes -> 8 bytes of nibbles
// (element 2i in the low nibble), the dense operand of kind::mxf4nvf4.
__global__ void pack_fp4_dense_kernel(const uint4* __restrict__ in, uint2* __restrict__ out,
                                      int64_t groups) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= groups) return;
  const uint4 v = in[i];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e)
    o[e >> 3] |= ((w[e >> 2] >> (8 * (e & 3))) & 0xFu) << (4 * (e & 7));
  out[i] = make_uint2(o[0], o[1]);
}
}  // namespace
}  // namespace lpfa

extern "C" lpfa_status lpfa_fp4_pack_dense(const void* codes, int64_t rows, int64_t cols,
                                           void* out, void* stream) {
  LPFA_CHECK_ARG(codes != nullptr && out != nullptr && aligned16(codes));
  LPFA_CHECK_ARG((reinterpret_cast<uintptr_t>(out) & 7u) == 0);
  LPFA_CHECK_ARG(rows >= 0 && cols >= 0 && cols % 16 == 0);
  const int64_t groups = rows * (cols / 16);
  if (groups == 0) return LPFA_OK;
  LPFA_CHECK_ARG(ceil_div(groups, 256) < (1ll << 31));
  pack_fp4_dense_kernel<<<static_cast<unsigned>(ceil_div(groups, 256)), 256, 0,
                          static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(codes), static_cast<uint2*>(out), groups);
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}

extern "C" lpfa_status lpfa_mx_gemm_fp4(const void* a, const void* sfa_mma, const void* b,
                                        const void* sfb_mma, float* d, int64_t M, int64_t N,
                                        int64_t K, int nvfp4, void* stream) {
  LPFA_CHECK_ARG(d != nullptr && (nvfp4 == 0 || nvfp4 == 1));
  LPFA_CHECK_ARG(K > 0 && K % 2 == 0);
  if (K % 256 != 0) return LPFA_ERR_UNSUPPORTED;
  return launch_gemm(a, sfa_mma, b, sfb_mma, d, M, N, K / 2, -1, nullptr, nullptr, nullptr,
                     nullptr, stream, LPFA_ELEM_E2M1, LPFA_ELEM_E2M1,
                     nvfp4 ? kKindNvf4 : kKindMxf4);
}

extern "C" lpfa_status lpfa_mx_pack_operand(const void* codes, int64_t rows, int64_t cols,
                                            lpfa_elem fmt, void* out, void* stream) {
  LPFA_CHECK_ARG(codes != nullptr && out != nullptr && aligned16(codes) && aligned16(out));
  LPFA_CHECK_ARG(rows >= 0 && cols >= 0 && cols % 16 == 0);
  LPFA_CHECK_ARG(fmt >= LPFA_ELEM_E4M3 && fmt <= LPFA_ELEM_E2M1);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int64_t groups = rows * (cols / 16);
  if (groups == 0) return LPFA_OK;
  if (fmt == LPFA_ELEM_E4M3 || fmt == LPFA_ELEM_E5M2) {
    if (codes != out)
      LPFA_CHECK_CUDA(cudaMemcpyAsync(out, codes, static_cast<size_t>(rows * cols),
                                      cudaMemcpyDeviceToDevice, cs));
    return LPFA_OK;
  }
  LPFA_CHECK_ARG(ceil_div(groups, 256) < (1ll << 31));
  const unsigned blocks = static_cast<unsigned>(ceil_div(groups, 256));
  if (fmt == LPFA_ELEM_E2M1)
    pack_operand_kernel<4><<<blocks, 256, 0, cs>>>(static_cast<const uint4*>(codes),
                                                   static_cast<uint4*>(out), groups);
  else
    pack_operand_kernel<6><<<blocks, 256, 0, cs>>>(static_cast<const uint4*>(codes),
                                                   static_cast<uint4*>(out), groups);
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}

extern "C" lpfa_status lpfa_mx_gemm_fmt(const void* a, const void* sfa_mma, const void* b,
                                        const void* sfb_mma, float* d, int64_t M, int64_t N,
                                        int64_t K, lpfa_elem a_fmt, lpfa_elem b_fmt,
                                        void* stream) {
  LPFA_CHECK_ARG(d != nullptr);
  LPFA_CHECK_ARG(a_fmt >= LPFA_ELEM_E4M3 && a_fmt <= LPFA_ELEM_E2M1);
  LPFA_CHECK_ARG(b_fmt >= LPFA_ELEM_E4M3 && b_fmt <= LPFA_ELEM_E2M1);
  return launch_gemm(a, sfa_mma, b, sfb_mma, d, M, N, K, -1, nullptr, nullptr, nullptr,
                     nullptr, stream, a_fmt, b_fmt);
}

extern "C" lpfa_status lpfa_mx_gemm_quantize(const void* a8, const void* sfa_mma,
                                             const void* b8, const void* sfb_mma,
                                             int64_t M, int64_t N, int64_t K, lpfa_block blk,
                                             void* out_e4m3, void* out_sf, void* out_sf_mma,
                                             void* out_sf_mma_t, float* d, void* stream) {
  LPFA_CHECK_ARG(out_e4m3 != nullptr && aligned16(out_e4m3));
  LPFA_CHECK_ARG(out_sf == nullptr || (reinterpret_cast<uintptr_t>(out_sf) & 7u) == 0);
  LPFA_CHECK_ARG(out_sf_mma == nullptr || aligned16(out_sf_mma));
  LPFA_CHECK_ARG(out_sf_mma_t == nullptr || blk == LPFA_BLK_32X32);
  if (blk != LPFA_BLK_1X32 && blk != LPFA_BLK_32X32) return LPFA_ERR_UNSUPPORTED;
  return launch_gemm(a8, sfa_mma, b8, sfb_mma, d, M, N, K, blk == LPFA_BLK_1X32 ? 0 : 2,
                     static_cast<uint8_t*>(out_e4m3), static_cast<uint8_t*>(out_sf),
                     static_cast<uint8_t*>(out_sf_mma), static_cast<uint8_t*>(out_sf_mma_t),
                     stream);
}
