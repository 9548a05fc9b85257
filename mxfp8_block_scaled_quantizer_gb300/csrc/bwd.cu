// MXFP8 block-scaled attention backward on tcgen05.
//
// Method ("Low Precision Flash Attention 4: End-to-End Block-Scaled Attention
// for Blackwell", paragraphs 2-3): Q, K, dO arrive quantized in square 32x32
// blocks, so one E4M3 payload serves both orientations of every GEMM (only
// the scale arrangement differs); V in 1x32 blocks along head_dim.  Per key
// tile the kernel recomputes P from the forward LSE, forms
// dS = P o (dP - D) with D_i = rowsum(dO o O), quantizes P and dS online in
// 32x32 blocks (per-lane max, then a warp-wide redux.sync max), and
// accumulates
//   dV += P^T dO,  dK += dS^T Q   (TMEM-resident over the query loop)
//   dQ^T = K^T dS^T               (per query step; scaled by softmax_scale *
//                                  dq_static_scale, rounded to FP16 and added
//                                  to the FP16 dQ in global memory with bulk
//                                  reduce-adds)
//
// CTA = one 128-key tile of one (sequence, kv head); it loops over the query
// heads of its GQA group and over 64-query steps (causal: from the diagonal).
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 2-9
// compute in two warpgroups, each owning 32 of the step's 64 queries (thread
// = key row for S^T/dP^T, = head_dim channel for dQ^T).  dQ partials leave
// as FP16 tensor reduce-adds, one per warp (32 queries x 32 channels).
//
// TMEM (512 columns):
//   [  0,128) dK      [128,256) dV      [256,320) S^T      [320,384) dP^T
//   [384,448) dQ^T, which between steps also holds the fp8 P^T / dS^T of
//             query block g at columns 32g / 32g + 8 (inside the slice that
//             warpgroup g alone reads back)
// The steps are software-pipelined: S^T / dP^T of step i+1 are issued as
// soon as step i's rows are in registers, and a warpgroup reads back dQ^T of
// step i-1 after computing step i, so the MMAs of one step overlap the
// elementwise work of the next.
//   [448,512) scale factors and the seed MMA's constant A tile (kCol* below)
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "lpfa_device.cuh"
#include "lpfa_internal.h"
#include "lpfa_seq.cuh"

namespace lpfa {
namespace {

constexpr int kBN = 128;         // keys per CTA
constexpr int kBQ = 64;          // queries per step
constexpr int kThreads = 320;
constexpr int kLseSlotsMax = 4;  // LSE / D row slots (see BwdCfg::kLseSlots)
constexpr int kTmemCols = 512;

// Layout for head_dim D (64 or 128).  B16 selects the bf16 variant (kind::f16
// MMAs on bf16 operands, P^T and dS^T rounded to bf16, no block scales),
// which exists to measure the MXFP8 kernel against the same algorithm in
// bf16.  Operand tiles are stored as chunks of at most 128 bytes per row (one
// swizzle span): a bf16 row of 128 channels is two chunks, [chunk][rows][128 B].
template <int D, bool B16>
struct BwdCfg {
  static constexpr int kEl = B16 ? 2 : 1;                // bytes per element
  static constexpr int kRowB = D * kEl;                  // bytes per token row
  static constexpr int kChunkB = kRowB < 128 ? kRowB : 128;
  static constexpr int kNCh = kRowB / kChunkB;           // chunks per row
  static constexpr uint32_t kSw = kChunkB == 128 ? 2u : 4u;   // 128B / 64B swizzle
  static constexpr uint32_t kSbo = 8 * kChunkB;               // 8 rows of a chunk
  static constexpr int kStages = B16 ? 3 : 5;   // Q / dO ring: loads run steps ahead
  // The producer builds a step's accumulator seed kLag steps after issuing
  // its copies from -log2 LSE / -D rows requested kLseAhead steps before
  // the copies (measured: the deep MXFP8 ring is fastest with the rows
  // requested beside the copies and the seed one step behind, the shallow
  // bf16 ring with the rows two steps ahead and no lag).  A slot is refilled
  // kLseSlots steps after its previous fill, by which time that fill's seed
  // must have been built: kLseSlots >= kLseAhead + kLag + 1.
  static constexpr int kLag = kStages >= 4 ? 1 : 0;
  static constexpr int kLseAhead = kStages >= 4 ? 0 : 2;
  static constexpr int kLseSlots = kLseAhead + kLag + 1;
  static_assert(kLseSlots <= kLseSlotsMax, "LSE slots");
  static constexpr int kDqBufs = 1;            // dQ staging tiles per compute warp (two ran 0.3 %, four 1.2 % slower)
  static constexpr int kKSteps = kRowB / 32;    // MMA K-steps over head_dim (32 bytes each)
  static constexpr int kQPerStep = 32 / kEl;    // queries / keys contracted per MMA
  // P^T and dS^T of a warpgroup's 32 queries: TMEM columns per key row
  static constexpr uint32_t kPCols = 8 * kEl;
  // TMEM columns
  static constexpr uint32_t kColDK = 0, kColDV = D, kColS = 2 * D,
                            kColDP = 2 * D + 64, kColDQ = 2 * D + 128;
  static constexpr uint32_t kColSF = 2 * D + 192;
  static constexpr uint32_t kColSFK = kColSF, kColSFV = kColSF + 4,
                            kColSFKt = kColSF + 8, kColSFQ = kColSF + 12,
                            kColSFdO = kColSF + 16, kColSFQt = kColSF + 20,
                            kColSFdOt = kColSF + 24, kColSFP = kColSF + 28 /* +4g */,
                            kColSFdS = kColSF + 36 /* +4g */, kColSFdSB = kColSF + 44;
  // constant A operand of the seed MMA: [128 keys][16 bf16], 8 columns,
  // 1.0 at k = 0, 1 (selects the hi, lo pair of a seed row)
  static constexpr uint32_t kColOnes = kColSF + 48;
  // shared memory (bytes from a 1024-aligned base)
  static constexpr int kSmK = 0;                                  // 128 x D
  static constexpr int kSmV = (kBN * kRowB + 1023) / 1024 * 1024; // 128 x D
  // A operand of dQ^T = K^T dS^T needs 128 rows (channels): for fp8 D = 64 a
  // copy of the K tile zero-padded to 128 channels (64..127 give rows of
  // zeros that are never read back); otherwise the K tile itself
  static constexpr int kSmKT = kSmV + kBN * kRowB;
  static constexpr int kKTBytes = kRowB == 64 ? kBN * 128 : 0;
  static constexpr int kSmStage0 = kSmKT + kKTBytes;              // Q, dO, SFs, seed
  static constexpr int kStQ = 0;
  static constexpr int kStdO = kBQ * kRowB;
  static constexpr int kStSF = 2 * kBQ * kRowB;                   // SFQ, SFQt, SFdO, SFdOt
  // accumulator seeds: [128 rows][16 bf16] K-major, 32-byte swizzle; row q
  // holds hi, lo of -LSE_q / c and row 64 + q those of -D_q (k = 0, 1), so
  // that one N = 128 MMA seeds the adjacent S^T and dP^T columns
  static constexpr int kStSeed = ((kStSF + (B16 ? 0 : 4 * 512)) + 255) / 256 * 256;
  static constexpr int kStageBytes = ((kStSeed + 2 * kBQ * 32) + 1023) / 1024 * 1024;
  static_assert(kColDP == kColS + kBQ, "the seed MMA spans S^T and dP^T");
  // dS^T tile [128 keys][64 queries]: 64-byte rows, 64B swizzle (fp8) or
  // 128-byte rows, 128B swizzle (bf16)
  static constexpr int kDsRowB = kBQ * kEl;
  static constexpr uint32_t kDsSw = kDsRowB == 128 ? 2u : 4u;
  static constexpr int kSmDS = kSmStage0 + kStages * kStageBytes;
  static constexpr int kSmSFdS = kSmDS + kBN * kDsRowB;           // 512 B
  static constexpr int kSmSFkv = kSmSFdS + 512;                   // SFK, SFKt, SFV
  // dQ staging: per compute warp kDqBufs [32 queries][32 channels] fp16
  // tiles, 64-byte rows, 64B swizzle (2 KB each, 1024-aligned)
  // -log2 LSE and -D rows of a step (64 + 64 floats), kLseSlots of them
  static constexpr int kLseSlotB = 2 * kBQ * 4;
  static constexpr int kSmLse = kSmSFkv + 3 * 512;
  static constexpr int kSmDQ = (kSmLse + kLseSlots * kLseSlotB + 1023) / 1024 * 1024;
  static constexpr int kSmBar = kSmDQ + 8 * kDqBufs * 32 * 32 * 2;
  static constexpr int kSmTotal = kSmBar + 256;
  static_assert(kSmTotal + 1024 <= 227 * 1024, "shared memory per CTA");
};

struct BwdParams {
  SeqView seqs;
  const uint8_t* sfq;    // [Tp/128, Hq, 512] contraction over head_dim
  const uint8_t* sfq_t;  // contraction over tokens
  const uint8_t* sfk;
  const uint8_t* sfk_t;
  const uint8_t* sfv;
  const uint8_t* sfdo;
  const uint8_t* sfdo_t;
  const float* lse2;     // [Hq, Tp]  -LSE * log2(e), padded rows
  const float* delta;    // [Hq, Tp]  -D
  __half* dq;            // [T, Hq, D] fp16, accumulated
  __nv_bfloat16* dk;     // [T, Hkv, D]
  __nv_bfloat16* dv;
  uint32_t* err;
  int32_t hq, hkv, group;
  int32_t causal;
  float scale_log2;      // softmax_scale * log2(e)
  float softmax_scale;
  float dq_mult;         // softmax_scale * dq_static_scale
};

template <int kStages>
struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[kStages];    // Q, dO, scales landed and the seed tile written
  uint64_t q_empty[kStages];
  uint64_t lse_full[kLseSlotsMax];  // a slot's -log2 LSE and -D rows landed
  uint64_t st_ready;
  uint64_t ds_ready;
  uint64_t dq_full;
  uint64_t st_loaded;
  uint64_t acc_done;
  uint64_t kt_ready;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct KvItem {
  int seq, ktile, kvh;
  int64_t start;
  int32_t len;
  int64_t sf_tile0;   // first padded 128-row tile of the sequence
};

__device__ __forceinline__ KvItem kv_item(const BwdParams& p) {
  KvItem w;
  const int64_t idx = blockIdx.x;
  w.kvh = static_cast<int>(idx % p.hkv);
  const int64_t t = idx / p.hkv;       // padded tile index
  w.seq = seq_of_sf_row(p.seqs, t * 128);
  const SeqInfo si = seq_info(p.seqs, w.seq);
  w.ktile = static_cast<int>((t * 128 - si.sf_start) / 128);
  w.start = si.start;
  w.len = si.len;
  w.sf_tile0 = si.sf_start / 128;
  return w;
}

// Scale 32 values (one thread's row of a 32x32 block) by 2^-e for the E8M0
// code of the block's amax (given as fp32 bits) and convert to E4M3; a block
// holding Inf or NaN gets code 0xFF and payloads 0x7F.  Writes 8 packed
// words, returns the code.
__device__ __forceinline__ uint32_t quant_block32(const float (&v)[32], uint32_t amax_bits,
                                                  uint32_t (&w)[8]) {
  const uint32_t code = e8m0_code_from_amax_bits(amax_bits);
  const float inv = inv_scale_from_code(code);
  const uint64_t inv2 = pack2(inv, inv);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t a = mul2(pack2(v[4 * i], v[4 * i + 1]), inv2);
    const uint64_t b = mul2(pack2(v[4 * i + 2], v[4 * i + 3]), inv2);
    w[i] = cvt_e4m3x4(lo2(a), hi2(a), lo2(b), hi2(b));
  }
  if (code == 0xFFu) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = 0x7F7F7F7Fu;
  }
  return code;
}

// max(|a|, |b|, |c|), NaN-propagating.
__device__ __forceinline__ float max3_abs_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Warp-wide maximum of non-negative fp32 values (NaN above +Inf), as bits:
// for such values the unsigned order of the bits is the numeric order.
__device__ __forceinline__ uint32_t warp_max_nonneg_bits(float x) {
  return __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(x));
}

// Shared-memory descriptor offset (16-byte units) of K-step kb (32 bytes of
// K) of a K-major operand tile stored in chunks of kChunkB-byte rows, `rows`
// rows each.
template <int kChunkB>
__device__ __forceinline__ constexpr uint64_t kstep_off(int kb, int rows) {
  return static_cast<uint64_t>((kb / (kChunkB / 32)) * rows * kChunkB +
                               (kb % (kChunkB / 32)) * 32) >> 4;
}

template <int D, bool B16>
__global__ void __launch_bounds__(kThreads, 1)
    mx_attn_bwd_kernel(const __grid_constant__ CUtensorMap tma_q,
                       const __grid_constant__ CUtensorMap tma_k,
                       const __grid_constant__ CUtensorMap tma_v,
                       const __grid_constant__ CUtensorMap tma_do,
                       const __grid_constant__ CUtensorMap tma_dq,
                       const BwdParams p) {
  using C = BwdCfg<D, B16>;
  constexpr int kStages = C::kStages;
  constexpr int kDqBufs = C::kDqBufs;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdBars<kStages>* bars = reinterpret_cast<BwdBars<kStages>*>(sm + C::kSmBar);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const KvItem w = kv_item(p);
  const int k0 = w.ktile * kBN;                    // first key (in sequence)
  if (k0 >= w.len) return;
  const int qstep0 = p.causal ? (k0 / kBQ) : 0;    // first 64-query step
  const int nqsteps = (w.len + kBQ - 1) / kBQ;
  const int steps_per_head = nqsteps - qstep0;
  const int nsteps = steps_per_head * p.group;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->q_full[s], 2);
      mbar_init(&bars->q_empty[s], 1);
    }
    for (int s = 0; s < C::kLseSlots; ++s) {
      mbar_init(&bars->lse_full[s], 1);
    }
    mbar_init(&bars->st_ready, 1);
    mbar_init(&bars->ds_ready, 8);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->st_loaded, 8);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->kt_ready, 4);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // the seed MMA's constant A operand (one warpgroup covers the 128 lanes)
  if (warp >= 2 && warp < 6) {
    const uint32_t lanes = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t one2 = 0x3F803F80u;   // bf16 pair (1.0, 1.0)
    const uint32_t ol[8] = {one2, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    tmem_st8(tmem + lanes + C::kColOnes, ol);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // step i -> (query head, first query of the step)
  auto step_head = [&](int i) { return w.kvh * p.group + i / steps_per_head; };
  auto step_q0 = [&](int i) { return (qstep0 + i % steps_per_head) * kBQ; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (converged); an elected lane issues the
    // copies.
    if (lane == 0) {
      tma_prefetch_desc(&tma_q);
      tma_prefetch_desc(&tma_k);
      tma_prefetch_desc(&tma_v);
      tma_prefetch_desc(&tma_do);
      tma_prefetch_desc(&tma_dq);
    }
    const int32_t row_k = static_cast<int32_t>(w.start + k0);
    const int64_t ksf = (w.sf_tile0 + w.ktile) * p.hkv + w.kvh;
    mbar_arrive_expect_tx_elect(&bars->kv_full, 2 * kBN * C::kRowB + (B16 ? 0 : 3 * 512));
#pragma unroll
    for (int c = 0; c < C::kNCh; ++c) {
      const int32_t x = c * (C::kChunkB / C::kEl);
      tma_load_3d_elect(sm + C::kSmK + c * kBN * C::kChunkB, &tma_k, x, w.kvh, row_k,
                        &bars->kv_full);
      tma_load_3d_elect(sm + C::kSmV + c * kBN * C::kChunkB, &tma_v, x, w.kvh, row_k,
                        &bars->kv_full);
    }
    if constexpr (!B16) {
      bulk_load_elect(sm + C::kSmSFkv, p.sfk + ksf * 512, 512, &bars->kv_full);
      bulk_load_elect(sm + C::kSmSFkv + 512, p.sfk_t + ksf * 512, 512, &bars->kv_full);
      bulk_load_elect(sm + C::kSmSFkv + 1024, p.sfv + ksf * 512, 512, &bars->kv_full);
    }
    // Zeroed seed tiles (32-byte swizzle: the 16-byte half k/8 of row r
    // sits at half (k/8) ^ ((r >> 2) & 1)).  The first q_full arrival below
    // publishes them to the tensor pipe.
    {
      for (int st = 0; st < kStages; ++st) {
        uint32_t* seed = reinterpret_cast<uint32_t*>(sm + C::kSmStage0 + st * C::kStageBytes + C::kStSeed);
        for (int i = lane; i < 2 * kBQ * 8; i += 32) seed[i] = 0u;
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    const float inv_c2 = 1.f / p.scale_log2;
    bool ok = true;
    int issued[kStages];
    for (int s = 0; s < kStages; ++s) issued[s] = -1;
    // The -log2 LSE and -D rows of a step run in a ring of their own,
    // requested ahead of the step's copies, so that the seed (and with it
    // the stage's q_full) does not wait a memory round trip behind them.
    // Only this warp reads the ring: a slot is free again once its seed is
    // built.
    constexpr int kLseAhead = C::kLseAhead, kLseSlots = C::kLseSlots, kLag = C::kLag;
    int lse_issued = 0, lse_used = 0;
    auto issue_lse = [&](int j) {
      const int slot = j % kLseSlots;
      const int64_t pr = w.sf_tile0 * 128 + step_q0(j);      // padded row of the step
      const int64_t rowoff = static_cast<int64_t>(step_head(j)) * p.seqs.total_sf_rows + pr;
      uint8_t* dst = sm + C::kSmLse + slot * C::kLseSlotB;
      mbar_arrive_expect_tx_elect(&bars->lse_full[slot], 2 * kBQ * 4);
      bulk_load_elect(dst, p.lse2 + rowoff, kBQ * 4, &bars->lse_full[slot]);
      bulk_load_elect(dst + kBQ * 4, p.delta + rowoff, kBQ * 4, &bars->lse_full[slot]);
      ++lse_issued;
    };
    // seed rows of step j (stage s) once its rows have landed: -LSE_q / c =
    // -log2LSE_q / c2 and -D_q, each as a bf16 pair hi + lo (hi = bf16(v),
    // lo = bf16(v - hi): ~16 significant bits); then the second q_full
    // arrival (also on abort, so that the phase can still complete once the
    // copies land)
    auto build_seed = [&](int j, int s) -> bool {
      const int slot = j % kLseSlots;
      const bool lok = mbar_wait_sleep(&bars->lse_full[slot], (j / kLseSlots) & 1, p.err, abort, 41);
      if (lok) {
        ++lse_used;
        const float* nl = reinterpret_cast<const float*>(sm + C::kSmLse + slot * C::kLseSlotB);
        const float* nd = nl + kBQ;
        uint8_t* seed = sm + C::kSmStage0 + s * C::kStageBytes + C::kStSeed;
#pragma unroll
        for (int k = 0; k < kBQ / 32; ++k) {
          const int r = lane + 32 * k;
          const float vl = nl[r] * inv_c2, vd = nd[r];
          const __nv_bfloat16 hl = __float2bfloat16_rn(vl);
          const __nv_bfloat16 ll = __float2bfloat16_rn(vl - __bfloat162float(hl));
          const __nv_bfloat16 hd = __float2bfloat16_rn(vd);
          const __nv_bfloat16 ld = __float2bfloat16_rn(vd - __bfloat162float(hd));
          const uint32_t w0 = static_cast<uint32_t>(__bfloat16_as_ushort(hl)) |
                              (static_cast<uint32_t>(__bfloat16_as_ushort(ll)) << 16);
          const uint32_t w1 = static_cast<uint32_t>(__bfloat16_as_ushort(hd)) |
                              (static_cast<uint32_t>(__bfloat16_as_ushort(ld)) << 16);
          // k = 0, 1 of rows r and 64 + r (same swizzle phase: 64 is a
          // multiple of 8 rows)
          *reinterpret_cast<uint32_t*>(seed + r * 32 + ((r >> 2) & 1) * 16) = w0;
          *reinterpret_cast<uint32_t*>(seed + (kBQ + r) * 32 + ((r >> 2) & 1) * 16) = w1;
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_full[s]);
      return lok;
    };
    for (int j = 0; j < kLseAhead && j < nsteps; ++j) issue_lse(j);
    for (int i = 0; i < nsteps + kLag; ++i) {
      if (i < nsteps) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        ok = mbar_wait_sleep(&bars->q_empty[s], ph ^ 1, p.err, abort, 40);
        if (!ok) {
          // the pending seed still arrives on its stage's q_full
          if (kLag > 0 && i > 0) build_seed(i - 1, (i - 1) % kStages);
          break;
        }
        const int h = step_head(i), q0 = step_q0(i);
        uint8_t* st = sm + C::kSmStage0 + s * C::kStageBytes;
        uint64_t* bar = &bars->q_full[s];
        mbar_arrive_expect_tx_elect(bar, 2 * kBQ * C::kRowB + (B16 ? 0 : 4 * 512));
        const int32_t row_q = static_cast<int32_t>(w.start + q0);
#pragma unroll
        for (int c = 0; c < C::kNCh; ++c) {
          const int32_t x = c * (C::kChunkB / C::kEl);
          tma_load_3d_elect(st + C::kStQ + c * kBQ * C::kChunkB, &tma_q, x, h, row_q, bar);
          tma_load_3d_elect(st + C::kStdO + c * kBQ * C::kChunkB, &tma_do, x, h, row_q, bar);
        }
        if constexpr (!B16) {
          const int64_t qsf = ((w.sf_tile0 * 128 + q0) / 128) * p.hq + h;
          bulk_load_elect(st + C::kStSF + 0 * 512, p.sfq + qsf * 512, 512, bar);
          bulk_load_elect(st + C::kStSF + 1 * 512, p.sfq_t + qsf * 512, 512, bar);
          bulk_load_elect(st + C::kStSF + 2 * 512, p.sfdo + qsf * 512, 512, bar);
          bulk_load_elect(st + C::kStSF + 3 * 512, p.sfdo_t + qsf * 512, 512, bar);
        }
        issued[s] = static_cast<int>(ph);
        if (i + kLseAhead < nsteps) issue_lse(i + kLseAhead);
      }
      const int j = i - kLag;                      // the step whose seed is built now
      if (j >= 0) {
        ok = build_seed(j, j % kStages);
        if (!ok) {
          if (kLag > 0 && i < nsteps) build_seed(i, i % kStages);
          break;
        }
      }
    }
    if (!ok) {
      // let every copy still in flight land before the CTA exits
      for (int s = 0; s < kStages; ++s)
        if (issued[s] >= 0)
          mbar_wait_sleep(&bars->q_full[s], static_cast<uint32_t>(issued[s]), nullptr, nullptr, 0);
      for (int j = lse_used; j < lse_issued; ++j)
        mbar_wait_sleep(&bars->lse_full[j % kLseSlots], (j / kLseSlots) & 1, nullptr, nullptr, 0);
      mbar_wait_sleep(&bars->kv_full, 0, nullptr, nullptr, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (converged); the lane elect.sync picks
    // issues each tcgen05 instruction (the cheapest issue form).  Shared
    // memory descriptors are built once and offset by constants: a stage
    // adds its byte offset / 16, a K-step 32 bytes (K-major operands) or 32
    // rows (MN-major operands) to the 14-bit address field, which never
    // carries (shared memory addresses stay below 256 KB).  The step loop is
    // unrolled by the ring depth so that stage indices are constants.
    constexpr uint32_t id_st = B16 ? idesc_bf16(128, kBQ, 0, 0)
                                   : idesc_mxf8(128, kBQ, 0, 0);   // S^T, dP^T
    constexpr uint32_t id_acc = B16 ? idesc_bf16(128, D, 0, 1)
                                    : idesc_mxf8(128, D, 0, 1);    // dV, dK (B MN-major)
    constexpr uint32_t id_dq = B16 ? idesc_bf16(128, kBQ, 1, 1)
                                   : idesc_mxf8(128, kBQ, 1, 1);   // dQ^T (A, B MN-major)
    // MN-major operands of several 128-byte chunks per row repeat the swizzle
    // pattern along MN every chunk (the leading offset); K-major operands
    // ignore it
    const uint64_t dk_ = make_sdesc(smem_u32(sm + C::kSmK), 16, C::kSbo, C::kSw);
    const uint64_t dv_ = make_sdesc(smem_u32(sm + C::kSmV), 16, C::kSbo, C::kSw);
    const uint64_t dkt = make_sdesc(C::kKTBytes == 0 ? smem_u32(sm + C::kSmK) : smem_u32(sm + C::kSmKT),
                                    C::kNCh > 1 ? kBN * C::kChunkB : 16, 1024, 2);
    const uint64_t dds = make_sdesc(smem_u32(sm + C::kSmDS), 16, 8 * C::kDsRowB, C::kDsSw);
    constexpr uint32_t kQLbo = C::kNCh > 1 ? kBQ * C::kChunkB : 16;
    const uint64_t dq_ = make_sdesc(smem_u32(sm + C::kSmStage0 + C::kStQ), kQLbo, C::kSbo, C::kSw);
    const uint64_t ddo = make_sdesc(smem_u32(sm + C::kSmStage0 + C::kStdO), kQLbo, C::kSbo, C::kSw);
    const uint64_t dsf = sf_tile_desc(smem_u32(sm + C::kSmStage0 + C::kStSF));
    // seed MMA (bf16, K = 16, N = 128 over S^T and dP^T)
    constexpr uint32_t id_seed = idesc_bf16(128, 2 * kBQ, 0, 0);
    const uint64_t dseed = make_sdesc(smem_u32(sm + C::kSmStage0 + C::kStSeed), 16, 256, 6);
    const uint64_t dsfds = sf_tile_desc(smem_u32(sm + C::kSmSFdS));
    bool ok = mbar_wait_sleep(&bars->kv_full, 0, p.err, abort, 50);
    if (ok) {
      tc_fence_after();
      if constexpr (!B16) {
        tc_cp_32x128b_warpx4_elect(tmem + C::kColSFK, sf_tile_desc(smem_u32(sm + C::kSmSFkv)));
        tc_cp_32x128b_warpx4_elect(tmem + C::kColSFKt, sf_tile_desc(smem_u32(sm + C::kSmSFkv + 512)));
        tc_cp_32x128b_warpx4_elect(tmem + C::kColSFV, sf_tile_desc(smem_u32(sm + C::kSmSFkv + 1024)));
      }
    }
    // S^T(i) = K Q_i^T and dP^T(i) = V dO_i^T (contraction over head_dim)
    auto issue_st = [&](int i, int s) -> bool {
      if (!mbar_wait_sleep(&bars->q_full[s], (i / kStages) & 1, p.err, abort, 51)) return false;
      tc_fence_after();
      const uint64_t so = static_cast<uint64_t>(s) * (C::kStageBytes >> 4);
      const uint32_t half = static_cast<uint32_t>((step_q0(i) / kBQ) & 1);
      if constexpr (!B16) {
        tc_cp_32x128b_warpx4_elect(tmem + C::kColSFQ, dsf + so);
        tc_cp_32x128b_warpx4_elect(tmem + C::kColSFdO, dsf + so + (1024 >> 4));
      }
      // S^T <- -LSE / c and dP^T <- -D, broadcast over keys, in one MMA
      mma_bf16_ts_elect(tmem + C::kColS, tmem + C::kColOnes, dseed + so, id_seed, 0);
#pragma unroll
      for (int kb = 0; kb < C::kKSteps; ++kb) {
        const uint64_t ka = kstep_off<C::kChunkB>(kb, kBN), kq = kstep_off<C::kChunkB>(kb, kBQ);
        if constexpr (B16)
          mma_bf16_ss_elect(tmem + C::kColS, dk_ + ka, dq_ + so + kq, id_st, 1);
        else
          mma_mxf8_ss_elect(tmem + C::kColS, dk_ + ka, dq_ + so + kq,
                            idesc_sf_ids(id_st, kb, kb), tmem + C::kColSFK,
                            tmem + C::kColSFQ + 2 * half, 1);
      }
#pragma unroll
      for (int kb = 0; kb < C::kKSteps; ++kb) {
        const uint64_t ka = kstep_off<C::kChunkB>(kb, kBN), kq = kstep_off<C::kChunkB>(kb, kBQ);
        if constexpr (B16)
          mma_bf16_ss_elect(tmem + C::kColDP, dv_ + ka, ddo + so + kq, id_st, 1);
        else
          mma_mxf8_ss_elect(tmem + C::kColDP, dv_ + ka, ddo + so + kq,
                            idesc_sf_ids(id_st, kb, kb), tmem + C::kColSFV,
                            tmem + C::kColSFdO + 2 * half, 1);
      }
      tc_commit_elect(&bars->st_ready);
      return true;
    };
    // dV += P^T dO_i, dK += dS^T Q_i, then dQ^T(i) = K^T dS^T over the same
    // columns the fp8 P^T / dS^T came from (MMAs execute in order)
    auto issue_acc = [&](int i, int s) -> bool {
      if (!mbar_wait_sleep(&bars->ds_ready, i & 1, p.err, abort, 52)) return false;
      tc_fence_after();
      const uint64_t so = static_cast<uint64_t>(s) * (C::kStageBytes >> 4);
      const uint32_t half = static_cast<uint32_t>((step_q0(i) / kBQ) & 1);
      // K-step (C::kQPerStep queries or keys) strides of the MN-major
      // operands: Q / dO rows, K rows (dQ^T's A), dS^T rows
      constexpr uint64_t kQStep = (C::kQPerStep * C::kChunkB) >> 4;
      constexpr uint64_t kKtStep = (C::kQPerStep * 128) >> 4;
      constexpr uint64_t kDsStep = (C::kQPerStep * C::kDsRowB) >> 4;
      if constexpr (B16) {
        // block g of the step's queries: P^T at dQ^T columns 32g, dS^T at
        // 32g + 16, 8 columns (16 queries) per K-step
#pragma unroll
        for (int kb = 0; kb < kBQ / C::kQPerStep; ++kb) {
          const uint32_t col = C::kColDQ + 32 * (kb >> 1) + 8 * (kb & 1);
          mma_bf16_ts_elect(tmem + C::kColDV, tmem + col, ddo + so + kb * kQStep, id_acc,
                            (i > 0) || (kb > 0));
          mma_bf16_ts_elect(tmem + C::kColDK, tmem + col + C::kPCols, dq_ + so + kb * kQStep,
                            id_acc, (i > 0) || (kb > 0));
        }
#pragma unroll
        for (int kb = 0; kb < kBN / C::kQPerStep; ++kb)
          mma_bf16_ss_elect(tmem + C::kColDQ, dkt + kb * kKtStep, dds + kb * kDsStep, id_dq,
                            kb > 0);
      } else {
        tc_cp_32x128b_warpx4_elect(tmem + C::kColSFQt, dsf + so + (512 >> 4));
        tc_cp_32x128b_warpx4_elect(tmem + C::kColSFdOt, dsf + so + (1536 >> 4));
        tc_cp_32x128b_warpx4_elect(tmem + C::kColSFdSB, dsfds);
#pragma unroll
        for (int kb = 0; kb < kBQ / 32; ++kb) {
          const uint32_t sfb = kb + 2 * half;
          mma_mxf8_ts_elect(tmem + C::kColDV, tmem + C::kColDQ + 32 * kb,
                            ddo + so + kb * kQStep, idesc_sf_ids(id_acc, 0, sfb),
                            tmem + C::kColSFP + 4 * kb, tmem + C::kColSFdOt, (i > 0) || (kb > 0));
          mma_mxf8_ts_elect(tmem + C::kColDK, tmem + C::kColDQ + 32 * kb + C::kPCols,
                            dq_ + so + kb * kQStep, idesc_sf_ids(id_acc, 0, sfb),
                            tmem + C::kColSFdS + 4 * kb, tmem + C::kColSFQt, (i > 0) || (kb > 0));
        }
        if (C::kKTBytes != 0 && i == 0) {
          if (!mbar_wait_sleep(&bars->kt_ready, 0, p.err, abort, 54)) return false;
        }
#pragma unroll
        for (int kb = 0; kb < kBN / 32; ++kb)
          mma_mxf8_ss_elect(tmem + C::kColDQ, dkt + kb * kKtStep, dds + kb * kDsStep,
                            idesc_sf_ids(id_dq, kb, kb), tmem + C::kColSFKt,
                            tmem + C::kColSFdSB, kb > 0);
      }
      // the compute warps release the Q / dO stage once they see dQ^T(i)
      tc_commit_elect(&bars->dq_full);
      return true;
    };
    if (ok) ok = issue_st(0, 0);
    for (int i0 = 0; i0 < nsteps && ok; i0 += kStages) {
#pragma unroll
      for (int ss = 0; ss < kStages; ++ss) {
        const int i = i0 + ss;                     // i % kStages == ss
        if (ok && i < nsteps) {
          // the next step's S^T / dP^T run while step i is in the compute
          // warps
          if (i + 1 < nsteps) {
            ok = mbar_wait_sleep(&bars->st_loaded, i & 1, p.err, abort, 53);
            if (ok) ok = issue_st(i + 1, (ss + 1) % kStages);
          }
          if (ok) ok = issue_acc(i, ss);
        }
      }
    }
    if (ok) tc_commit_elect(&bars->acc_done);
    if (!ok) *abort = 1;
    tc_commit_elect(&bars->drain);
    mbar_wait_sleep(&bars->drain, 0, nullptr, nullptr, 0);
  } else {
    // ------------------------------------------------------------- compute
    const int g = (warp - 2) >> 2;                // query block of the step
    const int quad = warp & 3;
    const int m = quad * 32 + lane;               // key row (and channel for dQ^T)
    const uint32_t lb = static_cast<uint32_t>(quad * 32) << 16;
    const int key = k0 + m;
    const int ctid = threadIdx.x - 64;            // 0..255 among compute threads
    bool ok = true;
    if (C::kKTBytes != 0 && g == 0) {
      // zero-padded 128-byte-row copy of the K tile (64B swizzle -> 128B)
      ok = mbar_wait_sleep(&bars->kv_full, 0, p.err, abort, 59);
      if (ok) {
        const uint8_t* src = sm + C::kSmK + m * D;
        uint8_t* dst = sm + C::kSmKT + m * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (c < D / 16) v = *reinterpret_cast<const uint4*>(src + 16 * (c ^ ((m >> 1) & 3)));
          *reinterpret_cast<uint4*>(dst + 16 * (c ^ (m & 7))) = v;
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->kt_ready);
    }
    // dQ^T(j) of this warp (32 channels x this warpgroup's 32 queries, fp32)
    // -> fp16 [query][channel] tile in one of the warp's own shared-memory
    // buffers -> one tensor reduce-add into global dQ, issued by lane 0
    // (bulk async groups belong to the issuing thread).  No other warp takes
    // part.  The values arrive in the accumulator-fragment arrangement
    // (16x256b loads: rq[16h + 4k + 2s + e] = channel 16h + 8s + lane/4,
    // query 8k + 2(lane%4) + e), which is what a transposing stmatrix takes:
    // one instruction writes the four 8-channel blocks of 8 queries.
    // Staging is split so that one proxy fence covers both this step's dS^T
    // tile and the previous step's dQ tile: stage_dq_store writes the tile
    // (slot j % kDqBufs), stage_dq_issue sends it after the fence.
    auto stage_dq_store = [&](int j, const uint32_t (&rq)[32]) {
      if (quad * 32 >= D) return;                  // no channels here (D = 64)
      const uint32_t sbase = smem_u32(sm + C::kSmDQ + ((warp - 2) * kDqBufs + (j & (kDqBufs - 1))) * 2048);
      // step j-kDqBufs's reduce has read the slot
      if (lane == 0) {
        if constexpr (kDqBufs == 4) bulk_wait_read_le3();
        else if constexpr (kDqBufs == 2) bulk_wait_read_le1();
        else bulk_wait_read0();
      }
      __syncwarp();
      const uint64_t mul = pack2(p.dq_mult, p.dq_mult);
      const int cb = lane >> 3;                   // channel block whose row this lane addresses
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t hv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {             // matrix i = channel block 2h + s
          const int r = 16 * (i >> 1) + 4 * k + 2 * (i & 1);
          const uint64_t v = mul2(pack2(__uint_as_float(rq[r]), __uint_as_float(rq[r + 1])), mul);
          const __half2 h2 = __floats2half2_rn(lo2(v), hi2(v));
          hv[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        const int q = 8 * k + (lane & 7);         // query row addressed by this lane
        stmatrix_x4_trans(sbase + q * 64 + 16 * (cb ^ ((q >> 1) & 3)), hv[0], hv[1], hv[2], hv[3]);
      }
    };
    auto stage_dq_issue = [&](int j, int hj, int q0j) {
      if (quad * 32 >= D) return;
      if (lane == 0) {
        // rows of the step beyond the sequence carry exact zeros
        tma_reduce_add_3d(&tma_dq, 32 * quad, hj, static_cast<int32_t>(w.start + q0j + 32 * g),
                          sm + C::kSmDQ + ((warp - 2) * kDqBufs + (j & (kDqBufs - 1))) * 2048);
        bulk_commit();
      }
    };
    auto read_dq = [&](int j, uint32_t (&rq)[32]) -> bool {
      if (!mbar_wait_sleep(&bars->dq_full, j & 1, p.err, abort, 61)) return false;
      tc_fence_after();
      // every MMA of step j has completed: its Q / dO stage may be refilled
      if (ctid == 0) mbar_arrive(&bars->q_empty[j % kStages]);
      tmem_ld_16x256b_x4(tmem + lb + C::kColDQ + 32 * g, rq);
      tmem_ld_16x256b_x4(tmem + lb + (16u << 16) + C::kColDQ + 32 * g, rq + 16);
      tmem_ld_wait();
      return true;
    };
    // (query head, first query) of step i and of step i-1, advanced without
    // divisions
    int cur_h = w.kvh * p.group, cur_qs = qstep0, prev_h = 0, prev_q0 = 0;
    for (int i = 0; i < nsteps && ok; ++i) {
      const int q0 = cur_qs * kBQ;
      ok = mbar_wait_sleep(&bars->st_ready, i & 1, p.err, abort, 60);
      if (!ok) break;
      tc_fence_after();
      uint32_t rs[32], rd[32];
      tmem_ld32(tmem + lb + C::kColS + 32 * g, rs);
      tmem_ld32(tmem + lb + C::kColDP + 32 * g, rd);
      tmem_ld_wait();
      // S^T / dP^T of this step are in registers: the next step's MMAs may go
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->st_loaded);
      float pv[32], dsv[32];
      const int qb0 = q0 + 32 * g;
      // visible queries of this key row within the block: [lo, hi)
      const int lo = p.causal ? max(0, key - qb0) : 0;
      const int hi = key < w.len ? min(32, w.len - qb0) : 0;
      const bool all_visible = __all_sync(0xFFFFFFFFu, lo == 0 && hi == 32);
      // TMEM holds S^T - LSE / c (seeded accumulator), so x = s * c2 - LSE2
      // is one multiply, two elements per instruction; invisible entries get
      // x = -inf, so P = 2^x = 0
      const uint64_t c2x2 = pack2(p.scale_log2, p.scale_log2);
      float xv[32];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const uint64_t x = mul2(pack2(__uint_as_float(rs[j]), __uint_as_float(rs[j + 1])), c2x2);
        xv[j] = lo2(x);
        xv[j + 1] = hi2(x);
      }
      if (!all_visible) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < lo || j >= hi) xv[j] = -INFINITY;
      }
      // P's block amax is 2^(max x) (2^x is monotonic); its warp reduction
      // is under way while the exponentials run
      uint32_t ap_bits = 0;
      if constexpr (!B16) {
        float mx = fmaxf(xv[0], xv[1]);
#pragma unroll
        for (int j = 2; j < 32; j += 2) mx = max3(mx, xv[j], xv[j + 1]);
        ap_bits = warp_max_nonneg_bits(ex2(mx));
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) pv[j] = ex2(xv[j]);
      // dS = P (dP - D); TMEM holds dP^T - D (seeded accumulator)
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const uint64_t ds = mul2(pack2(pv[j], pv[j + 1]),
                                 pack2(__uint_as_float(rd[j]), __uint_as_float(rd[j + 1])));
        dsv[j] = lo2(ds);
        dsv[j + 1] = hi2(ds);
      }
      // fp8: 32x32 block codes (warp maxima) and E4M3 payloads; bf16: pairs
      uint32_t wp[4 * C::kEl * 2], wd[4 * C::kEl * 2];
      uint32_t cp_ = 0, cd = 0;
      if constexpr (B16) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const __nv_bfloat162 a = __floats2bfloat162_rn(pv[2 * j], pv[2 * j + 1]);
          const __nv_bfloat162 b = __floats2bfloat162_rn(dsv[2 * j], dsv[2 * j + 1]);
          wp[j] = *reinterpret_cast<const uint32_t*>(&a);
          wd[j] = *reinterpret_cast<const uint32_t*>(&b);
        }
      } else {
        float md = max3_abs_nan(dsv[0], dsv[1], dsv[2]);
#pragma unroll
        for (int j = 3; j < 31; j += 2) md = max3_abs_nan(md, dsv[j], dsv[j + 1]);
        md = max3_abs_nan(md, dsv[31], 0.f);
        const uint32_t ad_bits = warp_max_nonneg_bits(md);
        cp_ = quant_block32(pv, ap_bits, wp);
        cd = quant_block32(dsv, ad_bits, wd);
      }
      // the previous step's dQ^T leaves TMEM before this step's fp8 P^T /
      // dS^T take its columns (and its MMA, the last reader of the dS^T
      // shared-memory tile, has completed)
      uint32_t rq[32];
      if (i > 0) {
        ok = read_dq(i - 1, rq);
        if (!ok) break;
      }
      // P^T, dS^T at dQ^T columns 32g and 32g + kPCols; (fp8) their
      // A-operand scales at lane m, column base + 4g + m/32
      if constexpr (B16) {
        tmem_st16(tmem + lb + C::kColDQ + 32 * g, wp);
        tmem_st16(tmem + lb + C::kColDQ + 32 * g + C::kPCols, wd);
      } else {
        tmem_st8(tmem + lb + C::kColDQ + 32 * g, wp);
        tmem_st8(tmem + lb + C::kColDQ + 32 * g + C::kPCols, wd);
        tmem_st1(tmem + lb + C::kColSFP + 4 * g + quad, cp_);
        tmem_st1(tmem + lb + C::kColSFdS + 4 * g + quad, cd);
      }
      // this warpgroup's 16-byte chunks of the key row -> the dS^T tile
      // (fp8: 64-byte rows, 64B swizzle; bf16: 128-byte rows, 128B swizzle)
      {
        constexpr int kCh = 2 * C::kEl;          // 16-byte chunks per 32 queries
        uint8_t* ds_row = sm + C::kSmDS + m * C::kDsRowB;
#pragma unroll
        for (int c = 0; c < kCh; ++c) {
          const int phys = B16 ? ((kCh * g + c) ^ (m & 7)) : ((kCh * g + c) ^ ((m >> 1) & 3));
          *reinterpret_cast<uint4*>(ds_row + 16 * phys) =
              make_uint4(wd[4 * c], wd[4 * c + 1], wd[4 * c + 2], wd[4 * c + 3]);
        }
      }
      // B-operand scale of dQ^T: (query n = 32 g + lane, key block quad)
      if constexpr (!B16) sm[C::kSmSFdS + lane * 16 + g * 4 + quad] = static_cast<uint8_t>(cd);
      // MXFP8: one proxy fence covers this step's dS^T tile and the previous
      // step's dQ tile; bf16 (whose accumulating MMAs take twice as long):
      // the accumulating MMAs are released first and the dQ tile is staged
      // behind a second fence (measured: MXFP8 7.50 vs 7.72 ms, bf16 9.3 vs
      // 8.9 ms)
      if constexpr (!B16) {
        if (i > 0) stage_dq_store(i - 1, rq);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_ready);
      if constexpr (B16) {
        if (i > 0) {
          stage_dq_store(i - 1, rq);
          fence_proxy_async_smem();
          __syncwarp();
        }
      }
      if (i > 0) stage_dq_issue(i - 1, prev_h, prev_q0);
      prev_h = cur_h;
      prev_q0 = q0;
      if (++cur_qs == nqsteps) {
        cur_qs = qstep0;
        ++cur_h;
      }
    }
    if (ok && nsteps > 0) {
      uint32_t rq[32];
      ok = read_dq(nsteps - 1, rq);
      if (ok) {
        stage_dq_store(nsteps - 1, rq);
        fence_proxy_async_smem();
        __syncwarp();
        stage_dq_issue(nsteps - 1, prev_h, prev_q0);
      }
    }
    if (lane == 0) bulk_wait0();
    // epilogue: warpgroup 0 writes dK (times softmax_scale), 1 writes dV
    if (ok) ok = mbar_wait_sleep(&bars->acc_done, 0, p.err, abort, 62);
    if (ok) {
      tc_fence_after();
      const bool valid = key < w.len;
      const int64_t tok = w.start + key;
      const uint32_t col = g == 0 ? C::kColDK : C::kColDV;
      const float mul = g == 0 ? p.softmax_scale : 1.f;
      __nv_bfloat16* out = (g == 0 ? p.dk : p.dv) + (tok * p.hkv + w.kvh) * D;
      uint4* dst = reinterpret_cast<uint4*>(out);
      uint32_t r[32];
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(tmem + lb + col + 32 * c, r);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint32_t wv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[8 * t + 2 * k]) * mul,
                                                        __uint_as_float(r[8 * t + 2 * k + 1]) * mul);
              wv[k] = *reinterpret_cast<uint32_t*>(&h2);
            }
            dst[4 * c + t] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// -D_i = -sum_d dO_id * O_id and -LSE in log2 units for every padded row
// (zeros on padding rows), negated so that the backward adds them in packed
// fp32x2 instructions; the FP16 dQ row of each token is cleared on the way.
// Rows in (padded row, head) order; head_dim / 8 lanes per row, one 16-byte
// chunk of O and of dO each.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const SeqView sv, const __nv_bfloat16* __restrict__ o,
                          const __nv_bfloat16* __restrict__ dout,
                          const float* __restrict__ lse, float* __restrict__ lse2,
                          float* __restrict__ delta, __half* __restrict__ dq, int32_t hq) {
  constexpr int kLanes = D / 8;
  const int64_t nrows = sv.total_sf_rows * hq;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gid / kLanes;
  const int sub = static_cast<int>(gid % kLanes);
  const bool in = row < nrows;
  float acc = 0.f;
  bool valid = false;
  int64_t tok = 0, pr = 0;
  int h = 0;
  if (in) {
    pr = row / hq;
    h = static_cast<int>(row % hq);
    const SeqInfo si = seq_info(sv, seq_of_sf_row(sv, pr));
    const int64_t off = pr - si.sf_start;
    valid = off < si.len;
    tok = si.start + off;
    if (valid) {
      const int64_t e = (tok * hq + h) * D + 8 * sub;
      const uint4 a = *reinterpret_cast<const uint4*>(o + e);
      const uint4 b = *reinterpret_cast<const uint4*>(dout + e);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 fa = __bfloat1622float2(a2[k]);
        const float2 fb = __bfloat1622float2(b2[k]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
      *reinterpret_cast<uint4*>(dq + e) = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (in && sub == 0) {
    const int64_t idx = static_cast<int64_t>(h) * sv.total_sf_rows + pr;
    delta[idx] = valid ? -acc : 0.f;
    lse2[idx] = valid ? -(lse[static_cast<int64_t>(h) * sv.total_tokens + tok] * 1.4426950408889634f)
                      : 0.f;
  }
}

__global__ void dq_unscale_kernel(__half2* __restrict__ dq, int64_t n2, float inv) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n2) {
    float2 f = __half22float2(dq[i]);
    dq[i] = __floats2half2_rn(f.x * inv, f.y * inv);
  }
}

}  // namespace
}  // namespace lpfa

using namespace lpfa;

namespace {
size_t bwd_ws_bytes(const lpfa_attn_desc* desc) {
  return 256 + 2 * static_cast<size_t>(desc->heads_q) *
                   static_cast<size_t>(desc->seqs.total_sf_rows) * sizeof(float);
}
}  // namespace

extern "C" size_t lpfa_bwd_workspace_size(const lpfa_attn_desc* desc) {
  if (desc == nullptr) return 0;
  return bwd_ws_bytes(desc);
}

namespace {

template <int D, bool B16>
lpfa_status launch_bwd_kernel(const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& tdo,
                              const CUtensorMap& tdq, const BwdParams& p, int64_t nblocks,
                              cudaStream_t cs) {
  const size_t smem = BwdCfg<D, B16>::kSmTotal + 1024;
  lpfa_status st = set_max_dynamic_smem(
      reinterpret_cast<const void*>(&mx_attn_bwd_kernel<D, B16>), static_cast<int>(smem));
  if (st != LPFA_OK) return st;
  mx_attn_bwd_kernel<D, B16><<<static_cast<unsigned>(nblocks), kThreads, smem, cs>>>(
      tq, tk, tv, tdo, tdq, p);
  return LPFA_OK;
}

lpfa_status bwd_impl(const lpfa_attn_desc* desc, const void* q8,
                     const void* sfq_mma, const void* sfq_mma_t,
                     const void* k8, const void* sfk_mma,
                     const void* sfk_mma_t, const void* v8,
                     const void* sfv_mma, const void* do8,
                     const void* sfdo_mma, const void* sfdo_mma_t,
                     const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, bool bf16,
                     void* stream) {
  SeqView sv;
  lpfa_status st = validate_attn(desc, &sv);
  if (st != LPFA_OK) return st;
  if (bf16 && desc->head_dim != 128) return LPFA_ERR_UNSUPPORTED;
  LPFA_CHECK_ARG(q8 && k8 && v8 && do8 && o && dout && lse && dq && dk && dv);
  LPFA_CHECK_ARG(bf16 || (sfq_mma && sfq_mma_t && sfk_mma && sfk_mma_t && sfv_mma &&
                          sfdo_mma && sfdo_mma_t));
  const void* ptrs[] = {q8, sfq_mma, sfq_mma_t, k8, sfk_mma, sfk_mma_t, v8, sfv_mma,
                        do8, sfdo_mma, sfdo_mma_t, o, dout, lse, dq, dk, dv};
  for (const void* ptr : ptrs) LPFA_CHECK_ARG(aligned16(ptr));
  LPFA_CHECK_ARG(workspace != nullptr &&
                 (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0);
  LPFA_CHECK_ARG(workspace_bytes >= bwd_ws_bytes(desc));
  LPFA_CHECK_ARG(desc->dq_static_scale > 0.f);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (sv.total_tokens == 0) return LPFA_OK;
  const int64_t hq = desc->heads_q, hkv = desc->heads_kv, D = desc->head_dim;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  float* lse2 = reinterpret_cast<float*>(ws + 256);
  float* delta = lse2 + hq * sv.total_sf_rows;
  // error words; the preprocess writes every log2-LSE / D row and clears dQ
  LPFA_CHECK_CUDA(cudaMemsetAsync(ws, 0, 256, cs));
  {
    const int64_t threads = sv.total_sf_rows * hq * (D / 8);
    LPFA_CHECK_ARG(ceil_div(threads, 256) < (1ll << 31));
    const unsigned blocks = static_cast<unsigned>(ceil_div(threads, 256));
    if (D == 128)
      bwd_preprocess_kernel<128><<<blocks, 256, 0, cs>>>(
          sv, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
          lse, lse2, delta, static_cast<__half*>(dq), static_cast<int32_t>(hq));
    else
      bwd_preprocess_kernel<64><<<blocks, 256, 0, cs>>>(
          sv, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
          lse, lse2, delta, static_cast<__half*>(dq), static_cast<int32_t>(hq));
    LPFA_CHECK_CUDA(cudaGetLastError());
  }

  CUtensorMap tq, tk, tv, tdo;
  // [tokens][heads][D] elements; a box is one chunk (<= 128 bytes) of `rows`
  // token rows of one head
  const int64_t el = bf16 ? 2 : 1;
  const int64_t chunk = D * el < 128 ? D * el : 128;
  const CUtensorMapSwizzle sw = chunk == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  auto make = [&](CUtensorMap* m, const void* base, int64_t heads, uint32_t rows) {
    uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(heads),
                        static_cast<uint64_t>(sv.total_tokens)};
    uint64_t strides[2] = {static_cast<uint64_t>(D * el), static_cast<uint64_t>(heads * D * el)};
    uint32_t box[3] = {static_cast<uint32_t>(chunk / el), 1u, rows};
    return encode_tmap(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                       3, base, dims, strides, box, sw);
  };
  if ((st = make(&tq, q8, hq, kBQ)) != LPFA_OK) return st;
  if ((st = make(&tdo, do8, hq, kBQ)) != LPFA_OK) return st;
  if ((st = make(&tk, k8, hkv, kBN)) != LPFA_OK) return st;
  if ((st = make(&tv, v8, hkv, kBN)) != LPFA_OK) return st;
  CUtensorMap tdq;
  {
    uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(hq),
                        static_cast<uint64_t>(sv.total_tokens)};
    uint64_t strides[2] = {static_cast<uint64_t>(D * 2), static_cast<uint64_t>(hq * D * 2)};
    uint32_t box[3] = {32u, 1u, 32u};   // one warp's [32 queries][32 channels]
    if ((st = encode_tmap(&tdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, dq, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_64B)) != LPFA_OK)
      return st;
  }

  BwdParams p;
  p.seqs = sv;
  p.sfq = static_cast<const uint8_t*>(sfq_mma);
  p.sfq_t = static_cast<const uint8_t*>(sfq_mma_t);
  p.sfk = static_cast<const uint8_t*>(sfk_mma);
  p.sfk_t = static_cast<const uint8_t*>(sfk_mma_t);
  p.sfv = static_cast<const uint8_t*>(sfv_mma);
  p.sfdo = static_cast<const uint8_t*>(sfdo_mma);
  p.sfdo_t = static_cast<const uint8_t*>(sfdo_mma_t);
  p.lse2 = lse2;
  p.delta = delta;
  p.dq = static_cast<__half*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.err = err;
  p.hq = static_cast<int32_t>(hq);
  p.hkv = static_cast<int32_t>(hkv);
  p.group = static_cast<int32_t>(hq / hkv);
  p.causal = desc->causal ? 1 : 0;
  p.scale_log2 = desc->softmax_scale * 1.4426950408889634f;
  p.softmax_scale = desc->softmax_scale;
  p.dq_mult = desc->softmax_scale * desc->dq_static_scale;

  const int64_t nblocks = (sv.total_sf_rows / 128) * hkv;
  LPFA_CHECK_ARG(nblocks > 0 && nblocks < (1ll << 31));
  if (bf16)
    st = launch_bwd_kernel<128, true>(tq, tk, tv, tdo, tdq, p, nblocks, cs);
  else if (D == 128)
    st = launch_bwd_kernel<128, false>(tq, tk, tv, tdo, tdq, p, nblocks, cs);
  else
    st = launch_bwd_kernel<64, false>(tq, tk, tv, tdo, tdq, p, nblocks, cs);
  if (st != LPFA_OK) return st;
  LPFA_CHECK_CUDA(cudaGetLastError());
  if (desc->dq_static_scale != 1.0f) {
    const int64_t n2 = sv.total_tokens * hq * D / 2;
    dq_unscale_kernel<<<static_cast<unsigned>(ceil_div(n2, 256)), 256, 0, cs>>>(
        static_cast<__half2*>(dq), n2, 1.0f / desc->dq_static_scale);
    LPFA_CHECK_CUDA(cudaGetLastError());
  }
  return LPFA_OK;
}

}  // namespace

extern "C" lpfa_status lpfa_bwd(const lpfa_attn_desc* desc, const void* q8,
                                const void* sfq_mma, const void* sfq_mma_t,
                                const void* k8, const void* sfk_mma,
                                const void* sfk_mma_t, const void* v8,
                                const void* sfv_mma, const void* do8,
                                const void* sfdo_mma, const void* sfdo_mma_t,
                                const void* o, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes,
                                void* stream) {
  return bwd_impl(desc, q8, sfq_mma, sfq_mma_t, k8, sfk_mma, sfk_mma_t, v8, sfv_mma, do8,
                  sfdo_mma, sfdo_mma_t, o, dout, lse, dq, dk, dv, workspace,
                  workspace_bytes, false, stream);
}

extern "C" lpfa_status lpfa_bwd_bf16(const lpfa_attn_desc* desc, const void* q,
                                     const void* k, const void* v, const void* o,
                                     const void* dout, const float* lse, void* dq,
                                     void* dk, void* dv, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return bwd_impl(desc, q, nullptr, nullptr, k, nullptr, nullptr, v, nullptr, dout,
                  nullptr, nullptr, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                  true, stream);
}

// ---------------------------------------------------------------------------
// lpfa_bwd_noalloc: the backward with its scratch in a static device array,
// for callers that cannot allocate (see include/lpfa.h).  It forwards to
// lpfa_bwd with the array as the workspace.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) uint8_t g_bwd_noalloc_scratch[LPFA_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDevices] = {nullptr};

// Device address of the array on the current device; looked up once per
// device, with that device current.
lpfa_status noalloc_scratch(void** out) {
  int dev = 0;
  LPFA_CHECK_CUDA(cudaGetDevice(&dev));
  LPFA_CHECK_ARG(dev >= 0 && dev < kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_addr[dev] == nullptr) {
    void* ptr = nullptr;
    LPFA_CHECK_CUDA(cudaGetSymbolAddress(&ptr, g_bwd_noalloc_scratch));
    g_noalloc_addr[dev] = ptr;
  }
  *out = g_noalloc_addr[dev];
  return LPFA_OK;
}

}  // namespace

extern "C" lpfa_status lpfa_bwd_noalloc(const lpfa_attn_desc* desc,
                                        const void* q8, const void* sfq_mma,
                                        const void* sfq_mma_t, const void* k8,
                                        const void* sfk_mma, const void* sfk_mma_t,
                                        const void* v8, const void* sfv_mma,
                                        const void* do8, const void* sfdo_mma,
                                        const void* sfdo_mma_t, const void* o,
                                        const void* dout, const float* lse,
                                        void* dq, void* dk, void* dv,
                                        void* stream) {
  LPFA_CHECK_ARG(desc != nullptr);
  LPFA_CHECK_ARG(desc->heads_q >= 1 && desc->seqs.total_sf_rows >= 0);
  const size_t need = bwd_ws_bytes(desc);
  if (need > LPFA_BWD_NOALLOC_SCRATCH_BYTES) {
    if (debug_enabled())
      std::fprintf(stderr,
                   "lpfa_bwd_noalloc: problem needs %zu scratch bytes, the static "
                   "array holds %u (heads_q * total_sf_rows too large)\n",
                   need, LPFA_BWD_NOALLOC_SCRATCH_BYTES);
    return LPFA_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  lpfa_status st = noalloc_scratch(&scratch);
  if (st != LPFA_OK) return st;
  return lpfa_bwd(desc, q8, sfq_mma, sfq_mma_t, k8, sfk_mma, sfk_mma_t, v8, sfv_mma,
                  do8, sfdo_mma, sfdo_mma_t, o, dout, lse, dq, dk, dv, scratch,
                  LPFA_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
