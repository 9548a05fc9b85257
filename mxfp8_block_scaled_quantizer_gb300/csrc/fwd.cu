// MXFP8 block-scaled attention forward on tcgen05.
//
// Method ("Low Precision Flash Attention 4: End-to-End Block-Scaled Attention
// for Blackwell", paragraphs 2-3; "Low-Precision FlashAttention-4 ...",
// "Key Algorithmic Innovations" 1-2; "FlashAttention-4 Adds Low-Precision
// Blackwell Support", "Technical Deep Dive"):
//   S = Q K^T           block-scaled MXFP8 MMA into TMEM (fp32)
//   online softmax      FP32 running reference max m and sum l per row in
//                       log2 units (softmax scale folded in); m moves only
//                       when a tile's max exceeds it by more than the
//                       rescale threshold (selective rescaling)
//   P -> MXFP8          1x32 blocks along keys; each block's scale comes from
//                       the block's logit maximum already reduced for the row
//                       max (amax(P) = 2^(max x - m)), and the block scale is
//                       folded into the exponent: p * 2^-e = 2^(x - m - e)
//   O += P V            block-scaled MMA, P read from TMEM as the A operand
//   epilogue            O / l -> bf16, LSE = (m + log2 l) ln 2
//
// Persistent: one CTA per SM walks work items (a 128-query tile of one
// (sequence, head)) in "snake" order (round r takes items r*G .. r*G+G-1,
// left to right on even rounds and right to left on odd ones), which
// balances heavy and light causal tiles across CTAs; key/value tiles of 256.
// Every barrier phase runs on across items, so the next item's Q, K/V loads
// and first S MMA overlap the current item's last tile and epilogue.
// Warp roles:
//   warp 0     TMA producer: per item Q, then K_j, V_j and their scale
//              tiles through a shared-memory ring.
//   warp 1     TMEM owner and issuer of the S = Q K^T MMAs.
//   warp 10    issuer of the O += P V MMAs.
//   warps 2-9  softmax: warps 2-5 take keys [0,128) of every tile, warps 6-9
//              keys [128,256); thread = query row = TMEM lane.  The two
//              threads of a row exchange their partial maxima (and, at the
//              end, their partial sums) through shared memory.
// The bf16 forward (fwd_pair.cu) keeps two query tiles in flight instead;
// for MXFP8 that structure leaves room in TMEM only for 64-key tiles beside
// the scale factors and measured slower (2.86 against 2.67 ms).
//
// Pipeline.  S has its own 256 columns and P its own 64, so S_{j+1} = Q
// K_{j+1}^T is issued as soon as the softmax has the row of S_j in
// registers; while the softmax works on tile j the tensor pipe runs PV_{j-1}
// and S_{j+1}.  The only waits on the softmax side are "S_j landed" and,
// before P_j overwrites P_{j-1}, "PV_{j-1} done".
//
// TMEM budget (all 512 columns; "TMEM allocation strategies that fit scale
// factors into the fully utilized 512-column TMEM with minimal new
// barriers", paragraph 2 of the first page):
//   S [0,256)   O [256,256+D)   P [384,448)   scale factors [448,476):
//   SFQ 4 columns, SFK 8 (two 128-key scale tiles), SFP 8 (one 4-column
//   group per softmax warpgroup), SFV 8.  The scale columns are rewritten by
//   tcgen05.cp (SFK, SFV) or tcgen05.st (SFP) every tile; the MMAs that read
//   them are ordered behind the copies by the issue order of the tensor pipe
//   and behind the stores by the P-full barrier that the PV MMA waits on.
#include <cuda_runtime.h>

#include "lpfa_device.cuh"
#include "lpfa_internal.h"
#include "lpfa_seq.cuh"

namespace lpfa {
namespace {

constexpr int kBlockM = 128;   // queries per CTA
constexpr int kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
constexpr uint32_t kColSFQ = 448, kColSFK = 452, kColSFP = 460;   // SFV after SFP

struct FwdParams {
  SeqView seqs;
  const uint8_t* sfq;   // [Tp/128, Hq, 512]
  const uint8_t* sfk;   // [Tp/128, Hkv, 512]
  const uint8_t* sfv;   // [Tp/128, Hkv, 512]
  __nv_bfloat16* o;     // [T, Hq, D]
  float* lse;           // [Hq, T]
  uint32_t* err;
  int32_t hq, hkv, group;
  int32_t nq;           // dense: query tiles per sequence
  int64_t nitems;       // work items (some may be empty: varlen tails)
  int32_t causal;
  float scale_log2;     // softmax_scale * log2(e)
  float threshold;      // log2 units
  uint64_t wait_ns;     // bound of every wait (kWaitLimitNs normally)
  int32_t withhold_kv;  // self-test: this CTA-local K/V tile is never loaded
                        // (-1 normally), so the waits on it must expire
};

// Tile plan for head_dim D.  Operand tiles are stored as chunks of at most
// 128 bytes per row (one swizzle span).
template <int D>
struct FwdCfg {
  static constexpr int kN = 256;                          // keys per tile
  // softmax warpgroups: each takes kWgN keys of every tile (all 128 query
  // rows, one per thread): 2 x 128 keys.  Four
  // warpgroups of 64 keys (608 threads, 96 registers) were measured slower
  // on the llm workload (2.88 against 2.73 ms): the four-way row-maximum
  // exchange and the 16-warp barriers cost more than the shorter chains gain.
  static constexpr int kWG = 2;
  static constexpr int kWgN = kN / kWG;                   // keys per softmax warpgroup
  static constexpr int kChunks = kWgN / 32;               // 32-key chunks per warpgroup
  static constexpr int kThreads = (3 + 4 * kWG) * 32;     // producer, S issuer, softmax, PV issuer
  static constexpr int kPvWarp = 2 + 4 * kWG;
  static constexpr uint32_t kColSFV = kColSFP + 4 * kWG;  // one 4-column SFP group per warpgroup
  static constexpr int kEl = 1;                           // bytes per element
  static constexpr int kRowB = D * kEl;                   // bytes per token row
  static constexpr int kChunkB = kRowB < 128 ? kRowB : 128;
  static constexpr int kNCh = kRowB / kChunkB;            // chunks per row
  static constexpr uint32_t kSw = kChunkB == 128 ? 2u : 4u;   // 128B / 64B swizzle
  static constexpr uint32_t kSbo = 8 * kChunkB;               // 8 rows of a chunk
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr int kQBytes = kBlockM * kRowB;
  static constexpr int kKVBytes = kN * kRowB;             // one of K, V
  static constexpr int kQ = 0;
  static constexpr int kStage0 = kQBytes;                 // stage s: K, V
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kSfQ = kStage0 + kStages * kStageBytes;
  static constexpr int kSfStage0 = kSfQ + 512;            // SFK[2], SFV[2]
  static constexpr int kSfStageBytes = 2048;
  static constexpr int kXMax = kSfStage0 + kStages * kSfStageBytes;  // float [2][kWG][128]
  static constexpr int kXSum = kXMax + 2 * kWG * 128 * 4;   // float [kWG][128]
  static constexpr int kBar = kXSum + kWG * 128 * 4;
  static constexpr int kTotal = kBar + 256;
  // one MMA instruction contracts 32 bytes of K (32 fp8 elements)
  static constexpr int kKStepsS = kRowB / 32;             // S = Q K^T over head_dim
  static constexpr int kKStepsPV = kN * kEl / 32;         // O += P V over the tile's keys
  static constexpr int kKeysPerStep = 32 / kEl;
};

template <int S>
struct FwdBars {
  uint64_t q_full;
  uint64_t q_empty;    // an item's last S MMA complete (MMA commit)
  uint64_t kv_full[S];
  uint64_t kv_empty[S];
  uint64_t s_full;     // S_j in TMEM (MMA commit)
  uint64_t s_free;     // every softmax warp holds its row of S_j (8 arrivals)
  uint64_t p_full;     // P_j, SFP_j in TMEM, O rescaled (8 arrivals)
  uint64_t pv_done;    // PV_j complete (MMA commit)
  uint64_t xchg[4];    // row maxima exchange, one per TMEM lane quarter (kWG)
  uint64_t drain[2];   // per MMA-issuing warp
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
      "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
      "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
      "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
      "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Work item idx: (sequence, q tile, head).  Items that share a key head are
// consecutive (their K/V tiles stay in L2 while the CTAs that read them run)
// and, for dense causal inputs, the heavy (late) q tiles of a group come
// first.
struct WorkItem {
  int seq, qtile, head;
  int64_t start;          // first token of the sequence
  int32_t len;
  int64_t sf_tile;        // padded 128-row tile index of the q tile
};

__device__ __forceinline__ bool work_item(const FwdParams& p, int64_t idx, WorkItem& w) {
  const int grp = p.group;
  int kvh;
  if (p.seqs.cu_seqlens == nullptr) {
    const int64_t per = static_cast<int64_t>(grp) * p.nq;
    const int64_t g = idx / per;
    const int r = static_cast<int>(idx % per);
    kvh = static_cast<int>(g % p.hkv);
    w.seq = static_cast<int>(g / p.hkv);
    w.qtile = p.nq - 1 - r / grp;
    w.head = kvh * grp + r % grp;
  } else {
    const int64_t ntiles = p.seqs.total_sf_rows / 128;
    const int64_t per = ntiles * grp;
    kvh = static_cast<int>(idx / per);
    const int64_t r = idx % per;
    const int64_t t = r / grp;
    w.head = kvh * grp + static_cast<int>(r % grp);
    w.seq = seq_of_sf_row(p.seqs, t * 128);
    const SeqInfo s0 = seq_info(p.seqs, w.seq);
    w.qtile = static_cast<int>((t * 128 - s0.sf_start) / 128);
  }
  const SeqInfo si = seq_info(p.seqs, w.seq);
  w.start = si.start;
  w.len = si.len;
  w.sf_tile = si.sf_start / 128 + w.qtile;
  return w.qtile * kBlockM < w.len;
}

// Item of round r for this CTA in snake order; -1 once the rounds run out.
__device__ __forceinline__ int64_t round_item(const FwdParams& p, int r) {
  const int64_t g = gridDim.x;
  const int64_t idx = static_cast<int64_t>(r) * g +
                      ((r & 1) ? (g - 1 - blockIdx.x) : static_cast<int64_t>(blockIdx.x));
  return idx < p.nitems ? idx : -1;
}

// Key/value tiles of an item (tiles of kN keys).
template <int kN>
__device__ __forceinline__ int item_tiles(const FwdParams& p, const WorkItem& w) {
  const int q0 = w.qtile * kBlockM;
  const int kv_len = p.causal ? min(w.len, q0 + kBlockM) : w.len;
  return (kv_len + kN - 1) / kN;
}

// Shared-memory descriptor offset (16-byte units) of K-step kb of a K-major
// operand tile stored in chunks of kChunkB-byte rows, `rows` rows each.
template <int kChunkB>
__device__ __forceinline__ constexpr uint64_t kstep_off(int kb, int rows) {
  return static_cast<uint64_t>((kb / (kChunkB / 32)) * rows * kChunkB +
                               (kb % (kChunkB / 32)) * 32) >> 4;
}

template <int D>
__global__ void __launch_bounds__(FwdCfg<D>::kThreads, 1)
    mx_attn_fwd_kernel(const __grid_constant__ CUtensorMap tma_q,
                       const __grid_constant__ CUtensorMap tma_k,
                       const __grid_constant__ CUtensorMap tma_v,
                       const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int kStages = C::kStages;
  constexpr int kBlockN = C::kN;
  constexpr int kWG = C::kWG;
  constexpr int kWgN = C::kWgN;
  constexpr uint32_t kColSFV = C::kColSFV;
  constexpr uint32_t kSw = C::kSw;
  constexpr uint32_t kSbo = C::kSbo;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBars<kStages>* bars = reinterpret_cast<FwdBars<kStages>*>(sm + C::kBar);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 4 * kWG);
    mbar_init(&bars->p_full, 4 * kWG);
    mbar_init(&bars->pv_done, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&bars->xchg[q], kWG);
    mbar_init(&bars->drain[0], 1);
    mbar_init(&bars->drain[1], 1);
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

  // Every role walks the same item sequence and counts the same key/value
  // tiles (gt) and items (k); barrier phases follow those counts.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (converged); an elected lane issues the
    // copies.
    if (lane == 0) {
      tma_prefetch_desc(&tma_q);
      tma_prefetch_desc(&tma_k);
      tma_prefetch_desc(&tma_v);
    }
    const int64_t sf_last = p.seqs.total_sf_rows / 128 - 1;
    bool ok = true;
    int gt = 0, k = 0, q_issued = -1;
    int issued[kStages];
    for (int s = 0; s < kStages; ++s) issued[s] = -1;
    for (int r = 0; ok; ++r) {
      const int64_t idx = round_item(p, r);
      if (idx < 0) break;
      WorkItem w;
      if (!work_item(p, idx, w)) continue;
      const int kvh = w.head / p.group;
      const int q0 = w.qtile * kBlockM;
      const int ntiles = item_tiles<kBlockN>(p, w);
      // the Q tile (and its scale tile) is free once the previous item's
      // last S MMA has completed
      if (k > 0) {
        ok = mbar_wait_sleep(&bars->q_empty, (k - 1) & 1, p.err, abort, 11, p.wait_ns);
        if (!ok) break;
      }
      mbar_arrive_expect_tx_elect(&bars->q_full, C::kQBytes + 512);
#pragma unroll
      for (int c = 0; c < C::kNCh; ++c)
        tma_load_3d_elect(sm + C::kQ + c * kBlockM * C::kChunkB, &tma_q,
                          c * (C::kChunkB / C::kEl), w.head,
                          static_cast<int32_t>(w.start + q0), &bars->q_full);
      bulk_load_elect(sm + C::kSfQ, p.sfq + (w.sf_tile * p.hq + w.head) * 512, 512,
                        &bars->q_full);
      q_issued = k & 1;
      ++k;
      // scale tiles of keys past the sequence's padded rows belong to the
      // next sequence (finite, and their keys are masked); past the tensor
      // the last tile stands in
      const int64_t kv_sf0 = w.sf_tile - w.qtile;
      for (int j = 0; j < ntiles; ++j, ++gt) {
        const int s = gt % kStages;
        const uint32_t ph = (gt / kStages) & 1;
        ok = mbar_wait_sleep(&bars->kv_empty[s], ph ^ 1, p.err, abort, 10, p.wait_ns);
        if (!ok) break;
        if (gt == p.withhold_kv) continue;
        uint8_t* kbuf = sm + C::kStage0 + s * C::kStageBytes;
        uint64_t* bar = &bars->kv_full[s];
        mbar_arrive_expect_tx_elect(bar, 2 * C::kKVBytes + C::kSfStageBytes);
        const int32_t row_k = static_cast<int32_t>(w.start + j * kBlockN);
#pragma unroll
        for (int c = 0; c < C::kNCh; ++c) {
          const int32_t x = c * (C::kChunkB / C::kEl);
          tma_load_3d_elect(kbuf + c * kBlockN * C::kChunkB, &tma_k, x, kvh, row_k, bar);
          tma_load_3d_elect(kbuf + C::kKVBytes + c * kBlockN * C::kChunkB, &tma_v, x, kvh,
                            row_k, bar);
        }
        {
          uint8_t* sfb = sm + C::kSfStage0 + s * 2048;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int64_t t = min(kv_sf0 + 2 * j + h, sf_last);
            const int64_t off = (t * p.hkv + kvh) * 512;
            bulk_load_elect(sfb + 512 * h, p.sfk + off, 512, bar);
            bulk_load_elect(sfb + 1024 + 512 * h, p.sfv + off, 512, bar);
          }
        }
        issued[s] = static_cast<int>(ph);
      }
    }
    // No copy may still be landing when the CTA exits, whichever warp ended
    // the loops: wait for the last phase issued on every buffer (already
    // complete in a run that did not abort).
    for (int s = 0; s < kStages; ++s)
      if (issued[s] >= 0)
        mbar_wait_sleep(&bars->kv_full[s], static_cast<uint32_t>(issued[s]), nullptr, nullptr, 0);
    if (q_issued >= 0)
      mbar_wait_sleep(&bars->q_full, static_cast<uint32_t>(q_issued), nullptr, nullptr, 0);
  } else if (warp == 1 || warp == C::kPvWarp) {
    // --------------------------------------------------------- MMA issuers
    // A warp issues at most one tcgen05 instruction every ~60-90 cycles, and
    // one tile needs 12 MMAs, 4 scale copies and 2 commits: more than a
    // single warp can issue in the ~1000 cycles the tensor pipe takes to run
    // them.  Warp 1 issues S = Q K^T, warp 10 (another scheduler) issues
    // O += P V; the two write disjoint TMEM columns (S | O, SFQ SFK | SFP
    // SFV), so their instructions need no mutual order.  Each warp runs its
    // loop converged and an elected lane issues.  Descriptors of stage 0 are
    // built once; a stage adds its byte offset / 16 and a K-step 32 bytes (S
    // operands) or 32 rows of V to the 14-bit address field, which never
    // carries (shared memory addresses stay below 256 KB).
    const uint64_t dsf = sf_tile_desc(smem_u32(sm + C::kSfStage0));
    bool ok = true;
    int gt = 0, k = 0;
    if (warp == 1) {
      constexpr uint32_t idesc_s = idesc_mxf8(kBlockM, kBlockN, 0, 0);
      const uint64_t dq = make_sdesc(smem_u32(sm + C::kQ), 16, kSbo, kSw);
      const uint64_t dk = make_sdesc(smem_u32(sm + C::kStage0), 16, kSbo, kSw);
      const uint32_t tS = tmem + kColS, tSFQ = tmem + kColSFQ, tSFK = tmem + kColSFK;
      // S = Q K^T (MXFP8: N = 256, two 128-key scale tiles side by side); S
      // may be overwritten once every softmax warp holds its row of the
      // previous S
      auto issue_s = [&](int g) -> bool {
        const int s = g % kStages;
        if (g > 0 && !mbar_wait_sleep(&bars->s_free, (g - 1) & 1, p.err, abort, 23, p.wait_ns)) return false;
        if (!mbar_wait_sleep(&bars->kv_full[s], (g / kStages) & 1, p.err, abort, 21, p.wait_ns)) return false;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(s) * (C::kStageBytes >> 4);
        {
          const uint64_t fo = static_cast<uint64_t>(s) * (2048 >> 4);
          tc_cp_32x128b_warpx4_elect(tSFK, dsf + fo);
          tc_cp_32x128b_warpx4_elect(tSFK + 4, dsf + fo + (512 >> 4));
#pragma unroll
          for (int kb = 0; kb < C::kKStepsS; ++kb)
            mma_mxf8_ss_elect(tS, dq + kstep_off<C::kChunkB>(kb, kBlockM),
                              dk + so + kstep_off<C::kChunkB>(kb, kBlockN),
                              idesc_sf_ids(idesc_s, kb, kb), tSFQ, tSFK, kb > 0);
        }
        tc_commit_elect(&bars->s_full);
        return true;
      };
      for (int r = 0; ok; ++r) {
        const int64_t idx = round_item(p, r);
        if (idx < 0) break;
        WorkItem w;
        if (!work_item(p, idx, w)) continue;
        const int ntiles = item_tiles<kBlockN>(p, w);
        ok = mbar_wait_sleep(&bars->q_full, k & 1, p.err, abort, 20, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        tc_cp_32x128b_warpx4_elect(tSFQ, sf_tile_desc(smem_u32(sm + C::kSfQ)));
        for (int j = 0; j < ntiles && ok; ++j, ++gt) ok = issue_s(gt);
        // the item's last reader of the Q tile is issued: the tile is free
        // once it completes
        if (ok) tc_commit_elect(&bars->q_empty);
        ++k;
      }
    } else {
      constexpr uint32_t idesc_o = idesc_mxf8(kBlockM, D, 0, 1);
      // V is MN-major (channels contiguous); a row of several 128-byte chunks
      // repeats the swizzle pattern along N every chunk (the leading offset)
      const uint64_t dv = make_sdesc(smem_u32(sm + C::kStage0 + C::kKVBytes),
                                     C::kNCh > 1 ? kBlockN * C::kChunkB : 16, kSbo, kSw);
      const uint32_t tO = tmem + kColO, tP = tmem + kColP;
      const uint32_t tSFP = tmem + kColSFP, tSFV = tmem + kColSFV;
      constexpr int kStepsWg = kWgN / C::kKeysPerStep;   // PV K-steps per softmax warpgroup
      // O (+)= P V over 256 keys (8 K-steps; scale group = K-step / 4); V
      // landed before its S could be computed, and P is written after the
      // softmax saw S, so P-full orders both.  An item's first PV overwrites
      // O: its P-full comes after the softmax read the previous item's O.
      auto issue_pv = [&](int g, bool first) -> bool {
        const int s = g % kStages;
        if (!mbar_wait_sleep(&bars->p_full, g & 1, p.err, abort, 22, p.wait_ns)) return false;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(s) * (C::kStageBytes >> 4);
        // K-step kb: P columns 8 kb (32 bytes of keys per lane), V rows
        // kKeysPerStep * kb of every chunk
        constexpr uint64_t kVStep = (C::kKeysPerStep * C::kChunkB) >> 4;
        {
          const uint64_t fo = static_cast<uint64_t>(s) * (2048 >> 4);
          tc_cp_32x128b_warpx4_elect(tSFV, dsf + fo + (1024 >> 4));
          tc_cp_32x128b_warpx4_elect(tSFV + 4, dsf + fo + (1536 >> 4));
#pragma unroll
          for (int kb = 0; kb < C::kKStepsPV; ++kb)
            // A (P) scales: warpgroup kb / kStepsWg's column group, byte
            // kb % kStepsWg; B (V) scales: 128-key tile kb / 4, byte kb % 4
            mma_mxf8_ts_elect(tO, tP + 8 * kb, dv + so + kb * kVStep,
                              idesc_sf_ids(idesc_o, kb % kStepsWg, kb & 3),
                              tSFP + 4 * (kb / kStepsWg), tSFV + 4 * (kb >> 2),
                              (!first) || (kb > 0));
        }
        tc_commit_elect(&bars->pv_done);
        // the tile's K / V stage is free once PV_g (and, before it in the
        // pipe, S_g) has completed
        tc_commit_elect(&bars->kv_empty[s]);
        return true;
      };
      for (int r = 0; ok; ++r) {
        const int64_t idx = round_item(p, r);
        if (idx < 0) break;
        WorkItem w;
        if (!work_item(p, idx, w)) continue;
        const int ntiles = item_tiles<kBlockN>(p, w);
        for (int j = 0; j < ntiles && ok; ++j, ++gt) ok = issue_pv(gt, j == 0);
      }
    }
    if (!ok) *abort = 1;
    uint64_t* dr = &bars->drain[warp == 1 ? 0 : 1];
    tc_commit_elect(dr);
    mbar_wait_sleep(dr, 0, nullptr, nullptr, 0);
  } else {
    // ------------------------------------------------------------- softmax
    const int wg = (warp - 2) >> 2;               // key half of every tile
    const int quad = warp & 3;                    // TMEM lane quarter
    const int row = quad * 32 + lane;             // query row within tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tSrow = tmem + kColS + kWgN * wg + lane_base;
    float* xmax = reinterpret_cast<float*>(sm + C::kXMax);   // [2][kWG][128]
    float* xsum = reinterpret_cast<float*>(sm + C::kXSum);   // [kWG][128]
    uint64_t* xbar = &bars->xchg[quad];
    const float c2 = p.scale_log2;
    const uint64_t c2x2 = pack2(c2, c2);
    bool ok = true;
    int gt = 0;                                   // tiles so far (all items)
    int gx = 0;                                   // row-pair exchanges so far
    for (int r = 0; ok; ++r) {
      const int64_t idx = round_item(p, r);
      if (idx < 0) break;
      WorkItem w;
      if (!work_item(p, idx, w)) continue;
      const int q0 = w.qtile * kBlockM;
      const int ntiles = item_tiles<kBlockN>(p, w);
      const int qi = q0 + row;                    // query index in sequence
      float m_ref = -INFINITY;                    // log2 units
      float l = 0.f;                              // this half's partial sum
      const int lim = p.causal ? min(w.len, qi + 1) : w.len;   // keys < lim visible
      for (int j = 0; j < ntiles && ok; ++j, ++gt) {
        ok = mbar_wait_sleep(&bars->s_full, gt & 1, p.err, abort, 30, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        constexpr int kCh = C::kChunks;
        uint32_t sv[kCh][32];
#pragma unroll
        for (int c = 0; c < kCh; ++c) tmem_ld32(tSrow + 32 * c, sv[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free);
        const int k0 = j * kBlockN + wg * kWgN;
        const bool need_mask = (k0 + kWgN > w.len) || (p.causal && k0 + kWgN - 1 > q0);
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < kCh; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (k0 + 32 * c + e >= lim) sv[c][e] = __float_as_uint(-INFINITY);
        }
        // chunk maxima of the raw logits (c2 > 0 keeps the order)
        float cmax[kCh];
#pragma unroll
        for (int c = 0; c < kCh; ++c) {
          float a = __uint_as_float(sv[c][0]);
#pragma unroll
          for (int e = 1; e < 31; e += 2)
            a = max3(a, __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
          cmax[c] = fmaxf(a, __uint_as_float(sv[c][31]));
        }
        // row maximum over both halves
        float hmax = cmax[0];
#pragma unroll
        for (int c = 1; c < kCh; ++c) hmax = fmaxf(hmax, cmax[c]);
        float* xm = xmax + (gx & 1) * (kWG * 128);
        xm[wg * 128 + row] = hmax;
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar);
        ok = mbar_wait_sleep(xbar, gx & 1, p.err, abort, 33, p.wait_ns);
        if (!ok) break;
        ++gx;
        float tmax = hmax;
#pragma unroll
        for (int o = 0; o < kWG; ++o)
          if (o != wg) tmax = fmaxf(tmax, xm[o * 128 + row]);
        const float mt = __fmul_rn(tmax, c2);
        float m_new = m_ref;
        if (m_ref == -INFINITY || mt > m_ref + p.threshold) m_new = mt;
        const bool moved = (m_new != m_ref);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (moved && m_ref != -INFINITY) ? ex2(m_ref - m_new) : 1.f;
        constexpr int kPW = 8 * kCh;                   // P words of this warpgroup's keys
        uint32_t pw[kPW];
        float lsum = 0.f;
        uint32_t sfp = 0;
        {
          // per-block scale codes: the exact decision 2^(fl(cmax*c2) - m)
          uint32_t code[kCh];
#pragma unroll
          for (int c = 0; c < kCh; ++c) {
            const float amax = ex2(__fsub_rn(__fmul_rn(cmax[c], c2), m_use));
            code[c] = e8m0_code_from_amax_bits(__float_as_uint(amax));
            sfp |= code[c] << (8 * c);
          }
          // P * 2^-e = 2^(s*c2 - (m + e)), two elements per instruction; l sums
          // the scaled values per block and rescales by 2^e
#pragma unroll
          for (int c = 0; c < kCh; ++c) {
            const int e = static_cast<int>(code[c]) - 127;
            const float nb = -(m_use + static_cast<float>(e));
            const uint64_t nb2 = pack2(nb, nb);
            uint64_t acc = 0;
#pragma unroll
            for (int kk = 0; kk < 16; kk += 2) {
              const uint64_t x0 = fma2(pack2(__uint_as_float(sv[c][2 * kk]), __uint_as_float(sv[c][2 * kk + 1])), c2x2, nb2);
              const uint64_t x1 = fma2(pack2(__uint_as_float(sv[c][2 * kk + 2]), __uint_as_float(sv[c][2 * kk + 3])), c2x2, nb2);
              const float p0 = ex2(lo2(x0)), p1 = ex2(hi2(x0));
              const float p2 = ex2(lo2(x1)), p3 = ex2(hi2(x1));
              acc = add2(acc, pack2(p0, p1));
              acc = add2(acc, pack2(p2, p3));
              pw[8 * c + kk / 2] = cvt_e4m3x4(p0, p1, p2, p3);
            }
            // 2^e as fp32 (e in [-127, 119]; 2^-127 flushes to 0, harmless: such
            // blocks hold only zeros)
            const float two_e = e > -127 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : 0.f;
            lsum = fmaf(lo2(acc) + hi2(acc), two_e, lsum);
          }
        }
        // the previous P must be consumed before this P overwrites it (and O
        // is stable only between two PVs); an item's first tile follows the
        // previous item's epilogue, which waited for its last PV
        if (j > 0) {
          ok = mbar_wait_sleep(&bars->pv_done, (gt - 1) & 1, p.err, abort, 31, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
        }
        if constexpr (kPW == 32) tmem_st32(tmem + kColP + kPW * wg + lane_base, pw);
        else tmem_st16(tmem + kColP + kPW * wg + lane_base, pw);
        tmem_st1(tmem + kColSFP + 4 * wg + quad + lane_base, sfp);
        // selective rescale of O (and l): only warps holding a moved row; each
        // half rescales half of the columns
        if (j > 0 && __any_sync(0xFFFFFFFFu, moved)) {
          constexpr int kOC = D / kWG;            // O columns of this warpgroup
          if constexpr (kOC >= 32) {
            uint32_t rr[32];
#pragma unroll 1
            for (int c = 0; c < kOC / 32; ++c) {
              const uint32_t ta = tmem + kColO + kOC * wg + 32 * c + lane_base;
              tmem_ld32(ta, rr);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
              tmem_st32(ta, rr);
            }
          } else {
            uint32_t rr[16];
            const uint32_t ta = tmem + kColO + kOC * wg + lane_base;
            tmem_ld16(ta, rr);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
            tmem_st16(ta, rr);
          }
        }
        tmem_st_wait();
        l = l * alpha + lsum;
        m_ref = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
      }
      if (!ok) break;
      // epilogue: O / l -> bf16 (each warpgroup writes D / kWG columns), LSE
      xsum[wg * 128 + row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      ok = mbar_wait_sleep(xbar, gx & 1, p.err, abort, 34, p.wait_ns);
      if (!ok) break;
      ++gx;
      ok = mbar_wait_sleep(&bars->pv_done, (gt - 1) & 1, p.err, abort, 32, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      // the row's sum over the warpgroups in a fixed order (every warpgroup
      // scales its O columns by the same 1 / l)
      float lt = 0.f;
#pragma unroll
      for (int o = 0; o < kWG; ++o) lt += xsum[o * 128 + row];
      const float inv_l = (lt > 0.f) ? 1.f / lt : 0.f;
      const bool valid = qi < w.len;
      const int64_t tok = w.start + qi;
      constexpr int kOC = D / kWG;                // O columns of this warpgroup
      uint4* dst = reinterpret_cast<uint4*>(p.o + (tok * p.hq + w.head) * D + kOC * wg);
      auto store8 = [&](const uint32_t* rv, int q) {
        uint32_t wv[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(rv[2 * kk]) * inv_l,
                                                    __uint_as_float(rv[2 * kk + 1]) * inv_l);
          wv[kk] = *reinterpret_cast<uint32_t*>(&h2);
        }
        dst[q] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      };
      if constexpr (kOC >= 32) {
        uint32_t rr[32];
#pragma unroll 1
        for (int c = 0; c < kOC / 32; ++c) {
          tmem_ld32(tmem + kColO + kOC * wg + 32 * c + lane_base, rr);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int i = 0; i < 4; ++i) store8(rr + 8 * i, 4 * c + i);
          }
        }
      } else {
        uint32_t rr[16];
        tmem_ld16(tmem + kColO + kOC * wg + lane_base, rr);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 2; ++i) store8(rr + 8 * i, i);
        }
      }
      if (valid && wg == 0) {
        const float lse2 = m_ref + __log2f(lt);
        p.lse[static_cast<int64_t>(w.head) * p.seqs.total_tokens + tok] =
            lse2 * 0.69314718055994531f;
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

template <int D>
lpfa_status launch_fwd(const lpfa_attn_desc* desc, const SeqView& sv,
                       const void* q8, const void* sfq, const void* k8,
                       const void* sfk, const void* v8, const void* sfv,
                       void* o, float* lse, uint32_t* err, uint64_t wait_ns,
                       int32_t withhold_kv, cudaStream_t cs) {
  using C = FwdCfg<D>;
  const CUtensorMapSwizzle sw =
      C::kChunkB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUtensorMap tq, tk, tv;
  // [tokens][heads][D] elements; a box is one chunk (<= 128 bytes) of `rows`
  // token rows of one head
  auto make = [&](CUtensorMap* m, const void* base, int64_t heads, uint32_t rows) {
    uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(heads),
                        static_cast<uint64_t>(sv.total_tokens)};
    uint64_t strides[2] = {static_cast<uint64_t>(C::kRowB),
                           static_cast<uint64_t>(heads * C::kRowB)};
    uint32_t box[3] = {static_cast<uint32_t>(C::kChunkB / C::kEl), 1u, rows};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                       3, base, dims, strides, box, sw);
  };
  lpfa_status st;
  if ((st = make(&tq, q8, desc->heads_q, kBlockM)) != LPFA_OK) return st;
  if ((st = make(&tk, k8, desc->heads_kv, C::kN)) != LPFA_OK) return st;
  if ((st = make(&tv, v8, desc->heads_kv, C::kN)) != LPFA_OK) return st;

  FwdParams p;
  p.seqs = sv;
  p.sfq = static_cast<const uint8_t*>(sfq);
  p.sfk = static_cast<const uint8_t*>(sfk);
  p.sfv = static_cast<const uint8_t*>(sfv);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = err;
  p.hq = static_cast<int32_t>(desc->heads_q);
  p.hkv = static_cast<int32_t>(desc->heads_kv);
  p.group = p.hq / p.hkv;
  p.nq = static_cast<int32_t>(ceil_div(sv.seqlen, kBlockM));
  p.causal = desc->causal ? 1 : 0;
  p.scale_log2 = desc->softmax_scale * 1.4426950408889634f;
  p.threshold = desc->rescale_threshold;
  p.wait_ns = wait_ns;
  p.withhold_kv = withhold_kv;

  const int64_t units = sv.cu_seqlens == nullptr
                            ? static_cast<int64_t>(sv.nseq) * p.nq
                            : sv.total_sf_rows / 128;
  const int64_t nitems = units * p.hq;
  LPFA_CHECK_ARG(nitems > 0 && nitems < (1ll << 31));
  p.nitems = nitems;
  const int nsm = num_sms();
  const int64_t nblocks = nitems < nsm ? nitems : nsm;   // one CTA per SM
  const size_t smem = C::kTotal + 1024;
  if ((st = set_max_dynamic_smem(reinterpret_cast<const void*>(&mx_attn_fwd_kernel<D>),
                                 static_cast<int>(smem))) != LPFA_OK)
    return st;
  mx_attn_fwd_kernel<D><<<static_cast<unsigned>(nblocks), C::kThreads, smem, cs>>>(tq, tk, tv, p);
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}

}  // namespace

lpfa_status validate_attn(const lpfa_attn_desc* desc, SeqView* sv) {
  LPFA_CHECK_ARG(desc != nullptr);
  lpfa_status st = make_seq_view(&desc->seqs, sv);
  if (st != LPFA_OK) return st;
  LPFA_CHECK_ARG(desc->heads_q >= 1 && desc->heads_kv >= 1 &&
                 desc->heads_q <= 1024 && desc->heads_q % desc->heads_kv == 0);
  if (desc->head_dim != 64 && desc->head_dim != 128) return LPFA_ERR_UNSUPPORTED;
  LPFA_CHECK_ARG(desc->softmax_scale > 0.f);
  LPFA_CHECK_ARG(desc->rescale_threshold >= 0.f);
  return LPFA_OK;
}

}  // namespace lpfa

using namespace lpfa;

extern "C" size_t lpfa_fwd_workspace_size(const lpfa_attn_desc* desc) {
  (void)desc;
  return 256;
}

namespace {

lpfa_status fwd_impl(const lpfa_attn_desc* desc, const void* q8, const void* sfq_mma,
                     const void* k8, const void* sfk_mma, const void* v8,
                     const void* sfv_mma, void* o, float* lse, void* workspace,
                     size_t workspace_bytes, uint64_t wait_ns, int32_t withhold_kv,
                     bool bf16, void* stream) {
  SeqView sv;
  lpfa_status st = validate_attn(desc, &sv);
  if (st != LPFA_OK) return st;
  LPFA_CHECK_ARG(q8 && k8 && v8 && o && lse);
  LPFA_CHECK_ARG(bf16 || (sfq_mma && sfk_mma && sfv_mma));
  LPFA_CHECK_ARG(aligned16(q8) && aligned16(k8) && aligned16(v8) &&
                 aligned16(sfq_mma) && aligned16(sfk_mma) && aligned16(sfv_mma) &&
                 aligned16(o));
  LPFA_CHECK_ARG(workspace != nullptr && workspace_bytes >= 256 &&
                 (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (sv.total_tokens == 0) return LPFA_OK;
  LPFA_CHECK_CUDA(cudaMemsetAsync(workspace, 0, 256, cs));
  uint32_t* err = static_cast<uint32_t*>(workspace);
  // bf16: the two-query-tile kernel (fwd_pair.cu), its faster structure
  if (bf16) return launch_fwd_pair_bf16(desc, sv, q8, k8, v8, o, lse, err, cs);
  if (desc->head_dim == 128)
    return launch_fwd<128>(desc, sv, q8, sfq_mma, k8, sfk_mma, v8, sfv_mma, o, lse, err,
                           wait_ns, withhold_kv, cs);
  return launch_fwd<64>(desc, sv, q8, sfq_mma, k8, sfk_mma, v8, sfv_mma, o, lse, err, wait_ns,
                        withhold_kv, cs);
}

}  // namespace

extern "C" lpfa_status lpfa_fwd(const lpfa_attn_desc* desc, const void* q8,
                                const void* sfq_mma, const void* k8,
                                const void* sfk_mma, const void* v8,
                                const void* sfv_mma, void* o, float* lse,
                                void* workspace, size_t workspace_bytes,
                                void* stream) {
  return fwd_impl(desc, q8, sfq_mma, k8, sfk_mma, v8, sfv_mma, o, lse, workspace,
                  workspace_bytes, kWaitLimitNs, -1, false, stream);
}

extern "C" lpfa_status lpfa_fwd_wait_expiry_selftest(
    const lpfa_attn_desc* desc, const void* q8, const void* sfq_mma, const void* k8,
    const void* sfk_mma, const void* v8, const void* sfv_mma, void* o, float* lse,
    void* workspace, size_t workspace_bytes, uint32_t wait_limit_us, void* stream) {
  LPFA_CHECK_ARG(wait_limit_us >= 1 && wait_limit_us <= 2000000u);
  return fwd_impl(desc, q8, sfq_mma, k8, sfk_mma, v8, sfv_mma, o, lse, workspace,
                  workspace_bytes, static_cast<uint64_t>(wait_limit_us) * 1000ull, 0,
                  false, stream);
}

extern "C" lpfa_status lpfa_fwd_bf16(const lpfa_attn_desc* desc, const void* q,
                                     const void* k, const void* v, void* o, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     void* stream) {
  return fwd_impl(desc, q, nullptr, k, nullptr, v, nullptr, o, lse, workspace,
                  workspace_bytes, kWaitLimitNs, -1, true, stream);
}
