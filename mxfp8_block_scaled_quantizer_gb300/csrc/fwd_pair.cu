// bf16 attention forward on tcgen05, two query tiles in flight.
//
// The bf16 counterpart of the MXFP8 forward (same online softmax with
// selective rescaling, same epilogue; "Low Precision Flash Attention 4 ...",
// paragraph 1 measures MXFP8 against bf16; "FlashAttention-4 Adds
// Low-Precision Blackwell Support", "Technical Deep Dive", overlap of the
// softmax with the MMAs).  Operands are bf16, the MMAs kind::f16, P is
// rounded to bf16 for the PV product and no scale factors exist.
//
// Structure.  A work item is a pair of 128-query tiles of one (sequence,
// head), sides A and B, each with its own softmax warpgroup (thread = query
// row = TMEM lane: a row is never split, so the softmax needs no exchange
// between warps); both sides walk the same 64-key K/V tiles, and while one
// side's warpgroup works on its tile the tensor pipe runs the other side's S
// and PV MMAs.  Persistent: one CTA per SM walks the items in "snake" order
// (round r takes items r*G .. r*G+G-1, left to right on even rounds and
// right to left on odd ones); every barrier phase runs on across items.
// Warp roles:
//   warp 0     TMA producer: per item Q_A, Q_B, then K_j, V_j through a
//              shared-memory ring.
//   warp 1     TMEM owner and issuer of the S_t = Q_t K^T MMAs.
//   warp 10    issuer of the O_t += P_t V MMAs.
//   warps 2-5  softmax of side A, warps 6-9 softmax of side B.
// S_t has its own 64 columns and P_t its own 32, so S_t(j+1) is issued as
// soon as side t's warpgroup holds its rows of S_t(j) in registers; the
// softmax waits only for "S_t(j) landed" and, before P_t(j) overwrites
// P_t(j-1) and O_t is rescaled, for "PV_t(j-1) done".
// TMEM (head_dim 128): S_A [0,64) S_B [64,128) O_A [128,256) O_B [256,384)
// P_A [384,416) P_B [416,448).
//
// The MXFP8 forward keeps one query tile and 256-key tiles: with two tiles
// in flight its scale factors leave room only for 64-key tiles, which
// double its MMA count per key and its per-tile softmax overhead (measured:
// 2.86 ms against 2.67 ms on the B8 H32 S8192 D128 causal workload), while
// the bf16 forward gains from the overlap (2.81 ms against 4.20 ms for the
// one-tile structure).
#include <cuda_runtime.h>

#include "lpfa_device.cuh"
#include "lpfa_internal.h"
#include "lpfa_seq.cuh"

namespace lpfa {
namespace {

constexpr int kBlockM = 128;   // queries per tile; a work item holds two
constexpr int kSides = 2;      // query tiles per work item
constexpr int kTmemCols = 512;

struct PairParams {
  SeqView seqs;
  __nv_bfloat16* o;     // [T, Hq, D]
  float* lse;           // [Hq, T]
  uint32_t* err;
  int32_t hq, hkv, group;
  int32_t npairs;       // dense: tile pairs per sequence
  int64_t nitems;       // work items (some may be empty: varlen tails)
  int32_t causal;
  float scale_log2;     // softmax_scale * log2(e)
  float threshold;      // log2 units
  uint64_t wait_ns;     // bound of every wait
};

// Tile plan for head_dim D.  Operand tiles are stored as chunks of at most
// 128 bytes per row (one swizzle span): a bf16 row of 128 channels is two
// chunks, [chunk][rows][128 B].
template <int D>
struct PairCfg {
  static constexpr int kN = 64;                           // keys per tile
  static constexpr int kThreads = (3 + 4 * kSides) * 32;  // producer, S issuer, softmax, PV issuer
  static constexpr int kPvWarp = 2 + 4 * kSides;
  static constexpr int kRowB = D * 2;                     // bytes per token row
  static constexpr int kChunkB = kRowB < 128 ? kRowB : 128;
  static constexpr int kNCh = kRowB / kChunkB;            // chunks per row
  static constexpr uint32_t kSw = kChunkB == 128 ? 2u : 4u;   // 128B / 64B swizzle
  static constexpr uint32_t kSbo = 8 * kChunkB;               // 8 rows of a chunk
  // TMEM columns (side t adds t times the region's per-side width)
  static constexpr uint32_t kColS = 0;                        // + kN t
  static constexpr uint32_t kColO = kSides * kN;              // + D t
  static constexpr uint32_t kPCols = kN * 2 / 4;              // P of one side (bf16 pairs)
  static constexpr uint32_t kColP = kColO + kSides * D;       // + kPCols t
  static_assert(kColP + kSides * kPCols <= kTmemCols, "TMEM budget");
  // shared memory: Q_A, Q_B, then the K/V ring
  static constexpr int kStages = 4;
  static constexpr int kQBytes = kBlockM * kRowB;         // one side's Q tile
  static constexpr int kKVBytes = kN * kRowB;             // one of K, V
  static constexpr int kQ = 0;                            // + kQBytes t
  static constexpr int kStage0 = kSides * kQBytes;        // stage s: K, V
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kBar = kStage0 + kStages * kStageBytes;
  static constexpr int kTotal = kBar + 256;
  static_assert(kTotal + 1024 <= 227 * 1024, "shared memory per CTA");
  // one MMA instruction contracts 32 bytes of K (16 bf16 elements)
  static constexpr int kKStepsS = kRowB / 32;             // S = Q K^T over head_dim
  static constexpr int kKStepsPV = kN * 2 / 32;           // O += P V over the tile's keys
  static constexpr int kKeysPerStep = 16;
  static constexpr int kChunks = kN / 32;                 // 32-key chunks of a row
};

template <int S>
struct PairBars {
  uint64_t q_full;
  uint64_t q_empty;           // an item's last S MMA complete (MMA commit)
  uint64_t kv_full[S];
  uint64_t kv_empty[S];
  uint64_t s_full[kSides];    // S_t(j) in TMEM (MMA commit)
  uint64_t s_free[kSides];    // side t's warpgroup holds its rows of S_t(j) (4 arrivals)
  uint64_t p_full[kSides];    // P_t(j) in TMEM, O_t rescaled (4 arrivals)
  uint64_t pv_done[kSides];   // PV_t(j) complete (MMA commit)
  uint64_t drain[2];          // per MMA-issuing warp
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

// Work item idx: a pair of 128-query tiles of one (sequence, head).  Items
// that share a key head are consecutive (their K/V tiles stay in L2 while the
// CTAs that read them run) and, for dense causal inputs, the heavy (late)
// pairs of a group come first.  A jagged batch enumerates 128-row tiles and
// lets the even tiles of each sequence lead a pair (an odd tile's item is
// empty).  Side B may lie past the sequence (an odd tile count).
struct WorkItem {
  int seq, qtile, head;   // qtile: side A's tile; side B is qtile + 1
  int64_t start;          // first token of the sequence
  int32_t len;
};

__device__ __forceinline__ bool work_item(const PairParams& p, int64_t idx, WorkItem& w) {
  const int grp = p.group;
  int kvh;
  if (p.seqs.cu_seqlens == nullptr) {
    const int64_t per = static_cast<int64_t>(grp) * p.npairs;
    const int64_t g = idx / per;
    const int r = static_cast<int>(idx % per);
    kvh = static_cast<int>(g % p.hkv);
    w.seq = static_cast<int>(g / p.hkv);
    w.qtile = 2 * (p.npairs - 1 - r / grp);
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
    if (w.qtile & 1) return false;
  }
  const SeqInfo si = seq_info(p.seqs, w.seq);
  w.start = si.start;
  w.len = si.len;
  return w.qtile * kBlockM < w.len;
}

// Item of round r for this CTA in snake order; -1 once the rounds run out.
__device__ __forceinline__ int64_t round_item(const PairParams& p, int r) {
  const int64_t g = gridDim.x;
  const int64_t idx = static_cast<int64_t>(r) * g +
                      ((r & 1) ? (g - 1 - blockIdx.x) : static_cast<int64_t>(blockIdx.x));
  return idx < p.nitems ? idx : -1;
}

// Key/value tiles (of kN keys) that side t of an item reads: 0 for a side
// past the sequence.
template <int kN>
__device__ __forceinline__ int side_tiles(const PairParams& p, const WorkItem& w, int t) {
  const int q0 = (w.qtile + t) * kBlockM;
  if (q0 >= w.len) return 0;
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
__global__ void __launch_bounds__(PairCfg<D>::kThreads, 1)
    bf16_attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tma_q,
                       const __grid_constant__ CUtensorMap tma_k,
                       const __grid_constant__ CUtensorMap tma_v,
                       const PairParams p) {
  using C = PairCfg<D>;
  constexpr int kStages = C::kStages;
  constexpr int kBlockN = C::kN;
  constexpr uint32_t kSw = C::kSw;
  constexpr uint32_t kSbo = C::kSbo;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairBars<kStages>* bars = reinterpret_cast<PairBars<kStages>*>(sm + C::kBar);
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
    for (int t = 0; t < kSides; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], 4);
      mbar_init(&bars->p_full[t], 4);
      mbar_init(&bars->pv_done[t], 1);
    }
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

  // Every role walks the same item sequence; the K/V ring counts the tiles
  // of all items (gkv) and each side its own tiles (gs, gp, gt); barrier
  // phases follow those counts.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (converged); an elected lane issues the
    // copies.
    if (lane == 0) {
      tma_prefetch_desc(&tma_q);
      tma_prefetch_desc(&tma_k);
      tma_prefetch_desc(&tma_v);
    }
    bool ok = true;
    int gkv = 0, k = 0, q_issued = -1;
    int issued[kStages];
    for (int s = 0; s < kStages; ++s) issued[s] = -1;
    for (int r = 0; ok; ++r) {
      const int64_t idx = round_item(p, r);
      if (idx < 0) break;
      WorkItem w;
      if (!work_item(p, idx, w)) continue;
      const int kvh = w.head / p.group;
      const int nt = max(side_tiles<kBlockN>(p, w, 0), side_tiles<kBlockN>(p, w, 1));
      // the Q tiles are free once the previous
      // item's last S MMA has completed
      if (k > 0) {
        ok = mbar_wait_sleep(&bars->q_empty, (k - 1) & 1, p.err, abort, 11, p.wait_ns);
        if (!ok) break;
      }
      // side B past the sequence reads rows of the next sequence or the
      // tensor's zero fill: finite, never used
      mbar_arrive_expect_tx_elect(&bars->q_full, kSides * C::kQBytes);
#pragma unroll
      for (int t = 0; t < kSides; ++t) {
        const int32_t row_q = static_cast<int32_t>(w.start + (w.qtile + t) * kBlockM);
#pragma unroll
        for (int c = 0; c < C::kNCh; ++c)
          tma_load_3d_elect(sm + C::kQ + t * C::kQBytes + c * kBlockM * C::kChunkB, &tma_q,
                            c * (C::kChunkB / 2), w.head, row_q, &bars->q_full);
      }
      q_issued = k & 1;
      ++k;
      for (int j = 0; j < nt; ++j, ++gkv) {
        const int s = gkv % kStages;
        const uint32_t ph = (gkv / kStages) & 1;
        ok = mbar_wait_sleep(&bars->kv_empty[s], ph ^ 1, p.err, abort, 10, p.wait_ns);
        if (!ok) break;
        uint8_t* kbuf = sm + C::kStage0 + s * C::kStageBytes;
        uint64_t* bar = &bars->kv_full[s];
        mbar_arrive_expect_tx_elect(bar, 2 * C::kKVBytes);
        const int32_t row_k = static_cast<int32_t>(w.start + j * kBlockN);
#pragma unroll
        for (int c = 0; c < C::kNCh; ++c) {
          const int32_t x = c * (C::kChunkB / 2);
          tma_load_3d_elect(kbuf + c * kBlockN * C::kChunkB, &tma_k, x, kvh, row_k, bar);
          tma_load_3d_elect(kbuf + C::kKVBytes + c * kBlockN * C::kChunkB, &tma_v, x, kvh,
                            row_k, bar);
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
    // Warp 1 issues S_t = Q_t K^T, warp 10 (another scheduler) issues
    // O_t += P_t V; the two write disjoint TMEM columns (S | O), so their
    // instructions need no mutual order.  Each warp runs
    // its loop converged and an elected lane issues.  Descriptors of stage 0
    // are built once; a stage adds its byte offset / 16 and a K-step 32 bytes
    // (S operands) or 32 rows of V to the 14-bit address field, which never
    // carries (shared memory addresses stay below 256 KB).
    bool ok = true;
    int gkv = 0;
    int gcnt[kSides] = {0, 0};                    // S (warp 1) or PV (warp 10) of side t so far
    if (warp == 1) {
      constexpr uint32_t idesc_s = idesc_bf16(kBlockM, kBlockN, 0, 0);
      const uint64_t dq = make_sdesc(smem_u32(sm + C::kQ), 16, kSbo, kSw);
      const uint64_t dk = make_sdesc(smem_u32(sm + C::kStage0), 16, kSbo, kSw);
      int k = 0;
      for (int r = 0; ok; ++r) {
        const int64_t idx = round_item(p, r);
        if (idx < 0) break;
        WorkItem w;
        if (!work_item(p, idx, w)) continue;
        int ntt[kSides];
#pragma unroll
        for (int t = 0; t < kSides; ++t) ntt[t] = side_tiles<kBlockN>(p, w, t);
        const int nt = max(ntt[0], ntt[1]);
        ok = mbar_wait_sleep(&bars->q_full, k & 1, p.err, abort, 20, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; j < nt && ok; ++j, ++gkv) {
          const int s = gkv % kStages;
          ok = mbar_wait_sleep(&bars->kv_full[s], (gkv / kStages) & 1, p.err, abort, 21, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint64_t so = static_cast<uint64_t>(s) * (C::kStageBytes >> 4);
#pragma unroll
          for (int t = 0; t < kSides; ++t) {
            if (j >= ntt[t]) continue;
            // S_t may be overwritten once side t's warpgroup holds its rows
            // of the previous S_t
            if (gcnt[t] > 0 &&
                !mbar_wait_sleep(&bars->s_free[t], (gcnt[t] - 1) & 1, p.err, abort, 23, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t qo = static_cast<uint64_t>(t) * (C::kQBytes >> 4);
            const uint32_t tS = tmem + C::kColS + kBlockN * t;
#pragma unroll
            for (int kb = 0; kb < C::kKStepsS; ++kb)
              mma_bf16_ss_elect(tS, dq + qo + kstep_off<C::kChunkB>(kb, kBlockM),
                                dk + so + kstep_off<C::kChunkB>(kb, kBlockN), idesc_s, kb > 0);
            tc_commit_elect(&bars->s_full[t]);
            ++gcnt[t];
          }
        }
        // the item's last readers of the Q tiles are issued: the tiles are
        // free once they complete
        if (ok) tc_commit_elect(&bars->q_empty);
        ++k;
      }
    } else {
      constexpr uint32_t idesc_o = idesc_bf16(kBlockM, D, 0, 1);
      // V is MN-major (channels contiguous); a row of several 128-byte chunks
      // repeats the swizzle pattern along N every chunk (the leading offset)
      const uint64_t dv = make_sdesc(smem_u32(sm + C::kStage0 + C::kKVBytes),
                                     C::kNCh > 1 ? kBlockN * C::kChunkB : 16, kSbo, kSw);
      constexpr uint64_t kVStep = (C::kKeysPerStep * C::kChunkB) >> 4;
      for (int r = 0; ok; ++r) {
        const int64_t idx = round_item(p, r);
        if (idx < 0) break;
        WorkItem w;
        if (!work_item(p, idx, w)) continue;
        int ntt[kSides];
#pragma unroll
        for (int t = 0; t < kSides; ++t) ntt[t] = side_tiles<kBlockN>(p, w, t);
        const int nt = max(ntt[0], ntt[1]);
        for (int j = 0; j < nt && ok; ++j, ++gkv) {
          const int s = gkv % kStages;
          const uint64_t so = static_cast<uint64_t>(s) * (C::kStageBytes >> 4);
#pragma unroll
          for (int t = 0; t < kSides; ++t) {
            if (j >= ntt[t]) continue;
            // P_t(j) written (hence S_t(j) complete and the tile's K / V
            // landed)
            if (!mbar_wait_sleep(&bars->p_full[t], gcnt[t] & 1, p.err, abort, 22, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t tO = tmem + C::kColO + D * t;
            const uint32_t tP = tmem + C::kColP + C::kPCols * t;
            // an item's first PV_t overwrites O_t: its P-full comes after
            // side t read the previous item's O_t
            // K-step kb: P columns 8 kb (16 keys per lane), V rows 16 kb
#pragma unroll
            for (int kb = 0; kb < C::kKStepsPV; ++kb)
              mma_bf16_ts_elect(tO, tP + 8 * kb, dv + so + kb * kVStep, idesc_o,
                                (j > 0) || (kb > 0));
            tc_commit_elect(&bars->pv_done[t]);
            ++gcnt[t];
          }
          // the tile's K / V stage is free once its PV MMAs (and, before
          // them in the pipe, its S MMAs) have completed
          if (ok) tc_commit_elect(&bars->kv_empty[s]);
        }
      }
    }
    if (!ok) *abort = 1;
    uint64_t* dr = &bars->drain[warp == 1 ? 0 : 1];
    tc_commit_elect(dr);
    mbar_wait_sleep(dr, 0, nullptr, nullptr, 0);
  } else {
    // ------------------------------------------------------------- softmax
    const int side = (warp - 2) >> 2;             // query tile of the item
    const int quad = warp & 3;                    // TMEM lane quarter
    const int row = quad * 32 + lane;             // query row within tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tSrow = tmem + C::kColS + kBlockN * side + lane_base;
    const uint32_t tOrow = tmem + C::kColO + D * side + lane_base;
    const float c2 = p.scale_log2;
    const uint64_t c2x2 = pack2(c2, c2);
    constexpr int kCh = C::kChunks;
    bool ok = true;
    int gt = 0;                                   // this side's tiles so far (all items)
    for (int r = 0; ok; ++r) {
      const int64_t idx = round_item(p, r);
      if (idx < 0) break;
      WorkItem w;
      if (!work_item(p, idx, w)) continue;
      const int ntiles = side_tiles<kBlockN>(p, w, side);
      if (ntiles == 0) continue;                  // side B past the sequence
      const int q0 = (w.qtile + side) * kBlockM;
      const int qi = q0 + row;                    // query index in sequence
      float m_ref = -INFINITY;                    // log2 units
      float l = 0.f;
      const int lim = p.causal ? min(w.len, qi + 1) : w.len;   // keys < lim visible
      for (int j = 0; j < ntiles && ok; ++j, ++gt) {
        ok = mbar_wait_sleep(&bars->s_full[side], gt & 1, p.err, abort, 30, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[kCh][32];
#pragma unroll
        for (int c = 0; c < kCh; ++c) tmem_ld32(tSrow + 32 * c, sv[c]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[side]);
        const int k0 = j * kBlockN;
        const bool need_mask = (k0 + kBlockN > w.len) || (p.causal && k0 + kBlockN - 1 > q0);
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
        float tmax = cmax[0];
#pragma unroll
        for (int c = 1; c < kCh; ++c) tmax = fmaxf(tmax, cmax[c]);
        const float mt = __fmul_rn(tmax, c2);
        float m_new = m_ref;
        if (m_ref == -INFINITY || mt > m_ref + p.threshold) m_new = mt;
        const bool moved = (m_new != m_ref);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (moved && m_ref != -INFINITY) ? ex2(m_ref - m_new) : 1.f;
        uint32_t pw[16 * kCh];                   // P words of the row (bf16 pairs)
        float lsum = 0.f;
        {
          // P = 2^(s*c2 - m) rounded to bf16 for the PV MMA; l sums the fp32
          // values
          const uint64_t nb2 = pack2(-m_use, -m_use);
          uint64_t acc = 0;
#pragma unroll
          for (int c = 0; c < kCh; ++c) {
#pragma unroll
            for (int kk = 0; kk < 32; kk += 4) {
              const uint64_t x0 = fma2(pack2(__uint_as_float(sv[c][kk]), __uint_as_float(sv[c][kk + 1])), c2x2, nb2);
              const uint64_t x1 = fma2(pack2(__uint_as_float(sv[c][kk + 2]), __uint_as_float(sv[c][kk + 3])), c2x2, nb2);
              const float p0 = ex2(lo2(x0)), p1 = ex2(hi2(x0));
              const float p2 = ex2(lo2(x1)), p3 = ex2(hi2(x1));
              acc = add2(acc, pack2(p0, p1));
              acc = add2(acc, pack2(p2, p3));
              const __nv_bfloat162 b0 = __floats2bfloat162_rn(p0, p1);
              const __nv_bfloat162 b1 = __floats2bfloat162_rn(p2, p3);
              pw[16 * c + kk / 2] = *reinterpret_cast<const uint32_t*>(&b0);
              pw[16 * c + kk / 2 + 1] = *reinterpret_cast<const uint32_t*>(&b1);
            }
          }
          lsum = lo2(acc) + hi2(acc);
        }
        // the previous P_t must be consumed before this P_t overwrites it
        // (and O_t is stable only between two PVs); an item's first tile
        // follows the previous item's epilogue, which waited for its last PV
        if (j > 0) {
          ok = mbar_wait_sleep(&bars->pv_done[side], (gt - 1) & 1, p.err, abort, 31, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t tProw = tmem + C::kColP + C::kPCols * side + lane_base;
        tmem_st32(tProw, pw);
        // selective rescale of O_t (and l): only warps holding a moved row
        if (j > 0 && __any_sync(0xFFFFFFFFu, moved)) {
          if constexpr (D >= 32) {
            uint32_t rr[32];
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              tmem_ld32(tOrow + 32 * c, rr);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
              tmem_st32(tOrow + 32 * c, rr);
            }
          }
        }
        tmem_st_wait();
        l = l * alpha + lsum;
        m_ref = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[side]);
      }
      if (!ok) break;
      // epilogue: O_t / l -> bf16, LSE
      ok = mbar_wait_sleep(&bars->pv_done[side], (gt - 1) & 1, p.err, abort, 32, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const bool valid = qi < w.len;
      const int64_t tok = w.start + qi;
      uint4* dst = reinterpret_cast<uint4*>(p.o + (tok * p.hq + w.head) * D);
      uint32_t rr[32];
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(tOrow + 32 * c, rr);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t wv[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(rr[8 * i + 2 * kk]) * inv_l,
                                                        __uint_as_float(rr[8 * i + 2 * kk + 1]) * inv_l);
              wv[kk] = *reinterpret_cast<uint32_t*>(&h2);
            }
            dst[4 * c + i] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
      if (valid) {
        const float lse2 = m_ref + __log2f(l);
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
lpfa_status launch_pair(const lpfa_attn_desc* desc, const SeqView& sv, const void* q,
                        const void* k, const void* v, void* o, float* lse, uint32_t* err,
                        cudaStream_t cs) {
  using C = PairCfg<D>;
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
    uint32_t box[3] = {static_cast<uint32_t>(C::kChunkB / 2), 1u, rows};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, sw);
  };
  lpfa_status st;
  if ((st = make(&tq, q, desc->heads_q, kBlockM)) != LPFA_OK) return st;
  if ((st = make(&tk, k, desc->heads_kv, C::kN)) != LPFA_OK) return st;
  if ((st = make(&tv, v, desc->heads_kv, C::kN)) != LPFA_OK) return st;

  PairParams p;
  p.seqs = sv;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = err;
  p.hq = static_cast<int32_t>(desc->heads_q);
  p.hkv = static_cast<int32_t>(desc->heads_kv);
  p.group = p.hq / p.hkv;
  p.npairs = static_cast<int32_t>((ceil_div(sv.seqlen, kBlockM) + 1) / 2);
  p.causal = desc->causal ? 1 : 0;
  p.scale_log2 = desc->softmax_scale * 1.4426950408889634f;
  p.threshold = desc->rescale_threshold;
  p.wait_ns = kWaitLimitNs;
  // dense: pairs of query tiles; jagged: 128-row tiles, the odd ones empty
  const int64_t units = sv.cu_seqlens == nullptr
                            ? static_cast<int64_t>(sv.nseq) * p.npairs
                            : sv.total_sf_rows / 128;
  const int64_t nitems = units * p.hq;
  LPFA_CHECK_ARG(nitems > 0 && nitems < (1ll << 31));
  p.nitems = nitems;
  const int nsm = num_sms();
  const int64_t nblocks = nitems < nsm ? nitems : nsm;   // one CTA per SM
  const size_t smem = C::kTotal + 1024;
  if ((st = set_max_dynamic_smem(reinterpret_cast<const void*>(&bf16_attn_fwd_pair_kernel<D>),
                                 static_cast<int>(smem))) != LPFA_OK)
    return st;
  bf16_attn_fwd_pair_kernel<D><<<static_cast<unsigned>(nblocks), C::kThreads, smem, cs>>>(tq, tk, tv, p);
  LPFA_CHECK_CUDA(cudaGetLastError());
  return LPFA_OK;
}

}  // namespace

// The bf16 forward (lpfa_fwd_bf16) after validation: arguments as there.
lpfa_status launch_fwd_pair_bf16(const lpfa_attn_desc* desc, const SeqView& sv,
                                 const void* q, const void* k, const void* v, void* o,
                                 float* lse, uint32_t* err, cudaStream_t cs) {
  if (desc->head_dim == 128) return launch_pair<128>(desc, sv, q, k, v, o, lse, err, cs);
  return launch_pair<64>(desc, sv, q, k, v, o, lse, err, cs);
}

}  // namespace lpfa
