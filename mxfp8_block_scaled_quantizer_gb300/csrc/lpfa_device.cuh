// Device primitives for sm_103a: shared-memory barriers, TMA, tcgen05
// (tensor memory, block-scaled MMA), bounded waits.  Inline PTX only.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace lpfa {

// ---------------------------------------------------------------- errors
// Error word layout (first 16 bytes of a workspace): word 0 = OR of error
// bits, word 1 = first failing site id, word 2 = blockIdx.x of that site.
enum : uint32_t {
  ERR_WAIT_TIMEOUT = 1u,
  ERR_TMEM_ALLOC = 2u,
};

__device__ __forceinline__ void report_error(uint32_t* err, uint32_t bits,
                                             uint32_t site) {
  if (err == nullptr) return;
  uint32_t prev = atomicOr(err, bits);
  if (prev == 0) {
    err[1] = site;
    err[2] = blockIdx.x;
  }
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete is suspended
// (up to `hint_ns`, or until the phase completes) instead of returning at
// once, so that a waiting warp does not take issue slots from the warps that
// share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wall-clock bound of every wait.  A correct pipeline never waits longer
// than microseconds; the bound only turns a logic error into a reported
// error instead of a hung GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Waits for `parity` on `bar`.  Returns false (after reporting) when the
// wait expires (after `limit_ns`) or when `abort` (shared flag) is already
// set by another warp.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint32_t* err, volatile int* abort,
                                          uint32_t site,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        if (abort != nullptr) *abort = 1;
        report_error(err, ERR_WAIT_TIMEOUT, site);
        return false;
      }
    }
  }
}


// mbar_wait for roles that wait long and share a scheduler with compute
// warps (producers, MMA issuers, waiting consumers): the same contract, with
// the polling thread suspended between tests.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity,
                                                uint32_t* err, volatile int* abort,
                                                uint32_t site,
                                                uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      if (abort != nullptr) *abort = 1;
      report_error(err, ERR_WAIT_TIMEOUT, site);
      return false;
    }
  }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap,
                                            int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap,
                                            int32_t x, int32_t y, int32_t z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// TMA tile store shared -> global (bulk group; out-of-range rows and
// columns of the box are not written).
__device__ __forceinline__ void tma_store_2d(const void* tmap, int32_t x, int32_t y,
                                             const void* smem_src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          tmap),
      "r"(x), "r"(y), "r"(smem_u32(smem_src))
      : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc,
                                          uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk reduce-add of packed fp16 from shared to global (16-byte aligned,
// bytes % 16 == 0).
__device__ __forceinline__ void bulk_reduce_add_f16(void* gdst,
                                                    const void* smem_src,
                                                    uint32_t bytes) {
  asm volatile(
      "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.noftz.f16 "
      "[%0], [%1], %2;" ::"l"(gdst),
      "r"(smem_u32(smem_src)), "r"(bytes)
      : "memory");
}

// Element-wise reduce-add of a shared-memory box into a tensor (the box and
// element type come from the tensor map; rows outside the tensor are skipped).
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap, int32_t x,
                                                  int32_t y, int32_t z,
                                                  const void* smem_src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group "
      "[%0, {%1, %2, %3}], [%4];" ::"l"(tmap),
      "r"(x), "r"(y), "r"(z), "r"(smem_u32(smem_src))
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// At most one committed bulk group may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// At most three committed bulk groups may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_le3() {
  asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Four 8x8 16-bit matrices to shared memory, transposed: lanes 8i..8i+7
// give the addresses of the 8 rows of matrix i; register ri of thread t holds
// its elements (t/4, 2(t%4)) and (t/4, 2(t%4)+1), which land in rows
// 2(t%4), 2(t%4)+1 at column t/4.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t saddr, uint32_t r0, uint32_t r1,
                                                  uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};"
               :: "r"(saddr), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------- tensor memory
// TMEM address: bits 31..16 lane, bits 15..0 column (32-bit columns).
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane,
                                              uint32_t col) {
  return base + (lane << 16) + col;
}

// Whole warp: allocate `ncols` (power of two >= 32) columns; the base
// address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::
          "r"(smem_u32(dst)),
      "r"(ncols)
      : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   base),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(smem_u32(bar))
      : "memory");
}

// ---- single-thread instructions issued from a converged warp: every lane
// of the warp makes the call and the lane that elect.sync picks issues the
// instruction.  The elected-lane predicate costs far fewer issue cycles per
// tcgen05 instruction than a branch on the lane index or a predicate derived
// from one (measured on sm_103a: ~39 cycles per MMA against ~62 and ~86),
// and keeps the warp converged.
#define LPFA_ELECT "elect.sync _|e, 0xffffffff;\n\t"

__device__ __forceinline__ void tc_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::
          "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_cp_32x128b_warpx4_elect(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}

__device__ __forceinline__ void mma_mxf8_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t" LPFA_ELECT
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
      "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_mxf8_ts_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t" LPFA_ELECT
      "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], [%1], %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
      "r"(accumulate)
      : "memory");
}

// D (tmem) (+)= A (smem) * B (smem), bf16 inputs, fp32 accumulation, K = 16.
__device__ __forceinline__ void mma_bf16_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t" LPFA_ELECT
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (tmem) (+)= A (tmem) * B (smem desc), bf16, K = 16; elected lane issues.
__device__ __forceinline__ void mma_bf16_ts_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t" LPFA_ELECT
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_elect(void* smem_dst, const void* tmap, int32_t x,
                                                  int32_t y, int32_t z, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%2, %3, %4}], [%5];\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_load_elect(void* smem_dst, const void* gsrc, uint32_t bytes,
                                                uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format).
//  swizzle: 0 none, 2 = 128-byte, 4 = 64-byte, 6 = 32-byte.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo,
                                               uint32_t sbo,
                                               uint32_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(swizzle & 7u) << 61;
  return d;
}

// Instruction descriptor, kind::mxf8f6f4 with E4M3 A and B, UE8M0 scales.
//  a_mn / b_mn: 1 when the operand is MN-major (M or N contiguous).
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t M, uint32_t N,
                                                 uint32_t a_mn, uint32_t b_mn) {
  return (0u << 7) | (0u << 10) | (a_mn << 15) | (b_mn << 16) |
         ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

// Instruction descriptor, kind::mxf8f6f4 with A / B element types given by
// their type codes (E4M3 0, E5M2 1, E2M3 3, E3M2 4, E2M1 5) and UE8M0 scales.
__host__ __device__ constexpr uint32_t idesc_mx_types(uint32_t M, uint32_t N, uint32_t atype,
                                                     uint32_t btype) {
  return (atype << 7) | (btype << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

// Set the scale-factor byte selectors (which byte of each 32-bit TMEM scale
// column feeds this MMA).
__device__ __forceinline__ uint32_t idesc_sf_ids(uint32_t idesc, uint32_t a_id,
                                                 uint32_t b_id) {
  return idesc | (b_id << 4) | (a_id << 29);
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N,
                                                 uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn << 15) | (b_mn << 16) |
         ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D (tmem) (+)= A (smem desc) * B (smem desc), block-scaled MXFP8, K = 32.
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t a_desc,
                                            uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem,
                                            uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
      "r"(accumulate)
      : "memory");
}

// D (tmem) (+)= A (tmem) * B (smem desc), block-scaled MXFP8, K = 32.
__device__ __forceinline__ void mma_mxf8_ts(uint32_t d_tmem, uint32_t a_tmem,
                                            uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem,
                                            uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], [%1], %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
      "r"(accumulate)
      : "memory");
}

// D (tmem) (+)= A (smem) * B (smem), dense FP4 (E2M1) operands, K = 64,
// 32-element E8M0 block scales (two per row per MMA).
__device__ __forceinline__ void mma_mxf4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem,
                                            uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// The same with 16-element E4M3 block scales (NVFP4; four per row per MMA).
__device__ __forceinline__ void mma_nvf4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem,
                                            uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// D (tmem) (+)= A (smem) * B (smem), bf16, K = 16.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc,
                                            uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (tmem) (+)= A (tmem) * B (smem), bf16, K = 16.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem,
                                            uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Copy a 32-row x 16-byte shared-memory block (rows 16 bytes apart) into
// 4 TMEM columns of every 32-lane quarter (the 512-byte scale tile).
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr,
                                                     uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr),
               "l"(sdesc)
               : "memory");
}

__device__ __forceinline__ uint64_t sf_tile_desc(uint32_t saddr) {
  // no swizzle; 8-row core matrices 128 bytes apart
  return make_sdesc(saddr, 0, 128, 0);
}

// ---- TMEM <-> registers (32x32b shape: thread i of the warp <-> lane
// base+i; .xN = N consecutive 32-bit columns)
#define LPFA_TMEM_LD_X8(taddr, r)                                            \
  asm volatile(                                                              \
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, "    \
      "[%8];"                                                                \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),          \
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7])                                   \
      : "r"(taddr))

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}

// 16x256b shape, four repetitions along columns: thread t gets, for
// repetition k (columns 8k..8k+7 from taddr), r[4k], r[4k+1] = lane
// base + t/4, columns 8k + 2(t%4) + {0, 1}, and r[4k+2], r[4k+3] = the same
// columns of lane base + 8 + t/4 (the accumulator-fragment arrangement)
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr,
                                         const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr),
               "r"(v)
               : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr,
                                          const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
      "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------ packed fp32 arithmetic
// Two lanes of fp32 math in one instruction (sm_100+ .f32x2 forms); a pair
// is carried as a 64-bit value, low half first.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ------------------------------------------------------ FP8 conversions
// Two fp32 -> packed e4m3x2 (lo = a, hi = b), round to nearest even,
// saturating to +-448.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c,
                                               float d) {
  return static_cast<uint32_t>(cvt_e4m3x2(a, b)) |
         (static_cast<uint32_t>(cvt_e4m3x2(c, d)) << 16);
}

// ---------------------------------------------- other MX element formats
// Quantizer element formats, one element per output byte (low bits, sign on
// top of the element's field): E4M3, E5M2 (IEEE-like Inf/NaN), FP6 E3M2 and
// E2M3, FP4 E2M1 (no Inf/NaN).  emax = exponent of the largest finite binade.
enum : int { kFmtE4M3 = 0, kFmtE5M2 = 1, kFmtE3M2 = 2, kFmtE2M3 = 3, kFmtE2M1 = 4 };

template <int F>
constexpr uint32_t fmt_emax() {
  return F == kFmtE4M3 ? 8u : F == kFmtE5M2 ? 15u : F == kFmtE3M2 ? 4u : 2u;
}

// Payload byte of a block whose scale code is 0xFF: the format's NaN, or for
// the formats without NaN their largest positive code.
template <int F>
constexpr uint32_t fmt_nan_byte() {
  return F == kFmtE4M3 || F == kFmtE5M2 ? 0x7Fu : F == kFmtE2M1 ? 0x07u : 0x1Fu;
}

// E8M0 code floor(log2 amax) - emax + 127 from amax's fp32 bits (clamped at
// 0; Inf/NaN -> 0xFF).
template <int F>
__device__ __forceinline__ uint32_t scale_code_from_amax_bits(uint32_t bits) {
  constexpr uint32_t emax = fmt_emax<F>();
  const uint32_t ef = (bits >> 23) & 0xFFu;
  if (ef == 0xFFu) return 0xFFu;
  return ef > emax ? ef - emax : 0u;
}

// Four fp32 -> four element bytes (a in byte 0), round to nearest even,
// saturating to the format's largest finite magnitude.
template <int F>
__device__ __forceinline__ uint32_t cvt_x4(float a, float b, float c, float d) {
  if constexpr (F == kFmtE4M3) {
    return cvt_e4m3x4(a, b, c, d);
  } else if constexpr (F == kFmtE2M1) {
    uint16_t lo, hi;   // two FP4 codes per byte: first operand in the low nibble
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(lo) : "f"(a), "f"(b));
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(hi) : "f"(c), "f"(d));
    return (lo & 0xFu) | ((lo >> 4) & 0xFu) << 8 | (hi & 0xFu) << 16 | ((hi >> 4) & 0xFu) << 24;
  } else {
    uint16_t lo, hi;
    if constexpr (F == kFmtE5M2) {
      asm("cvt.rn.satfinite.e5m2x2.f32 %0, %2, %1;" : "=h"(lo) : "f"(a), "f"(b));
      asm("cvt.rn.satfinite.e5m2x2.f32 %0, %2, %1;" : "=h"(hi) : "f"(c), "f"(d));
    } else if constexpr (F == kFmtE3M2) {
      asm("cvt.rn.satfinite.e3m2x2.f32 %0, %2, %1;" : "=h"(lo) : "f"(a), "f"(b));
      asm("cvt.rn.satfinite.e3m2x2.f32 %0, %2, %1;" : "=h"(hi) : "f"(c), "f"(d));
    } else {
      asm("cvt.rn.satfinite.e2m3x2.f32 %0, %2, %1;" : "=h"(lo) : "f"(a), "f"(b));
      asm("cvt.rn.satfinite.e2m3x2.f32 %0, %2, %1;" : "=h"(hi) : "f"(c), "f"(d));
    }
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
}

// Warp-wide maximum of |x| (NaN-propagating).
__device__ __forceinline__ float warp_max_abs(float x) {
  float r;
  asm volatile("redux.sync.max.abs.NaN.f32 %0, %1, 0xffffffff;"
               : "=f"(r)
               : "f"(x));
  return r;
}

// E8M0 code of a block maximum given as fp32 bits (sign ignored):
// floor(log2 amax) - 8 + 127, clamped at 0; non-finite -> 0xFF.
__device__ __forceinline__ uint32_t e8m0_code_from_amax_bits(uint32_t bits) {
  uint32_t ef = (bits >> 23) & 0xFFu;
  if (ef == 0xFFu) return 0xFFu;
  return ef > 8u ? ef - 8u : 0u;
}

// 2^-e as fp32 for e = code - 127 (code in [0, 254]).
__device__ __forceinline__ float inv_scale_from_code(uint32_t code) {
  return __uint_as_float((254u - code) << 23);
}


// ------------------------------------------------- CTA pairs (cta_group::2)
// Two CTAs of a cluster whose ranks differ in bit 0 form a pair; one
// tcgen05.mma.cta_group::2 issued by the even CTA computes an M = 256 tile
// whose A rows, B rows (N) and D rows are split between the two CTAs' shared
// and tensor memory at the same offsets.  Every tcgen05 instruction of a
// kernel that uses pairs carries cta_group::2.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster (address from mapa).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// As mbar_wait, with cluster-scope acquire (the phase is completed by
// arrivals from the other CTA of the pair).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* err,
                                                  volatile int* abort, uint32_t site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        if (abort != nullptr) *abort = 1;
        report_error(err, ERR_WAIT_TIMEOUT, site);
        return false;
      }
    }
  }
}

// TMA tile load into this CTA's shared memory whose completion is signalled
// on the mbarrier at `bar_cluster` (a cluster address: this CTA's or the
// pair peer's).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const void* tmap, int32_t x,
                                                 int32_t y, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// Whole warp of each CTA of the pair: allocate the same `ncols` columns in
// both tensor memories.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols)
               : "memory");
}

// Arrive on `bar` (this CTA) once the pair's tcgen05 operations issued so far
// by this thread have completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// The same, arriving on the mbarrier at this offset in every CTA of `mask`.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Scale tile copy shared -> tensor memory in each CTA of the pair (same
// offsets).
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// D (M = 256 over the pair) (+)= A * B, block-scaled, K = 32 per MMA.
__device__ __forceinline__ void mma_pair_mxf8_ss(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Elected-lane forms of the pair instructions (whole converged warp calls).
__device__ __forceinline__ void mma_pair_mxf8_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                       uint64_t b_desc, uint32_t idesc,
                                                       uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t" LPFA_ELECT
      "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4_elect(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_mc_elect(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Dense FP4 pair MMAs (kind::mxf4nvf4, K = 64): MXFP4 (scale_vec::2X) and
// NVFP4 (scale_vec::4X).
__device__ __forceinline__ void mma_pair_mxf4_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                       uint64_t b_desc, uint32_t idesc,
                                                       uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t" LPFA_ELECT
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_pair_nvf4_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                       uint64_t b_desc, uint32_t idesc,
                                                       uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t" LPFA_ELECT
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Elected-lane forms of the pair TMA loads (whole converged warp calls).
__device__ __forceinline__ void tma_load_2d_pair_elect(void* smem_dst, const void* tmap, int32_t x,
                                                       int32_t y, uint32_t bar_cluster) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair_elect(void* smem_dst, const void* tmap, int32_t x,
                                                       int32_t y, int32_t z, uint32_t bar_cluster) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t" LPFA_ELECT
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3, %4}], [%5];\n\t}" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
      : "memory");
}

}  // namespace lpfa
