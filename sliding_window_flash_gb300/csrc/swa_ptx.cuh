// swa_ptx.cuh — thin inline-PTX layer for sm_103a: mbarriers, TMA tile loads, tcgen05 MMA/TMEM.
//
// Everything the attention kernels need from the Blackwell execution model, written as small
// device functions over PTX instructions:
//   * mbarrier init / arrive / expect-tx / bounded parity wait,
//   * cp.async.bulk.tensor (TMA) 3-D tile loads with 128-byte swizzle,
//   * tcgen05.alloc / dealloc of tensor memory (TMEM), tcgen05.mma (kind::f16, bf16 in, fp32 acc,
//     cta_group::1), tcgen05.commit to an mbarrier, tcgen05.ld / st of 32 lanes x 32 columns,
//   * the shared-memory matrix descriptor and the instruction descriptor of tcgen05.mma.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "swa_kernels.h"

namespace swa {

// ------------------------------------------------------------------------------------------------
// Error reporting of bounded waits.
// ------------------------------------------------------------------------------------------------

// A wait gives up after this many SM clock cycles (~1 s at 2 GHz) or this many polls.
constexpr long long kWaitCycleLimit = 2000000000ll;
constexpr unsigned kWaitPollLimit = 1u << 30;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }

// ------------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tensor cores) and other threads.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Slow path of the waits below: keeps polling until the phase completes, the abort flag rises, or
// the bound runs out (then raises the abort flag and the device error word).  Kept out of line so
// that a wait whose phase has already completed costs one try_wait.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            unsigned* err_word) {
  const long long t0 = clock64();
  for (unsigned it = 0; it < kWaitPollLimit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (clock64() - t0 > kWaitCycleLimit) break;
    }
  }
  *abort_flag = 1;
  atomicOr(err_word, kErrWaitTimeout);
  return false;
}

// Waits until the phase with the given parity has completed.  Bounded: returns false (and raises
// the CTA's abort flag and the device error word) when the wait runs out, or returns false at once
// when another role of the CTA has already raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* err_word) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, err_word);
}

// ------------------------------------------------------------------------------------------------
// Proxy fences and named barriers
// ------------------------------------------------------------------------------------------------

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------------------------------------
// TMA
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tile load (x innermost).  Out-of-range elements are written as zero; the barrier's
// transaction count is charged the full box.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 3-D tile store from shared memory (same box and swizzle as the loads).  Elements outside the
// tensor are not written.  Completion is tracked with the bulk async-group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// dst[0..3] += {a, b, c, d} in fp32, performed at the L2 (relaxed, no return value); dst 16-byte
// aligned.
__device__ __forceinline__ void red_add_v4_f32(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// ------------------------------------------------------------------------------------------------
// tcgen05: TMEM allocation
// ------------------------------------------------------------------------------------------------

// Whole warp.  Writes the allocated TMEM base address to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------------------------------------
// tcgen05: descriptors
// ------------------------------------------------------------------------------------------------

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits  0-13 start address >> 4      bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 descriptor version (1 on sm_100 family)
//   bits 49-51 base offset (0: atoms 1024-byte aligned)   bits 61-63 layout (2 = 128B swizzle)
// K-major operand: rows of 128 bytes (64 bf16 along K), 8-row atoms of 1024 bytes; SBO = distance
// between 8-row groups, LBO unused.  MN-major operand: 128-byte rows hold 64 consecutive M/N
// elements, one row per K index; SBO = distance between 8-K-row groups, LBO = distance between
// 64-element M/N blocks.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32)   bits 7-9 A format (1 = bf16)   bits 10-12 B format (1 = bf16)
//   bit 15 A major (0 K, 1 MN)    bit 16 B major                  bits 17-22 N >> 3
//   bits 24-28 M >> 4
// `fmt` is the A/B operand format of kind::f16: 0 = fp16, 1 = bf16 (both operands the same).
__host__ __device__ constexpr uint32_t idesc_f16kind(uint32_t fmt, int M, int N, bool a_mn_major,
                                                     bool b_mn_major) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------------------------------------
// tcgen05: MMA and commit
// ------------------------------------------------------------------------------------------------

// Warp-converged forms: every lane of the issuing warp executes these, one elected lane issues.
// Keeping the MMA warp converged (rather than running its loop on one lane) keeps the tensor pipe
// fed: branches inside a single-lane region stall the issue of the next MMA.

// Arrives once on `bar` when every tcgen05 operation issued so far by the issuing thread has
// completed.
__device__ __forceinline__ void umma_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// 8 MMAs along K (16 each) with A and B both K-major, 128B-swizzled, 128-row tiles in shared
// memory: K-step ks starts 32 bytes further inside a 64-column chunk, and every fourth step moves
// to the next 16 KB chunk.  One elect.sync for the whole group; descriptor offsets (16-byte units)
// are immediate adds.  The first MMA accumulates iff `accumulate`, the others always do.
__device__ __forceinline__ void umma_ss_kmajor_x8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b64 ra, rb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 1024;\n\tadd.s64 rb, %2, 1024;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 1026;\n\tadd.s64 rb, %2, 1026;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 1028;\n\tadd.s64 rb, %2, 1028;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 1030;\n\tadd.s64 rb, %2, 1030;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "}" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 4 MMAs along K (16 each) with A and B both K-major, 128B-swizzled, 128-row tiles in shared
// memory: K-step ks starts 32 bytes further inside a 64-column chunk, and every fourth step moves
// to the next 16 KB chunk.  One elect.sync for the whole group; descriptor offsets (16-byte units)
// are immediate adds.  The first MMA accumulates iff `accumulate`, the others always do.
__device__ __forceinline__ void umma_ss_kmajor_x4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b64 ra, rb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "}" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// S-type product over the head dimension D (64 or 128; D = 256 runs as two 128 halves): D / 16
// MMAs.
template <int D>
__device__ __forceinline__ void umma_ss_kmajor_d(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  static_assert(D == 64 || D == 128, "head dim");
  if constexpr (D == 128)
    umma_ss_kmajor_x8(d_tmem, a_desc, b_desc, idesc, accumulate);
  else
    umma_ss_kmajor_x4(d_tmem, a_desc, b_desc, idesc, accumulate);
}

// 8 MMAs along K = 128 with A (bf16 pairs) in TMEM and B MN-major, 128B-swizzled in shared memory
// (one 128-byte row per K index, so K-step ks starts 2048 bytes further).  A's K-step ks sits at
// column 8 ks (contiguous packing) or 8 ks + 32 (ks / 4) (two 32-column halves 64 columns apart).
__device__ __forceinline__ void umma_ts_mnmajor_x8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 ra;\n\t.reg .b64 rb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 ra, %1, 8;\n\tadd.s64 rb, %2, 128;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 16;\n\tadd.s64 rb, %2, 256;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 24;\n\tadd.s64 rb, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 32;\n\tadd.s64 rb, %2, 512;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 40;\n\tadd.s64 rb, %2, 640;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 48;\n\tadd.s64 rb, %2, 768;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 56;\n\tadd.s64 rb, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_ts_mnmajor_x8_split(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 ra;\n\t.reg .b64 rb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.u32 ra, %1, 8;\n\tadd.s64 rb, %2, 128;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 16;\n\tadd.s64 rb, %2, 256;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 24;\n\tadd.s64 rb, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 64;\n\tadd.s64 rb, %2, 512;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 72;\n\tadd.s64 rb, %2, 640;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 80;\n\tadd.s64 rb, %2, 768;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.u32 ra, %1, 88;\n\tadd.s64 rb, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 8 MMAs along K = 128 with A K-major (128B-swizzled, two 64-column chunks 16 KB apart: K-step ks
// at 32 (ks % 4) bytes inside chunk ks / 4) and B MN-major (one 128-byte row per K index, so K-step
// ks starts 2048 bytes further).  Both operands in shared memory.
__device__ __forceinline__ void umma_ss_kA_mnB_x8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                  uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b64 ra, rb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 128;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 256;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 1024;\n\tadd.s64 rb, %2, 512;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 1026;\n\tadd.s64 rb, %2, 640;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 1028;\n\tadd.s64 rb, %2, 768;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 1030;\n\tadd.s64 rb, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "}" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 8 MMAs along K = 128 with A and B both MN-major in shared memory (one 128-byte row per K index:
// K-step ks starts 2048 bytes further in both).
__device__ __forceinline__ void umma_ss_mnA_mnB_x8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b64 ra, rb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "add.s64 ra, %1, 128;\n\tadd.s64 rb, %2, 128;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 256;\n\tadd.s64 rb, %2, 256;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 384;\n\tadd.s64 rb, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 512;\n\tadd.s64 rb, %2, 512;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 640;\n\tadd.s64 rb, %2, 640;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 768;\n\tadd.s64 rb, %2, 768;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "add.s64 ra, %1, 896;\n\tadd.s64 rb, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
      "}" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ------------------------------------------------------------------------------------------------
// tcgen05: TMEM <-> registers, 32 lanes x 32 columns of 32 bits (one lane per thread of the warp).
// A warp may only touch the 32-lane quarter (warp_id % 4) of TMEM.
// ------------------------------------------------------------------------------------------------

#define SWA_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), \
                  "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
#define SWA_W8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), \
                  "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])

// Issues the load; the registers are valid only after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : SWA_R8(0), SWA_R8(8), SWA_R8(16), SWA_R8(24)
      : "r"(taddr));
}

// 16 lanes x 8 groups of 8 columns (16x256b shape, 8 repetitions): with L the lane in taddr,
// thread t receives, for group j, r[4j], r[4j+1] = columns 8j + 2(t%4), +1 of lane L + t/4 and
// r[4j+2], r[4j+3] = the same columns of lane L + 8 + t/4.  Issues the load (no wait).
__device__ __forceinline__ void tmem_ld16x256_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : SWA_R8(0), SWA_R8(8), SWA_R8(16), SWA_R8(24)
      : "r"(taddr));
}

// Waits for this thread's outstanding TMEM loads; `r` is passed through so that no use of the
// loaded registers can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}

// Waits for all of this thread's outstanding TMEM loads (use reg_fence on every loaded array
// afterwards, so that no use of those registers is scheduled above the wait).
__device__ __forceinline__ void tmem_wait_ld_all() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      SWA_W8(0), SWA_W8(8), SWA_W8(16), SWA_W8(24)
      : "memory");
}

// The store counterpart of tmem_ld16x256_x8 (same register layout).
__device__ __forceinline__ void tmem_st16x256_x8(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      SWA_W8(0), SWA_W8(8), SWA_W8(16), SWA_W8(24)
      : "memory");
}

// 16 lanes x 16 groups of 4 columns (16x128b shape, 16 repetitions): thread t writes r[2j] to
// column 4j + t%4 of lane L + t/4 and r[2j+1] to the same column of lane L + 8 + t/4.
__device__ __forceinline__ void tmem_st16x128_x16(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      SWA_W8(0), SWA_W8(8), SWA_W8(16), SWA_W8(24)
      : "memory");
}

// 32 lanes x 16 columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      SWA_W8(0), SWA_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef SWA_R8
#undef SWA_W8

// ------------------------------------------------------------------------------------------------
// Small arithmetic helpers
// ------------------------------------------------------------------------------------------------

// 2^x with the hardware approximation (MUFU.EX2); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Element type of the attention tensors: bf16 (F16 = false) or fp16.  Both are kind::f16
// tensor-core operands; P and dS are rounded to the element type (round to nearest even) and
// every accumulator is fp32 either way.
template <bool F16>
struct Elem {
  static constexpr uint32_t kMmaFmt = F16 ? 0u : 1u;  // A/B format field of the MMA descriptor
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    if constexpr (F16) {
      __half2 h = __floats2half2_rn(lo, hi);
      return *reinterpret_cast<uint32_t*>(&h);
    } else {
      return pack_bf16x2(lo, hi);
    }
  }
  static __device__ __forceinline__ float2 unpack(uint32_t v) {
    if constexpr (F16)
      return __half22float2(*reinterpret_cast<const __half2*>(&v));
    else
      return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  }
};

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t a) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(a) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Byte offset of 16-byte unit `unit` (0..7) of row `row` inside a 128B-swizzled K-major tile
// whose rows are 128 bytes (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t unit) {
  return row * 128u + ((unit ^ (row & 7u)) << 4);
}

// ------------------------------------------------------------------------------------------------
// Kernel-side helpers shared by the attention kernels
// ------------------------------------------------------------------------------------------------

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
#define SWA_NEG_INF (-__int_as_float(0x7f800000))
#define SWA_POS_INF (__int_as_float(0x7f800000))

// True when the dynamic shared-memory window starts on a 1024-byte boundary, which the
// 128-byte-swizzled tiles require.  Kernels declare no static shared memory and request exactly
// their layout's size, so the window is aligned; a kernel that finds it is not raises
// kErrSmemLayout and returns at once, before any barrier or tensor-memory use.
__device__ __forceinline__ bool smem_base_ok(const uint8_t* smem, unsigned* err) {
  if ((smem_u32(smem) & 1023u) == 0u) return true;
  if (threadIdx.x == 0) atomicOr(err, kErrSmemLayout);
  return false;
}

// Bounded wait that ignores the abort flag: used to drain a CTA's own copies before it exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned* err) {
  int never = 0;
  mbar_wait(bar, parity, &never, err);
}

// drain_wait for all 32 lanes of a warp.
__device__ __forceinline__ void warp_drain_wait(uint32_t bar, uint32_t parity, unsigned* err) {
  int never = 0;
  const bool ok = mbar_wait(bar, parity, &never, err);
  __all_sync(0xffffffffu, ok);
}

// One arrival per warp: every lane has finished its own tcgen05 loads/stores (wait::ld / wait::st)
// and shared-memory writes before this; the before_thread_sync fence and __syncwarp order them
// ahead of lane 0's release-arrive.  Barriers fed this way count warps, not threads, which keeps
// the shared-memory atomics per phase at one per warp.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31u) == 0u) mbar_arrive(bar);
}

// All 32 lanes wait; the result is uniform across the warp.  Fast path: one try_wait per lane and
// one vote.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* err) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const bool ok = mbar_wait_slow(bar, parity, abort_flag, err);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------------------------------------
// CTA pairs (cluster of two CTAs on one TPC sharing tcgen05.mma.cta_group::2 operations)
// ------------------------------------------------------------------------------------------------
// An M = 256 pair MMA issued by rank 0 computes rows [0, 128) into rank 0's TMEM and rows
// [128, 256) into rank 1's, each from its own CTA's A operand (shared memory or TMEM, at the same
// address in both); B's N columns are split between the pair, [0, N/2) in rank 0's shared memory
// and [N/2, N) in rank 1's, at the same address.  A kernel that uses pairs uses cta_group::2 for
// every tcgen05 allocation, MMA and commit.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs; orders each CTA's prior shared-memory writes (barrier inits
// included) before the other's later accesses.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the cluster window, of the same shared-memory offset in rank 0 of the pair.
__device__ __forceinline__ uint32_t mapa_rank0(uint32_t saddr) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(saddr));
  return r;
}

// Arrive on a barrier given by its cluster-window address (default semantics: the data handed
// over is TMEM, ordered by the tcgen05 fences around the arrive and the wait, or shared memory
// written by TMA and read by the tensor core).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// mbar_wait_slow with acquire at cluster scope (barriers that the other CTA of a pair arrives on).
static __device__ __noinline__ bool mbar_wait_cluster_slow(uint32_t bar, uint32_t parity,
                                                           volatile int* abort_flag,
                                                           unsigned* err_word) {
  const long long t0 = clock64();
  for (unsigned it = 0; it < kWaitPollLimit; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (clock64() - t0 > kWaitCycleLimit) break;
    }
  }
  *abort_flag = 1;
  atomicOr(err_word, kErrWaitTimeout);
  return false;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, unsigned* err_word) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return mbar_wait_cluster_slow(bar, parity, abort_flag, err_word);
}

__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, unsigned* err) {
  if (__all_sync(0xffffffffu, mbar_try_wait_cluster(bar, parity))) return true;
  const bool ok = mbar_wait_cluster_slow(bar, parity, abort_flag, err);
  return __all_sync(0xffffffffu, ok);
}

// warp_arrive on the barrier at the same offset in rank 0 of the pair.
__device__ __forceinline__ void warp_arrive_rank0(uint32_t bar) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31u) == 0u) mbar_arrive_cluster(mapa_rank0(bar));
}

// One warp in each CTA of the pair, collectively: both receive the same TMEM address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Arrives once on the barrier at offset `bar` in both CTAs of the pair when every tcgen05
// operation issued so far by the issuing thread has completed.
__device__ __forceinline__ void umma2_commit_w(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar),
      "h"(static_cast<unsigned short>(3))
      : "memory");
}

// Pair MMAs along K over the head dimension D (64 or 128): A and B K-major, 128B-swizzled.  A is
// each CTA's 128-row tile (64-column chunks 16 KB apart), B each CTA's 64-row half (chunks 8 KB
// apart).  K-step ks starts 32 bytes further inside a chunk; every fourth step moves to the next.
template <int D>
__device__ __forceinline__ void umma2_ss_kmajor_d(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                  uint32_t idesc, uint32_t accumulate) {
  static_assert(D == 64 || D == 128, "head dim");
  if constexpr (D == 128) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b64 ra, rb;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, %3, %3;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "add.s64 ra, %1, 1024;\n\tadd.s64 rb, %2, 512;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "add.s64 ra, %1, 1026;\n\tadd.s64 rb, %2, 514;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "add.s64 ra, %1, 1028;\n\tadd.s64 rb, %2, 516;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "add.s64 ra, %1, 1030;\n\tadd.s64 rb, %2, 518;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "}" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b64 ra, rb;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, %3, %3;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], ra, rb, %3, t;\n\t"
        "}" ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// umma2_ts_mnmajor_x8 with A's K-step ks at column 8 ks + 32 (ks / 4): two 32-column halves 64
// columns apart.
__device__ __forceinline__ void umma2_ts_mnmajor_x8_split(uint32_t d_tmem, uint32_t a_tmem,
                                                          uint64_t b_desc, uint32_t idesc,
                                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 ra;\n\t.reg .b64 rb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.s32 ra, %1, 8;\n\tadd.s64 rb, %2, 128;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 16;\n\tadd.s64 rb, %2, 256;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 24;\n\tadd.s64 rb, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 64;\n\tadd.s64 rb, %2, 512;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 72;\n\tadd.s64 rb, %2, 640;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 80;\n\tadd.s64 rb, %2, 768;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 88;\n\tadd.s64 rb, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 8 pair MMAs along K = 128 with A (bf16 pairs, K-step ks at column 8 ks) in each CTA's TMEM and
// B MN-major, 128B-swizzled in each CTA's shared memory (one 128-byte row per K index: K-step ks
// starts 2048 bytes further).
__device__ __forceinline__ void umma2_ts_mnmajor_x8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                    uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t.reg .b32 ra;\n\t.reg .b64 rb;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, %3, %3;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "add.s32 ra, %1, 8;\n\tadd.s64 rb, %2, 128;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 16;\n\tadd.s64 rb, %2, 256;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 24;\n\tadd.s64 rb, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 32;\n\tadd.s64 rb, %2, 512;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 40;\n\tadd.s64 rb, %2, 640;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 48;\n\tadd.s64 rb, %2, 768;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "add.s32 ra, %1, 56;\n\tadd.s64 rb, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [ra], rb, %3, t;\n\t"
      "}" ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Stages 16 packed bf16 pairs = columns [c0, c0 + 32) of row `row` of a 128-row tile whose
// 64-column chunks (128 rows x 128 bytes, 128B-swizzled) start at `tile` + chunk * 16 KB.
__device__ __forceinline__ void stage_row32_sw128(uint32_t tile, uint32_t row, uint32_t c0,
                                                  const uint32_t (&pk)[16]) {
  const uint32_t chunk = tile + (c0 >> 6) * (128u * 128u);
  const uint32_t unit0 = (c0 & 63u) >> 3;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    st_shared_v4(chunk + sw128_offset(row, unit0 + u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                 pk[4 * u + 3]);
}

// Writes zeros to rows [k0, min(k0 + 128, L)) of plane `bh` of one or two (t1 may be null)
// [BH, L, D] 16-bit tensors, with 16-byte stores spread over the whole block.
__device__ __forceinline__ void zero_key_rows(uint16_t* t0, uint16_t* t1, int bh, int k0, int L,
                                              int D) {
  const int rows = min(128, L - k0);
  if (rows <= 0) return;
  const size_t base = (static_cast<size_t>(bh) * L + k0) * D;
  const int units = rows * D / 8;  // 16-byte units per tensor
  const int total = t1 ? 2 * units : units;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int u = static_cast<int>(threadIdx.x); u < total; u += static_cast<int>(blockDim.x)) {
    uint16_t* t = u < units ? t0 : t1;
    reinterpret_cast<uint4*>(t + base)[u < units ? u : u - units] = z;
  }
}

}  // namespace swa
