// swa_d256.cuh — device helpers shared by the head-dimension-256 kernels (swa_d256.cu and the
// CTA-pair kernels next to it): the score-column mask, the transposed probabilities and dS of
// the key-block kernels and their accumulator epilogue.
#pragma once
#include "swa_kernels.h"
#include "swa_ptx.cuh"

namespace swa {
namespace d256 {

constexpr int kChunk = kBlockM * 128;  // one 64-column chunk: 128 rows x 128 bytes

// Column mask of one half-row of scores: keeps columns [lo, hi] of 64, sets the rest to `fill`.
__device__ __forceinline__ void mask64(float (&x)[64], int lo, int hi, float fill) {
#pragma unroll
  for (int c = 0; c < 64; ++c) x[c] = (c >= lo && c <= hi) ? x[c] : fill;
}

// P^T = 2^(scale log2(e) S^T - LSE log2(e)) for this thread's 64 query columns, from the S^T
// columns at `s_col` and the negated LSE log2(e) of those queries in shared memory; queries the key
// row does not see get 0 (queries past the end have -LSE = -inf, so P = 0 there already).
__device__ __forceinline__ void p_transposed(float (&p)[64], uint32_t s_col, const float* nl2,
                                             float sl2, bool masked, int lo, int hi) {
  const float4* l4 = reinterpret_cast<const float4*>(nl2);
  float4 lv[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) lv[c] = l4[c];
  uint32_t rr[2][32];
  tmem_ld32(s_col, rr[0]);
  tmem_ld32(s_col + 32u, rr[1]);
  tmem_wait_ld_all();
  reg_fence(rr[0]);
  reg_fence(rr[1]);
  const float2 scale2 = make_float2(sl2, sl2);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint32_t* src = &rr[c >> 3][(4 * c) & 31];
    const float2 t0 = __ffma2_rn(make_float2(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                 scale2, make_float2(lv[c].x, lv[c].y));
    const float2 t1 = __ffma2_rn(make_float2(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                 scale2, make_float2(lv[c].z, lv[c].w));
    p[4 * c + 0] = ex2(t0.x);
    p[4 * c + 1] = ex2(t0.y);
    p[4 * c + 2] = ex2(t1.x);
    p[4 * c + 3] = ex2(t1.y);
  }
  if (masked) mask64(p, lo, hi, 0.f);
}

// dS^T = P^T (dP^T - Delta) for this thread's 64 query columns: dP^T from the TMEM columns at
// `dcol`, the negated Delta of those queries in shared memory at `nd`; the result goes back as
// packed 16-bit pairs over the first 32 of those columns (the A operand of dK += dS^T Q).
template <bool F16>
__device__ __forceinline__ void ds_transposed(uint32_t dcol, const float* nd, const float (&p)[64]) {
  const float4* d4 = reinterpret_cast<const float4*>(nd);
  float4 dv4[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) dv4[c] = d4[c];
  uint32_t rr[2][32];
  tmem_ld32(dcol, rr[0]);
  tmem_ld32(dcol + 32u, rr[1]);
  tmem_wait_ld_all();
  reg_fence(rr[0]);
  reg_fence(rr[1]);
  uint32_t pk[32];
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint32_t* src = &rr[c >> 3][(4 * c) & 31];
    const float2 d0 = __fadd2_rn(make_float2(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                 make_float2(dv4[c].x, dv4[c].y));
    const float2 d1 = __fadd2_rn(make_float2(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                 make_float2(dv4[c].z, dv4[c].w));
    const float2 s0 = __fmul2_rn(make_float2(p[4 * c], p[4 * c + 1]), d0);
    const float2 s1 = __fmul2_rn(make_float2(p[4 * c + 2], p[4 * c + 3]), d1);
    pk[2 * c] = Elem<F16>::pack(s0.x, s0.y);
    pk[2 * c + 1] = Elem<F16>::pack(s1.x, s1.y);
  }
  tmem_st32(dcol, pk);
}

// Epilogue of the key-block kernels: acc (TMEM columns [256, 512), this thread's 128-column half)
// times `mul` -> 16-bit, staged into the 64 KB tile at `stage`, then one warp stores it with four
// tensor stores (rows past Lk are not written).  With no visiting query the tile is zeros.
template <bool F16>
__device__ __forceinline__ void key_epilogue(uint32_t tmem_row, uint32_t stage, int r, uint32_t h,
                                             float mul, bool zero, uint32_t out_full_bar,
                                             const CUtensorMap* map, int k0, int bhk,
                                             volatile int* abort_flag, unsigned* err) {
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    uint32_t rr[32];
    if (!zero) {
      tmem_ld32(tmem_row + 128u * h + 32u * c4, rr);
      tmem_wait_ld(rr);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) rr[c] = 0u;
    }
    uint32_t o16[16];
#pragma unroll
    for (int c = 0; c < 16; ++c)
      o16[c] = Elem<F16>::pack(__uint_as_float(rr[2 * c]) * mul,
                               __uint_as_float(rr[2 * c + 1]) * mul);
    stage_row32_sw128(stage, static_cast<uint32_t>(r), 128u * h + 32u * c4, o16);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31u) == 0) mbar_arrive(out_full_bar);
  if (threadIdx.x < 32 && warp_wait(out_full_bar, 0, abort_flag, err) && threadIdx.x == 0) {
    for (int c = 0; c < 4; ++c) tma_store_3d(map, stage + c * kChunk, 64 * c, k0, bhk);
    bulk_commit_group();
    bulk_wait_group_read0();
  }
}

}  // namespace d256
}  // namespace swa
