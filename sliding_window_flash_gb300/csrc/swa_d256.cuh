// swa_d256.cuh — device code shared by the head-dimension-256 kernels (swa_d256.cu and the
// CTA-pair kernels next to it): the score-column mask, the transposed probabilities and dS of
// the key-block kernels and their accumulator epilogue, and the compute warps of the forward and
// dQ kernels (one routine each for the single-CTA and the pair kernel).
#pragma once
#include "swa_kernels.h"
#include "swa_ptx.cuh"

namespace swa {
namespace d256 {

constexpr int kChunk = kBlockM * 128;  // one 64-column chunk: 128 rows x 128 bytes

// Before a CTA exits no copy may be in flight.  Called by all 32 lanes of both producer warps of
// a two-producer ring (p = 0, 1), `last` being lane 0's last item per slot and full(i) the
// barrier item i completes: the two warps publish their `last` in `s_last` ([2][kSlots] ints),
// meet at named barrier 1, then one lane waits (bounded) for the final fill of every slot.  Only
// the final fill's phase parity (item / kSlots) is unambiguous: the producers alternate within a
// slot, so a producer's own last fill may be followed by the other's, after which the barrier has
// moved two phases on.
template <int kSlots, typename FullOf>
__device__ __forceinline__ void drain_ring(const int (&last)[kSlots], int* s_last, int p,
                                           uint32_t lane, FullOf full, unsigned* err) {
  if (lane == 0)
    for (int s = 0; s < kSlots; ++s) s_last[p * kSlots + s] = last[s];
  __syncwarp();
  named_barrier_sync(1, 64);
  if (p == 0 && lane == 0) {
    for (int s = 0; s < kSlots; ++s) {
      const int fin = max(s_last[s], s_last[kSlots + s]);
      if (fin >= 0) drain_wait(full(fin), static_cast<uint32_t>((fin / kSlots) & 1), err);
    }
  }
}

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

// ------------------------------------------------------------------------------------------------
// The forward's softmax warps (warps 0-7 of the D = 256 forward kernels, single-CTA and pair):
// two threads per query row (warp w: TMEM lanes 32 (w % 4).., score columns [64 h, 64 h + 64),
// h = w / 4); per key block S is read from TMEM, masked at the window's edges, exponentiated
// against the running reference max (redone exactly on a tile's first block or when a row's block
// sum exceeds 2^12, the row's halves swapping their block sums and maxima through shared memory),
// and P goes back over S as packed pairs; each tile's epilogue divides O by the row sum, writes the
// natural-log LSE and stages O (16-bit, swizzled) in the Q buffer for the store warp.
// ------------------------------------------------------------------------------------------------
constexpr float kRescaleThreshold = 8.0f;  // exact path: move the max only past 2^8
constexpr float kFastSumLimit = 4096.0f;   // one-pass block stands if its row sum <= 2^12

// Addresses the softmax warps use.  S / P buffers at tmem + 0 and + 128, O at tmem + 256.  The
// kernels keep their softmax barriers as one run of 8-byte mbarriers starting at `bars`, in the
// order of FwdBar below.
struct FwdSoftmax {
  uint32_t tmem, sQ;
  float* s_red;   // [2 slots][2 halves][128] fp32
  uint32_t bars;  // address of the first S-full barrier
  volatile int* abort_flag;
  unsigned* err;
  float scale_log2;
  float* lse;
};
struct FwdBar {
  static constexpr int kSFull = 0;    // 2: S of block g landed in buffer g & 1
  static constexpr int kPFull = 2;    // 2: P of block g written (rank 0's in a pair)
  static constexpr int kPVDone = 4;   // 2: P V of block g completed
  static constexpr int kXch = 6;      // [4 lane quarters][2 slots]: row-half swaps
  static constexpr int kOEmpty = 14;  // O read out (rank 0's in a pair)
  static constexpr int kOutFull = 15; // staged O tile complete
};

// Runs the softmax warps over the CTA's tiles tile0, tile0 + tile_step, .. < ntiles, with the
// addresses in cx; tile_of(t) gives the tile's plane bh, first query q0, first key block kb_lo and
// block count nkv.  With kPair the P-written and O-read handshakes go to rank 0 of the CTA pair
// (whose MMA warp issues for both SMs).
template <bool F16, bool kPair, typename TileOf>
__device__ __forceinline__ void fwd_softmax(const FwdSoftmax& cx, const Span& sp, int tile0,
                                            int tile_step, int ntiles, TileOf tile_of) {
  const uint32_t warp = warp_id(), lane = lane_id();
  auto bar = [&](int i) { return cx.bars + 8u * static_cast<uint32_t>(i); };
  auto arrive = [](uint32_t b) {
    if constexpr (kPair)
      warp_arrive_rank0(b);
    else
      warp_arrive(b);
  };
  const int r = static_cast<int>(threadIdx.x & 127);  // row within the tile == TMEM lane
  const uint32_t h = warp >> 2;                          // column half of every score tile
  const uint32_t quarter = warp & 3u;
  const uint32_t lane_base = (quarter * 32u) << 16;
  const float sl2 = cx.scale_log2;
  int xn = 0;  // exchanges done so far
  // Swap a per-row value with the thread that owns the other half of the row (slot xn & 1 was
  // last used two exchanges ago, and the partner passed the exchange in between only after
  // reading it).
  auto exchange = [&](float v, float* other) -> bool {
    float* red = cx.s_red + (xn & 1) * 2 * kBlockM;
    red[h * kBlockM + r] = v;
    __syncwarp();
    const uint32_t xb = bar(FwdBar::kXch + quarter * 2 + (xn & 1));
    if (lane == 0) mbar_arrive(xb);
    if (!warp_wait(xb, (xn >> 1) & 1, cx.abort_flag, cx.err)) return false;
    *other = red[(h ^ 1u) * kBlockM + r];
    ++xn;
    return true;
  };
  int g = 0;
  bool ok = true;
  for (int t = tile0, it = 0; ok && t < ntiles; t += tile_step, ++it) {
    const auto f = tile_of(t);
    const int q0 = f.q0;
    const int row = q0 + r;
    float m_ref = SWA_NEG_INF;  // reference max (log2 domain) that P and l are taken against
    float l = 0.f;              // partial row sum over this thread's half of the columns
    for (int j = 0; j < f.nkv; ++j) {
      const int gg = g + j;
      const int k0 = (f.kb_lo + j) * kBlockN;
      const int sb = gg & 1;
      if (!(ok = warp_wait(bar(FwdBar::kSFull + sb), (gg >> 1) & 1, cx.abort_flag, cx.err))) break;
      tc_fence_after();
      const uint32_t s_col = cx.tmem + lane_base + 128u * sb + 64u * h;
      float x[64];  // raw scores S (the scale is applied inside the exponent)
      {
        uint32_t rr[2][32];
        tmem_ld32(s_col, rr[0]);
        tmem_ld32(s_col + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(rr[c >> 5][c & 31]);
      }
      if (!sp.interior(q0, k0)) {
        // Columns c (keys k0 + 64h + c) visible to row `row`, and inside the key sequence.
        const int rel = row + sp.off - k0 - 64 * static_cast<int>(h);
        mask64(x, rel - sp.dmax, min(rel - sp.dmin, sp.Lk - 1 - k0 - 64 * static_cast<int>(h)),
               SWA_NEG_INF);
      }
      uint32_t pk[32];
      auto exponentiate = [&](float m) -> float {
        const float2 scale2 = make_float2(sl2, sl2), neg_m2 = make_float2(-m, -m);
        float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 tt = __ffma2_rn(make_float2(x[2 * c], x[2 * c + 1]), scale2, neg_m2);
          const float2 e = make_float2(ex2(tt.x), ex2(tt.y));
          rs2[c & 3] = __fadd2_rn(rs2[c & 3], e);
          pk[c] = Elem<F16>::pack(e.x, e.y);
        }
        return ((rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y)) +
               ((rs2[2].x + rs2[2].y) + (rs2[3].x + rs2[3].y));
      };
      // One pass against the running reference max; redone exactly on a tile's first block or
      // when a row's block sum exceeds 2^12 (both halves of a row decide alike).
      bool redo = true;
      float bsum = 0.f;
      if (__all_sync(0xffffffffu, m_ref != SWA_NEG_INF)) {
        bsum = exponentiate(m_ref);
        float other;
        if (!(ok = exchange(bsum, &other))) break;
        redo = __any_sync(0xffffffffu, !(bsum + other <= kFastSumLimit));
      }
      bool resc = false;
      float factor = 1.f;
      if (redo) {
        float m8[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) m8[c] = x[c];
#pragma unroll
        for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], x[c]);
        float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                         fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
        float mx_other;
        if (!(ok = exchange(mx, &mx_other))) break;
        mx = fmaxf(mx, mx_other);
        const float m_new = fmaxf(m_ref, mx);
        resc = m_new > m_ref + kRescaleThreshold;
        if (resc) {
          factor = ex2(m_ref - m_new);  // 0 when m_ref is -inf
          l *= factor;
          m_ref = m_new;
        }
        bsum = exponentiate((m_ref == SWA_NEG_INF) ? 0.f : m_ref);
      }
      l += bsum;
      // Rescaling O needs this tile's P V of block gg - 1 (and so every earlier one) to have
      // landed; a tile's first block needs none (its P V overwrites O).
      if (j >= 1 && __any_sync(0xffffffffu, resc)) {
        if (!(ok = warp_wait(bar(FwdBar::kPVDone + (sb ^ 1)), ((gg - 1) >> 1) & 1, cx.abort_flag,
                             cx.err)))
          break;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          const uint32_t oc = cx.tmem + lane_base + 256u + 128u * h + c0;
          uint32_t rr[32];
          tmem_ld32(oc, rr);
          tmem_wait_ld(rr);
#pragma unroll
          for (int c = 0; c < 32; ++c) rr[c] = __float_as_uint(__uint_as_float(rr[c]) * factor);
          tmem_st32(oc, rr);
        }
      } else {
        tc_fence_after();
      }
      // keys [64h, 64h + 64) -> packed P over the first 32 of this thread's S columns (the
      // landing of S_gg implies P V_{gg-2}, which read the previous P here, has completed).
      tmem_st32(s_col, pk);
      tmem_wait_st();
      arrive(bar(FwdBar::kPFull + sb));
    }
    if (!ok) break;
    g += f.nkv;

    // ---------------------------------------------------------- tile epilogue
    float l_other = 0.f;
    if (!(ok = exchange(l, &l_other))) break;
    const int last = g - 1;
    if (!(ok = warp_wait(bar(FwdBar::kPVDone + (last & 1)), (last >> 1) & 1, cx.abort_flag, cx.err)))
      break;
    tc_fence_after();
    const float l_row = l + l_other;
    const float inv_l = 1.f / l_row;
    const float m_use = (m_ref == SWA_NEG_INF) ? 0.f : m_ref;
    if (row < sp.Lq && h == 0)
      cx.lse[static_cast<size_t>(f.bh) * sp.Lq + row] = (m_use + log2f(l_row)) * kLn2;
    // O / l -> 16-bit, staged in the Q buffer (every S of the tile has completed) in the
    // swizzled layout of the TMA map; warp 10 stores it.
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t rr[32];
      tmem_ld32(cx.tmem + lane_base + 256u + 128u * h + 32u * c4, rr);
      tmem_wait_ld(rr);
      uint32_t o16[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        o16[c] = Elem<F16>::pack(__uint_as_float(rr[2 * c]) * inv_l,
                                 __uint_as_float(rr[2 * c + 1]) * inv_l);
      stage_row32_sw128(cx.sQ, r, 128u * h + 32u * c4, o16);
    }
    arrive(bar(FwdBar::kOEmpty));  // the next tile's first P V may overwrite O now
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(FwdBar::kOutFull));
  }
}

// ------------------------------------------------------------------------------------------------
// The dQ kernels' compute warps (warps 0-7 of the D = 256 dQ kernels, single-CTA and pair): two
// threads per query row as in the forward; per key block P = exp(scale S - LSE) (window-masked)
// and dS = P (dP - Delta) go back over the dP columns as packed pairs; each tile's dQ * scale is
// read out of TMEM and stored to global memory directly (rows past Lq are not written).
// ------------------------------------------------------------------------------------------------
struct DqBar {
  static constexpr int kSFull = 0;   // S of the block landed
  static constexpr int kSEmpty = 1;  // S read (rank 0's in a pair)
  static constexpr int kDPFull = 2;  // dP of the block landed
  static constexpr int kDSFull = 3;  // dS written (rank 0's in a pair)
  static constexpr int kDQDone = 4;  // the tile's last dQ product has completed
  static constexpr int kDQEmpty = 5; // dQ read out (rank 0's in a pair)
};

// Runs the compute warps over the CTA's tiles tile0, tile0 + tile_step, .. < a.ntiles.  TMEM: S at
// tmem + 0, dP / dS at + 128, dQ at + 256; `bars` is the address of the first of the six
// consecutive barriers of DqBar.  `a` supplies lse, delta, dq, scale, scale_log2, err and ntiles;
// tile_of(t) the tile's plane bh, first query q0, first key block kb_lo and block count nkv.
template <bool F16, bool kPair, typename Args, typename TileOf>
__device__ __forceinline__ void dq_compute(const Args& a, const Span& sp, uint32_t tmem,
                                           uint32_t bars, volatile int* abort_flag, int tile0,
                                           int tile_step, TileOf tile_of) {
  const uint32_t warp = warp_id();
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  auto arrive = [](uint32_t b) {
    if constexpr (kPair)
      warp_arrive_rank0(b);
    else
      warp_arrive(b);
  };
  const int r = static_cast<int>(threadIdx.x & 127);  // query row within the tile = TMEM lane
  const uint32_t h = warp >> 2;                          // column half of every score tile
  const uint32_t lane_base = ((warp & 3u) * 32u) << 16;
  const float sl2 = a.scale_log2;
  int g = 0;
  bool ok = true;
  // LSE and Delta of this thread's row in the next tile, loaded a whole tile ahead so that
  // the loads' latency hides behind the current tile.  Rows past the end see P = 0 (their LSE
  // is taken as +inf), so they add nothing.
  float nxt_lse = SWA_POS_INF, nxt_dlt = 0.f;
  auto fetch_rows = [&](int tn) {
    if (tn >= a.ntiles) return;
    const auto fn = tile_of(tn);
    const int rn = fn.q0 + r;
    if (rn < sp.Lq) {
      const size_t gn = static_cast<size_t>(fn.bh) * sp.Lq + rn;
      nxt_lse = a.lse[gn];
      nxt_dlt = a.delta[gn];
    } else {
      nxt_lse = SWA_POS_INF;
      nxt_dlt = 0.f;
    }
  };
  fetch_rows(tile0);
  for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
    const auto f = tile_of(t);
    const int q0 = f.q0;
    const int row = q0 + r;
    const bool in_range = row < sp.Lq;
    const size_t grow = static_cast<size_t>(f.bh) * sp.Lq + row;
    const float lse2 = nxt_lse == SWA_POS_INF ? SWA_POS_INF : nxt_lse * kLog2e;
    const float dlt = nxt_dlt;
    fetch_rows(t + tile_step);
    for (int j = 0; j < f.nkv; ++j) {
      const int gg = g + j;
      const int k0 = (f.kb_lo + j) * kBlockN;
      if (!(ok = warp_wait(bar(DqBar::kSFull), gg & 1, abort_flag, a.err))) break;
      tc_fence_after();
      float p[64];
      {
        uint32_t rr[2][32];
        tmem_ld32(tmem + lane_base + 64u * h, rr[0]);
        tmem_ld32(tmem + lane_base + 64u * h + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = __uint_as_float(rr[c >> 5][c & 31]);
      }
      arrive(bar(DqBar::kSEmpty));
      if (!sp.interior(q0, k0)) {
        const int rel = row + sp.off - k0 - 64 * static_cast<int>(h);
        mask64(p, rel - sp.dmax, min(rel - sp.dmin, sp.Lk - 1 - k0 - 64 * static_cast<int>(h)),
               SWA_NEG_INF);
      }
      {
        const float2 scale2 = make_float2(sl2, sl2), neg_l2 = make_float2(-lse2, -lse2);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 tt = __ffma2_rn(make_float2(p[2 * c], p[2 * c + 1]), scale2, neg_l2);
          p[2 * c] = ex2(tt.x);
          p[2 * c + 1] = ex2(tt.y);
        }
      }
      // dP_gg landing also means dQ_{gg-1} has finished reading the previous dS here.
      if (!(ok = warp_wait(bar(DqBar::kDPFull), gg & 1, abort_flag, a.err))) break;
      tc_fence_after();
      {
        const uint32_t dcol = tmem + lane_base + 128u + 64u * h;
        uint32_t rr[2][32];
        tmem_ld32(dcol, rr[0]);
        tmem_ld32(dcol + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
        uint32_t pk[32];
        const float2 neg_d2 = make_float2(-dlt, -dlt);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const uint32_t d0 = rr[c >> 4][(2 * c) & 31], d1 = rr[c >> 4][(2 * c + 1) & 31];
          const float2 ds = __fmul2_rn(
              make_float2(p[2 * c], p[2 * c + 1]),
              __fadd2_rn(make_float2(__uint_as_float(d0), __uint_as_float(d1)), neg_d2));
          pk[c] = Elem<F16>::pack(ds.x, ds.y);
        }
        tmem_st32(dcol, pk);  // over the first 32 of this thread's dP columns
      }
      tmem_wait_st();
      arrive(bar(DqBar::kDSFull));
    }
    if (!ok) break;
    g += f.nkv;

    // ---------------------------------------------------------- tile epilogue
    if (!(ok = warp_wait(bar(DqBar::kDQDone), it & 1, abort_flag, a.err))) break;
    tc_fence_after();
    uint16_t* dst_row = a.dq + grow * 256 + 128 * h;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      uint32_t rr[32];
      tmem_ld32(tmem + lane_base + 256u + 128u * h + 32u * c4, rr);
      tmem_wait_ld(rr);
      if (in_range) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = Elem<F16>::pack(__uint_as_float(rr[2 * c]) * a.scale,
                                  __uint_as_float(rr[2 * c + 1]) * a.scale);
        uint4* dst = reinterpret_cast<uint4*>(dst_row + 32 * c4);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      }
    }
    arrive(bar(DqBar::kDQEmpty));  // the next tile's first dQ may overwrite the accumulator
  }
}

}  // namespace d256
}  // namespace swa
