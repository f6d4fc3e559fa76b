// swa_bwd_dq.cuh — the compute warps of the dQ kernels for D <= 128 (swa_bwd_dq.cu, one CTA per
// tile, and swa_bwd_dq_pair.cu, CTA pairs): per query tile, for each key block the window reaches,
// P = exp(scale S - LSE) (window-masked) and dS = P (dP - Delta) go back over the dP columns as
// packed pairs for dQ += dS K; each tile's dQ * scale is read out of TMEM and stored to global
// memory straight from registers once the next tile's first S has been read ("Off NVIDIA, you fix
// the platform yourself", Lab 28, "What did fixing it take?").
#pragma once
#include "swa_kernels.h"
#include "swa_ptx.cuh"

namespace swa {
namespace dqc {

// The compute warps' barriers: one run of consecutive 8-byte mbarriers in this order.
struct DqBar {
  static constexpr int kSFull = 0;    // S of the block landed
  static constexpr int kSEmpty = 1;   // S read (rank 0's in a pair)
  static constexpr int kDPFull = 2;   // 2, per dP buffer: dP of the block landed
  static constexpr int kDSFull = 4;   // 2, per dP buffer: dS written (rank 0's in a pair)
  static constexpr int kDQDone = 6;   // the tile's last dQ product has completed
  static constexpr int kDQEmpty = 7;  // dQ read out (rank 0's in a pair)
};

// TMEM columns: S at [0,128), dP buffers at [128,256) and [256,384) (dS written over the first 32
// of each half-row's 64 columns), dQ at [384, 384 + D).
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 384;

// Runs the compute warps (warps 0-7: two threads per query row, warp w on TMEM lanes 32 (w % 4)..
// and columns [64 h, 64 h + 64), h = w / 4) over the CTA's tiles tile0, tile0 + tile_step, ..
// < a.ntiles.  `bars` is the address of the first barrier of DqBar; `a` supplies lse, delta, dq,
// scale, scale_log2, err and ntiles; tile_of(t) the tile's plane bh, first query q0, first key block
// kb_lo and block count nkv.  With kPair the S-read, dS-written and dQ-read handshakes go to rank
// 0 of the CTA pair (whose MMA warp issues for both SMs).
template <int D, bool F16, bool kPair, typename Args, typename TileOf>
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
  const uint32_t h = warp >> 2;                          // column half of every tile
  const uint32_t lane_base = ((warp & 3u) * 32u) << 16;
  const float sl2 = a.scale_log2;
  // dQ * scale of tile `pit` -> 16-bit, written straight from registers: each thread owns 64
  // or 128 contiguous bytes of its row.
  auto epilogue = [&](int pit, size_t pgrow, bool pin) -> bool {
    if (!warp_wait(bar(DqBar::kDQDone), pit & 1, abort_flag, a.err)) return false;
    tc_fence_after();
    constexpr int kHalf = D / 2;
    uint32_t rr[kHalf / 32][32];
#pragma unroll
    for (int c4 = 0; c4 < kHalf / 32; ++c4)
      tmem_ld32(tmem + lane_base + kColDQ + kHalf * h + 32u * c4, rr[c4]);
    tmem_wait_ld_all();
#pragma unroll
    for (int c4 = 0; c4 < kHalf / 32; ++c4) reg_fence(rr[c4]);
    arrive(bar(DqBar::kDQEmpty));  // the next tile's first dQ may overwrite the accumulator
    if (pin) {
      uint16_t* dst_row = a.dq + pgrow * D + kHalf * h;
#pragma unroll
      for (int c4 = 0; c4 < kHalf / 32; ++c4) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = Elem<F16>::pack(__uint_as_float(rr[c4][2 * i]) * a.scale,
                                  __uint_as_float(rr[c4][2 * i + 1]) * a.scale);
        uint4* dst = reinterpret_cast<uint4*>(dst_row + 32 * c4);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      }
    }
    return true;
  };
  int prev_it = -1;  // tile whose epilogue is still to run
  size_t prev_grow = 0;
  bool prev_in = false;
  int g = 0;  // key blocks consumed so far by this CTA
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
        tmem_ld32(tmem + lane_base + kColS + 64u * h, rr[0]);
        tmem_ld32(tmem + lane_base + kColS + 64u * h + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
#pragma unroll
        for (int i = 0; i < 64; ++i) p[i] = __uint_as_float(rr[i >> 5][i & 31]);
      }
      arrive(bar(DqBar::kSEmpty));
      if (j == 0 && prev_it >= 0) {  // the previous tile's epilogue (see below)
        if (!(ok = epilogue(prev_it, prev_grow, prev_in))) break;
        prev_it = -1;
      }
      // Masked cells get S = -inf, so P = 0 there.
      if (!sp.interior(q0, k0)) {
        // Columns c (keys k0 + 64h + c) visible to row `row`, and inside the key sequence.
        const int rel = row + sp.off - k0 - 64 * static_cast<int>(h);
        const int lo = rel - sp.dmax;
        const int hi = min(rel - sp.dmin, sp.Lk - 1 - k0 - 64 * static_cast<int>(h));
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = (c >= lo && c <= hi) ? p[c] : SWA_NEG_INF;
      }
      // P = 2^(scale log2(e) S - LSE log2(e)), two scores per packed FFMA.
      {
        const float2 scale2 = make_float2(sl2, sl2), neg_l2 = make_float2(-lse2, -lse2);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 t = __ffma2_rn(make_float2(p[2 * c], p[2 * c + 1]), scale2, neg_l2);
          p[2 * c] = ex2(t.x);
          p[2 * c + 1] = ex2(t.y);
        }
      }

      const uint32_t dp_col = tmem + lane_base + kColDP + 128u * (gg & 1) + 64u * h;
      if (!(ok = warp_wait(bar(DqBar::kDPFull + (gg & 1)), (gg >> 1) & 1, abort_flag, a.err))) break;
      tc_fence_after();
      {
        uint32_t rr[2][32];
        tmem_ld32(dp_col, rr[0]);
        tmem_ld32(dp_col + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
        // dS = P (dP - Delta), two columns per packed FADD / FMUL.
        uint32_t pk[32];
        const float2 neg_d2 = make_float2(-dlt, -dlt);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t d0 = rr[i >> 4][(2 * i) & 31], d1 = rr[i >> 4][(2 * i + 1) & 31];
          const float2 ds = __fmul2_rn(make_float2(p[2 * i], p[2 * i + 1]),
                                       __fadd2_rn(make_float2(__uint_as_float(d0),
                                                              __uint_as_float(d1)),
                                                  neg_d2));
          pk[i] = Elem<F16>::pack(ds.x, ds.y);
        }
        // dS columns [64h, 64h+64) -> packed over the first 32 of the 64 dP columns just read.
        tmem_st32(dp_col, pk);
      }
      tmem_wait_st();
      arrive(bar(DqBar::kDSFull + (gg & 1)));
    }
    if (!ok) break;
    g += f.nkv;

    // The epilogue of this tile runs once the next tile's first S has been read (or after the
    // last tile): the MMA computes that tile's next scores while these stores drain.
    prev_it = it;
    prev_grow = grow;
    prev_in = in_range;
  }
  if (ok && prev_it >= 0) epilogue(prev_it, prev_grow, prev_in);
}

}  // namespace dqc
}  // namespace swa
