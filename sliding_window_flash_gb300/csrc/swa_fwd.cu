// swa_fwd.cu — forward of causal sliding-window attention on sm_103a.
//
// A tile is one 128-row query block of one (batch, query head):
//   O[q0:q0+128] = softmax(scale * Q K^T, window mask) V,  LSE = natural-log row log-sum-exp,
// walking only the key blocks kb_lo..kb_hi that the window reaches ("Off NVIDIA, you fix the
// platform yourself", Lab 28, "What did fixing it take?": blocks outside the window are not visited,
// blocks its boundary crosses are masked, and a query tile's walk can start past block 0).
// Only O and LSE are written (mlx-train-perf README, flash-attention section: the saved state is
// the output and the log-sum-exp).
//
// The kernel is persistent: one CTA per SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// (heaviest first).  Q is double-buffered, so the next tile's Q and first key blocks load, and its
// first score tiles are computed, while the softmax warps finish the current tile.
//
// Warp roles (384 threads):
//   warps 0-7  softmax: warp w owns TMEM lanes 32(w%4)..+31 (query rows) and columns
//              [64 h, 64 h + 64) of every score tile, h = w / 4, so each row is split over two
//              threads.  Each masks its half and exponentiates it against the row's running
//              reference max in one pass (packed fp32x2 arithmetic); the two halves swap their
//              block sums through shared memory, and only a tile's first block or a block whose
//              sum shows the max has risen far is redone exactly, with the halves' maxima
//              swapped first.  Each keeps the running max m and its partial sum l in registers,
//              writes bf16 P back to TMEM (packed pairs), rescales its half of the O row in TMEM
//              when the max grows by more than 2^8, and at the end of a tile stages its half of
//              O / l in the tile's Q buffer (and writes LSE).
//   warp 8     TMA producer of Q (per tile) and of the K ring (K_j is released as soon as S_j is
//              computed).
//   warp 11    TMA producer of the V ring (V_j is released after P_j V_j).  Loads are issued
//              from two warps because one warp's TMA copies complete at only ~40 B/clk on this
//              GPU, less than one key block (64 KB of K and V) per MMA period needs.
//   warp 9     MMA issuer and TMEM owner (converged warp, one elected lane issues): S_j = Q K_j^T
//              into one of kSBufs TMEM S buffers; O += P_j V_j with P_j read from TMEM (A operand).
//              The S products run kSBufs blocks ahead of the P V products, across tiles, so the
//              tensor core computes the next scores while the softmax warps work on this block.
//              tcgen05.mma operations of one thread run in issue order, which orders every TMEM
//              reuse below.
//   warp 10    output: one TMA tensor store per staged O tile, then frees that Q buffer.
// TMEM columns: D = 64: three S buffers at [0,384), P_j over the first 32 of each half-row's 64
// columns of its S buffer, O at [384,448).  D = 128: two S buffers at [0,256), O at [256,384), two
// 64-column P buffers at [384,512).
// D = 128 with an even number of query heads per kv head runs on CTA pairs instead
// (swa_fwd_pair.cu).
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

// In the exact path the running max is only moved (and O rescaled) when it grows by more than
// this many powers of 2; otherwise P is computed against the stale max (exact softmax either way).
constexpr float kRescaleThreshold = 8.0f;
// A block exponentiated against the running reference max stands when its row sum is at most
// this (so every P <= 2^12); otherwise it is redone against the block's own max.
constexpr float kFastSumLimit = 4096.0f;

template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = kBlockM * D * 2;  // one 128 x D bf16 tile
  static constexpr int kChunkBytes = kBlockM * 128;   // 128 rows x 64 columns (128-byte rows)
  static constexpr int kChunks = D / 64;
  static constexpr int kKStages = (D == 128) ? 3 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;  // 2 buffers
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffRed = kOffV + kVStages * kTileBytes;  // [2 slots][2 halves][128] fp32
  static constexpr int kOffBar = kOffRed + 2 * 2 * kBlockM * 4;
  // barrier indices
  static constexpr int kQFull = 0;   // 2
  static constexpr int kQEmpty = 2;  // 2
  static constexpr int kKFull = 4;
  static constexpr int kKEmpty = kKFull + kKStages;
  static constexpr int kVFull = kKEmpty + kKStages;
  static constexpr int kVEmpty = kVFull + kVStages;
  // S buffers in TMEM: the S products run kSBufs blocks ahead of the P V products, which the K
  // ring must keep fed (a K tile lands ~2,400 cycles after its copy is issued, longer than one
  // block's softmax).  D = 64 (four K stages): three buffers, P written over S.  D = 128 (three K
  // stages): two S buffers and two P buffers of their own (P over S with two buffers measured
  // slower).
  static constexpr bool kPOverS = (D == 64);
  static constexpr int kSBufs = kPOverS ? 3 : 2;
  static constexpr int kSFull = kVEmpty + kVStages;  // kSBufs
  static constexpr int kPFull = kSFull + kSBufs;     // kSBufs
  static constexpr int kPVDone = kPFull + kSBufs;    // kSBufs
  static constexpr int kXch = kPVDone + kSBufs;      // [4 lane quarters][2 slots]
  static constexpr int kOEmpty = kXch + 8;           // the O accumulator has been read
  static constexpr int kOutFull = kOEmpty + 1;       // 2: staged O tile complete, per Q buffer
  static constexpr int kDrain = kOutFull + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;  // + TMEM address and abort flag
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  // Buffer b at kColS + 128 b holds S_g (fp32) for blocks g = b mod kSBufs; P_g (bf16 pairs) goes
  // over the first 32 of each half-row's 64 columns (kPOverS) or into P buffer g & 1 at kColP.
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 128 * kSBufs;
  static constexpr uint32_t kColP = kColO + D;  // two 64-column buffers (D = 128 only)
  static constexpr int kThreads = 384;
  static constexpr int kComputeThreads = 256;
};

struct FwdArgs {
  float* lse;
  int BH;  // B * Hq
  int Hq, Hkv, G, nqb, ntiles;
  Span span;
  float scale_log2;  // scale * log2(e)
  unsigned* err;
  FastDiv divBH, divHq, divG;  // tile index decomposition
};

struct FwdTile {
  int bh, bhk, q0, kb_lo, nkv;
};

// Tile t: heaviest query blocks first (the causal case gives later blocks more key blocks).
__device__ __forceinline__ FwdTile fwd_tile(int t, const FwdArgs& a, const Span sp) {
  FwdTile f;
  const uint32_t tq = a.divBH.div(static_cast<uint32_t>(t));
  const int qb = a.nqb - 1 - static_cast<int>(tq);
  f.bh = t - static_cast<int>(tq) * a.BH;
  const uint32_t b = a.divHq.div(static_cast<uint32_t>(f.bh));
  f.bhk = static_cast<int>(b) * a.Hkv +
          static_cast<int>(a.divG.div(static_cast<uint32_t>(f.bh) - b * static_cast<uint32_t>(a.Hq)));
  f.q0 = qb * kBlockM;
  f.kb_lo = sp.first_kblock(f.q0);
  f.nkv = sp.last_kblock(f.q0) - f.kb_lo + 1;
  return f;
}

template <int D, bool F16>
__global__ void __launch_bounds__(384, 1)
    swa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (!smem_base_ok(smem, a.err)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);  // raised by a failed wait
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ0 = smem_u32(smem + C::kOffQ);
  const uint32_t sK0 = smem_u32(smem + C::kOffK);
  const uint32_t sV0 = smem_u32(smem + C::kOffV);
  float* s_red = reinterpret_cast<float*>(smem + C::kOffRed);
  const int tile_step = static_cast<int>(gridDim.x);
  const Span sp = a.span;  // window geometry, held in registers

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kQFull + b), 1);
      mbar_init(bar(C::kQEmpty + b), 1);
      mbar_init(bar(C::kOutFull + b), C::kComputeThreads / 32);
    }
    for (int b = 0; b < C::kSBufs; ++b) {
      mbar_init(bar(C::kSFull + b), 1);
      mbar_init(bar(C::kPFull + b), C::kComputeThreads / 32);
      mbar_init(bar(C::kPVDone + b), 1);
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar(C::kKFull + s), 1);
      mbar_init(bar(C::kKEmpty + s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar(C::kVFull + s), 1);
      mbar_init(bar(C::kVEmpty + s), 1);
    }
    for (int x = 0; x < 8; ++x) mbar_init(bar(C::kXch + x), 2);  // the two warps of a lane quarter
    mbar_init(bar(C::kOEmpty), C::kComputeThreads / 32);
    mbar_init(bar(C::kDrain), 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      int last_q[2] = {-1, -1};
      int last_k[C::kKStages];
      for (int s = 0; s < C::kKStages; ++s) last_k[s] = -1;
      int g = 0;  // key blocks loaded so far by this CTA
      bool ok = true;
      for (int t = blockIdx.x, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
        const FwdTile f = fwd_tile(t, a, sp);
        const int qbuf = it & 1;
        // The Q buffer was last the staging tile of tile it - 2's output.
        if (it >= 2 && !mbar_wait(bar(C::kQEmpty + qbuf), ((it - 2) >> 1) & 1, &abort_flag, a.err))
          break;
        const uint32_t sQ = sQ0 + qbuf * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kQFull + qbuf), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(sQ + h * C::kChunkBytes, &tm_q, bar(C::kQFull + qbuf), 64 * h, f.q0, f.bh);
        last_q[qbuf] = it;
        for (int j = 0; j < f.nkv; ++j, ++g) {
          const int k0 = (f.kb_lo + j) * kBlockN;
          const int sk = g % C::kKStages, nk = g / C::kKStages;
          if (g >= C::kKStages &&
              !(ok = mbar_wait(bar(C::kKEmpty + sk), (nk - 1) & 1, &abort_flag, a.err)))
            break;
          const uint32_t sK = sK0 + sk * C::kTileBytes;
          mbar_arrive_expect_tx(bar(C::kKFull + sk), C::kTileBytes);
          for (int h = 0; h < C::kChunks; ++h)
            tma_load_3d(sK + h * C::kChunkBytes, &tm_k, bar(C::kKFull + sk), 64 * h, k0, f.bhk);
          last_k[sk] = g;
        }
      }
      // Never leave a copy in flight: wait for the last fill of every buffer.
      for (int b = 0; b < 2; ++b)
        if (last_q[b] >= 0) drain_wait(bar(C::kQFull + b), (last_q[b] >> 1) & 1, a.err);
      for (int s = 0; s < C::kKStages; ++s)
        if (last_k[s] >= 0) drain_wait(bar(C::kKFull + s), (last_k[s] / C::kKStages) & 1, a.err);
    }
  } else if (warp == 11) {
    // ------------------------------------------------------------------ TMA producer (V ring)
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      int last_v[C::kVStages];
      for (int s = 0; s < C::kVStages; ++s) last_v[s] = -1;
      int g = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < a.ntiles; t += tile_step) {
        const FwdTile f = fwd_tile(t, a, sp);
        for (int j = 0; j < f.nkv; ++j, ++g) {
          const int sv = g % C::kVStages, nv = g / C::kVStages;
          if (g >= C::kVStages &&
              !(ok = mbar_wait(bar(C::kVEmpty + sv), (nv - 1) & 1, &abort_flag, a.err)))
            break;
          const uint32_t sV = sV0 + sv * C::kTileBytes;
          mbar_arrive_expect_tx(bar(C::kVFull + sv), C::kTileBytes);
          for (int h = 0; h < C::kChunks; ++h)
            tma_load_3d(sV + h * C::kChunkBytes, &tm_v, bar(C::kVFull + sv), 64 * h,
                        (f.kb_lo + j) * kBlockN, f.bhk);
          last_v[sv] = g;
        }
      }
      for (int s = 0; s < C::kVStages; ++s)
        if (last_v[s] >= 0) drain_wait(bar(C::kVFull + s), (last_v[s] / C::kVStages) & 1, a.err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdO = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockM, D, false, true);
    // S_gg = Q K_gg^T into buffer gg mod kSBufs.  The buffer last held P_{gg-kSBufs}, which the P V
    // of that block, issued before this, reads: tcgen05.mma operations of one thread run in issue
    // order.
    auto issue_s = [&](int gg, uint32_t sQ) -> bool {
      const int s = gg % C::kKStages, n = gg / C::kKStages, sb = gg % C::kSBufs;
      if (!warp_wait(bar(C::kKFull + s), n & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      umma_ss_kmajor_d<D>(tmem + C::kColS + 128u * sb, smem_desc_sw128(sQ, 16, 1024),
                          smem_desc_sw128(sK0 + s * C::kTileBytes, 16, 1024), kIdS, 0u);
      umma_commit_w(bar(C::kSFull + sb));
      umma_commit_w(bar(C::kKEmpty + s));
      return true;
    };
    // O += P_gg V_gg.  P over S: keys 16 ks .. 16 ks + 15 at packed column 8 ks + 32 (ks / 4) of
    // buffer gg mod kSBufs (each half-row's P over the first 32 of its 64 columns); else at column
    // 8 ks of P buffer gg & 1.
    auto issue_pv = [&](int gg, bool first) -> bool {
      const int s = gg % C::kVStages, n = gg / C::kVStages, pb = gg % C::kSBufs;
      if (!warp_wait(bar(C::kPFull + pb), (gg / C::kSBufs) & 1, &abort_flag, a.err)) return false;
      if (!warp_wait(bar(C::kVFull + s), n & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      const uint64_t vdesc = smem_desc_sw128(sV0 + s * C::kTileBytes, C::kChunkBytes, 1024);
      if constexpr (C::kPOverS)
        umma_ts_mnmajor_x8_split(tmem + C::kColO, tmem + C::kColS + 128u * pb, vdesc, kIdO,
                                 first ? 0u : 1u);
      else
        umma_ts_mnmajor_x8(tmem + C::kColO, tmem + C::kColP + 64u * pb, vdesc, kIdO,
                           first ? 0u : 1u);
      umma_commit_w(bar(C::kPVDone + pb));
      umma_commit_w(bar(C::kVEmpty + s));
      return true;
    };
    // The S products run up to kSBufs blocks ahead of the P V products over the CTA's whole walk
    // (across tiles): S of block gg + kSBufs is issued right after P_gg V_gg, so the softmax warps do
    // not wait for scores, and no extra barrier is needed.  S of a tile may be issued only once
    // every P V of the tile two before it has been: its Q buffer is that tile's output staging
    // area, refilled after the store.
    int s_t = static_cast<int>(blockIdx.x), s_it = 0, s_j = 0, s_g = 0;
    FwdTile s_f = fwd_tile(s_t < a.ntiles ? s_t : 0, a, sp);
    auto issue_next_s = [&]() -> bool {
      if (s_t >= a.ntiles) return true;
      if (s_j == 0 &&
          !warp_wait(bar(C::kQFull + (s_it & 1)), (s_it >> 1) & 1, &abort_flag, a.err))
        return false;
      if (!issue_s(s_g, sQ0 + (s_it & 1) * C::kTileBytes)) return false;
      ++s_g;
      if (++s_j == s_f.nkv) {
        s_j = 0;
        s_t += tile_step;
        ++s_it;
        if (s_t < a.ntiles) s_f = fwd_tile(s_t, a, sp);
      }
      return true;
    };
    // Issues S up to (excluding) block s_limit, for tiles below tiles_done + 2.
    auto fill_s = [&](int s_limit, int tiles_done) -> bool {
      while (s_t < a.ntiles && s_g < s_limit && s_it < tiles_done + 2)
        if (!issue_next_s()) return false;
      return true;
    };
    bool ok = fill_s(C::kSBufs, 0);
    int g = 0;  // key blocks whose P V has been issued
    for (int t = blockIdx.x, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const FwdTile f = fwd_tile(t, a, sp);
      for (int j = 0; ok && j < f.nkv; ++j) {
        // The first P V of a tile overwrites O: the previous tile's epilogue must have read it.
        if (j == 0 && it > 0) ok = warp_wait(bar(C::kOEmpty), (it - 1) & 1, &abort_flag, a.err);
        if (ok) ok = issue_pv(g + j, j == 0);
        if (ok) ok = fill_s(g + j + 1 + C::kSBufs, it + (j + 1 == f.nkv ? 1 : 0));
      }
      g += f.nkv;
    }
    // Every issued MMA completes before TMEM is released.
    umma_commit_w(bar(C::kDrain));
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else if (warp == 10) {
    // ------------------------------------------------------------------ output stores
    for (int t = blockIdx.x, it = 0; t < a.ntiles; t += tile_step, ++it) {
      const FwdTile f = fwd_tile(t, a, sp);
      const int b = it & 1;
      if (!warp_wait(bar(C::kOutFull + b), (it >> 1) & 1, &abort_flag, a.err)) break;
      if (lane == 0) {
        const uint32_t sQ = sQ0 + b * C::kTileBytes;
        for (int h = 0; h < C::kChunks; ++h)
          tma_store_3d(&tm_o, sQ + h * C::kChunkBytes, 64 * h, f.q0, f.bh);
        bulk_commit_group();
        bulk_wait_group_read0();  // the Q buffer may be refilled once the store has read it
        mbar_arrive(bar(C::kQEmpty + b));
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-7)
    const int r = static_cast<int>(threadIdx.x & 127);  // row within the tile == TMEM lane
    const uint32_t h = warp >> 2;                          // column half of every tile
    const uint32_t quarter = warp & 3u;
    const uint32_t lane_base = (quarter * 32u) << 16;
    const float sl2 = a.scale_log2;
    int xn = 0;  // exchanges done so far
    // Swap a per-row value with the thread that owns the other half of the row.  Slot `xn & 1`
    // was last used two exchanges ago, and the partner arrived at the exchange in between only
    // after reading it.
    auto exchange = [&](float v, float* other) -> bool {
      float* red = s_red + (xn & 1) * 2 * kBlockM;
      red[h * kBlockM + r] = v;
      __syncwarp();
      const uint32_t xb = bar(C::kXch + quarter * 2 + (xn & 1));
      if (lane == 0) mbar_arrive(xb);
      if (!warp_wait(xb, (xn >> 1) & 1, &abort_flag, a.err)) return false;
      *other = red[(h ^ 1u) * kBlockM + r];
      ++xn;
      return true;
    };
    int g = 0;  // key blocks consumed so far by this CTA
    bool ok = true;
    for (int t = blockIdx.x, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const FwdTile f = fwd_tile(t, a, sp);
      const int q0 = f.q0;
      const int row = q0 + r;
      float m_ref = SWA_NEG_INF;  // reference max (log2 domain) that P and l are taken against
      float l = 0.f;              // partial row sum over this thread's half of the columns
      for (int j = 0; j < f.nkv; ++j) {
        const int gg = g + j;
        const int k0 = (f.kb_lo + j) * kBlockN;
        const int sb = gg % C::kSBufs;
        if (!(ok = warp_wait(bar(C::kSFull + sb), (gg / C::kSBufs) & 1, &abort_flag, a.err))) break;
        tc_fence_after();
        float x[64];  // raw scores S (the scale is applied inside the exponent below)
        {
          uint32_t rr[2][32];
          tmem_ld32(tmem + lane_base + C::kColS + 128u * sb + 64u * h, rr[0]);
          tmem_ld32(tmem + lane_base + C::kColS + 128u * sb + 64u * h + 32u, rr[1]);
          tmem_wait_ld_all();
          reg_fence(rr[0]);
          reg_fence(rr[1]);
#pragma unroll
          for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(rr[i >> 5][i & 31]);
        }
        // Window mask (the tile is not wholly visible): keep the cells row `row` sees.
        if (!sp.interior(q0, k0)) {
          // Columns c (keys k0 + 64h + c) visible to row `row`, and inside the key sequence.
          const int rel = row + sp.off - k0 - 64 * static_cast<int>(h);
          const int lo = rel - sp.dmax;
          const int hi = min(rel - sp.dmin, sp.Lk - 1 - k0 - 64 * static_cast<int>(h));
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = (c >= lo && c <= hi) ? x[c] : SWA_NEG_INF;
        }
        // p = 2^(scale log2(e) S - m) for this half, two scores per step: one packed FFMA, two
        // MUFU.EX2, one packed FADD into the row sum and one bf16 pack.  Returns the half's sum.
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
        // Fast path: one pass against the reference max, taken when every row of the warp has a
        // reference.  It stands unless some row's block sum exceeds 2^12; a sum within that bound
        // keeps every P of the block <= 2^12, so the result is the exact softmax either way.  The
        // two halves of a row swap their partial sums, so both take the same decision.
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
          // Exact path (a tile's first block, or a large rise of the max): the row max first
          // (a tree of eight chains per half, then swapped between the halves), then the
          // exponentials against it.
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = x[i];
#pragma unroll
          for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], x[c]);
          float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                           fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
          float mx_other;
          if (!(ok = exchange(mx, &mx_other))) break;
          mx = fmaxf(mx, mx_other);
          // Both halves of a row see the same maxima, so they take the same decisions below.
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

        // A P buffer of its own was last read by the P V of block gg - 2.
        if constexpr (!C::kPOverS) {
          if (gg >= 2 &&
              !(ok = warp_wait(bar(C::kPVDone + sb), ((gg - 2) >> 1) & 1, &abort_flag, a.err)))
            break;
        }
        // Rescaling O needs this tile's P V of block gg - 1 (and so every earlier one) to have
        // landed; a tile's first block needs none (its P V overwrites O).
        if (j >= 1 && __any_sync(0xffffffffu, resc)) {
          if (!(ok = warp_wait(bar(C::kPVDone + (gg - 1) % C::kSBufs), ((gg - 1) / C::kSBufs) & 1,
                               &abort_flag, a.err)))
            break;
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            const uint32_t oc = tmem + lane_base + C::kColO + (D / 2) * h + c0;
            uint32_t rr[32];
            tmem_ld32(oc, rr);
            tmem_wait_ld(rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * factor);
            tmem_st32(oc, rr);
          }
        } else {
          tc_fence_after();
        }
        // keys [64h, 64h+64) -> packed P over the first 32 of the 64 S columns this thread read, or
        // columns [32h, 32h+32) of P buffer gg & 1
        if constexpr (C::kPOverS)
          tmem_st32(tmem + lane_base + C::kColS + 128u * sb + 64u * h, pk);
        else
          tmem_st32(tmem + lane_base + C::kColP + 64u * sb + 32u * h, pk);
        tmem_wait_st();
        warp_arrive(bar(C::kPFull + sb));
      }
      if (!ok) break;
      g += f.nkv;

      // ---------------------------------------------------------------- tile epilogue
      float l_other = 0.f;
      if (!(ok = exchange(l, &l_other))) break;
      const int last = g - 1;
      if (!(ok = warp_wait(bar(C::kPVDone + last % C::kSBufs), (last / C::kSBufs) & 1, &abort_flag,
                           a.err)))
        break;
      tc_fence_after();
      constexpr int kHalf = D / 2;
      uint32_t rr[kHalf / 32][32];
#pragma unroll
      for (int c4 = 0; c4 < kHalf / 32; ++c4)
        tmem_ld32(tmem + lane_base + C::kColO + kHalf * h + 32u * c4, rr[c4]);
      tmem_wait_ld_all();
#pragma unroll
      for (int c4 = 0; c4 < kHalf / 32; ++c4) reg_fence(rr[c4]);
      warp_arrive(bar(C::kOEmpty));  // the next tile's first P V may overwrite O now

      const float l_row = l + l_other;
      const float inv_l = 1.f / l_row;
      const float m_use = (m_ref == SWA_NEG_INF) ? 0.f : m_ref;
      if (row < sp.Lq && h == 0)
        a.lse[static_cast<size_t>(f.bh) * sp.Lq + row] = (m_use + log2f(l_row)) * kLn2;
      // O / l -> bf16, staged in this tile's Q buffer (free: every S MMA of the tile has
      // completed) in the swizzled layout of the TMA map; warp 10 stores it.
      const uint32_t sQ = sQ0 + (it & 1) * C::kTileBytes;
#pragma unroll
      for (int c4 = 0; c4 < kHalf / 32; ++c4) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = Elem<F16>::pack(__uint_as_float(rr[c4][2 * i]) * inv_l,
                              __uint_as_float(rr[c4][2 * i + 1]) * inv_l);
        stage_row32_sw128(sQ, r, kHalf * h + 32u * c4, pk);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kOutFull + (it & 1)));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool F16>
cudaError_t launch_fwd_d(const Problem& pb, const void* q, const void* k, const void* v, void* o,
                         float* lse, cudaStream_t stream) {
  using C = FwdCfg<D>;
  CUtensorMap tq, tk, tv, to;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_3d(&tq, q, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&to, o, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tk, k, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tv, v, bhk, pb.span.Lk, D, kBlockN, F16))
    return cudaErrorInvalidValue;
  auto kern = swa_fwd_kernel<D, F16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  FwdArgs a;
  a.lse = lse;
  a.BH = pb.B * pb.Hq;
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.G = pb.Hq / pb.Hkv;
  a.span = pb.span;
  a.nqb = (pb.span.Lq + kBlockM - 1) / kBlockM;
  a.ntiles = a.nqb * a.BH;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  a.divBH = FastDiv(static_cast<uint32_t>(a.BH));
  a.divHq = FastDiv(static_cast<uint32_t>(a.Hq));
  a.divG = FastDiv(static_cast<uint32_t>(a.G));
  const int grid = a.ntiles < sm_count() ? a.ntiles : sm_count();
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Problem& pb, const void* q, const void* k, const void* v, void* o,
                       float* lse, cudaStream_t stream) {
  if (pb.D == 256) return launch_fwd_d256(pb, q, k, v, o, lse, stream);
  if (fwd_pair_applies(pb)) return launch_fwd_pair(pb, q, k, v, o, lse, stream);
  if (pb.D == 64)
    return pb.f16 ? launch_fwd_d<64, true>(pb, q, k, v, o, lse, stream)
                  : launch_fwd_d<64, false>(pb, q, k, v, o, lse, stream);
  if (pb.D == 128)
    return pb.f16 ? launch_fwd_d<128, true>(pb, q, k, v, o, lse, stream)
                  : launch_fwd_d<128, false>(pb, q, k, v, o, lse, stream);
  return cudaErrorInvalidValue;
}

}  // namespace swa
