// swa_fwd_pair.cu — forward of causal sliding-window attention on CTA pairs (sm_103a).
//
// The same computation as swa_fwd.cu (O = softmax(scale Q K^T, window mask) V and the natural-log
// LSE per query row, over only the key blocks kb_lo..kb_hi the window reaches: "Off NVIDIA, you fix
// the platform yourself", Lab 28, "What did fixing it take?"), for D = 128 and an even number G of
// query heads per kv head.  The two CTAs of a cluster run on one TPC and take the two query heads
// 2p and 2p + 1 of one kv group at the same query block, so they need the same K and V blocks and
// walk the same window.  Rank 0 issues every MMA for both SMs as tcgen05.mma.cta_group::2 with
// M = 256 (each SM computes its own 128 query rows into its own TMEM):
//   S = Q K^T     B = K block: rank r holds keys [64 r, 64 r + 64) (K-major, 16 KB),
//   O += P V      B = V block: rank r holds head dims [64 r, 64 r + 64) (MN-major, 16 KB),
// so each SM loads and reads half of every key block, and one MMA instruction feeds both tensor
// cores.  Q, P, O, the softmax and the epilogue stay per CTA, as in swa_fwd.cu.
//
// Warp roles (384 threads per CTA):
//   warps 0-7  softmax of this CTA's rows: warp w owns 16 whole rows (TMEM lanes 32 (w % 4) +
//              16 (w / 4) ..), read with the 16x256b TMEM shape, so that each row lies in four
//              threads of one warp; the P and O-read handshakes arrive on rank 0's barriers (16
//              arrivals: both CTAs' softmax warps).
//   warp 8     TMA producer of this CTA's Q and K halves; warp 11 of its V halves.
//   warp 9     rank 0: MMA issuer for the pair; commits arrive on the barriers of both CTAs.
//              rank 1: relay — waits for each of its own Q / K / V copies, in the order rank 0
//              consumes them, and arrives on rank 0's matching barrier (rank 0's full barriers
//              count its own copy and rank 1's relay).
//   warp 10    output: TMA store of this CTA's O tile.
// TMEM (each CTA, allocated for the pair): three 128-column S buffers at [0,384) — buffer b holds
// S_g for the blocks g = b mod 3, then P_g over its first 64 columns (16-bit pairs: keys 2c and
// 2c + 1 in column c) — and O at [384,512).  With three buffers and the deep K ring that half-tiles leave room
// for, the S products run up to three blocks ahead of the P V products.
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

// The running-max policy of the single-CTA forward (exact softmax either way).
constexpr float kRescaleThreshold = 8.0f;
constexpr float kFastSumLimit = 4096.0f;

template <int D>
struct FwdPairCfg {
  static_assert(D == 128, "pair forward: D = 128 (one 64-column V chunk per CTA)");
  static constexpr int kTileBytes = kBlockM * D * 2;        // this CTA's Q tile
  static constexpr int kChunkBytes = kBlockM * 128;         // 128 rows x 64 columns
  static constexpr int kChunks = D / 64;
  static constexpr int kKHalfRows = kBlockN / 2;
  static constexpr int kKChunkBytes = kKHalfRows * 128;     // 64 rows x 64 columns
  static constexpr int kKHalfBytes = kKHalfRows * D * 2;    // 64 keys x D
  static constexpr int kVHalfBytes = kBlockN * 128;         // 128 keys x 64 head dims
  static constexpr int kKStages = 5;
  static constexpr int kVStages = 4;
  static constexpr int kOffQ = 0;  // 2 buffers
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kKHalfBytes;
  static constexpr int kOffBar = kOffV + kVStages * kVHalfBytes;
  static constexpr int kQFull = 0;   // 2
  static constexpr int kQEmpty = 2;  // 2
  static constexpr int kKFull = 4;
  static constexpr int kKEmpty = kKFull + kKStages;
  static constexpr int kVFull = kKEmpty + kKStages;
  static constexpr int kVEmpty = kVFull + kVStages;
  static constexpr int kSBufs = 3;
  static constexpr int kSFull = kVEmpty + kVStages;  // kSBufs
  static constexpr int kPFull = kSFull + kSBufs;     // kSBufs (rank 0's: both CTAs' softmax warps)
  static constexpr int kPVDone = kPFull + kSBufs;    // kSBufs
  static constexpr int kOEmpty = kPVDone + kSBufs;   // rank 0's: both CTAs have read O
  static constexpr int kOutFull = kOEmpty + 1;       // 2
  static constexpr int kDrain = kOutFull + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;  // + TMEM address and abort flag
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;  // buffer b at kColS + 128 b
  static constexpr uint32_t kColO = 128 * kSBufs;
  static constexpr int kThreads = 384;
  static constexpr int kComputeThreads = 256;
  static constexpr uint32_t kPairWarps = 2 * kComputeThreads / 32;  // arrivals on rank 0's barriers
};

struct FwdPairArgs {
  float* lse;
  int BHKP;  // B * Hkv * G / 2: head pairs per query block
  int Hq, Hkv, G, nqb, ntiles;
  Span span;
  float scale_log2;
  unsigned* err;
  FastDiv divBHKP, divGP, divHkv;  // tile index decomposition (divGP: G / 2)
};

struct PairTile {
  int bh, bhk, q0, kb_lo, nkv;
};

// Pair tile t (heaviest query blocks first); rank r takes query head 2 p + r of the kv group.
__device__ __forceinline__ PairTile fwd_pair_tile(int t, const FwdPairArgs& a, const Span sp,
                                                  uint32_t rank) {
  PairTile f;
  const uint32_t tq = a.divBHKP.div(static_cast<uint32_t>(t));
  const int qb = a.nqb - 1 - static_cast<int>(tq);
  const uint32_t rem = static_cast<uint32_t>(t) - tq * static_cast<uint32_t>(a.BHKP);
  f.bhk = static_cast<int>(a.divGP.div(rem));
  const int gp = static_cast<int>(rem) - f.bhk * (a.G / 2);
  const int b = static_cast<int>(a.divHkv.div(static_cast<uint32_t>(f.bhk)));
  const int hk = f.bhk - b * a.Hkv;
  f.bh = b * a.Hq + hk * a.G + 2 * gp + static_cast<int>(rank);
  f.q0 = qb * kBlockM;
  f.kb_lo = sp.first_kblock(f.q0);
  f.nkv = sp.last_kblock(f.q0) - f.kb_lo + 1;
  return f;
}

template <int D, bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    swa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, const FwdPairArgs a) {
  using C = FwdPairCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  // Both CTAs of the pair always reach the cluster barriers and the collective TMEM allocation;
  // a misaligned window only disables the work (and is reported).
  const bool smem_ok = (smem_u32(smem) & 1023u) == 0u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);  // raised by a failed wait
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ0 = smem_u32(smem + C::kOffQ);
  const uint32_t sK0 = smem_u32(smem + C::kOffK);
  const uint32_t sV0 = smem_u32(smem + C::kOffV);
  const uint32_t rank = cluster_rank();
  const bool lead = rank == 0u;
  const int tile0 = static_cast<int>(blockIdx.x >> 1);
  const int tile_step = static_cast<int>(gridDim.x >> 1);
  const Span sp = a.span;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = smem_ok ? 0 : 1;
    if (!smem_ok) atomicOr(a.err, kErrSmemLayout);
    const uint32_t full_count = lead ? 2u : 1u;  // rank 0: own copy + rank 1's relay
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kQFull + b), full_count);
      mbar_init(bar(C::kQEmpty + b), 1);
      mbar_init(bar(C::kOutFull + b), C::kComputeThreads / 32);
    }
    for (int b = 0; b < C::kSBufs; ++b) {
      mbar_init(bar(C::kSFull + b), 1);
      mbar_init(bar(C::kPFull + b), C::kPairWarps);
      mbar_init(bar(C::kPVDone + b), 1);
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar(C::kKFull + s), full_count);
      mbar_init(bar(C::kKEmpty + s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar(C::kVFull + s), full_count);
      mbar_init(bar(C::kVEmpty + s), 1);
    }
    mbar_init(bar(C::kOEmpty), C::kPairWarps);
    mbar_init(bar(C::kDrain), 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The pair's MMA schedule, run by rank 0's MMA warp (issuing) and rank 1's relay warp
  // (forwarding its copies, in the same order): S for up to kSBufs key blocks ahead of P V over the
  // whole walk, across tiles, but never for a tile whose Q buffer is still the output staging area
  // of a tile with P V outstanding (S of tile i waits until every P V of tile i - 2 is issued).
  // on_s(g, tile index, first block of its tile) and on_pv(g, tile index, block within the tile).
  auto walk = [&](auto&& on_s, auto&& on_pv) -> bool {
    int s_t = tile0, s_it = 0, s_j = 0, s_g = 0;
    PairTile s_f = fwd_pair_tile(s_t < a.ntiles ? s_t : 0, a, sp, rank);
    auto fill_s = [&](int s_limit, int tiles_done) -> bool {
      while (s_t < a.ntiles && s_g < s_limit && s_it < tiles_done + 2) {
        if (!on_s(s_g, s_it, s_j == 0)) return false;
        ++s_g;
        if (++s_j == s_f.nkv) {
          s_j = 0;
          s_t += tile_step;
          ++s_it;
          if (s_t < a.ntiles) s_f = fwd_pair_tile(s_t, a, sp, rank);
        }
      }
      return true;
    };
    bool ok = fill_s(C::kSBufs, 0);
    int g = 0;
    for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const PairTile f = fwd_pair_tile(t, a, sp, rank);
      for (int j = 0; ok && j < f.nkv; ++j) {
        ok = on_pv(g + j, it, j);
        if (ok) ok = fill_s(g + j + 1 + C::kSBufs, it + (j + 1 == f.nkv ? 1 : 0));
      }
      g += f.nkv;
    }
    return ok;
  };

  if (!smem_ok) {
    // nothing to do: fall through to the final barrier and the collective release
  } else if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer (Q, K half)
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      int last_q[2] = {-1, -1};
      int last_k[C::kKStages];
      for (int s = 0; s < C::kKStages; ++s) last_k[s] = -1;
      int g = 0;
      bool ok = true;
      for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
        const PairTile f = fwd_pair_tile(t, a, sp, rank);
        const int qbuf = it & 1;
        if (it >= 2 && !mbar_wait(bar(C::kQEmpty + qbuf), ((it - 2) >> 1) & 1, &abort_flag, a.err))
          break;
        const uint32_t sQ = sQ0 + qbuf * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kQFull + qbuf), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(sQ + h * C::kChunkBytes, &tm_q, bar(C::kQFull + qbuf), 64 * h, f.q0, f.bh);
        last_q[qbuf] = it;
        for (int j = 0; j < f.nkv; ++j, ++g) {
          const int k0 = (f.kb_lo + j) * kBlockN + C::kKHalfRows * static_cast<int>(rank);
          const int sk = g % C::kKStages, nk = g / C::kKStages;
          if (g >= C::kKStages &&
              !(ok = mbar_wait(bar(C::kKEmpty + sk), (nk - 1) & 1, &abort_flag, a.err)))
            break;
          const uint32_t sK = sK0 + sk * C::kKHalfBytes;
          mbar_arrive_expect_tx(bar(C::kKFull + sk), C::kKHalfBytes);
          for (int h = 0; h < C::kChunks; ++h)
            tma_load_3d(sK + h * C::kKChunkBytes, &tm_k, bar(C::kKFull + sk), 64 * h, k0, f.bhk);
          last_k[sk] = g;
        }
      }
      for (int b = 0; b < 2; ++b)
        if (last_q[b] >= 0) drain_wait(bar(C::kQFull + b), (last_q[b] >> 1) & 1, a.err);
      for (int s = 0; s < C::kKStages; ++s)
        if (last_k[s] >= 0) drain_wait(bar(C::kKFull + s), (last_k[s] / C::kKStages) & 1, a.err);
    }
  } else if (warp == 11) {
    // ------------------------------------------------------------------ TMA producer (V half)
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      int last_v[C::kVStages];
      for (int s = 0; s < C::kVStages; ++s) last_v[s] = -1;
      int g = 0;
      bool ok = true;
      for (int t = tile0; ok && t < a.ntiles; t += tile_step) {
        const PairTile f = fwd_pair_tile(t, a, sp, rank);
        for (int j = 0; j < f.nkv; ++j, ++g) {
          const int sv = g % C::kVStages, nv = g / C::kVStages;
          if (g >= C::kVStages &&
              !(ok = mbar_wait(bar(C::kVEmpty + sv), (nv - 1) & 1, &abort_flag, a.err)))
            break;
          const uint32_t sV = sV0 + sv * C::kVHalfBytes;
          mbar_arrive_expect_tx(bar(C::kVFull + sv), C::kVHalfBytes);
          tma_load_3d(sV, &tm_v, bar(C::kVFull + sv), 64 * static_cast<int>(rank),
                      (f.kb_lo + j) * kBlockN, f.bhk);
          last_v[sv] = g;
        }
      }
      for (int s = 0; s < C::kVStages; ++s)
        if (last_v[s] >= 0) drain_wait(bar(C::kVFull + s), (last_v[s] / C::kVStages) & 1, a.err);
    }
  } else if (warp == 9 && lead) {
    // ------------------------------------------------------------------ MMA issuer (the pair)
    constexpr uint32_t kIdS = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdO = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockM, D, false, true);
    // S_gg = Q K_gg^T into buffer gg mod 3, which last held P_{gg-3}: the P V of block gg - 3 was
    // issued before this, and tcgen05.mma operations of one thread run in issue order.
    auto on_s = [&](int gg, int qit, bool first_of_tile) -> bool {
      const int s = gg % C::kKStages, n = gg / C::kKStages, sb = gg % C::kSBufs;
      if (first_of_tile &&
          !warp_wait_cluster(bar(C::kQFull + (qit & 1)), (qit >> 1) & 1, &abort_flag, a.err))
        return false;
      if (!warp_wait_cluster(bar(C::kKFull + s), n & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ss_kmajor_d<D>(tmem + C::kColS + 128u * sb,
                           smem_desc_sw128(sQ0 + (qit & 1) * C::kTileBytes, 16, 1024),
                           smem_desc_sw128(sK0 + s * C::kKHalfBytes, 16, 1024), kIdS, 0u);
      umma2_commit_w(bar(C::kSFull + sb));
      umma2_commit_w(bar(C::kKEmpty + s));
      return true;
    };
    // O += P_gg V_gg with P_gg in buffer gg mod 3 (keys 16 ks .. 16 ks + 15 at packed columns
    // 8 ks .. 8 ks + 7); a tile's first P V overwrites O once both CTAs' epilogues have read it.
    auto on_pv = [&](int gg, int it, int j) -> bool {
      const int s = gg % C::kVStages, n = gg / C::kVStages, pb = gg % C::kSBufs;
      if (j == 0 && it > 0 &&
          !warp_wait_cluster(bar(C::kOEmpty), (it - 1) & 1, &abort_flag, a.err))
        return false;
      if (!warp_wait_cluster(bar(C::kPFull + pb), (gg / C::kSBufs) & 1, &abort_flag, a.err))
        return false;
      if (!warp_wait_cluster(bar(C::kVFull + s), n & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ts_mnmajor_x8(tmem + C::kColO, tmem + C::kColS + 128u * pb,
                                smem_desc_sw128(sV0 + s * C::kVHalfBytes, C::kVHalfBytes, 1024),
                                kIdO, j == 0 ? 0u : 1u);
      umma2_commit_w(bar(C::kPVDone + pb));
      umma2_commit_w(bar(C::kVEmpty + s));
      return true;
    };
    walk(on_s, on_pv);
    umma2_commit_w(bar(C::kDrain));
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else if (warp == 9) {
    // ------------------------------------------------------------------ relay (rank 1)
    // Forwards each of this CTA's copies in the order rank 0's MMA warp consumes them.
    auto relay = [&](int idx, uint32_t parity) -> bool {
      if (!warp_wait(bar(idx), parity, &abort_flag, a.err)) return false;
      if (lane == 0) mbar_arrive_cluster(mapa_rank0(bar(idx)));
      __syncwarp();
      return true;
    };
    auto on_s = [&](int gg, int qit, bool first_of_tile) -> bool {
      if (first_of_tile && !relay(C::kQFull + (qit & 1), (qit >> 1) & 1)) return false;
      return relay(C::kKFull + gg % C::kKStages, (gg / C::kKStages) & 1);
    };
    auto on_pv = [&](int gg, int, int) -> bool {
      return relay(C::kVFull + gg % C::kVStages, (gg / C::kVStages) & 1);
    };
    walk(on_s, on_pv);
  } else if (warp == 10) {
    // ------------------------------------------------------------------ output stores
    for (int t = tile0, it = 0; t < a.ntiles; t += tile_step, ++it) {
      const PairTile f = fwd_pair_tile(t, a, sp, rank);
      const int b = it & 1;
      if (!warp_wait(bar(C::kOutFull + b), (it >> 1) & 1, &abort_flag, a.err)) break;
      if (lane == 0) {
        const uint32_t sQ = sQ0 + b * C::kTileBytes;
        for (int h = 0; h < C::kChunks; ++h)
          tma_store_3d(&tm_o, sQ + h * C::kChunkBytes, 64 * h, f.q0, f.bh);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(bar(C::kQEmpty + b));
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-7)
    // Thread t of warp w holds rows R0 = 32 (w % 4) + 16 (w / 4) + t / 4 and R1 = R0 + 8 of the
    // tile, and of every group j (0..15) of 8 columns the columns 8j + 2kq, 8j + 2kq + 1 (kq =
    // t % 4): x[4j], x[4j+1] of R0 and x[4j+2], x[4j+3] of R1.  Row maxima and sums combine the four
    // threads kq = 0..3 with two shuffles; P goes back as packed pairs, column 4j + kq of each row,
    // which is the 16x128b store layout.
    const uint32_t lane0 = 32u * (warp & 3u) + 16u * (warp >> 2);
    const uint32_t lane_base = lane0 << 16;
    const int r0 = static_cast<int>(lane0 + (lane >> 2));  // R0 (R1 = R0 + 8)
    const int kq = static_cast<int>(lane & 3u);
    const float sl2 = a.scale_log2;
    auto row_max = [](float v) {
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
      return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
    };
    auto row_sum = [](float v) {
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      return v + __shfl_xor_sync(0xffffffffu, v, 2);
    };
    int g = 0;
    bool ok = true;
    for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const PairTile f = fwd_pair_tile(t, a, sp, rank);
      const int q0 = f.q0;
      const int row0 = q0 + r0, row1 = row0 + 8;
      float m0 = SWA_NEG_INF, m1 = SWA_NEG_INF;  // reference max (log2 domain) of rows R0, R1
      float l0 = 0.f, l1 = 0.f;                  // partial sums over this thread's columns
      for (int j = 0; j < f.nkv; ++j) {
        const int gg = g + j;
        const int k0 = (f.kb_lo + j) * kBlockN;
        const int sb = gg % C::kSBufs;
        if (!(ok = warp_wait(bar(C::kSFull + sb), (gg / C::kSBufs) & 1, &abort_flag, a.err))) break;
        tc_fence_after();
        const uint32_t s_addr = tmem + lane_base + C::kColS + 128u * sb;
        float x[64];
        {
          uint32_t rr[2][32];
          tmem_ld16x256_x8(s_addr, rr[0]);
          tmem_ld16x256_x8(s_addr + 64u, rr[1]);
          tmem_wait_ld_all();
          reg_fence(rr[0]);
          reg_fence(rr[1]);
#pragma unroll
          for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(rr[i >> 5][i & 31]);
        }
        if (!sp.interior(q0, k0)) {
          // column 8 (i / 4) + 2 kq + (i & 1) of row R0 (i % 4 < 2) or R1, visible to that row and
          // inside the key sequence
          const int rel0 = row0 + sp.off - k0 - 2 * kq, rel1 = rel0 + 8;
          const int lo0 = rel0 - sp.dmax, hi0 = min(rel0 - sp.dmin, sp.Lk - 1 - k0 - 2 * kq);
          const int lo1 = rel1 - sp.dmax, hi1 = min(rel1 - sp.dmin, sp.Lk - 1 - k0 - 2 * kq);
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const int c = 8 * (i >> 2) + (i & 1);
            const bool vis = (i & 2) ? (c >= lo1 && c <= hi1) : (c >= lo0 && c <= hi0);
            x[i] = vis ? x[i] : SWA_NEG_INF;
          }
        }
        uint32_t pk[32];  // pk[2j] row R0, pk[2j+1] row R1: packed column 4j + kq
        float b0 = 0.f, b1 = 0.f;
        auto exponentiate = [&](float mu0, float mu1) {
          const float2 scale2 = make_float2(sl2, sl2);
          const float2 n0 = make_float2(-mu0, -mu0), n1 = make_float2(-mu1, -mu1);
          float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
          float2 u0 = make_float2(0.f, 0.f), u1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const float2 t0 = __ffma2_rn(make_float2(x[4 * jj], x[4 * jj + 1]), scale2, n0);
            const float2 t1 = __ffma2_rn(make_float2(x[4 * jj + 2], x[4 * jj + 3]), scale2, n1);
            const float2 e0 = make_float2(ex2(t0.x), ex2(t0.y));
            const float2 e1 = make_float2(ex2(t1.x), ex2(t1.y));
            if (jj & 1) {
              u0 = __fadd2_rn(u0, e0);
              u1 = __fadd2_rn(u1, e1);
            } else {
              s0 = __fadd2_rn(s0, e0);
              s1 = __fadd2_rn(s1, e1);
            }
            pk[2 * jj] = Elem<F16>::pack(e0.x, e0.y);
            pk[2 * jj + 1] = Elem<F16>::pack(e1.x, e1.y);
          }
          b0 = (s0.x + s0.y) + (u0.x + u0.y);
          b1 = (s1.x + s1.y) + (u1.x + u1.y);
        };
        // One pass against the running reference max; redone exactly on a tile's first block or
        // when a row's block sum exceeds 2^12 (the four threads of a row decide alike).
        bool redo = true;
        if (__all_sync(0xffffffffu, m0 != SWA_NEG_INF && m1 != SWA_NEG_INF)) {
          exponentiate(m0, m1);
          redo = __any_sync(0xffffffffu,
                            !(row_sum(b0) <= kFastSumLimit) || !(row_sum(b1) <= kFastSumLimit));
        }
        bool resc = false;
        float f0 = 1.f, f1 = 1.f;  // rescale factors of rows R0, R1
        if (redo) {
          float a0 = x[0], a1 = x[2], c0 = x[1], c1 = x[3];
#pragma unroll
          for (int jj = 1; jj < 16; ++jj) {
            a0 = fmaxf(a0, x[4 * jj]);
            c0 = fmaxf(c0, x[4 * jj + 1]);
            a1 = fmaxf(a1, x[4 * jj + 2]);
            c1 = fmaxf(c1, x[4 * jj + 3]);
          }
          const float mx0 = row_max(fmaxf(a0, c0)) * sl2, mx1 = row_max(fmaxf(a1, c1)) * sl2;
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          if (mn0 > m0 + kRescaleThreshold) {
            f0 = ex2(m0 - mn0);  // 0 when m0 is -inf
            l0 *= f0;
            m0 = mn0;
            resc = true;
          }
          if (mn1 > m1 + kRescaleThreshold) {
            f1 = ex2(m1 - mn1);
            l1 *= f1;
            m1 = mn1;
            resc = true;
          }
          exponentiate((m0 == SWA_NEG_INF) ? 0.f : m0, (m1 == SWA_NEG_INF) ? 0.f : m1);
        }
        l0 += b0;
        l1 += b1;

        // Rescaling O needs this tile's P V of block gg - 1 to have landed.
        if (j >= 1 && __any_sync(0xffffffffu, resc)) {
          if (!(ok = warp_wait(bar(C::kPVDone + (gg - 1) % C::kSBufs), ((gg - 1) / C::kSBufs) & 1,
                               &abort_flag, a.err)))
            break;
          tc_fence_after();
#pragma unroll
          for (int hc = 0; hc < D / 64; ++hc) {
            const uint32_t oc = tmem + lane_base + C::kColO + 64u * hc;
            uint32_t rr[32];
            tmem_ld16x256_x8(oc, rr);
            tmem_wait_ld(rr);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              rr[i] = __float_as_uint(__uint_as_float(rr[i]) * ((i & 2) ? f1 : f0));
            tmem_st16x256_x8(oc, rr);
          }
        } else {
          tc_fence_after();
        }
        // packed P over the first 64 columns of the buffer (this warp's rows of S have been read)
        tmem_st16x128_x16(s_addr, pk);
        tmem_wait_st();
        warp_arrive_rank0(bar(C::kPFull + sb));
      }
      if (!ok) break;
      g += f.nkv;

      // ---------------------------------------------------------------- tile epilogue
      const float lr0 = row_sum(l0), lr1 = row_sum(l1);
      const int last = g - 1;
      if (!(ok = warp_wait(bar(C::kPVDone + last % C::kSBufs), (last / C::kSBufs) & 1, &abort_flag,
                           a.err)))
        break;
      tc_fence_after();
      uint32_t ro[D / 64][32];
#pragma unroll
      for (int hc = 0; hc < D / 64; ++hc) tmem_ld16x256_x8(tmem + lane_base + C::kColO + 64u * hc, ro[hc]);
      tmem_wait_ld_all();
#pragma unroll
      for (int hc = 0; hc < D / 64; ++hc) reg_fence(ro[hc]);
      warp_arrive_rank0(bar(C::kOEmpty));

      const float inv0 = 1.f / lr0, inv1 = 1.f / lr1;
      if (kq == 0) {
        const size_t base = static_cast<size_t>(f.bh) * sp.Lq;
        if (row0 < sp.Lq)
          a.lse[base + row0] = (((m0 == SWA_NEG_INF) ? 0.f : m0) + log2f(lr0)) * kLn2;
        if (row1 < sp.Lq)
          a.lse[base + row1] = (((m1 == SWA_NEG_INF) ? 0.f : m1) + log2f(lr1)) * kLn2;
      }
      // O / l -> 16-bit, staged in the Q buffer in the swizzled layout of the TMA map: group j of
      // 64-column chunk hc is 16-byte unit j of the row, this thread's pair its word kq.
      const uint32_t sQ = sQ0 + (it & 1) * C::kTileBytes;
#pragma unroll
      for (int hc = 0; hc < D / 64; ++hc) {
        const uint32_t chunk = sQ + hc * C::kChunkBytes + 4u * kq;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          st_shared_b32(chunk + sw128_offset(r0, jj),
                        Elem<F16>::pack(__uint_as_float(ro[hc][4 * jj]) * inv0,
                                        __uint_as_float(ro[hc][4 * jj + 1]) * inv0));
          st_shared_b32(chunk + sw128_offset(r0 + 8, jj),
                        Elem<F16>::pack(__uint_as_float(ro[hc][4 * jj + 2]) * inv1,
                                        __uint_as_float(ro[hc][4 * jj + 3]) * inv1));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kOutFull + (it & 1)));
    }
  }

  // Every cross-CTA arrival and every pair MMA (rank 0 waited for its drain) is complete once both
  // CTAs are here; then the pair releases its TMEM together.
  tc_fence_before();
  cluster_sync_all();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

template <int D, bool F16>
cudaError_t launch_fwd_pair_d(const Problem& pb, const void* q, const void* k, const void* v,
                              void* o, float* lse, cudaStream_t stream) {
  using C = FwdPairCfg<D>;
  CUtensorMap tq, tk, tv, to;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_3d(&tq, q, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&to, o, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tk, k, bhk, pb.span.Lk, D, C::kKHalfRows, F16) ||
      !make_tmap_3d(&tv, v, bhk, pb.span.Lk, D, kBlockN, F16))
    return cudaErrorInvalidValue;
  auto kern = swa_fwd_pair_kernel<D, F16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  FwdPairArgs a;
  a.lse = lse;
  a.G = pb.Hq / pb.Hkv;
  a.BHKP = pb.B * pb.Hkv * (a.G / 2);
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.span = pb.span;
  a.nqb = (pb.span.Lq + kBlockM - 1) / kBlockM;
  a.ntiles = a.nqb * a.BHKP;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  a.divBHKP = FastDiv(static_cast<uint32_t>(a.BHKP));
  a.divGP = FastDiv(static_cast<uint32_t>(a.G / 2));
  a.divHkv = FastDiv(static_cast<uint32_t>(a.Hkv));
  const int clusters = max_pair_clusters<swa_fwd_pair_kernel<D, F16>>(C::kThreads, C::kSmemBytes);
  const int nclusters = a.ntiles < clusters ? a.ntiles : clusters;
  kern<<<2 * nclusters, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

bool fwd_pair_applies(const Problem& pb) {
  const int G = pb.Hq / pb.Hkv;
  return pb.D == 128 && G % 2 == 0;
}

cudaError_t launch_fwd_pair(const Problem& pb, const void* q, const void* k, const void* v,
                            void* o, float* lse, cudaStream_t stream) {
  if (!fwd_pair_applies(pb)) return cudaErrorInvalidValue;
  return pb.f16 ? launch_fwd_pair_d<128, true>(pb, q, k, v, o, lse, stream)
                : launch_fwd_pair_d<128, false>(pb, q, k, v, o, lse, stream);
}

}  // namespace swa
