// swa_bwd_dq_pair.cu — dQ of causal sliding-window attention on CTA pairs (sm_103a).
//
// The same computation as swa_bwd_dq.cu — per key block of a query tile's window walk
//   S = Q K_j^T,  P = exp(scale S - LSE) (window-masked),  dP = dO V_j^T,  dS = P (dP - Delta),
//   dQ += dS K_j,  and a final dQ *= scale
// ("Off NVIDIA, you fix the platform yourself", Lab 28, "Method and disclosure": a query tile's dQ
// starts at the first key tile it visits) — for D = 128 and an even number of query heads per kv
// head.  The two CTAs of a cluster run on one TPC and take the query heads 2p and 2p + 1 of one kv
// group at the same query block, so they walk the same K and V blocks.  Rank 0 issues every MMA
// for both SMs as tcgen05.mma.cta_group::2 with M = 256 (each SM computes its own 128 query rows):
//   S  = Q K^T     B = keys [64 r, 64 r + 64) of the block, all head dims (K-major, 16 KB),
//   dP = dO V^T    B = the same key half of V (K-major, 16 KB),
//   dQ += dS K     B = head dims [64 r, 64 r + 64) of the block, all keys (MN-major, 16 KB),
// r = the CTA's rank.  A K stage holds both K pieces (32 KB, a quarter of the tile loaded twice),
// so each SM loads 48 KB per key block instead of 64, which leaves room for a fourth K stage: a K
// tile is held from S_j until dQ_j completes, and three stages could not cover the copy latency.
//
// Warp roles (352 threads per CTA): warps 0-7 compute (as swa_bwd_dq.cu; the S-read, dS-written
// and dQ-read handshakes arrive on rank 0's barriers, 16 arrivals from both CTAs);
// warp 8 TMA producer of this CTA's Q and dO (per tile) and K pieces; warp 10 of its V halves;
// warp 9 rank 0: MMA issuer for the pair (commits arrive on the barriers of both CTAs), rank 1:
// relay — waits for each of its own copies in the order rank 0 consumes them and arrives on rank
// 0's matching barrier.
// TMEM (each CTA, allocated for the pair): [0,128) S, [128,384) two dP buffers, [384,512) dQ.  dS_g
// (bf16 pairs) goes over the first 32 of each half-row's 64 columns of dP buffer g & 1, so dP of
// the next block is computed into the other buffer while the compute warps work on this one.
#include "swa_bwd_dq.cuh"
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

template <int D>
struct DqPairCfg {
  static_assert(D == 128, "pair dQ: D = 128");
  static constexpr int kTileBytes = kBlockM * D * 2;    // Q or dO tile of this CTA's head
  static constexpr int kChunkBytes = kBlockM * 128;     // 128 rows x 64 columns
  static constexpr int kChunks = D / 64;
  static constexpr int kHalfRows = kBlockN / 2;
  static constexpr int kHalfChunkBytes = kHalfRows * 128;  // 64 rows x 64 columns
  static constexpr int kHalfBytes = kHalfRows * D * 2;     // 64 keys x D (S / dP operand)
  static constexpr int kKColBytes = kBlockN * 128;         // 128 keys x 64 head dims (dQ operand)
  static constexpr int kKStageBytes = kHalfBytes + kKColBytes;
  static constexpr int kKStages = 4;
  static constexpr int kVStages = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffK = kOffDO + kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kKStageBytes;
  static constexpr int kOffBar = kOffV + kVStages * kHalfBytes;
  static constexpr int kQDFull = 0;
  static constexpr int kQDEmpty = 1;
  static constexpr int kKFull = 2;
  static constexpr int kKEmpty = kKFull + kKStages;
  static constexpr int kVFull = kKEmpty + kKStages;
  static constexpr int kVEmpty = kVFull + kVStages;
  static constexpr int kSFull = kVEmpty + kVStages;
  static constexpr int kSEmpty = kSFull + 1;    // rank 0's: both CTAs have read S
  static constexpr int kDPFull = kSEmpty + 1;   // 2 (one per dP buffer)
  static constexpr int kDSFull = kDPFull + 2;   // 2, rank 0's: both CTAs' dS written
  static constexpr int kDQDone = kDSFull + 2;
  static constexpr int kDQEmpty = kDQDone + 1;  // rank 0's: both epilogues have read dQ
  static constexpr int kDrain = kDQEmpty + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;  // + TMEM address and abort flag
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 384;  // dP buffer b at kColDP + 128 b
  static constexpr int kThreads = 352;
  static constexpr int kComputeThreads = 256;
  static constexpr uint32_t kPairWarps = 2 * kComputeThreads / 32;
};

struct DqPairArgs {
  const float* lse;
  const float* delta;
  uint16_t* dq;
  int BHKP;  // B * Hkv * G / 2: head pairs per query block
  int Hq, Hkv, G, nqb, ntiles;
  Span span;
  float scale, scale_log2;
  unsigned* err;
  FastDiv divBHKP, divGP, divHkv;  // tile index decomposition (divGP: G / 2)
};

struct DqPairTile {
  int bh, bhk, q0, kb_lo, nkv;
};

// Pair tile t (heaviest query blocks first); rank r takes query head 2 p + r of the kv group.
__device__ __forceinline__ DqPairTile dq_pair_tile(int t, const DqPairArgs& a, const Span sp,
                                                   uint32_t rank) {
  DqPairTile f;
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
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(352, 1)
    swa_dq_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k64,   // K, 64-row boxes
                       const __grid_constant__ CUtensorMap tm_k128,  // K, 128-row boxes
                       const __grid_constant__ CUtensorMap tm_v64,   // V, 64-row boxes
                       const DqPairArgs a) {
  using C = DqPairCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  // Both CTAs always reach the cluster barriers and the collective TMEM allocation; a misaligned
  // window only disables the work (and is reported).
  const bool smem_ok = (smem_u32(smem) & 1023u) == 0u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sK0 = smem_u32(smem + C::kOffK);
  const uint32_t sV0 = smem_u32(smem + C::kOffV);
  // K stage s: the key half for S at sKS(s), the head-dim chunk for dQ at sKQ(s).
  auto sKS = [&](int s) { return sK0 + s * C::kKStageBytes; };
  auto sKQ = [&](int s) { return sK0 + s * C::kKStageBytes + C::kHalfBytes; };
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
    mbar_init(bar(C::kQDFull), full_count);
    mbar_init(bar(C::kQDEmpty), 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar(C::kKFull + s), full_count);
      mbar_init(bar(C::kKEmpty + s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar(C::kVFull + s), full_count);
      mbar_init(bar(C::kVEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSEmpty), C::kPairWarps);
    mbar_init(bar(C::kDPFull + 0), 1);
    mbar_init(bar(C::kDPFull + 1), 1);
    mbar_init(bar(C::kDSFull + 0), C::kPairWarps);
    mbar_init(bar(C::kDSFull + 1), C::kPairWarps);
    mbar_init(bar(C::kDQDone), 1);
    mbar_init(bar(C::kDQEmpty), C::kPairWarps);
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

  if (!smem_ok) {
    // nothing to do: fall through to the final barrier and the collective release
  } else if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer (Q, dO, K)
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k64);
      tma_prefetch_desc(&tm_k128);
      int last_qd = -1;
      int last_k[C::kKStages];
      for (int s = 0; s < C::kKStages; ++s) last_k[s] = -1;
      int g = 0;
      bool ok = true;
      for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
        const DqPairTile f = dq_pair_tile(t, a, sp, rank);
        // Q / dO of the previous tile are free once its last dP has been computed.
        if (it >= 1 && !mbar_wait(bar(C::kQDEmpty), (it - 1) & 1, &abort_flag, a.err)) break;
        mbar_arrive_expect_tx(bar(C::kQDFull), 2 * C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h) {
          tma_load_3d(sQ + h * C::kChunkBytes, &tm_q, bar(C::kQDFull), 64 * h, f.q0, f.bh);
          tma_load_3d(sDO + h * C::kChunkBytes, &tm_do, bar(C::kQDFull), 64 * h, f.q0, f.bh);
        }
        last_qd = it;
        for (int j = 0; j < f.nkv; ++j, ++g) {
          const int k0 = (f.kb_lo + j) * kBlockN;
          const int sk = g % C::kKStages, nk = g / C::kKStages;
          if (g >= C::kKStages &&
              !(ok = mbar_wait(bar(C::kKEmpty + sk), (nk - 1) & 1, &abort_flag, a.err)))
            break;
          mbar_arrive_expect_tx(bar(C::kKFull + sk), C::kKStageBytes);
          for (int h = 0; h < C::kChunks; ++h)
            tma_load_3d(sKS(sk) + h * C::kHalfChunkBytes, &tm_k64, bar(C::kKFull + sk), 64 * h,
                        k0 + C::kHalfRows * static_cast<int>(rank), f.bhk);
          tma_load_3d(sKQ(sk), &tm_k128, bar(C::kKFull + sk), 64 * static_cast<int>(rank), k0,
                      f.bhk);
          last_k[sk] = g;
        }
      }
      if (last_qd >= 0) drain_wait(bar(C::kQDFull), last_qd & 1, a.err);
      for (int s = 0; s < C::kKStages; ++s)
        if (last_k[s] >= 0) drain_wait(bar(C::kKFull + s), (last_k[s] / C::kKStages) & 1, a.err);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------------ TMA producer (V half)
    if (lane == 0) {
      tma_prefetch_desc(&tm_v64);
      int last_v[C::kVStages];
      for (int s = 0; s < C::kVStages; ++s) last_v[s] = -1;
      int g = 0;
      bool ok = true;
      for (int t = tile0; ok && t < a.ntiles; t += tile_step) {
        const DqPairTile f = dq_pair_tile(t, a, sp, rank);
        for (int j = 0; j < f.nkv; ++j, ++g) {
          const int sv = g % C::kVStages, nv = g / C::kVStages;
          if (g >= C::kVStages &&
              !(ok = mbar_wait(bar(C::kVEmpty + sv), (nv - 1) & 1, &abort_flag, a.err)))
            break;
          const uint32_t sV = sV0 + sv * C::kHalfBytes;
          mbar_arrive_expect_tx(bar(C::kVFull + sv), C::kHalfBytes);
          for (int h = 0; h < C::kChunks; ++h)
            tma_load_3d(sV + h * C::kHalfChunkBytes, &tm_v64, bar(C::kVFull + sv), 64 * h,
                        (f.kb_lo + j) * kBlockN + C::kHalfRows * static_cast<int>(rank), f.bhk);
          last_v[sv] = g;
        }
      }
      for (int s = 0; s < C::kVStages; ++s)
        if (last_v[s] >= 0) drain_wait(bar(C::kVFull + s), (last_v[s] / C::kVStages) & 1, a.err);
    }
  } else if (warp == 9 && lead) {
    // ------------------------------------------------------------------ MMA issuer (the pair)
    // Per tile: S_0, dP_0, then per block j: S_{j+1}, dP_{j+1}, dQ += dS_j K_j (as swa_bwd_dq.cu).
    // dP_gg goes into buffer gg & 1, which last held dS_{gg-2}: dQ_{gg-2} was issued before it and
    // tcgen05.mma operations of one thread run in issue order, so no wait is needed.
    constexpr uint32_t kIdSq = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdDq = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockM, D, false, true);
    auto issue_s = [&](int gg) -> bool {  // S = Q K_gg^T once S_{gg-1} has been read
      const int s = gg % C::kKStages, n = gg / C::kKStages;
      if (!warp_wait_cluster(bar(C::kKFull + s), n & 1, &abort_flag, a.err)) return false;
      if (gg >= 1 && !warp_wait_cluster(bar(C::kSEmpty), (gg - 1) & 1, &abort_flag, a.err))
        return false;
      tc_fence_after();
      umma2_ss_kmajor_d<D>(tmem + C::kColS, smem_desc_sw128(sQ, 16, 1024),
                           smem_desc_sw128(sKS(s), 16, 1024), kIdSq, 0u);
      umma2_commit_w(bar(C::kSFull));
      return true;
    };
    auto issue_dp = [&](int gg, bool tile_last) -> bool {  // dP = dO V_gg^T into buffer gg & 1
      const int s = gg % C::kVStages, n = gg / C::kVStages;
      if (!warp_wait_cluster(bar(C::kVFull + s), n & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ss_kmajor_d<D>(tmem + C::kColDP + 128u * (gg & 1), smem_desc_sw128(sDO, 16, 1024),
                           smem_desc_sw128(sV0 + s * C::kHalfBytes, 16, 1024), kIdSq, 0u);
      umma2_commit_w(bar(C::kDPFull + (gg & 1)));
      umma2_commit_w(bar(C::kVEmpty + s));
      if (tile_last) umma2_commit_w(bar(C::kQDEmpty));  // every S and dP of the tile is issued
      return true;
    };
    // dQ += dS_gg K_gg with dS_gg in dP buffer gg & 1: keys 16 ks .. 16 ks + 15 at packed column
    // 8 ks + 32 (ks / 4).
    auto issue_dq = [&](int gg, bool first, bool tile_last) -> bool {
      const int s = gg % C::kKStages, db = gg & 1;
      if (!warp_wait_cluster(bar(C::kDSFull + db), (gg >> 1) & 1, &abort_flag, a.err))
        return false;
      tc_fence_after();
      umma2_ts_mnmajor_x8_split(tmem + C::kColDQ, tmem + C::kColDP + 128u * db,
                                smem_desc_sw128(sKQ(s), C::kKColBytes, 1024), kIdDq,
                                first ? 0u : 1u);
      umma2_commit_w(bar(C::kKEmpty + s));
      if (tile_last) umma2_commit_w(bar(C::kDQDone));
      return true;
    };
    int g = 0;
    bool ok = true;
    for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const DqPairTile f = dq_pair_tile(t, a, sp, rank);
      const int n = f.nkv;
      ok = warp_wait_cluster(bar(C::kQDFull), it & 1, &abort_flag, a.err);
      if (ok) ok = issue_s(g);
      if (ok) ok = issue_dp(g, n == 1);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          ok = issue_s(g + j + 1);
          if (ok) ok = issue_dp(g + j + 1, j + 2 == n);
        }
        // The first dQ of a tile overwrites the accumulator: both epilogues must have read it.
        if (ok && j == 0 && it > 0)
          ok = warp_wait_cluster(bar(C::kDQEmpty), (it - 1) & 1, &abort_flag, a.err);
        if (ok) ok = issue_dq(g + j, j == 0, j + 1 == n);
      }
      g += n;
    }
    umma2_commit_w(bar(C::kDrain));
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else if (warp == 9) {
    // ------------------------------------------------------------------ relay (rank 1)
    // Rank 0 consumes, per tile: Q and dO, K_0, V_0, then K_{j+1} and V_{j+1} for each block j.
    auto relay = [&](int idx, uint32_t parity) -> bool {
      if (!warp_wait(bar(idx), parity, &abort_flag, a.err)) return false;
      if (lane == 0) mbar_arrive_cluster(mapa_rank0(bar(idx)));
      __syncwarp();
      return true;
    };
    auto relay_kv = [&](int gg) -> bool {
      return relay(C::kKFull + gg % C::kKStages, (gg / C::kKStages) & 1) &&
             relay(C::kVFull + gg % C::kVStages, (gg / C::kVStages) & 1);
    };
    int g = 0;
    bool ok = true;
    for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const DqPairTile f = dq_pair_tile(t, a, sp, rank);
      ok = relay(C::kQDFull, it & 1);
      for (int j = 0; ok && j < f.nkv; ++j) ok = relay_kv(g + j);
      g += f.nkv;
    }
  } else {
    // ------------------------------------------------------------------ compute (warps 0-7)
    static_assert(C::kSEmpty - C::kSFull == dqc::DqBar::kSEmpty &&
                      C::kDPFull - C::kSFull == dqc::DqBar::kDPFull &&
                      C::kDSFull - C::kSFull == dqc::DqBar::kDSFull &&
                      C::kDQDone - C::kSFull == dqc::DqBar::kDQDone &&
                      C::kDQEmpty - C::kSFull == dqc::DqBar::kDQEmpty && C::kColS == dqc::kColS &&
                      C::kColDP == dqc::kColDP && C::kColDQ == dqc::kColDQ,
                  "dQ compute layout");
    dqc::dq_compute<D, F16, true>(a, sp, tmem, bar(C::kSFull), &abort_flag, tile0, tile_step,
                                  [&](int t) { return dq_pair_tile(t, a, sp, rank); });
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
cudaError_t launch_dq_pair_d(const Problem& pb, const void* q, const void* k, const void* v,
                             const void* dO, const float* lse, const float* delta, void* dq,
                             cudaStream_t stream) {
  using C = DqPairCfg<D>;
  CUtensorMap tq, tdo, tk64, tk128, tv64;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_3d(&tq, q, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tdo, dO, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tk64, k, bhk, pb.span.Lk, D, C::kHalfRows, F16) ||
      !make_tmap_3d(&tk128, k, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tv64, v, bhk, pb.span.Lk, D, C::kHalfRows, F16))
    return cudaErrorInvalidValue;
  auto kern = swa_dq_pair_kernel<D, F16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  DqPairArgs a;
  a.lse = lse;
  a.delta = delta;
  a.dq = static_cast<uint16_t*>(dq);
  a.G = pb.Hq / pb.Hkv;
  a.BHKP = pb.B * pb.Hkv * (a.G / 2);
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.span = pb.span;
  a.nqb = (pb.span.Lq + kBlockM - 1) / kBlockM;
  a.ntiles = a.nqb * a.BHKP;
  a.scale = pb.scale;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  a.divBHKP = FastDiv(static_cast<uint32_t>(a.BHKP));
  a.divGP = FastDiv(static_cast<uint32_t>(a.G / 2));
  a.divHkv = FastDiv(static_cast<uint32_t>(a.Hkv));
  const int clusters = max_pair_clusters<swa_dq_pair_kernel<D, F16>>(C::kThreads, C::kSmemBytes);
  const int nclusters = a.ntiles < clusters ? a.ntiles : clusters;
  kern<<<2 * nclusters, C::kThreads, C::kSmemBytes, stream>>>(tq, tdo, tk64, tk128, tv64, a);
  return cudaGetLastError();
}

}  // namespace

bool dq_pair_applies(const Problem& pb) {
  const int G = pb.Hq / pb.Hkv;
  return pb.D == 128 && G % 2 == 0;
}

cudaError_t launch_dq_pair(const Problem& pb, const void* q, const void* k, const void* v,
                           const void* dO, const float* lse, const float* delta, void* dq,
                           cudaStream_t stream) {
  if (!dq_pair_applies(pb)) return cudaErrorInvalidValue;
  return pb.f16 ? launch_dq_pair_d<128, true>(pb, q, k, v, dO, lse, delta, dq, stream)
                : launch_dq_pair_d<128, false>(pb, q, k, v, dO, lse, delta, dq, stream);
}

}  // namespace swa
