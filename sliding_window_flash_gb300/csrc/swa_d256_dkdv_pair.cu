// swa_d256_dkdv_pair.cu — dV and dK with head dimension 256 on CTA pairs (sm_103a).
//
// The same sums as the key-block kernels of swa_d256.cu — dV = sum P^T dO and
// dK = scale sum dS^T Q over the G query heads of a kv head and the query blocks that see a key
// block, P and dS recomputed from LSE and Delta ("Off NVIDIA, you fix the platform yourself",
// Lab 28 record, numbers entry "Attention backward memory": Gemma 4's sliding layers use
// 256-wide heads).  A cluster of two CTAs takes two neighbouring 128-row key blocks of one
// (batch, kv head), rank r the block 2 p + r, and both walk the union of the two blocks' query
// blocks (for a causal window of W keys: W / 128 + 2 query blocks where each block alone sees
// W / 128 + 1; the extra one is fully masked for one of the two and contributes exact zeros).
// Rank 0 issues every MMA for both SMs as tcgen05.mma.cta_group::2 with M = 256, each SM
// computing its own 128 key rows:
//   S^T = K Q^T, dP^T = V dO^T   over D in two halves; B = queries [64 r, 64 r + 64) (32 KB),
//   dV += P^T dO, dK += dS^T Q   one N = 256 product; B = head dims [128 r, 128 r + 128) (32 KB).
// Each SM thus moves half the query-side bytes the single-CTA kernels move per query block, and
// its MMAs read half their B operand from shared memory.
//
// Warp roles (352 threads per CTA): warps 0-7 compute (as swa_d256.cu: warp w owns key rows
// 32 (w % 4).. and query columns [64 h, 64 h + 64), h = w / 4; the arrivals that let rank 0 issue
// an MMA reading their output go to rank 0's barriers, 16 arrivals); warps 8 and 10 load this
// CTA's ring items (even / odd) and the CTA's K (dV) or K and V (dK) once; warp 9 rank 0: MMA
// issuer for the pair, rank 1: relay — waits for each of its own copies in the order rank 0
// consumes them and arrives on rank 0's matching barrier (rank 0's full barriers count its own
// copies and the relay).
#include "swa_d256.cuh"
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

using d256::ds_transposed;
using d256::key_epilogue;
using d256::p_transposed;

constexpr int kD = 256;
constexpr int kChunk = kBlockM * 128;       // 128 rows x 64 columns
constexpr int kHalfRows = kBlockM / 2;
constexpr int kHalfChunk = kHalfRows * 128;  // 64 rows x 64 columns
constexpr int kItemBytes = 32768;
constexpr int kFullBytes = kBlockN * kD * 2;  // a whole 128 x 256 key-side tile
constexpr uint32_t kPairWarps = 16;

struct PairArgs {
  const float* lse;
  const float* delta;
  uint16_t* dk;  // outputs, for key blocks no query sees (zeros)
  uint16_t* dv;
  int Hq, Hkv, G, BHK;  // BHK = B * Hkv
  Span span;
  float scale, scale_log2;
  unsigned* err;
};

// The pair's walk: G query heads x the union [qb_lo, qb_lo + nq) of the two key blocks' query
// blocks; tile t = g nq + (query block - qb_lo).  Own-block fields describe this CTA's keys.
struct PairWalk {
  int bhk, b, hk, k0, qb_lo, nq, T;
  bool valid;                // this CTA's key block starts inside the key sequence
  int q_int_lo, q_int_hi;    // query tiles q0 in [q_int_lo, q_int_hi] need no mask for own keys
};

__device__ __forceinline__ PairWalk pair_walk(const PairArgs& a, const Span& sp, uint32_t rank) {
  PairWalk w;
  const int c = static_cast<int>(blockIdx.x >> 1);
  const int kp = c / a.BHK;
  w.bhk = c - kp * a.BHK;
  w.b = w.bhk / a.Hkv;
  w.hk = w.bhk - w.b * a.Hkv;
  int lo = 0, hi = -1;
  bool any = false;
  for (int r = 0; r < 2; ++r) {
    const int k0 = (2 * kp + r) * kBlockN;
    if (k0 >= sp.Lk) continue;
    const int f = sp.first_qblock(k0), l = sp.last_qblock(k0);
    if (f > l) continue;
    if (!any) lo = f;  // first_qblock and last_qblock grow with k0
    hi = l;
    any = true;
  }
  w.qb_lo = lo;
  w.nq = any ? hi - lo + 1 : 0;
  w.T = a.G * w.nq;
  w.k0 = (2 * kp + static_cast<int>(rank)) * kBlockN;
  w.valid = w.k0 < sp.Lk;
  w.q_int_lo = w.k0 + kBlockN - 1 + sp.dmin - sp.off;
  w.q_int_hi = (w.k0 + kBlockN <= sp.Lk)
                   ? min(w.k0 + sp.dmax - sp.off - (kBlockM - 1), sp.Lq - kBlockM)
                   : -1;
  return w;
}

// Query position and (batch, query head) plane of walk tile t.
__device__ __forceinline__ int pw_q0(const PairWalk& w, int t) {
  return (w.qb_lo + t % w.nq) * kBlockM;
}
__device__ __forceinline__ int pw_bhq(const PairWalk& w, const PairArgs& a, int t) {
  return w.b * a.Hq + w.hk * a.G + t / w.nq;
}

// Ring item kinds: query half of Q (B of S^T), query half of dO (B of dP^T), head-dim half of
// Q or dO (B of dK or dV).
enum : int { kQH = 0, kDOH = 1, kQC = 2, kDOC = 3 };

__device__ __forceinline__ void load_item(uint32_t dst, uint32_t full_bar, int kind, int q0,
                                          int bhq, uint32_t rank, const CUtensorMap* tm_q64,
                                          const CUtensorMap* tm_do64, const CUtensorMap* tm_q128,
                                          const CUtensorMap* tm_do128) {
  mbar_arrive_expect_tx(full_bar, kItemBytes);
  if (kind == kQC || kind == kDOC) {
    const CUtensorMap* m = kind == kQC ? tm_q128 : tm_do128;
    for (int c = 0; c < 2; ++c)
      tma_load_3d(dst + c * kChunk, m, full_bar, 128 * static_cast<int>(rank) + 64 * c, q0, bhq);
  } else {
    const CUtensorMap* m = kind == kQH ? tm_q64 : tm_do64;
    for (int c = 0; c < 4; ++c)
      tma_load_3d(dst + c * kHalfChunk, m, full_bar, 64 * c,
                  q0 + kHalfRows * static_cast<int>(rank), bhq);
  }
}

// ================================================================================================
// dV.  Ring order: QH_0, then per tile t: QH_{t+1} (if any), dOC_t.
// TMEM (each CTA): [0,128) S^T / P^T buffer 0, [128,256) buffer 1, [256,512) dV.
// ================================================================================================
struct VP {
  static constexpr int kSlots = 5;
  static constexpr int kOffK = 0;
  static constexpr int kOffRing = kOffK + kFullBytes;
  static constexpr int kOffRow = kOffRing + kSlots * kItemBytes;  // [2 slots][128] -LSE log2(e)
  static constexpr int kOffBar = kOffRow + 2 * kBlockM * 4;
  static constexpr int kKFull = 0;
  static constexpr int kFull = 1;
  static constexpr int kEmpty = kFull + kSlots;
  static constexpr int kSFull = kEmpty + kSlots;  // 2
  static constexpr int kPFull = kSFull + 2;       // 2, rank 0's
  static constexpr int kVecFull = kPFull + 2;     // 2
  static constexpr int kDone = kVecFull + 2;
  static constexpr int kOutFull = kDone + 1;
  static constexpr int kDrain = kOutFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 48;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kColS = 0, kColAcc = 256;
  static constexpr int kThreads = 352;
};

template <bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(352, 1)
    swa_dv256_pair_kernel(const __grid_constant__ CUtensorMap tm_q64,
                          const __grid_constant__ CUtensorMap tm_do128,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_dv, const PairArgs a) {
  using C = VP;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const Span sp = a.span;
  const uint32_t rank = cluster_rank();
  const bool lead = rank == 0u;
  const PairWalk w = pair_walk(a, sp, rank);
  if (w.T == 0) {  // neither key block is seen by any query (both CTAs return here)
    zero_key_rows(a.dv, nullptr, w.bhk, w.k0, sp.Lk, kD);
    return;
  }
  const bool smem_ok = (smem_u32(smem) & 1023u) == 0u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 4);  // [2][kSlots]: producers' last fills
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sRing = smem_u32(smem + C::kOffRing);
  float* s_rows = reinterpret_cast<float*>(smem + C::kOffRow);
  auto slot = [&](int i) { return sRing + (i % C::kSlots) * kItemBytes; };
  auto full = [&](int i) { return bar(C::kFull + i % C::kSlots); };
  auto empty = [&](int i) { return bar(C::kEmpty + i % C::kSlots); };
  auto parity = [&](int i) { return static_cast<uint32_t>((i / C::kSlots) & 1); };

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = smem_ok ? 0 : 1;
    if (!smem_ok) atomicOr(a.err, kErrSmemLayout);
    const uint32_t full_count = lead ? 2u : 1u;  // rank 0: own copy + rank 1's relay
    mbar_init(bar(C::kKFull), full_count);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kFull + s), full_count);
      mbar_init(bar(C::kEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kSFull + b), 1);
      mbar_init(bar(C::kPFull + b), kPairWarps);
      mbar_init(bar(C::kVecFull + b), 8);
    }
    mbar_init(bar(C::kDone), 1);
    mbar_init(bar(C::kOutFull), 8);
    mbar_init(bar(C::kDrain), 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // This CTA's ring items in consumption order: on_item(index, kind, tile).
  auto walk_items = [&](auto&& on_item) -> bool {
    int i = 0;
    if (!on_item(i++, kQH, 0)) return false;
    for (int t = 0; t < w.T; ++t) {
      if (t + 1 < w.T && !on_item(i++, kQH, t + 1)) return false;
      if (!on_item(i++, kDOC, t)) return false;
    }
    return true;
  };

  if (!smem_ok) {
    // nothing to do: fall through to the final barrier and the collective release
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ K once; ring items
    const int p = warp == 8 ? 0 : 1;
    int last[C::kSlots];  // lane 0: last item loaded per slot
    for (int s = 0; s < C::kSlots; ++s) last[s] = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q64);
      tma_prefetch_desc(&tm_do128);
      if (p == 0) {
        tma_prefetch_desc(&tm_k);
        mbar_arrive_expect_tx(bar(C::kKFull), kFullBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_3d(sK + c * kChunk, &tm_k, bar(C::kKFull), 64 * c, w.k0, w.bhk);
      }
      walk_items([&](int i, int kind, int t) -> bool {
        if ((i & 1) != p) return true;
        if (i >= C::kSlots &&
            !mbar_wait(empty(i), ((i / C::kSlots) - 1) & 1, &abort_flag, a.err))
          return false;
        load_item(slot(i), full(i), kind, pw_q0(w, t), pw_bhq(w, a, t), rank, &tm_q64, nullptr,
                  nullptr, &tm_do128);
        last[i % C::kSlots] = i;
        return true;
      });
      if (p == 0) drain_wait(bar(C::kKFull), 0, a.err);
    }
    d256::drain_ring<C::kSlots>(last, s_last, p, lane, full, a.err);
  } else if (warp == 9 && lead) {
    // ------------------------------------------------------------ MMA issuer (the pair)
    constexpr uint32_t kIdS = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockN, kBlockM, false, false);
    constexpr uint32_t kIdAcc = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockN, kD, false, true);
    int i = 0;
    // S^T_t = K Q_t^T into buffer t & 1 (which last held P^T_{t-2}, read by dV_{t-2}, issued
    // before this).
    auto issue_s = [&](int t) -> bool {
      if (!warp_wait_cluster(full(i), parity(i), &abort_flag, a.err)) return false;
      tc_fence_after();
      const uint32_t d = tmem + C::kColS + 128u * (t & 1);
      umma2_ss_kmajor_d<128>(d, smem_desc_sw128(sK, 16, 1024), smem_desc_sw128(slot(i), 16, 1024),
                             kIdS, 0u);
      umma2_ss_kmajor_d<128>(d, smem_desc_sw128(sK + 2 * kChunk, 16, 1024),
                             smem_desc_sw128(slot(i) + 2 * kHalfChunk, 16, 1024), kIdS, 1u);
      umma2_commit_w(empty(i));
      ++i;
      umma2_commit_w(bar(C::kSFull + (t & 1)));
      return true;
    };
    // dV (+)= P^T_t dO_t: P^T packed over S^T buffer t & 1, B = this CTA's 128 head dims of dO.
    auto issue_dv = [&](int t) -> bool {
      const int pb = t & 1;
      if (!warp_wait_cluster(bar(C::kPFull + pb), (t >> 1) & 1, &abort_flag, a.err)) return false;
      if (!warp_wait_cluster(full(i), parity(i), &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ts_mnmajor_x8_split(tmem + C::kColAcc, tmem + C::kColS + 128u * pb,
                                smem_desc_sw128(slot(i), kChunk, 1024), kIdAcc, t > 0 ? 1u : 0u);
      umma2_commit_w(empty(i));
      ++i;
      return true;
    };
    bool ok = warp_wait_cluster(bar(C::kKFull), 0, &abort_flag, a.err);
    if (ok) ok = issue_s(0);
    for (int t = 0; ok && t < w.T; ++t) {
      if (t + 1 < w.T) ok = issue_s(t + 1);
      if (ok) ok = issue_dv(t);
    }
    if (ok) umma2_commit_w(bar(C::kDone));
    umma2_commit_w(bar(C::kDrain));
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else if (warp == 9) {
    // ------------------------------------------------------------ relay (rank 1)
    auto relay = [&](uint32_t b, uint32_t par) -> bool {
      if (!warp_wait(b, par, &abort_flag, a.err)) return false;
      if (lane == 0) mbar_arrive_cluster(mapa_rank0(b));
      __syncwarp();
      return true;
    };
    if (relay(bar(C::kKFull), 0))
      walk_items([&](int i, int, int) { return relay(full(i), parity(i)); });
  } else {
    // ------------------------------------------------------------ compute (warps 0-7)
    const int r = static_cast<int>(threadIdx.x & 127);  // key row within the block = TMEM lane
    const uint32_t h = warp >> 2;
    const int key = w.k0 + r;
    const int vis_lo = key + sp.dmin - sp.off, vis_hi = key + sp.dmax - sp.off;
    const uint32_t lane_base = ((warp & 3u) * 32u) << 16;
    float nxt = 0.f;  // LSE of query q0(t) + r, fetched a tile ahead (h = 0 threads)
    auto fetch_row = [&](int t) {
      const int q = pw_q0(w, t) + r;
      nxt = q < sp.Lq ? a.lse[static_cast<size_t>(pw_bhq(w, a, t)) * sp.Lq + q] : SWA_POS_INF;
    };
    if (h == 0) fetch_row(0);
    bool ok = true;
    for (int t = 0; t < w.T; ++t) {
      const int q0 = pw_q0(w, t);
      // Slot t & 1 was last read in tile t - 2; every warp has since arrived for tile t - 1.
      float* nl2 = s_rows + (t & 1) * kBlockM;
      if (h == 0) nl2[r] = -nxt * kLog2e;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kVecFull + (t & 1)));
      if (!(ok = warp_wait(bar(C::kVecFull + (t & 1)), (t >> 1) & 1, &abort_flag, a.err))) break;
      if (t + 1 < w.T && h == 0) fetch_row(t + 1);
      if (!(ok = warp_wait(bar(C::kSFull + (t & 1)), (t >> 1) & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      const uint32_t s_col = tmem + lane_base + C::kColS + 128u * (t & 1) + 64u * h;
      float p[64];
      const int base = q0 + 64 * static_cast<int>(h);
      p_transposed(p, s_col, nl2 + 64 * h, a.scale_log2, !(q0 >= w.q_int_lo && q0 <= w.q_int_hi),
                   vis_lo - base, vis_hi - base);
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pk[c] = Elem<F16>::pack(p[2 * c], p[2 * c + 1]);
      tmem_st32(s_col, pk);
      tmem_wait_st();
      warp_arrive_rank0(bar(C::kPFull + (t & 1)));
    }
    if (ok && warp_wait(bar(C::kDone), 0, &abort_flag, a.err) && w.valid) {
      tc_fence_after();
      // dV -> 16-bit, staged in the K buffer (every MMA of the pair has completed).
      key_epilogue<F16>(tmem + lane_base + C::kColAcc, sK, r, h, 1.f, false, bar(C::kOutFull),
                        &tm_dv, w.k0, w.bhk, &abort_flag, a.err);
    }
  }

  // Every cross-CTA arrival and every pair MMA (rank 0 waited for its drain) is complete once both
  // CTAs are here; then the pair releases its TMEM together.
  tc_fence_before();
  cluster_sync_all();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// ================================================================================================
// dK.  S^T_{t+1} is issued once the compute warps of both CTAs have read S^T_t; dS^T goes over
// the dP^T columns it came from and is the A operand of dK += dS^T Q_t, after which dP^T_{t+1}
// is issued.
// Ring order: QH_0, dOH_0, then per tile t: QH_{t+1} (if any), QC_t, dOH_{t+1} (if any).
// TMEM (each CTA): [0,128) S^T, [128,256) dP^T / dS^T, [256,512) dK.
// ================================================================================================
struct KP {
  static constexpr int kSlots = 3;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kFullBytes;
  static constexpr int kOffRing = kOffV + kFullBytes;
  static constexpr int kOffRow = kOffRing + kSlots * kItemBytes;  // [2 slots][-LSE log2e | -Delta]
  static constexpr int kOffBar = kOffRow + 2 * 2 * kBlockM * 4;
  static constexpr int kKVFull = 0;
  static constexpr int kFull = 1;
  static constexpr int kEmpty = kFull + kSlots;
  static constexpr int kSFull = kEmpty + kSlots;
  static constexpr int kSEmpty = kSFull + 1;   // rank 0's
  static constexpr int kDPFull = kSEmpty + 1;
  static constexpr int kDSFull = kDPFull + 1;  // rank 0's
  static constexpr int kVecFull = kDSFull + 1;  // 2
  static constexpr int kDone = kVecFull + 2;
  static constexpr int kOutFull = kDone + 1;
  static constexpr int kDrain = kOutFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 48;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc = 256;
  static constexpr int kThreads = 352;
};

template <bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(352, 1)
    swa_dk256_pair_kernel(const __grid_constant__ CUtensorMap tm_q64,
                          const __grid_constant__ CUtensorMap tm_do64,
                          const __grid_constant__ CUtensorMap tm_q128,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_dk, const PairArgs a) {
  using C = KP;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const Span sp = a.span;
  const uint32_t rank = cluster_rank();
  const bool lead = rank == 0u;
  const PairWalk w = pair_walk(a, sp, rank);
  if (w.T == 0) {  // neither key block is seen by any query (both CTAs return here)
    zero_key_rows(a.dk, nullptr, w.bhk, w.k0, sp.Lk, kD);
    return;
  }
  const bool smem_ok = (smem_u32(smem) & 1023u) == 0u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 4);  // [2][kSlots]: producers' last fills
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const uint32_t sRing = smem_u32(smem + C::kOffRing);
  float* s_rows = reinterpret_cast<float*>(smem + C::kOffRow);
  auto slot = [&](int i) { return sRing + (i % C::kSlots) * kItemBytes; };
  auto full = [&](int i) { return bar(C::kFull + i % C::kSlots); };
  auto empty = [&](int i) { return bar(C::kEmpty + i % C::kSlots); };
  auto parity = [&](int i) { return static_cast<uint32_t>((i / C::kSlots) & 1); };

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = smem_ok ? 0 : 1;
    if (!smem_ok) atomicOr(a.err, kErrSmemLayout);
    // K and V: one arrival per producer warp (+ rank 1's relay on rank 0)
    mbar_init(bar(C::kKVFull), lead ? 3u : 2u);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kFull + s), lead ? 2u : 1u);
      mbar_init(bar(C::kEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSEmpty), kPairWarps);
    mbar_init(bar(C::kDPFull), 1);
    mbar_init(bar(C::kDSFull), kPairWarps);
    mbar_init(bar(C::kVecFull + 0), 8);
    mbar_init(bar(C::kVecFull + 1), 8);
    mbar_init(bar(C::kDone), 1);
    mbar_init(bar(C::kOutFull), 8);
    mbar_init(bar(C::kDrain), 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // This CTA's ring items in consumption order: on_item(index, kind, tile).
  auto walk_items = [&](auto&& on_item) -> bool {
    int i = 0;
    if (!on_item(i++, kQH, 0)) return false;
    if (!on_item(i++, kDOH, 0)) return false;
    for (int t = 0; t < w.T; ++t) {
      if (t + 1 < w.T && !on_item(i++, kQH, t + 1)) return false;
      if (!on_item(i++, kQC, t)) return false;
      if (t + 1 < w.T && !on_item(i++, kDOH, t + 1)) return false;
    }
    return true;
  };

  if (!smem_ok) {
    // nothing to do: fall through to the final barrier and the collective release
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ K / V once; ring items
    const int p = warp == 8 ? 0 : 1;
    int last[C::kSlots];  // lane 0: last item loaded per slot
    for (int s = 0; s < C::kSlots; ++s) last[s] = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q64);
      tma_prefetch_desc(&tm_do64);
      tma_prefetch_desc(&tm_q128);
      {
        const CUtensorMap* m = p == 0 ? &tm_k : &tm_v;
        const uint32_t dst = p == 0 ? sK : sV;
        mbar_arrive_expect_tx(bar(C::kKVFull), kFullBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_3d(dst + c * kChunk, m, bar(C::kKVFull), 64 * c, w.k0, w.bhk);
      }
      walk_items([&](int i, int kind, int t) -> bool {
        if ((i & 1) != p) return true;
        if (i >= C::kSlots &&
            !mbar_wait(empty(i), ((i / C::kSlots) - 1) & 1, &abort_flag, a.err))
          return false;
        load_item(slot(i), full(i), kind, pw_q0(w, t), pw_bhq(w, a, t), rank, &tm_q64, &tm_do64,
                  &tm_q128, nullptr);
        last[i % C::kSlots] = i;
        return true;
      });
      drain_wait(bar(C::kKVFull), 0, a.err);
    }
    d256::drain_ring<C::kSlots>(last, s_last, p, lane, full, a.err);
  } else if (warp == 9 && lead) {
    // ------------------------------------------------------------ MMA issuer (the pair)
    constexpr uint32_t kIdS = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockN, kBlockM, false, false);
    constexpr uint32_t kIdAcc = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockN, kD, false, true);
    int i = 0;
    auto product_d = [&](uint32_t d, uint32_t a_tile) -> bool {  // A B^T over D, B = ring item
      if (!warp_wait_cluster(full(i), parity(i), &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ss_kmajor_d<128>(d, smem_desc_sw128(a_tile, 16, 1024),
                             smem_desc_sw128(slot(i), 16, 1024), kIdS, 0u);
      umma2_ss_kmajor_d<128>(d, smem_desc_sw128(a_tile + 2 * kChunk, 16, 1024),
                             smem_desc_sw128(slot(i) + 2 * kHalfChunk, 16, 1024), kIdS, 1u);
      umma2_commit_w(empty(i));
      ++i;
      return true;
    };
    auto issue_s = [&](int t) -> bool {  // S^T = K Q_t^T once S^T_{t-1} has been read
      if (t >= 1 && !warp_wait_cluster(bar(C::kSEmpty), (t - 1) & 1, &abort_flag, a.err))
        return false;
      if (!product_d(tmem + C::kColS, sK)) return false;
      umma2_commit_w(bar(C::kSFull));
      return true;
    };
    auto issue_dp = [&]() -> bool {  // dP^T = V dO_t^T, after dK of the previous tile
      if (!product_d(tmem + C::kColDP, sV)) return false;
      umma2_commit_w(bar(C::kDPFull));
      return true;
    };
    auto issue_dk = [&](int t) -> bool {  // dK (+)= dS_t^T Q_t, B = this CTA's 128 head dims of Q
      if (!warp_wait_cluster(bar(C::kDSFull), t & 1, &abort_flag, a.err)) return false;
      if (!warp_wait_cluster(full(i), parity(i), &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ts_mnmajor_x8_split(tmem + C::kColAcc, tmem + C::kColDP,
                                smem_desc_sw128(slot(i), kChunk, 1024), kIdAcc, t > 0 ? 1u : 0u);
      umma2_commit_w(empty(i));
      ++i;
      return true;
    };
    bool ok = warp_wait_cluster(bar(C::kKVFull), 0, &abort_flag, a.err);
    if (ok) ok = issue_s(0);
    if (ok) ok = issue_dp();
    for (int t = 0; ok && t < w.T; ++t) {
      if (t + 1 < w.T) ok = issue_s(t + 1);
      if (ok) ok = issue_dk(t);
      if (ok && t + 1 < w.T) ok = issue_dp();
    }
    if (ok) umma2_commit_w(bar(C::kDone));
    umma2_commit_w(bar(C::kDrain));
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else if (warp == 9) {
    // ------------------------------------------------------------ relay (rank 1)
    auto relay = [&](uint32_t b, uint32_t par) -> bool {
      if (!warp_wait(b, par, &abort_flag, a.err)) return false;
      if (lane == 0) mbar_arrive_cluster(mapa_rank0(b));
      __syncwarp();
      return true;
    };
    if (relay(bar(C::kKVFull), 0))
      walk_items([&](int i, int, int) { return relay(full(i), parity(i)); });
  } else {
    // ------------------------------------------------------------ compute (warps 0-7)
    const int r = static_cast<int>(threadIdx.x & 127);
    const uint32_t h = warp >> 2;
    const int key = w.k0 + r;
    const int vis_lo = key + sp.dmin - sp.off, vis_hi = key + sp.dmax - sp.off;
    const uint32_t lane_base = ((warp & 3u) * 32u) << 16;
    // h = 0 threads fetch LSE, h = 1 threads Delta, of query q0(t) + r, a tile ahead.
    float nxt = 0.f;
    auto fetch_row = [&](int t) {
      const int q = pw_q0(w, t) + r;
      if (q < sp.Lq) {
        const size_t gi = static_cast<size_t>(pw_bhq(w, a, t)) * sp.Lq + q;
        nxt = h == 0 ? a.lse[gi] : a.delta[gi];
      } else {
        nxt = h == 0 ? SWA_POS_INF : 0.f;
      }
    };
    fetch_row(0);
    bool ok = true;
    for (int t = 0; t < w.T; ++t) {
      const int q0 = pw_q0(w, t);
      float* nl2 = s_rows + (t & 1) * 2 * kBlockM;  // -LSE log2(e)
      float* nd = nl2 + kBlockM;                     // -Delta
      if (h == 0)
        nl2[r] = -nxt * kLog2e;
      else
        nd[r] = -nxt;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kVecFull + (t & 1)));
      if (!(ok = warp_wait(bar(C::kVecFull + (t & 1)), (t >> 1) & 1, &abort_flag, a.err))) break;
      if (t + 1 < w.T) fetch_row(t + 1);
      if (!(ok = warp_wait(bar(C::kSFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      float p[64];
      const int base = q0 + 64 * static_cast<int>(h);
      p_transposed(p, tmem + lane_base + C::kColS + 64u * h, nl2 + 64 * h, a.scale_log2,
                   !(q0 >= w.q_int_lo && q0 <= w.q_int_hi), vis_lo - base, vis_hi - base);
      warp_arrive_rank0(bar(C::kSEmpty));  // S^T_{t+1} may overwrite S^T_t now
      if (!(ok = warp_wait(bar(C::kDPFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      ds_transposed<F16>(tmem + lane_base + C::kColDP + 64u * h, nd + 64 * h, p);
      tmem_wait_st();
      warp_arrive_rank0(bar(C::kDSFull));
    }
    if (ok && warp_wait(bar(C::kDone), 0, &abort_flag, a.err) && w.valid) {
      tc_fence_after();
      // dK * scale -> 16-bit, staged in the K buffer (every MMA of the pair has completed).
      key_epilogue<F16>(tmem + lane_base + C::kColAcc, sK, r, h, a.scale, false, bar(C::kOutFull),
                        &tm_dk, w.k0, w.bhk, &abort_flag, a.err);
    }
  }

  tc_fence_before();
  cluster_sync_all();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

template <bool F16>
cudaError_t launch_t(const Problem& pb, const void* q, const void* k, const void* v,
                     const void* dO, const float* lse, const float* delta, void* dk, void* dv,
                     cudaStream_t stream) {
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq;
  const uint64_t bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  const int Lq = pb.span.Lq, Lk = pb.span.Lk;
  CUtensorMap tq64, tdo64, tq128, tdo128, tk, tv, tdk, tdv;
  if (!make_tmap_3d(&tq64, q, bhq, Lq, kD, kHalfRows, F16) ||
      !make_tmap_3d(&tdo64, dO, bhq, Lq, kD, kHalfRows, F16) ||
      !make_tmap_3d(&tq128, q, bhq, Lq, kD, kBlockM, F16) ||
      !make_tmap_3d(&tdo128, dO, bhq, Lq, kD, kBlockM, F16) ||
      !make_tmap_3d(&tk, k, bhk, Lk, kD, kBlockN, F16) ||
      !make_tmap_3d(&tv, v, bhk, Lk, kD, kBlockN, F16) ||
      !make_tmap_3d(&tdk, dk, bhk, Lk, kD, kBlockN, F16) ||
      !make_tmap_3d(&tdv, dv, bhk, Lk, kD, kBlockN, F16))
    return cudaErrorInvalidValue;
  PairArgs a;
  a.lse = lse;
  a.delta = delta;
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.G = pb.Hq / pb.Hkv;
  a.BHK = pb.B * pb.Hkv;
  a.span = pb.span;
  a.scale = pb.scale;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  const int nkb = (Lk + kBlockN - 1) / kBlockN;
  const unsigned grid = 2u * static_cast<unsigned>((nkb + 1) / 2) * static_cast<unsigned>(a.BHK);
  auto kk = swa_dk256_pair_kernel<F16>;
  cudaError_t e = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       KP::kSmemBytes);
  if (e != cudaSuccess) return e;
  kk<<<grid, KP::kThreads, KP::kSmemBytes, stream>>>(tq64, tdo64, tq128, tk, tv, tdk, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto kv = swa_dv256_pair_kernel<F16>;
  e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, VP::kSmemBytes);
  if (e != cudaSuccess) return e;
  kv<<<grid, VP::kThreads, VP::kSmemBytes, stream>>>(tq64, tdo128, tk, tdv, a);
  return cudaGetLastError();
}

}  // namespace

bool dkdv256_pair_applies(const Problem& pb) { return pb.D == 256; }

cudaError_t launch_dkdv256_pair(const Problem& pb, const void* q, const void* k, const void* v,
                                const void* dO, const float* lse, const float* delta, void* dk,
                                void* dv, cudaStream_t stream) {
  if (!dkdv256_pair_applies(pb)) return cudaErrorInvalidValue;
  return pb.f16 ? launch_t<true>(pb, q, k, v, dO, lse, delta, dk, dv, stream)
                : launch_t<false>(pb, q, k, v, dO, lse, delta, dk, dv, stream);
}

}  // namespace swa
