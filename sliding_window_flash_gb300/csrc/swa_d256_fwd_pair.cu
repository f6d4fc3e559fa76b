// swa_d256_fwd_pair.cu — forward with head dimension 256 on CTA pairs (sm_103a).
//
// The same computation as the D = 256 forward of swa_d256.cu — per 128-row query tile,
// O = softmax(scale Q K^T, window mask) V and the natural-log LSE, over the key blocks the window
// reaches ("Off NVIDIA, you fix the platform yourself", Lab 28 record, numbers entry "Attention
// backward memory": Gemma 4's sliding layers use 256-wide heads) — for an even number of query
// heads per kv head.  The two CTAs of a cluster take the query heads 2p and 2p + 1 of one kv group
// at the same query block; rank 0 issues every MMA for both SMs as tcgen05.mma.cta_group::2 with
// M = 256, each SM computing its own 128 query rows:
//   S = Q K^T     over D in two halves; B = keys [64 r, 64 r + 64) of the block (32 KB),
//   O += P V      one N = 256 product; B = head dims [128 r, 128 r + 128) of V, all keys (32 KB),
// r the CTA's rank.  The single-CTA kernel moves four 32 KB half-tiles per key block through its
// five-slot ring; here each SM moves two, so the same ring runs twice as many blocks ahead.
//
// Warp roles (384 threads per CTA): warps 0-7 softmax (as swa_d256.cu: two threads per row, the
// halves swapping block sums and maxima through shared memory; the P-written and O-read
// handshakes arrive on rank 0's barriers, 16 arrivals); warps 8 and 11 load this CTA's ring items
// (even / odd); warp 10 loads each tile's Q and stores its O (staged in the Q buffer once every S
// of the tile has completed); warp 9 rank 0: MMA issuer for the pair, rank 1: relay — waits for
// each of its own copies in the order rank 0 consumes them and arrives on rank 0's matching
// barrier (rank 0's full barriers count its own copy and the relay).
// Ring order per tile of n key blocks: KH_0, then per block j: KH_{j+1} (if any), VC_j — KH the key
// half of K, VC the head-dim half of V.
// TMEM (each CTA, allocated for the pair): [0,128) S / P buffer 0, [128,256) S / P buffer 1,
// [256,512) O.
#include "swa_d256.cuh"
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

struct FwdP256 {
  static constexpr int kD = 256;
  static constexpr int kTileBytes = kBlockM * kD * 2;  // Q of this CTA's head: 4 chunks
  static constexpr int kChunk = kBlockM * 128;         // 128 rows x 64 columns
  static constexpr int kHalfRows = kBlockN / 2;
  static constexpr int kHalfChunk = kHalfRows * 128;   // 64 rows x 64 columns
  static constexpr int kItemBytes = 32768;
  static constexpr int kSlots = 5;
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kOffQ + kTileBytes;
  static constexpr int kOffRed = kOffRing + kSlots * kItemBytes;  // [2 slots][2 halves][128] fp32
  static constexpr int kOffBar = kOffRed + 2 * 2 * kBlockM * 4;
  static constexpr int kQFull = 0;
  static constexpr int kFull = 1;
  static constexpr int kEmpty = kFull + kSlots;
  static constexpr int kSFull = kEmpty + kSlots;  // 2
  static constexpr int kPFull = kSFull + 2;       // 2, rank 0's: both CTAs' P written
  static constexpr int kPVDone = kPFull + 2;      // 2
  static constexpr int kXch = kPVDone + 2;        // [4 lane quarters][2 slots]
  static constexpr int kOEmpty = kXch + 8;        // rank 0's: both CTAs have read O
  static constexpr int kOutFull = kOEmpty + 1;    // staged O tile complete
  static constexpr int kDrain = kOutFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  // + TMEM address, abort flag, and the producers' last fills ([2][kSlots] ints)
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 48;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kColS = 0, kColO = 256;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kPairWarps = 16;
};

struct FwdP256Args {
  float* lse;
  int BHKP;  // B * Hkv * G / 2: head pairs per query block
  int Hq, Hkv, G, nqb, ntiles;
  Span span;
  float scale_log2;
  unsigned* err;
  FastDiv divBHKP, divGP, divHkv;  // tile index decomposition (divGP: G / 2)
};

struct FwdP256Tile {
  int bh, bhk, q0, kb_lo, nkv;
};

// Pair tile t (heaviest query blocks first); rank r takes query head 2 p + r of the kv group.
__device__ __forceinline__ FwdP256Tile fwdp256_tile(int t, const FwdP256Args& a, const Span sp,
                                                    uint32_t rank) {
  FwdP256Tile f;
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

template <bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    swa_fwd256_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k64,   // K, 64-row boxes
                           const __grid_constant__ CUtensorMap tm_v128,  // V, 128-row boxes
                           const __grid_constant__ CUtensorMap tm_o, const FwdP256Args a) {
  using C = FwdP256;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  // Both CTAs always reach the cluster barriers and the collective TMEM allocation; a misaligned
  // window only disables the work (and is reported).
  const bool smem_ok = (smem_u32(smem) & 1023u) == 0u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 4);  // [2][kSlots]: producers' last fills
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sRing = smem_u32(smem + C::kOffRing);
  float* s_red = reinterpret_cast<float*>(smem + C::kOffRed);
  auto slot = [&](int i) { return sRing + (i % C::kSlots) * C::kItemBytes; };
  auto full = [&](int i) { return bar(C::kFull + i % C::kSlots); };
  auto empty = [&](int i) { return bar(C::kEmpty + i % C::kSlots); };
  auto parity = [&](int i) { return static_cast<uint32_t>((i / C::kSlots) & 1); };
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
    mbar_init(bar(C::kQFull), full_count);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kFull + s), full_count);
      mbar_init(bar(C::kEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kSFull + b), 1);
      mbar_init(bar(C::kPFull + b), C::kPairWarps);
      mbar_init(bar(C::kPVDone + b), 1);
    }
    for (int x = 0; x < 8; ++x) mbar_init(bar(C::kXch + x), 2);  // the two warps of a quarter
    mbar_init(bar(C::kOEmpty), C::kPairWarps);
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

  // This CTA's ring items in consumption order: on_item(index, is V, key block start, kv plane);
  // on_tile(tile iteration) before each tile's first item.
  auto walk_items = [&](auto&& on_tile, auto&& on_item) -> bool {
    int i = 0;
    for (int t = tile0, it = 0; t < a.ntiles; t += tile_step, ++it) {
      const FwdP256Tile f = fwdp256_tile(t, a, sp, rank);
      if (!on_tile(it)) return false;
      if (!on_item(i++, false, f.kb_lo * kBlockN, f.bhk)) return false;
      for (int j = 0; j < f.nkv; ++j) {
        const int k0 = (f.kb_lo + j) * kBlockN;
        if (j + 1 < f.nkv && !on_item(i++, false, k0 + kBlockN, f.bhk)) return false;
        if (!on_item(i++, true, k0, f.bhk)) return false;
      }
    }
    return true;
  };

  if (!smem_ok) {
    // nothing to do: fall through to the final barrier and the collective release
  } else if (warp == 8 || warp == 11) {
    // ------------------------------------------------------------ ring items (even / odd)
    const int p = warp == 8 ? 0 : 1;
    int last[C::kSlots];  // lane 0: last item loaded per slot
    for (int s = 0; s < C::kSlots; ++s) last[s] = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_k64);
      tma_prefetch_desc(&tm_v128);
      walk_items([&](int) { return true; },
                 [&](int i, bool is_v, int k0, int bhk) -> bool {
                   if ((i & 1) != p) return true;
                   if (i >= C::kSlots &&
                       !mbar_wait(empty(i), ((i / C::kSlots) - 1) & 1, &abort_flag, a.err))
                     return false;
                   const uint32_t dst = slot(i);
                   mbar_arrive_expect_tx(full(i), C::kItemBytes);
                   if (is_v) {
                     for (int c = 0; c < 2; ++c)
                       tma_load_3d(dst + c * C::kChunk, &tm_v128, full(i),
                                   128 * static_cast<int>(rank) + 64 * c, k0, bhk);
                   } else {
                     for (int c = 0; c < 4; ++c)
                       tma_load_3d(dst + c * C::kHalfChunk, &tm_k64, full(i), 64 * c,
                                   k0 + C::kHalfRows * static_cast<int>(rank), bhk);
                   }
                   last[i % C::kSlots] = i;
                   return true;
                 });
    }
    d256::drain_ring<C::kSlots>(last, s_last, p, lane, full, a.err);
  } else if (warp == 10) {
    // ------------------------------------------------------------ Q loads, O stores
    auto load_q = [&](int t) {
      const FwdP256Tile f = fwdp256_tile(t, a, sp, rank);
      mbar_arrive_expect_tx(bar(C::kQFull), C::kTileBytes);
      for (int c = 0; c < 4; ++c)
        tma_load_3d(sQ + c * C::kChunk, &tm_q, bar(C::kQFull), 64 * c, f.q0, f.bh);
    };
    int last_q = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_o);
      if (tile0 < a.ntiles) {
        load_q(tile0);
        last_q = 0;
      }
    }
    for (int t = tile0, it = 0; t < a.ntiles; t += tile_step, ++it) {
      if (!warp_wait(bar(C::kOutFull), it & 1, &abort_flag, a.err)) break;
      if (lane == 0) {
        const FwdP256Tile f = fwdp256_tile(t, a, sp, rank);
        for (int c = 0; c < 4; ++c) tma_store_3d(&tm_o, sQ + c * C::kChunk, 64 * c, f.q0, f.bh);
        bulk_commit_group();
        bulk_wait_group_read0();  // the Q buffer may be refilled once the store has read it
        if (t + tile_step < a.ntiles) {
          load_q(t + tile_step);
          last_q = it + 1;
        }
      }
      __syncwarp();
    }
    if (lane == 0 && last_q >= 0) drain_wait(bar(C::kQFull), last_q & 1, a.err);
  } else if (warp == 9 && lead) {
    // ------------------------------------------------------------ MMA issuer (the pair)
    constexpr uint32_t kIdS = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdO = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockM, C::kD, false, true);
    int i = 0;  // ring items consumed
    // S_gg = Q K_gg^T into S buffer gg & 1 (over D in two 8-step groups).  That buffer last held
    // P_{gg-2}, whose P V was issued before this.
    auto issue_s = [&](int gg) -> bool {
      if (!warp_wait_cluster(full(i), parity(i), &abort_flag, a.err)) return false;
      tc_fence_after();
      const uint32_t d = tmem + C::kColS + 128u * (gg & 1);
      umma2_ss_kmajor_d<128>(d, smem_desc_sw128(sQ, 16, 1024), smem_desc_sw128(slot(i), 16, 1024),
                             kIdS, 0u);
      umma2_ss_kmajor_d<128>(d, smem_desc_sw128(sQ + 2 * C::kChunk, 16, 1024),
                             smem_desc_sw128(slot(i) + 2 * C::kHalfChunk, 16, 1024), kIdS, 1u);
      umma2_commit_w(empty(i));
      ++i;
      umma2_commit_w(bar(C::kSFull + (gg & 1)));
      return true;
    };
    // O (+)= P_gg V_gg: P packed over S buffer gg & 1 (keys 16 ks .. 16 ks + 15 at packed column
    // 8 ks + 32 (ks / 4)), B = this CTA's 128 head dims of V (two 128 x 64 chunks, MN-major).
    auto issue_pv = [&](int gg, bool first) -> bool {
      const int pb = gg & 1;
      if (!warp_wait_cluster(bar(C::kPFull + pb), (gg >> 1) & 1, &abort_flag, a.err)) return false;
      if (!warp_wait_cluster(full(i), parity(i), &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ts_mnmajor_x8_split(tmem + C::kColO, tmem + C::kColS + 128u * pb,
                                smem_desc_sw128(slot(i), C::kChunk, 1024), kIdO, first ? 0u : 1u);
      umma2_commit_w(empty(i));
      ++i;
      umma2_commit_w(bar(C::kPVDone + pb));
      return true;
    };
    int g = 0;
    bool ok = true;
    for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const FwdP256Tile f = fwdp256_tile(t, a, sp, rank);
      ok = warp_wait_cluster(bar(C::kQFull), it & 1, &abort_flag, a.err);
      if (ok) ok = issue_s(g);
      for (int j = 0; ok && j < f.nkv; ++j) {
        if (j + 1 < f.nkv) ok = issue_s(g + j + 1);
        // The first P V of a tile overwrites O: both CTAs' epilogues must have read it.
        if (ok && j == 0 && it > 0)
          ok = warp_wait_cluster(bar(C::kOEmpty), (it - 1) & 1, &abort_flag, a.err);
        if (ok) ok = issue_pv(g + j, j == 0);
      }
      g += f.nkv;
    }
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
    walk_items([&](int it) { return relay(bar(C::kQFull), static_cast<uint32_t>(it & 1)); },
               [&](int i, bool, int, int) { return relay(full(i), parity(i)); });
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    static_assert(C::kPFull - C::kSFull == d256::FwdBar::kPFull &&
                      C::kPVDone - C::kSFull == d256::FwdBar::kPVDone &&
                      C::kXch - C::kSFull == d256::FwdBar::kXch &&
                      C::kOEmpty - C::kSFull == d256::FwdBar::kOEmpty &&
                      C::kOutFull - C::kSFull == d256::FwdBar::kOutFull,
                  "softmax barrier layout");
    const d256::FwdSoftmax cx{tmem + C::kColS, sQ,        s_red,      bar(C::kSFull),
                              &abort_flag,     a.err,     a.scale_log2, a.lse};
    d256::fwd_softmax<F16, true>(cx, sp, tile0, tile_step, a.ntiles,
                                 [&](int t) { return fwdp256_tile(t, a, sp, rank); });
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

template <bool F16>
cudaError_t launch_fwd256_pair_t(const Problem& pb, const void* q, const void* k, const void* v,
                                 void* o, float* lse, cudaStream_t stream) {
  using C = FwdP256;
  CUtensorMap tq, to, tk64, tv128;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_3d(&tq, q, bhq, pb.span.Lq, C::kD, kBlockM, F16) ||
      !make_tmap_3d(&to, o, bhq, pb.span.Lq, C::kD, kBlockM, F16) ||
      !make_tmap_3d(&tk64, k, bhk, pb.span.Lk, C::kD, C::kHalfRows, F16) ||
      !make_tmap_3d(&tv128, v, bhk, pb.span.Lk, C::kD, kBlockN, F16))
    return cudaErrorInvalidValue;
  auto kern = swa_fwd256_pair_kernel<F16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  FwdP256Args a;
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
  const int clusters = max_pair_clusters<swa_fwd256_pair_kernel<F16>>(C::kThreads, C::kSmemBytes);
  const int nclusters = a.ntiles < clusters ? a.ntiles : clusters;
  kern<<<2 * nclusters, C::kThreads, C::kSmemBytes, stream>>>(tq, tk64, tv128, to, a);
  return cudaGetLastError();
}

}  // namespace

bool fwd256_pair_applies(const Problem& pb) {
  return pb.D == 256 && (pb.Hq / pb.Hkv) % 2 == 0;
}

cudaError_t launch_fwd256_pair(const Problem& pb, const void* q, const void* k, const void* v,
                               void* o, float* lse, cudaStream_t stream) {
  if (!fwd256_pair_applies(pb)) return cudaErrorInvalidValue;
  return pb.f16 ? launch_fwd256_pair_t<true>(pb, q, k, v, o, lse, stream)
                : launch_fwd256_pair_t<false>(pb, q, k, v, o, lse, stream);
}

}  // namespace swa
