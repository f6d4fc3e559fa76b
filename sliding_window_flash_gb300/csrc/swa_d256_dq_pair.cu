// swa_d256_dq_pair.cu — dQ with head dimension 256 on CTA pairs (sm_103a).
//
// The same computation as the D = 256 dQ kernel of swa_d256.cu — per key block of a query tile's
// window walk
//   S = Q K_j^T,  P = exp(scale S - LSE) (window-masked),  dP = dO V_j^T,  dS = P (dP - Delta),
//   dQ += dS K_j,  and a final dQ *= scale
// ("Off NVIDIA, you fix the platform yourself", Lab 28 record, numbers entry "Attention backward
// memory": Gemma 4's sliding layers use 256-wide heads) — for an even number of query heads per kv
// head.  The two CTAs of a cluster take the query heads 2p and 2p + 1 of one kv group at the same
// query block and walk the same key blocks; rank 0 issues every MMA for both SMs as
// tcgen05.mma.cta_group::2 with M = 256, each SM computing its own 128 query rows:
//   S  = Q K^T    over D in two halves; B = keys [64 r, 64 r + 64) of the block (32 KB),
//   dP = dO V^T   likewise with the key half of V (32 KB),
//   dQ += dS K    one N = 256 product; B = head dims [128 r, 128 r + 128) of K, all keys (32 KB),
// r the CTA's rank.  The single-CTA kernel streams K twice per block as four 32 KB half-tiles plus
// two of V; here each SM takes three 32 KB items per block through the same three-slot ring.
//
// Shared memory per CTA: Q and dO of its head (64 KB each, held for the tile) and the ring.
// Warp roles (384 threads per CTA): warps 0-7 compute (two threads per row, as swa_d256.cu; the
// S-read, dS-written and dQ-read handshakes arrive on rank 0's barriers, 16 arrivals); warps 8 and
// 11 load this CTA's ring items (even / odd); warp 10 its Q and dO; warp 9 rank 0: MMA issuer for
// the pair, rank 1: relay — waits for each of its own copies in the order rank 0 consumes them and
// arrives on rank 0's matching barrier (rank 0's full barriers count its own copy and the relay).
// Ring order per tile of n key blocks: KH_0, VH_0, then per block j: KH_{j+1} (if any), KC_j,
// VH_{j+1} (if any) — KH / VH the key halves of K / V, KC the head-dim half of K.
// TMEM (each CTA, allocated for the pair): [0,128) S, [128,256) dP / dS, [256,512) dQ.
#include "swa_d256.cuh"
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

struct DqP256 {
  static constexpr int kD = 256;
  static constexpr int kTileBytes = kBlockM * kD * 2;  // Q or dO of this CTA's head: 4 chunks
  static constexpr int kChunk = kBlockM * 128;         // 128 rows x 64 columns
  static constexpr int kHalfRows = kBlockN / 2;
  static constexpr int kHalfChunk = kHalfRows * 128;   // 64 rows x 64 columns
  static constexpr int kItemBytes = 32768;             // one ring item
  static constexpr int kSlots = 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffRing = kOffDO + kTileBytes;
  static constexpr int kOffBar = kOffRing + kSlots * kItemBytes;
  static constexpr int kQDFull = 0;
  static constexpr int kQDEmpty = 1;
  static constexpr int kFull = 2;
  static constexpr int kEmpty = kFull + kSlots;
  static constexpr int kSFull = kEmpty + kSlots;
  static constexpr int kSEmpty = kSFull + 1;    // rank 0's: both CTAs have read S
  static constexpr int kDPFull = kSEmpty + 1;
  static constexpr int kDSFull = kDPFull + 1;   // rank 0's: both CTAs' dS written
  static constexpr int kDQDone = kDSFull + 1;
  static constexpr int kDQEmpty = kDQDone + 1;  // rank 0's: both epilogues have read dQ
  static constexpr int kDrain = kDQEmpty + 1;
  static constexpr int kNumBars = kDrain + 1;
  // + TMEM address, abort flag, and the producers' last fills ([2][kSlots] ints)
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 32;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
  static constexpr int kThreads = 384;
  static constexpr uint32_t kPairWarps = 16;
};

struct DqP256Args {
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

struct DqP256Tile {
  int bh, bhk, q0, kb_lo, nkv;
};

// Pair tile t (heaviest query blocks first); rank r takes query head 2 p + r of the kv group.
__device__ __forceinline__ DqP256Tile dqp256_tile(int t, const DqP256Args& a, const Span sp,
                                                  uint32_t rank) {
  DqP256Tile f;
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

// Ring item kinds: key half of K or V (four 64 x 64 boxes), head-dim half of K (two 128 x 64).
enum ItemKind : int { kKH = 0, kVH = 1, kKC = 2 };

template <bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    swa_dq256_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_k64,   // K, 64-row boxes
                          const __grid_constant__ CUtensorMap tm_v64,   // V, 64-row boxes
                          const __grid_constant__ CUtensorMap tm_k128,  // K, 128-row boxes
                          const DqP256Args a) {
  using C = DqP256;
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
  const uint32_t sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sRing = smem_u32(smem + C::kOffRing);
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
    mbar_init(bar(C::kQDFull), full_count);
    mbar_init(bar(C::kQDEmpty), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kFull + s), full_count);
      mbar_init(bar(C::kEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSEmpty), C::kPairWarps);
    mbar_init(bar(C::kDPFull), 1);
    mbar_init(bar(C::kDSFull), C::kPairWarps);
    mbar_init(bar(C::kDQDone), 1);
    mbar_init(bar(C::kDQEmpty), C::kPairWarps);
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

  // Walks this CTA's ring items in consumption order: on_item(index, kind, key block start,
  // kv plane); on_tile(tile iteration) before each tile's first item.
  auto walk_items = [&](auto&& on_tile, auto&& on_item) -> bool {
    int i = 0;
    for (int t = tile0, it = 0; t < a.ntiles; t += tile_step, ++it) {
      const DqP256Tile f = dqp256_tile(t, a, sp, rank);
      if (!on_tile(it)) return false;
      const int kb = f.kb_lo * kBlockN;
      if (!on_item(i++, kKH, kb, f.bhk) || !on_item(i++, kVH, kb, f.bhk)) return false;
      for (int j = 0; j < f.nkv; ++j) {
        const int k0 = (f.kb_lo + j) * kBlockN;
        if (j + 1 < f.nkv && !on_item(i++, kKH, k0 + kBlockN, f.bhk)) return false;
        if (!on_item(i++, kKC, k0, f.bhk)) return false;
        if (j + 1 < f.nkv && !on_item(i++, kVH, k0 + kBlockN, f.bhk)) return false;
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
      tma_prefetch_desc(&tm_v64);
      tma_prefetch_desc(&tm_k128);
      walk_items([&](int) { return true; },
                 [&](int i, int kind, int k0, int bhk) -> bool {
                   if ((i & 1) != p) return true;
                   if (i >= C::kSlots &&
                       !mbar_wait(empty(i), ((i / C::kSlots) - 1) & 1, &abort_flag, a.err))
                     return false;
                   const uint32_t dst = slot(i);
                   mbar_arrive_expect_tx(full(i), C::kItemBytes);
                   if (kind == kKC) {
                     for (int c = 0; c < 2; ++c)
                       tma_load_3d(dst + c * C::kChunk, &tm_k128, full(i),
                                   128 * static_cast<int>(rank) + 64 * c, k0, bhk);
                   } else {
                     const CUtensorMap* m = kind == kKH ? &tm_k64 : &tm_v64;
                     for (int c = 0; c < 4; ++c)
                       tma_load_3d(dst + c * C::kHalfChunk, m, full(i), 64 * c,
                                   k0 + C::kHalfRows * static_cast<int>(rank), bhk);
                   }
                   last[i % C::kSlots] = i;
                   return true;
                 });
    }
    d256::drain_ring<C::kSlots>(last, s_last, p, lane, full, a.err);
  } else if (warp == 10) {
    // ------------------------------------------------------------ Q and dO of each tile
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      int last = -1;
      for (int t = tile0, it = 0; t < a.ntiles; t += tile_step, ++it) {
        const DqP256Tile f = dqp256_tile(t, a, sp, rank);
        // Q / dO of the previous tile are free once its last S and dP have completed.
        if (it >= 1 && !mbar_wait(bar(C::kQDEmpty), (it - 1) & 1, &abort_flag, a.err)) break;
        mbar_arrive_expect_tx(bar(C::kQDFull), 2 * C::kTileBytes);
        for (int c = 0; c < 4; ++c) {
          tma_load_3d(sQ + c * C::kChunk, &tm_q, bar(C::kQDFull), 64 * c, f.q0, f.bh);
          tma_load_3d(sDO + c * C::kChunk, &tm_do, bar(C::kQDFull), 64 * c, f.q0, f.bh);
        }
        last = it;
      }
      if (last >= 0) drain_wait(bar(C::kQDFull), last & 1, a.err);
    }
  } else if (warp == 9 && lead) {
    // ------------------------------------------------------------ MMA issuer (the pair)
    constexpr uint32_t kIdS = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdQ = idesc_f16kind(Elem<F16>::kMmaFmt, 2 * kBlockM, C::kD, false, true);
    int i = 0;  // ring items consumed
    // d = A B^T over D, A this CTA's 64 KB tile (four 64-column chunks), B the next ring item (a
    // key half: four 64 x 64 chunks); two 8-step groups, one per 128 columns of D.
    auto product_d = [&](uint32_t d, uint32_t a_tile) -> bool {
      if (!warp_wait_cluster(full(i), parity(i), &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ss_kmajor_d<128>(d, smem_desc_sw128(a_tile, 16, 1024),
                             smem_desc_sw128(slot(i), 16, 1024), kIdS, 0u);
      umma2_ss_kmajor_d<128>(d, smem_desc_sw128(a_tile + 2 * C::kChunk, 16, 1024),
                             smem_desc_sw128(slot(i) + 2 * C::kHalfChunk, 16, 1024), kIdS, 1u);
      umma2_commit_w(empty(i));
      ++i;
      return true;
    };
    auto issue_s = [&](int gg) -> bool {  // S = Q K_gg^T once S_{gg-1} has been read
      if (gg >= 1 && !warp_wait_cluster(bar(C::kSEmpty), (gg - 1) & 1, &abort_flag, a.err))
        return false;
      if (!product_d(tmem + C::kColS, sQ)) return false;
      umma2_commit_w(bar(C::kSFull));
      return true;
    };
    auto issue_dp = [&](bool tile_last) -> bool {  // dP = dO V^T (after dQ of the previous block)
      if (!product_d(tmem + C::kColDP, sDO)) return false;
      umma2_commit_w(bar(C::kDPFull));
      if (tile_last) umma2_commit_w(bar(C::kQDEmpty));  // every S and dP of the tile is issued
      return true;
    };
    // dQ += dS K_gg: dS over the dP columns (keys 16 ks .. 16 ks + 15 at packed column
    // 8 ks + 32 (ks / 4)), B = this CTA's 128 head dims of K (two 128 x 64 chunks, MN-major).
    auto issue_dq = [&](int gg, bool first, bool tile_last) -> bool {
      if (!warp_wait_cluster(bar(C::kDSFull), gg & 1, &abort_flag, a.err)) return false;
      if (!warp_wait_cluster(full(i), parity(i), &abort_flag, a.err)) return false;
      tc_fence_after();
      umma2_ts_mnmajor_x8_split(tmem + C::kColDQ, tmem + C::kColDP,
                                smem_desc_sw128(slot(i), C::kChunk, 1024), kIdQ, first ? 0u : 1u);
      umma2_commit_w(empty(i));
      ++i;
      if (tile_last) umma2_commit_w(bar(C::kDQDone));
      return true;
    };
    int g = 0;  // key blocks issued so far by this CTA
    bool ok = true;
    for (int t = tile0, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const DqP256Tile f = dqp256_tile(t, a, sp, rank);
      const int n = f.nkv;
      ok = warp_wait_cluster(bar(C::kQDFull), it & 1, &abort_flag, a.err);
      if (ok) ok = issue_s(g);
      if (ok) ok = issue_dp(n == 1);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) ok = issue_s(g + j + 1);
        // The first dQ of a tile overwrites the accumulator: both epilogues must have read it.
        if (ok && j == 0 && it > 0)
          ok = warp_wait_cluster(bar(C::kDQEmpty), (it - 1) & 1, &abort_flag, a.err);
        if (ok) ok = issue_dq(g + j, j == 0, j + 1 == n);
        if (ok && j + 1 < n) ok = issue_dp(j + 2 == n);
      }
      g += n;
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
    walk_items([&](int it) { return relay(bar(C::kQDFull), static_cast<uint32_t>(it & 1)); },
               [&](int i, int, int, int) { return relay(full(i), parity(i)); });
  } else {
    // ------------------------------------------------------------ compute (warps 0-7)
    static_assert(C::kSEmpty - C::kSFull == d256::DqBar::kSEmpty &&
                      C::kDPFull - C::kSFull == d256::DqBar::kDPFull &&
                      C::kDSFull - C::kSFull == d256::DqBar::kDSFull &&
                      C::kDQDone - C::kSFull == d256::DqBar::kDQDone &&
                      C::kDQEmpty - C::kSFull == d256::DqBar::kDQEmpty && C::kColDP == 128 &&
                      C::kColDQ == 256,
                  "dQ compute layout");
    d256::dq_compute<F16, true>(a, sp, tmem + C::kColS, bar(C::kSFull), &abort_flag, tile0,
                                tile_step, [&](int t) { return dqp256_tile(t, a, sp, rank); });
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
cudaError_t launch_dq256_pair_t(const Problem& pb, const void* q, const void* k, const void* v,
                                const void* dO, const float* lse, const float* delta, void* dq,
                                cudaStream_t stream) {
  using C = DqP256;
  CUtensorMap tq, tdo, tk64, tv64, tk128;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_3d(&tq, q, bhq, pb.span.Lq, C::kD, kBlockM, F16) ||
      !make_tmap_3d(&tdo, dO, bhq, pb.span.Lq, C::kD, kBlockM, F16) ||
      !make_tmap_3d(&tk64, k, bhk, pb.span.Lk, C::kD, C::kHalfRows, F16) ||
      !make_tmap_3d(&tv64, v, bhk, pb.span.Lk, C::kD, C::kHalfRows, F16) ||
      !make_tmap_3d(&tk128, k, bhk, pb.span.Lk, C::kD, kBlockN, F16))
    return cudaErrorInvalidValue;
  auto kern = swa_dq256_pair_kernel<F16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  DqP256Args a;
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
  const int clusters = max_pair_clusters<swa_dq256_pair_kernel<F16>>(C::kThreads, C::kSmemBytes);
  const int nclusters = a.ntiles < clusters ? a.ntiles : clusters;
  kern<<<2 * nclusters, C::kThreads, C::kSmemBytes, stream>>>(tq, tdo, tk64, tv64, tk128, a);
  return cudaGetLastError();
}

}  // namespace

bool dq256_pair_applies(const Problem& pb) {
  return pb.D == 256 && (pb.Hq / pb.Hkv) % 2 == 0;
}

cudaError_t launch_dq256_pair(const Problem& pb, const void* q, const void* k, const void* v,
                              const void* dO, const float* lse, const float* delta, void* dq,
                              cudaStream_t stream) {
  if (!dq256_pair_applies(pb)) return cudaErrorInvalidValue;
  return pb.f16 ? launch_dq256_pair_t<true>(pb, q, k, v, dO, lse, delta, dq, stream)
                : launch_dq256_pair_t<false>(pb, q, k, v, dO, lse, delta, dq, stream);
}

}  // namespace swa
