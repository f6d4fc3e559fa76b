// swa_bwd_dq.cu — dQ of causal sliding-window attention on sm_103a.
//
// A tile is one 128-row query block of one (batch, query head).  dQ for it walks only the key
// blocks inside the tile's window (the same walk as the forward), recomputing per block
//   S = Q K_j^T,  P = exp(scale S - LSE) (window-masked),  dP = dO V_j^T,  dS = P (dP - Delta),
//   dQ += dS K_j,
// with a final dQ *= scale.  dQ accumulates in TMEM (fp32) and is initialised by the first visited
// key block rather than block zero ("Off NVIDIA, you fix the platform yourself", Lab 28, "Method and
// disclosure": a query tile's dQ starts at the first key tile it visits).  One bf16 rounding
// at the store; S and dP stay fp32 in TMEM and only dS is rounded to bf16 as an MMA operand (the
// lab's fp32-score-tile experiment showed the error of bf16 score scratch).
//
// The kernel is persistent: one CTA per SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// (heaviest first).  A tile's Q and dO are released as soon as its last dP has been computed, so
// the next tile's Q, dO and first key blocks load while the current tile finishes.
//
// Warp roles (352 threads): warps 0-7 compute — warp w handles TMEM lanes 32(w%4)..+31 (query
// rows) and columns [64 h, 64 h + 64) of every 128-column tile, h = w / 4, so each score row is
// split over two threads; warp 8 TMA producer of Q and dO (per tile) and of the K ring; warp 10
// TMA producer of the V ring; warp 9 MMA issuer and TMEM owner.  Loads are issued from two warps
// because one warp's TMA copies complete at only ~40 B/clk on this GPU, less than one key block
// (64 KB of K and V) per MMA period needs.  dS goes back to TMEM over the dP it was formed from and
// is the A operand of dQ += dS K_j.
// TMEM columns: [0,128) S, [128,384) two dP buffers, [384, 384+D) dQ.  dS_g (bf16 pairs) goes over
// the first 32 of each half-row's 64 columns of dP buffer g & 1, so dP of the next block is
// computed into the other buffer while the compute warps work on this one.
#include "swa_bwd_dq.cuh"
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

template <int D>
struct DqCfg {
  static constexpr int kTileBytes = kBlockM * D * 2;
  static constexpr int kChunkBytes = kBlockM * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kKStages = (D == 128) ? 3 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffK = kOffDO + kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * kTileBytes;
  static constexpr int kQDFull = 0;
  static constexpr int kQDEmpty = 1;
  static constexpr int kKFull = 2;
  static constexpr int kKEmpty = kKFull + kKStages;
  static constexpr int kVFull = kKEmpty + kKStages;
  static constexpr int kVEmpty = kVFull + kVStages;
  static constexpr int kSFull = kVEmpty + kVStages;
  static constexpr int kSEmpty = kSFull + 1;
  static constexpr int kDPFull = kSEmpty + 1;   // 2 (one per dP buffer)
  static constexpr int kDSFull = kDPFull + 2;   // 2 (one per dP buffer)
  static constexpr int kDQDone = kDSFull + 2;   // a tile's last dQ MMA has completed
  static constexpr int kDQEmpty = kDQDone + 1;  // the epilogue has read the dQ accumulator
  static constexpr int kDrain = kDQEmpty + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;  // + TMEM address and abort flag
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 384;  // dP buffer b at kColDP + 128 b
  static constexpr int kThreads = 352;
  static constexpr int kComputeThreads = 256;
};

struct DqArgs {
  const float* lse;
  const float* delta;
  uint16_t* dq;  // bf16 or fp16 elements
  int BH, Hq, Hkv, G, nqb, ntiles;
  Span span;
  float scale, scale_log2;
  unsigned* err;
  FastDiv divBH, divHq, divG;  // tile index decomposition
};

struct DqTile {
  int bh, bhk, q0, kb_lo, nkv;
};

// Tile t: heaviest query blocks first (the causal case gives later blocks more key blocks).
__device__ __forceinline__ DqTile dq_tile(int t, const DqArgs& a, const Span sp) {
  DqTile f;
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
__global__ void __launch_bounds__(352, 1)
    swa_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DqArgs a) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (!smem_base_ok(smem, a.err)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);  // raised by a failed wait
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sK0 = smem_u32(smem + C::kOffK);
  const uint32_t sV0 = smem_u32(smem + C::kOffV);
  const int tile_step = static_cast<int>(gridDim.x);
  const Span sp = a.span;  // window geometry, held in registers

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(C::kQDFull), 1);
    mbar_init(bar(C::kQDEmpty), 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar(C::kKFull + s), 1);
      mbar_init(bar(C::kKEmpty + s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar(C::kVFull + s), 1);
      mbar_init(bar(C::kVEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSEmpty), C::kComputeThreads / 32);
    mbar_init(bar(C::kDPFull + 0), 1);
    mbar_init(bar(C::kDPFull + 1), 1);
    mbar_init(bar(C::kDSFull + 0), C::kComputeThreads / 32);
    mbar_init(bar(C::kDSFull + 1), C::kComputeThreads / 32);
    mbar_init(bar(C::kDQDone), 1);
    mbar_init(bar(C::kDQEmpty), C::kComputeThreads / 32);
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
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      int last_qd = -1;
      int last_k[C::kKStages];
      for (int s = 0; s < C::kKStages; ++s) last_k[s] = -1;
      int g = 0;  // key blocks loaded so far by this CTA
      bool ok = true;
      for (int t = blockIdx.x, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
        const DqTile f = dq_tile(t, a, sp);
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
          const uint32_t sK = sK0 + sk * C::kTileBytes;
          mbar_arrive_expect_tx(bar(C::kKFull + sk), C::kTileBytes);
          for (int h = 0; h < C::kChunks; ++h)
            tma_load_3d(sK + h * C::kChunkBytes, &tm_k, bar(C::kKFull + sk), 64 * h, k0, f.bhk);
          last_k[sk] = g;
        }
      }
      if (last_qd >= 0) drain_wait(bar(C::kQDFull), last_qd & 1, a.err);
      for (int s = 0; s < C::kKStages; ++s)
        if (last_k[s] >= 0) drain_wait(bar(C::kKFull + s), (last_k[s] / C::kKStages) & 1, a.err);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------------ TMA producer (V ring)
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      int last_v[C::kVStages];
      for (int s = 0; s < C::kVStages; ++s) last_v[s] = -1;
      int g = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < a.ntiles; t += tile_step) {
        const DqTile f = dq_tile(t, a, sp);
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
    // Per tile: S_0, dP_0, then per block j: S_{j+1}, dP_{j+1}, dQ += dS_j K_j.  The next block's
    // S and dP are computed as soon as the compute warps have read this block's, so they never
    // wait on dQ_j.  dP_g goes into buffer g & 1, which last held dS_{g-2}: dQ_{g-2} was issued
    // before it and tcgen05.mma operations of one thread run in issue order, so no wait is needed.
    // Block counters run across tiles.
    constexpr uint32_t kIdSq = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockM, kBlockN, false, false);  // S, dP
    constexpr uint32_t kIdDq = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockM, D, false, true);         // dQ += dS K
    auto issue_s = [&](int gg) -> bool {  // S = Q K_gg^T once S_{gg-1} has been read
      const int s = gg % C::kKStages, n = gg / C::kKStages;
      if (!warp_wait(bar(C::kKFull + s), n & 1, &abort_flag, a.err)) return false;
      if (gg >= 1 && !warp_wait(bar(C::kSEmpty), (gg - 1) & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      umma_ss_kmajor_d<D>(tmem + C::kColS, smem_desc_sw128(sQ, 16, 1024),
                          smem_desc_sw128(sK0 + s * C::kTileBytes, 16, 1024), kIdSq, 0u);
      umma_commit_w(bar(C::kSFull));
      return true;
    };
    auto issue_dp = [&](int gg, bool tile_last) -> bool {  // dP = dO V_gg^T into buffer gg & 1
      const int s = gg % C::kVStages, n = gg / C::kVStages;
      if (!warp_wait(bar(C::kVFull + s), n & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      umma_ss_kmajor_d<D>(tmem + C::kColDP + 128u * (gg & 1), smem_desc_sw128(sDO, 16, 1024),
                          smem_desc_sw128(sV0 + s * C::kTileBytes, 16, 1024), kIdSq, 0u);
      umma_commit_w(bar(C::kDPFull + (gg & 1)));
      umma_commit_w(bar(C::kVEmpty + s));
      if (tile_last) umma_commit_w(bar(C::kQDEmpty));  // every S and dP of the tile is issued
      return true;
    };
    // dQ += dS_gg K_gg with dS_gg in dP buffer gg & 1: keys 16 ks .. 16 ks + 15 at packed column
    // 8 ks + 32 (ks / 4).
    auto issue_dq = [&](int gg, bool first, bool tile_last) -> bool {
      const int s = gg % C::kKStages, db = gg & 1;
      if (!warp_wait(bar(C::kDSFull + db), (gg >> 1) & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      umma_ts_mnmajor_x8_split(tmem + C::kColDQ, tmem + C::kColDP + 128u * db,
                               smem_desc_sw128(sK0 + s * C::kTileBytes, C::kChunkBytes, 1024),
                               kIdDq, first ? 0u : 1u);
      umma_commit_w(bar(C::kKEmpty + s));
      if (tile_last) umma_commit_w(bar(C::kDQDone));
      return true;
    };
    int g = 0;  // key blocks issued so far by this CTA
    bool ok = true;
    for (int t = blockIdx.x, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const DqTile f = dq_tile(t, a, sp);
      const int n = f.nkv;
      ok = warp_wait(bar(C::kQDFull), it & 1, &abort_flag, a.err);
      if (ok) ok = issue_s(g);
      if (ok) ok = issue_dp(g, n == 1);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          ok = issue_s(g + j + 1);
          if (ok) ok = issue_dp(g + j + 1, j + 2 == n);
        }
        // The first dQ of a tile overwrites the accumulator: the previous tile's epilogue must
        // have read it.
        if (ok && j == 0 && it > 0)
          ok = warp_wait(bar(C::kDQEmpty), (it - 1) & 1, &abort_flag, a.err);
        if (ok) ok = issue_dq(g + j, j == 0, j + 1 == n);
      }
      g += n;
    }
    umma_commit_w(bar(C::kDrain));
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else {
    // ------------------------------------------------------------------ compute (warps 0-7)
    static_assert(C::kSEmpty - C::kSFull == dqc::DqBar::kSEmpty &&
                      C::kDPFull - C::kSFull == dqc::DqBar::kDPFull &&
                      C::kDSFull - C::kSFull == dqc::DqBar::kDSFull &&
                      C::kDQDone - C::kSFull == dqc::DqBar::kDQDone &&
                      C::kDQEmpty - C::kSFull == dqc::DqBar::kDQEmpty && C::kColS == dqc::kColS &&
                      C::kColDP == dqc::kColDP && C::kColDQ == dqc::kColDQ,
                  "dQ compute layout");
    dqc::dq_compute<D, F16, false>(a, sp, tmem, bar(C::kSFull), &abort_flag,
                                   static_cast<int>(blockIdx.x), tile_step,
                                   [&](int t) { return dq_tile(t, a, sp); });
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool F16>
cudaError_t launch_dq_d(const Problem& pb, const void* q, const void* k, const void* v,
                        const void* dO, const float* lse, const float* delta, void* dq,
                        cudaStream_t stream) {
  using C = DqCfg<D>;
  CUtensorMap tq, tdo, tk, tv;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_3d(&tq, q, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tdo, dO, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tk, k, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tv, v, bhk, pb.span.Lk, D, kBlockN, F16))
    return cudaErrorInvalidValue;
  auto kern = swa_dq_kernel<D, F16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  DqArgs a;
  a.lse = lse;
  a.delta = delta;
  a.dq = static_cast<uint16_t*>(dq);
  a.BH = pb.B * pb.Hq;
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.G = pb.Hq / pb.Hkv;
  a.span = pb.span;
  a.nqb = (pb.span.Lq + kBlockM - 1) / kBlockM;
  a.ntiles = a.nqb * a.BH;
  a.scale = pb.scale;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  a.divBH = FastDiv(static_cast<uint32_t>(a.BH));
  a.divHq = FastDiv(static_cast<uint32_t>(a.Hq));
  a.divG = FastDiv(static_cast<uint32_t>(a.G));
  const int grid = a.ntiles < sm_count() ? a.ntiles : sm_count();
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tdo, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const Problem& pb, const void* q, const void* k, const void* v,
                          const void* dO, const float* lse, const float* delta, void* dq,
                          cudaStream_t stream) {
  if (pb.D == 256) return launch_dq_d256(pb, q, k, v, dO, lse, delta, dq, stream);
  if (dq_pair_applies(pb)) return launch_dq_pair(pb, q, k, v, dO, lse, delta, dq, stream);
  if (pb.D == 64)
    return pb.f16 ? launch_dq_d<64, true>(pb, q, k, v, dO, lse, delta, dq, stream)
                  : launch_dq_d<64, false>(pb, q, k, v, dO, lse, delta, dq, stream);
  if (pb.D == 128)
    return pb.f16 ? launch_dq_d<128, true>(pb, q, k, v, dO, lse, delta, dq, stream)
                  : launch_dq_d<128, false>(pb, q, k, v, dO, lse, delta, dq, stream);
  return cudaErrorInvalidValue;
}

}  // namespace swa
