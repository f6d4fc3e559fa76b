// swa_bwd_fused.cu — dK, dV and dQ of sliding-window attention in one pass over the key blocks, on
// sm_103a.
//
// One CTA owns one 128-row key block of one (batch, kv head) and walks, for each of the G query
// heads of the group, the query blocks inside the block's window, as the dK/dV kernel does
// ("Off NVIDIA, you fix the platform yourself", Lab 28, "What did fixing it take?": tiles wholly
// outside the window are skipped, edge tiles are masked, dK / dV of a key tile no query visits are
// written as zeros).  Per (query head, query block) tile it computes
//   S^T = K Q^T,  P^T = exp(scale S^T - LSE),  dV += P^T dO,  dP^T = V dO^T,
//   dS^T = P^T (dP^T - Delta),  dK += dS^T Q,  dQ_tile = dS K,
// so the backward's five contractions run once each; the split backward's dQ kernel recomputes S
// and dP, seven per tile.  dK and dV accumulate in TMEM across the group (the grouped-query
// reduction, no atomics), as in the dK/dV kernel.  A query block's dQ gets one partial per key
// block of its window; each partial (fp32) is added into a caller-owned fp32 accumulator with
// vector reduce-adds at the L2, and a small kernel scales and rounds the sum (swa_bwd_dq_acc.cu).
// The order of those fp32 additions varies between runs, so dQ is not bit-reproducible on this
// path; dK and dV are (the split path stays the deterministic option).
//
// Warp roles (352 threads): warps 0-7 compute — warp w handles TMEM lanes 32(w%4)..+31 and columns
// [64 h, 64 h + 64) of every 128-column tile, h = w / 4; warp 8 TMA producer of K (once) and of the
// Q ring; warp 10 TMA producer of V (once) and of the dO ring; warp 9 MMA issuer and TMEM owner.
//
// TMEM (512 columns): A = [0,128) holds S^T, then P^T (each half-row thread packs its 64 P values
// as bf16 pairs into the first 32 of its 64 columns), the A operand of dV += P^T dO;
// B = [128,256) holds dP^T, then the tile's dQ partial (lanes = query rows, D fp32 columns);
// [256, 256+D) dK, [256+D, 256+2D) dV.
// Shared memory: K, V, a ring of Q tiles, a ring of two dO tiles, the per-query LSE / Delta slots.
// dS^T (bf16, rows = keys, 128 query columns in two 64-column swizzled chunks) is written over the
// tile's own dO slot once dV has read it (D = 128, where a dO tile is exactly dS^T's 32 KB; D = 64
// has its own dS^T buffer); it is the K-major A operand of dK += dS^T Q and, read MN-major, the
// A operand of dQ = dS K.  The compute warps read a tile's dQ partial out of TMEM (each thread its
// half-row, which frees B for the next dP^T at once) and add it into the accumulator straight from
// registers with 16-byte vector reduce-adds; the accumulator's layout makes one warp's reduce-add
// (4 columns of 32 consecutive rows) a contiguous 512-byte span, so the L2 works on whole sectors.
// A Q slot is free once dK has read it, a dO slot once dQ has completed (dS^T may sit there).
//
// MMA issue order (steady state): dK_t, dQ_t, dV_{t+1}, dP_{t+1}, S_{t+2}.  S_{t+2} overwrites A
// after dV_{t+1} has read P_{t+1}; dQ_t overwrites B after the compute warps have read dP_t (dS_t
// depends on it); dP_{t+1} waits until they have read dQ_t out.  One thread's tcgen05.mma
// operations run in issue order.
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

template <int D>
struct FusedCfg {
  static constexpr int kTileBytes = kBlockM * D * 2;      // Q, dO, K, V tiles (16-bit elements)
  static constexpr int kChunkBytes = kBlockM * 128;       // one 64-column chunk of a 128-row tile
  static constexpr int kChunks = D / 64;
  static constexpr int kDSBytes = kBlockN * kBlockM * 2;  // dS^T: 128 keys x 128 queries, 16-bit
  static constexpr int kDSChunkBytes = kBlockN * 128;     // one 64-query chunk of dS^T
  static constexpr int kQStages = (D == 128) ? 3 : 4;
  static constexpr int kDOStages = 2;
  static constexpr bool kDSInDO = (kTileBytes == kDSBytes);
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kDOStages * kTileBytes;  // own buffer unless kDSInDO
  static constexpr int kOffRow = kOffDS + (kDSInDO ? 0 : kDSBytes);
  static constexpr int kOffBar = kOffRow + 2 * 2 * kBlockM * 4;  // two {lse2, delta} slots
  // barriers
  static constexpr int kKVFull = 0;
  static constexpr int kQFull = 1;
  static constexpr int kDOFull = kQFull + kQStages;
  static constexpr int kQEmpty = kDOFull + kDOStages;  // per Q slot: dK has read it
  static constexpr int kSFull = kQEmpty + kQStages;
  static constexpr int kPFull = kSFull + 1;
  static constexpr int kDPFull = kPFull + 1;
  static constexpr int kDVDone = kDPFull + 1;
  static constexpr int kDSFull = kDVDone + 1;
  static constexpr int kBFree = kDSFull + 1;
  static constexpr int kDQDone = kBFree + 1;  // 2 (tile parity)
  static constexpr int kVecFull = kDQDone + 2;  // 2 slots
  static constexpr int kDone = kVecFull + 2;
  static constexpr int kOutFull = kDone + 1;
  static constexpr int kDrain = kOutFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;  // + TMEM address, abort flag
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColA = 0, kColB = 128, kColDK = 256, kColDV = 256 + D;
  static constexpr int kThreads = 352;
  static constexpr int kComputeThreads = 256;
};

struct FusedArgs {
  const float* lse;
  const float* delta;
  float* dq_acc;  // fp32 accumulator, tile-major (see swa_kernels.h: dq_acc_offset)
  uint16_t* dk;   // bf16 or fp16 elements
  uint16_t* dv;
  int BHK, Hq, Hkv, G, nqb;
  Span span;
  float scale, scale_log2;
  unsigned* err;
};

template <int D, bool F16>
__global__ void __launch_bounds__(352, 1)
    swa_fused_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_dk,
                         const __grid_constant__ CUtensorMap tm_dv, const FusedArgs a) {
  using C = FusedCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (!smem_base_ok(smem, a.err)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  float* s_rows = reinterpret_cast<float*>(smem + C::kOffRow);  // [slot][lse2 | delta][128]
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);  // raised by a failed wait
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const uint32_t sQ0 = smem_u32(smem + C::kOffQ);
  const uint32_t sDO0 = smem_u32(smem + C::kOffDO);
  auto q_slot = [&](int t) { return sQ0 + static_cast<uint32_t>(t % C::kQStages) * C::kTileBytes; };
  auto do_slot = [&](int t) { return sDO0 + static_cast<uint32_t>(t % C::kDOStages) * C::kTileBytes; };
  auto ds_tile = [&](int t) {
    return C::kDSInDO ? do_slot(t) : smem_u32(smem + C::kOffDS);
  };

  const int kb = static_cast<int>(blockIdx.x) / a.BHK;
  const int bhk = static_cast<int>(blockIdx.x) % a.BHK;
  const int b = bhk / a.Hkv, hk = bhk % a.Hkv;
  const int k0 = kb * kBlockN;
  const Span sp = a.span;
  const int qb_lo = sp.first_qblock(k0);
  const int qb_hi = sp.last_qblock(k0);
  const int nq = qb_hi >= qb_lo ? qb_hi - qb_lo + 1 : 0;
  const int T = a.G * nq;  // (query head, query block) tiles of the walk
  const int q_int_lo = k0 + kBlockN - 1 + sp.dmin - sp.off;
  const int q_int_hi = (k0 + kBlockN <= sp.Lk)
                           ? min(k0 + sp.dmax - sp.off - (kBlockM - 1), sp.Lq - kBlockM)
                           : -1;
  auto tile_qb = [&](int t) { return qb_lo + t % nq; };
  auto tile_q0 = [&](int t) { return tile_qb(t) * kBlockM; };
  auto tile_bhq = [&](int t) { return b * a.Hq + hk * a.G + t / nq; };

  if (T == 0) {
    // No query sees this key block: dK = dV = 0 and no dQ partial.
    zero_key_rows(a.dk, a.dv, bhk, k0, sp.Lk, D);
    return;
  }

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(C::kKVFull), 2);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(bar(C::kQFull + s), 1);
      mbar_init(bar(C::kQEmpty + s), 1);
    }
    for (int s = 0; s < C::kDOStages; ++s) mbar_init(bar(C::kDOFull + s), 1);
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kPFull), C::kComputeThreads / 32);
    mbar_init(bar(C::kDPFull), 1);
    mbar_init(bar(C::kDVDone), 1);
    mbar_init(bar(C::kDSFull), C::kComputeThreads / 32);
    mbar_init(bar(C::kBFree), C::kComputeThreads / 32);
    mbar_init(bar(C::kDQDone + 0), 1);
    mbar_init(bar(C::kDQDone + 1), 1);
    mbar_init(bar(C::kVecFull + 0), C::kComputeThreads / 32);
    mbar_init(bar(C::kVecFull + 1), C::kComputeThreads / 32);
    mbar_init(bar(C::kDone), 1);
    mbar_init(bar(C::kOutFull), C::kComputeThreads / 32);
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
    // ------------------------------------------------------- TMA producer (K, Q ring)
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(bar(C::kKVFull), C::kTileBytes);
      for (int h = 0; h < C::kChunks; ++h)
        tma_load_3d(sK + h * C::kChunkBytes, &tm_k, bar(C::kKVFull), 64 * h, k0, bhk);
      int last_q[C::kQStages];
      for (int s = 0; s < C::kQStages; ++s) last_q[s] = -1;
      for (int t = 0; t < T; ++t) {
        const int sq = t % C::kQStages, nqs = t / C::kQStages;
        if (t >= C::kQStages && !mbar_wait(bar(C::kQEmpty + sq), (nqs - 1) & 1, &abort_flag, a.err))
          break;
        mbar_arrive_expect_tx(bar(C::kQFull + sq), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(q_slot(t) + h * C::kChunkBytes, &tm_q, bar(C::kQFull + sq), 64 * h,
                      tile_q0(t), tile_bhq(t));
        last_q[sq] = t;
      }
      drain_wait(bar(C::kKVFull), 0, a.err);
      for (int s = 0; s < C::kQStages; ++s)
        if (last_q[s] >= 0) drain_wait(bar(C::kQFull + s), (last_q[s] / C::kQStages) & 1, a.err);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------- TMA producer (V, dO ring)
    if (lane == 0) {
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(C::kKVFull), C::kTileBytes);
      for (int h = 0; h < C::kChunks; ++h)
        tma_load_3d(sV + h * C::kChunkBytes, &tm_v, bar(C::kKVFull), 64 * h, k0, bhk);
      int last_do[C::kDOStages];
      for (int s = 0; s < C::kDOStages; ++s) last_do[s] = -1;
      for (int t = 0; t < T; ++t) {
        const int sd = t % C::kDOStages;
        // The slot's previous tile t - 2 is done with it once its dQ has completed (its dS^T may
        // live there, read by dK and dQ).
        if (t >= C::kDOStages &&
            !mbar_wait(bar(C::kDQDone + (t & 1)), ((t - 2) >> 1) & 1, &abort_flag, a.err))
          break;
        mbar_arrive_expect_tx(bar(C::kDOFull + sd), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(do_slot(t) + h * C::kChunkBytes, &tm_do, bar(C::kDOFull + sd), 64 * h,
                      tile_q0(t), tile_bhq(t));
        last_do[sd] = t;
      }
      drain_wait(bar(C::kKVFull), 0, a.err);
      for (int s = 0; s < C::kDOStages; ++s)
        if (last_do[s] >= 0)
          drain_wait(bar(C::kDOFull + s), (last_do[s] / C::kDOStages) & 1, a.err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------- MMA issuer
    constexpr uint32_t fmt = Elem<F16>::kMmaFmt;
    constexpr uint32_t kIdS = idesc_f16kind(fmt, kBlockN, kBlockM, false, false);  // S^T, dP^T
    constexpr uint32_t kIdAcc = idesc_f16kind(fmt, kBlockN, D, false, true);       // dV, dK
    constexpr uint32_t kIdDq = idesc_f16kind(fmt, kBlockM, D, true, true);         // dQ = dS K
    auto issue_s = [&](int t) -> bool {  // S^T = K Q_t^T into A
      if (!warp_wait(bar(C::kQFull + t % C::kQStages), (t / C::kQStages) & 1, &abort_flag, a.err))
        return false;
      tc_fence_after();
      umma_ss_kmajor_d<D>(tmem + C::kColA, smem_desc_sw128(sK, 16, 1024),
                          smem_desc_sw128(q_slot(t), 16, 1024), kIdS, 0u);
      umma_commit_w(bar(C::kSFull));
      return true;
    };
    auto issue_dp = [&](int t) -> bool {  // dP^T = V dO_t^T into B
      if (!warp_wait(bar(C::kDOFull + t % C::kDOStages), (t / C::kDOStages) & 1, &abort_flag,
                     a.err))
        return false;
      tc_fence_after();
      umma_ss_kmajor_d<D>(tmem + C::kColB, smem_desc_sw128(sV, 16, 1024),
                          smem_desc_sw128(do_slot(t), 16, 1024), kIdS, 0u);
      umma_commit_w(bar(C::kDPFull));
      return true;
    };
    auto issue_dv = [&](int t) -> bool {  // dV += P_t^T dO_t (P^T in A, split packing)
      // dV_t goes out before dP_t (except for the first tile), so it waits for dO_t itself.
      if (!warp_wait(bar(C::kPFull), t & 1, &abort_flag, a.err) ||
          !warp_wait(bar(C::kDOFull + t % C::kDOStages), (t / C::kDOStages) & 1, &abort_flag,
                     a.err))
        return false;
      tc_fence_after();
      umma_ts_mnmajor_x8_split(tmem + C::kColDV, tmem + C::kColA,
                               smem_desc_sw128(do_slot(t), C::kChunkBytes, 1024), kIdAcc,
                               t > 0 ? 1u : 0u);
      umma_commit_w(bar(C::kDVDone));
      return true;
    };
    bool ok = warp_wait(bar(C::kKVFull), 0, &abort_flag, a.err);
    if (ok) ok = issue_s(0);
    if (ok) ok = issue_dp(0);
    if (ok) ok = issue_dv(0);
    if (ok && T > 1) ok = issue_s(1);
    for (int t = 0; ok && t < T; ++t) {
      if (!(ok = warp_wait(bar(C::kDSFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      // dK += dS_t^T Q_t (dS^T K-major in shared memory, Q_t MN-major)
      umma_ss_kA_mnB_x8(tmem + C::kColDK, smem_desc_sw128(ds_tile(t), 16, 1024),
                        smem_desc_sw128(q_slot(t), C::kChunkBytes, 1024), kIdAcc, t > 0 ? 1u : 0u);
      umma_commit_w(bar(C::kQEmpty + t % C::kQStages));
      // dQ_t = dS_t K into B (dS read MN-major: queries along M in two 64-column chunks)
      umma_ss_mnA_mnB_x8(tmem + C::kColB, smem_desc_sw128(ds_tile(t), C::kDSChunkBytes, 1024),
                         smem_desc_sw128(sK, C::kChunkBytes, 1024), kIdDq, 0u);
      umma_commit_w(bar(C::kDQDone + (t & 1)));
      if (t + 1 < T) {
        if (!(ok = issue_dv(t + 1))) break;
        // dP_{t+1} overwrites B once dQ_t has been read out of it.
        if (!(ok = warp_wait(bar(C::kBFree), t & 1, &abort_flag, a.err))) break;
        if (!(ok = issue_dp(t + 1))) break;
        if (t + 2 < T && !(ok = issue_s(t + 2))) break;
      }
    }
    if (ok) umma_commit_w(bar(C::kDone));
    umma_commit_w(bar(C::kDrain));
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else {
    // ------------------------------------------------------- compute (warps 0-7)
    const int r = static_cast<int>(threadIdx.x & 127);  // TMEM lane: key row (A, B) or query row
    const uint32_t h = warp >> 2;                          // column half of every tile
    const int key = k0 + r;
    const int vis_lo = key + sp.dmin - sp.off, vis_hi = key + sp.dmax - sp.off;
    const uint32_t lane_base = ((warp & 3u) * 32u) << 16;
    const float sl2 = a.scale_log2;
    float nxt = 0.f;
    auto fetch_row = [&](int t) {
      const int q = tile_q0(t) + r;
      if (q < sp.Lq) {
        const size_t gi = static_cast<size_t>(tile_bhq(t)) * sp.Lq + q;
        nxt = h == 0 ? a.lse[gi] : a.delta[gi];
      } else {
        nxt = h == 0 ? SWA_POS_INF : 0.f;
      }
    };
    // Reads this thread's half-row of tile tt's dQ partial out of B (releasing B for the next
    // dP^T at once) and adds it into the accumulator, 4 columns per vector reduce-add.
    auto readout = [&](int tt) -> bool {
      if (!warp_wait(bar(C::kDQDone + (tt & 1)), (tt >> 1) & 1, &abort_flag, a.err)) return false;
      tc_fence_after();
      constexpr int kHalfCols = D / 2;
      uint32_t rr[kHalfCols / 32][32];
#pragma unroll
      for (int c4 = 0; c4 < kHalfCols / 32; ++c4)
        tmem_ld32(tmem + lane_base + C::kColB + kHalfCols * h + 32u * c4, rr[c4]);
      tmem_wait_ld_all();
#pragma unroll
      for (int c4 = 0; c4 < kHalfCols / 32; ++c4) reg_fence(rr[c4]);
      warp_arrive(bar(C::kBFree));
      float* row0 = a.dq_acc + dq_acc_offset(tile_bhq(tt), tile_qb(tt), r,
                                             kHalfCols * static_cast<int>(h), a.nqb, D);
#pragma unroll
      for (int c4 = 0; c4 < kHalfCols / 32; ++c4)
#pragma unroll
        for (int g = 0; g < 8; ++g)  // columns kHalfCols h + 32 c4 + 4 g .. + 3
          red_add_v4_f32(row0 + (8 * c4 + g) * (kBlockM * 4),
                         __uint_as_float(rr[c4][4 * g]), __uint_as_float(rr[c4][4 * g + 1]),
                         __uint_as_float(rr[c4][4 * g + 2]), __uint_as_float(rr[c4][4 * g + 3]));
      return true;
    };
    fetch_row(0);
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int q0 = tile_q0(t);
      float* s_lse2 = s_rows + (t & 1) * 2 * kBlockM;
      float* s_delta = s_lse2 + kBlockM;
      if (h == 0)
        s_lse2[r] = -nxt * kLog2e;
      else
        s_delta[r] = -nxt;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kVecFull + (t & 1)));
      if (!(ok = warp_wait(bar(C::kVecFull + (t & 1)), (t >> 1) & 1, &abort_flag, a.err))) break;
      if (t + 1 < T) fetch_row(t + 1);

      // ---- P^T = exp(scale S^T - LSE), written back over A as bf16 pairs
      if (!(ok = warp_wait(bar(C::kSFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      float p[64];
      {
        const float4* l4 = reinterpret_cast<const float4*>(s_lse2 + 64 * h);
        float4 lv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) lv[i] = l4[i];
        uint32_t rr[2][32];
        tmem_ld32(tmem + lane_base + C::kColA + 64u * h, rr[0]);
        tmem_ld32(tmem + lane_base + C::kColA + 64u * h + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
        const float2 scale2 = make_float2(sl2, sl2);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t* src = &rr[i >> 3][(4 * i) & 31];
          const float2 t0 = __ffma2_rn(make_float2(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                       scale2, make_float2(lv[i].x, lv[i].y));
          const float2 t1 = __ffma2_rn(make_float2(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                       scale2, make_float2(lv[i].z, lv[i].w));
          p[4 * i + 0] = ex2(t0.x);
          p[4 * i + 1] = ex2(t0.y);
          p[4 * i + 2] = ex2(t1.x);
          p[4 * i + 3] = ex2(t1.y);
        }
      }
      if (!(q0 >= q_int_lo && q0 <= q_int_hi)) {
        const int base = q0 + 64 * static_cast<int>(h);
        const int lo = vis_lo - base, hi = vis_hi - base;
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = (c >= lo && c <= hi) ? p[c] : 0.f;
      }
      {
        uint32_t pk_p[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk_p[c] = Elem<F16>::pack(p[2 * c], p[2 * c + 1]);
        tmem_st32(tmem + lane_base + C::kColA + 64u * h, pk_p);
        tmem_wait_st();
      }
      warp_arrive(bar(C::kPFull));

      // ---- the previous tile's dQ partial out of B, into its Q slot
      if (t >= 1 && !(ok = readout(t - 1))) break;

      // ---- dS^T = P^T (dP^T - Delta), into shared memory once dV_t has read this tile's dO
      if (!(ok = warp_wait(bar(C::kDPFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      uint32_t pk_ds[32];
      {
        uint32_t rr[2][32];
        tmem_ld32(tmem + lane_base + C::kColB + 64u * h, rr[0]);
        tmem_ld32(tmem + lane_base + C::kColB + 64u * h + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
        const float4* d4 = reinterpret_cast<const float4*>(s_delta + 64 * h);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 4 * i;
          const float4 nd = d4[i];
          const uint32_t* src = &rr[i >> 3][(4 * i) & 31];
          const float2 d0 = __fadd2_rn(make_float2(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                       make_float2(nd.x, nd.y));
          const float2 d1 = __fadd2_rn(make_float2(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                       make_float2(nd.z, nd.w));
          const float2 s0 = __fmul2_rn(make_float2(p[c], p[c + 1]), d0);
          const float2 s1 = __fmul2_rn(make_float2(p[c + 2], p[c + 3]), d1);
          pk_ds[2 * i] = Elem<F16>::pack(s0.x, s0.y);
          pk_ds[2 * i + 1] = Elem<F16>::pack(s1.x, s1.y);
        }
      }
      if (!(ok = warp_wait(bar(C::kDVDone), t & 1, &abort_flag, a.err))) break;
      {
        const uint32_t dst = ds_tile(t);
        uint32_t half0[16], half1[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          half0[i] = pk_ds[i];
          half1[i] = pk_ds[16 + i];
        }
        stage_row32_sw128(dst, static_cast<uint32_t>(r), 64u * h, half0);
        stage_row32_sw128(dst, static_cast<uint32_t>(r), 64u * h + 32u, half1);
      }
      fence_proxy_async_smem();
      warp_arrive(bar(C::kDSFull));
    }
    if (ok) ok = readout(T - 1);
    if (ok && warp_wait(bar(C::kDone), 0, &abort_flag, a.err)) {
      tc_fence_after();
      // dK * scale and dV -> 16-bit, staged in the two dO slots (every MMA has completed) and
      // written with tensor stores, one per 64-column chunk.
      constexpr int kHalf = D / 2;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which == 0 ? C::kColDK : C::kColDV) + kHalf * h;
        const float mul = which == 0 ? a.scale : 1.f;
        const uint32_t stage = sDO0 + which * C::kTileBytes;
        uint32_t rr[kHalf / 32][32];
#pragma unroll
        for (int c4 = 0; c4 < kHalf / 32; ++c4) tmem_ld32(tmem + lane_base + col + 32u * c4, rr[c4]);
        tmem_wait_ld_all();
#pragma unroll
        for (int c4 = 0; c4 < kHalf / 32; ++c4) {
          reg_fence(rr[c4]);
          uint32_t o16[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o16[i] = Elem<F16>::pack(__uint_as_float(rr[c4][2 * i]) * mul,
                                     __uint_as_float(rr[c4][2 * i + 1]) * mul);
          stage_row32_sw128(stage, r, kHalf * h + 32u * c4, o16);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kOutFull));
      if (warp == 0 && warp_wait(bar(C::kOutFull), 0, &abort_flag, a.err) && lane == 0) {
        for (int hh = 0; hh < C::kChunks; ++hh) {
          tma_store_3d(&tm_dk, sDO0 + hh * C::kChunkBytes, 64 * hh, k0, bhk);
          tma_store_3d(&tm_dv, sDO0 + C::kTileBytes + hh * C::kChunkBytes, 64 * hh, k0, bhk);
        }
        bulk_commit_group();
        bulk_wait_group_read0();
      }
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
cudaError_t launch_fused_d(const Problem& pb, const void* q, const void* k, const void* v,
                           const void* dO, const float* lse, const float* delta, float* dq_acc,
                           void* dk, void* dv, cudaStream_t stream) {
  using C = FusedCfg<D>;
  CUtensorMap tq, tdo, tk, tv, tdk, tdv;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_3d(&tq, q, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tdo, dO, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tk, k, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tv, v, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tdk, dk, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tdv, dv, bhk, pb.span.Lk, D, kBlockN, F16))
    return cudaErrorInvalidValue;
  auto kern = swa_fused_bwd_kernel<D, F16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  FusedArgs a;
  a.lse = lse;
  a.delta = delta;
  a.dq_acc = dq_acc;
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.BHK = pb.B * pb.Hkv;
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.G = pb.Hq / pb.Hkv;
  a.nqb = (pb.span.Lq + kBlockM - 1) / kBlockM;
  a.span = pb.span;
  a.scale = pb.scale;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  const int nkb = (pb.span.Lk + kBlockN - 1) / kBlockN;
  const unsigned grid = static_cast<unsigned>(nkb) * static_cast<unsigned>(a.BHK);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tdo, tk, tv, tdk, tdv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_fused(const Problem& pb, const void* q, const void* k, const void* v,
                             const void* dO, const float* lse, const float* delta, float* dq_acc,
                             void* dk, void* dv, cudaStream_t stream) {
  if (pb.D == 64)
    return pb.f16 ? launch_fused_d<64, true>(pb, q, k, v, dO, lse, delta, dq_acc, dk, dv, stream)
                  : launch_fused_d<64, false>(pb, q, k, v, dO, lse, delta, dq_acc, dk, dv, stream);
  if (pb.D == 128)
    return pb.f16 ? launch_fused_d<128, true>(pb, q, k, v, dO, lse, delta, dq_acc, dk, dv, stream)
                  : launch_fused_d<128, false>(pb, q, k, v, dO, lse, delta, dq_acc, dk, dv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace swa
