// swa_bwd_dkdv.cu — dK and dV of causal sliding-window attention on sm_103a.
//
// One CTA owns one 128-row key block of one (batch, kv head).  It walks, for each of the G query
// heads that share this kv head, only the query blocks that can see the block — keys j see queries
// i in [j, j+W-1] — and recomputes per query tile (transposed, so the key rows sit on TMEM lanes)
//   S^T = K Q^T,  P^T = exp(scale S^T - LSE) (window-masked),  dV += P^T dO,
//   dP^T = V dO^T,  dS^T = P^T (dP^T - Delta),  dK += dS^T Q,
// with a final dK *= scale.  dK and dV accumulate in TMEM (fp32) across the whole group, which is
// the grouped-query reduction: no atomics and no per-query-head partial buffers.  The walk follows
// "Off NVIDIA, you fix the platform yourself" (Lab 28), "What did fixing it take?" and "Method and
// disclosure": tiles wholly outside the window are skipped, edge tiles are masked, and dK / dV of
// a key tile that no query visits are still written (as zeros).
//
// Warp roles (352 threads): warps 0-7 compute — warp w handles TMEM lanes 32(w%4)..+31 (key rows)
// and query columns [64 h, 64 h + 64) of every tile, h = w / 4; warp 8 TMA producer of K (once)
// and of the Q_t ring, warp 10 of V (once) and of the dO_t ring — two issuing warps, because one
// warp's TMA copies complete at only ~40 B/clk on this GPU; warp 9 MMA issuer and TMEM owner.
// A compute thread reads its S^T values and releases the S^T columns at once, so the next tile's
// S^T is computed while it exponentiates; once dP^T has landed and been read, P^T and dS^T go
// back to TMEM as bf16 pairs over the dP^T columns (each half of a row: P^T over the first 32 of
// its 64 columns, dS^T over the last 32) and are the A operands of dV += P^T dO and dK += dS^T Q.
// TMEM columns: [0,128) S^T, [128,256) dP^T / P^T + dS^T, [256, 256+D) dK, [256+D, 256+2D) dV.
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

template <int D>
struct DkdvCfg {
  static constexpr int kTileBytes = kBlockM * D * 2;
  static constexpr int kChunkBytes = kBlockM * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kQStages = (D == 128) ? 3 : 4;
  static constexpr int kDOStages = (D == 128) ? 2 : 4;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
  // two slots of the per-query vectors {lse2[128], delta[128]}
  static constexpr int kOffRow = kOffDO + kDOStages * kTileBytes;
  static constexpr int kOffBar = kOffRow + 2 * 2 * kBlockM * 4;
  static constexpr int kKVFull = 0;
  static constexpr int kQFull = 1;
  static constexpr int kQEmpty = kQFull + kQStages;
  static constexpr int kDOFull = kQEmpty + kQStages;
  static constexpr int kDOEmpty = kDOFull + kDOStages;
  static constexpr int kSFull = kDOEmpty + kDOStages;
  static constexpr int kSEmpty = kSFull + 1;  // every compute warp has read S^T
  static constexpr int kDPFull = kSEmpty + 1;
  static constexpr int kPFull = kDPFull + 1;  // P^T and dS^T written (one arrival per warp)
  static constexpr int kVecFull = kPFull + 1;  // 2 slots
  static constexpr int kDone = kVecFull + 2;
  static constexpr int kOutFull = kDone + 1;  // staged dK / dV tiles complete (one arrival per warp)
  static constexpr int kDrain = kOutFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;  // + TMEM address and abort flag
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  // Once dP^T has been read, P^T and dS^T go over its columns: in each half-row's 64 columns,
  // P^T over the first 32 and dS^T over the last 32 (bf16 pairs).
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 256 + D;
  static constexpr int kThreads = 352;
  static constexpr int kComputeThreads = 256;
};

struct DkdvArgs {
  const float* lse;
  const float* delta;
  uint16_t* dk;  // bf16 or fp16 elements
  uint16_t* dv;
  int BHK, Hq, Hkv, G, nkb;
  Span span;
  float scale, scale_log2;
  unsigned* err;
};

template <int D, bool F16>
__global__ void __launch_bounds__(352, 1)
    swa_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv, const DkdvArgs a) {
  using C = DkdvCfg<D>;
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

  // Key blocks with the longest walks (lowest index under a full causal window) go first.
  const int kb = static_cast<int>(blockIdx.x) / a.BHK;
  const int bhk = static_cast<int>(blockIdx.x) % a.BHK;
  const int b = bhk / a.Hkv, hk = bhk % a.Hkv;
  const int k0 = kb * kBlockN;
  const Span sp = a.span;  // window geometry, held in registers
  const int qb_lo = sp.first_qblock(k0);
  const int qb_hi = sp.last_qblock(k0);
  // No query sees this key block when the queries are a short suffix of the keys: then nq <= 0,
  // nothing is computed and dK = dV = 0 is written.
  const int nq = qb_hi >= qb_lo ? qb_hi - qb_lo + 1 : 0;
  const int T = a.G * nq;  // (query head, query block) tiles of the walk
  // A query tile q0 needs no mask iff q_int_lo <= q0 <= q_int_hi (Span::interior for this key
  // block, solved for q0 once).
  const int q_int_lo = k0 + kBlockN - 1 + sp.dmin - sp.off;
  const int q_int_hi = (k0 + kBlockN <= sp.Lk)
                           ? min(k0 + sp.dmax - sp.off - (kBlockM - 1), sp.Lq - kBlockM)
                           : -1;
  // Tile t of the walk is query head gi of the group and query block qb_lo + qi, t = gi nq + qi.
  // Each role advances (qi, gi) tile by tile: dividing t by nq costs an integer division per tile,
  // whose reciprocal queues behind the compute warps' exponentials.
  struct WalkPos {
    int qi = 0, gi = 0;
  };
  auto advance = [&](WalkPos& w) {
    if (++w.qi == nq) {
      w.qi = 0;
      ++w.gi;
    }
  };
  const int bhq0 = b * a.Hq + hk * a.G;
  auto pos_q0 = [&](const WalkPos& w) { return (qb_lo + w.qi) * kBlockM; };
  auto pos_bhq = [&](const WalkPos& w) { return bhq0 + w.gi; };

  if (T == 0) {
    // No query sees this key block: its dK and dV rows are zero.  Written straight from the
    // threads, before any barrier, tensor memory or copy is set up.
    zero_key_rows(a.dk, a.dv, bhk, k0, sp.Lk, D);
    return;
  }

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(C::kKVFull), 2);  // one arrival per producer warp
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(bar(C::kQFull + s), 1);
      mbar_init(bar(C::kQEmpty + s), 1);
    }
    for (int s = 0; s < C::kDOStages; ++s) {
      mbar_init(bar(C::kDOFull + s), 1);
      mbar_init(bar(C::kDOEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSEmpty), C::kComputeThreads / 32);
    mbar_init(bar(C::kDPFull), 1);
    mbar_init(bar(C::kPFull), C::kComputeThreads / 32);
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
    // ------------------------------------------------------------------ TMA producer (K, Q ring)
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(bar(C::kKVFull), C::kTileBytes);
      for (int h = 0; h < C::kChunks; ++h)
        tma_load_3d(sK + h * C::kChunkBytes, &tm_k, bar(C::kKVFull), 64 * h, k0, bhk);
      int last_q[C::kQStages];
      for (int s = 0; s < C::kQStages; ++s) last_q[s] = -1;
      WalkPos wp;
      for (int t = 0; t < T; ++t, advance(wp)) {
        const int sq = t % C::kQStages, nqs = t / C::kQStages;
        if (t >= C::kQStages && !mbar_wait(bar(C::kQEmpty + sq), (nqs - 1) & 1, &abort_flag, a.err))
          break;
        const uint32_t sQ = sQ0 + sq * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kQFull + sq), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(sQ + h * C::kChunkBytes, &tm_q, bar(C::kQFull + sq), 64 * h, pos_q0(wp),
                      pos_bhq(wp));
        last_q[sq] = t;
      }
      drain_wait(bar(C::kKVFull), 0, a.err);
      for (int s = 0; s < C::kQStages; ++s)
        if (last_q[s] >= 0) drain_wait(bar(C::kQFull + s), (last_q[s] / C::kQStages) & 1, a.err);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------------ TMA producer (V, dO ring)
    if (lane == 0) {
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(C::kKVFull), C::kTileBytes);
      for (int h = 0; h < C::kChunks; ++h)
        tma_load_3d(sV + h * C::kChunkBytes, &tm_v, bar(C::kKVFull), 64 * h, k0, bhk);
      int last_do[C::kDOStages];
      for (int s = 0; s < C::kDOStages; ++s) last_do[s] = -1;
      WalkPos wp;
      for (int t = 0; t < T; ++t, advance(wp)) {
        const int sd = t % C::kDOStages, nds = t / C::kDOStages;
        if (t >= C::kDOStages &&
            !mbar_wait(bar(C::kDOEmpty + sd), (nds - 1) & 1, &abort_flag, a.err))
          break;
        const uint32_t sDO = sDO0 + sd * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kDOFull + sd), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(sDO + h * C::kChunkBytes, &tm_do, bar(C::kDOFull + sd), 64 * h, pos_q0(wp),
                      pos_bhq(wp));
        last_do[sd] = t;
      }
      drain_wait(bar(C::kKVFull), 0, a.err);
      for (int s = 0; s < C::kDOStages; ++s)
        if (last_do[s] >= 0)
          drain_wait(bar(C::kDOFull + s), (last_do[s] / C::kDOStages) & 1, a.err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    // Issue order: S_0, dP_0, then per tile t: S_{t+1}, dV += P_t^T dO_t, dK += dS_t^T Q_t,
    // dP_{t+1}.  S_{t+1} overwrites the S^T columns once every compute warp has read S_t^T
    // (S_EMPTY); the MMAs run in issue order, so dP_{t+1} overwrites P_t^T / dS_t^T only after
    // dV_t and dK_t have read them.
    {  // the whole warp, converged; one elected lane issues
      constexpr uint32_t kIdS = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockN, kBlockM, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockN, D, false, true);       // dV, dK
      auto issue_s = [&](int t) -> bool {  // S^T = K Q_t^T
        const int s = t % C::kQStages;
        if (t > 0 && !warp_wait(bar(C::kSEmpty), (t - 1) & 1, &abort_flag, a.err)) return false;
        if (!warp_wait(bar(C::kQFull + s), (t / C::kQStages) & 1, &abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t sQ = sQ0 + s * C::kTileBytes;
        umma_ss_kmajor_d<D>(tmem + C::kColS, smem_desc_sw128(sK, 16, 1024),
                            smem_desc_sw128(sQ, 16, 1024), kIdS, 0u);
        umma_commit_w(bar(C::kSFull));
        return true;
      };
      auto issue_dp = [&](int t) -> bool {  // dP^T = V dO_t^T
        const int s = t % C::kDOStages;
        if (!warp_wait(bar(C::kDOFull + s), (t / C::kDOStages) & 1, &abort_flag, a.err))
          return false;
        tc_fence_after();
        const uint32_t sDO = sDO0 + s * C::kTileBytes;
        umma_ss_kmajor_d<D>(tmem + C::kColDP, smem_desc_sw128(sV, 16, 1024),
                            smem_desc_sw128(sDO, 16, 1024), kIdS, 0u);
        umma_commit_w(bar(C::kDPFull));
        return true;
      };
      // acc += X^T B_t with X^T (bf16 pairs) in TMEM at column a_col and B_t = dO_t or Q_t (MN-major)
      // (wait_bar < 0: no wait, the operand's barrier has already been waited for)
      auto issue_acc = [&](int t, int wait_bar, uint32_t a_col, uint32_t b_tile,
                           uint32_t d_col) -> bool {
        if (wait_bar >= 0) {
          if (!warp_wait(bar(wait_bar), t & 1, &abort_flag, a.err)) return false;
          tc_fence_after();
        }
        // query columns 16 ks .. 16 ks + 15 sit at packed column 8 ks + 32 (ks / 4)
        umma_ts_mnmajor_x8_split(tmem + d_col, tmem + a_col,
                                 smem_desc_sw128(b_tile, C::kChunkBytes, 1024), kIdAcc,
                                 t > 0 ? 1u : 0u);
        return true;
      };
      bool ok = warp_wait(bar(C::kKVFull), 0, &abort_flag, a.err);
      if (ok && T > 0) ok = issue_s(0);
      if (ok && T > 0) ok = issue_dp(0);
      for (int t = 0; ok && t < T; ++t) {
        const int sq = t % C::kQStages, sd = t % C::kDOStages;
        if (t + 1 < T && !(ok = issue_s(t + 1))) break;
        ok = issue_acc(t, C::kPFull, C::kColDP, sDO0 + sd * C::kTileBytes, C::kColDV);  // dV
        if (!ok) break;
        umma_commit_w(bar(C::kDOEmpty + sd));
        // dK: dS^T was written with P^T, under the same barrier
        ok = issue_acc(t, -1, C::kColDP + 32u, sQ0 + sq * C::kTileBytes, C::kColDK);
        if (!ok) break;
        umma_commit_w(bar(C::kQEmpty + sq));
        if (t + 1 < T) ok = issue_dp(t + 1);
      }
      if (ok) umma_commit_w(bar(C::kDone));
      umma_commit_w(bar(C::kDrain));
      warp_drain_wait(bar(C::kDrain), 0, a.err);
    }
  } else {
    // ------------------------------------------------------------------ compute (warps 0-7)
    const int r = static_cast<int>(threadIdx.x & 127);  // key row within the block = TMEM lane
    const uint32_t h = warp >> 2;                          // query-column half of every tile
    const int key = k0 + r;
    const int vis_lo = key + sp.dmin - sp.off, vis_hi = key + sp.dmax - sp.off;  // visible queries
    const uint32_t lane_base = ((warp & 3u) * 32u) << 16;
    const float sl2 = a.scale_log2;
    // Per-query vectors of the next tile: the h = 0 threads fetch LSE, the h = 1 threads Delta,
    // for query q0 + r.  The raw value is kept until it is stored, so the load's latency hides
    // behind a whole tile.
    float nxt = 0.f;
    auto fetch_row = [&](const WalkPos& w) {
      const int q = pos_q0(w) + r;
      if (q < sp.Lq) {
        const size_t gi = static_cast<size_t>(pos_bhq(w)) * sp.Lq + q;
        nxt = h == 0 ? a.lse[gi] : a.delta[gi];
      } else {  // queries past the end contribute P = 0
        nxt = h == 0 ? SWA_POS_INF : 0.f;
      }
    };
    WalkPos wcur, wnext;  // tiles t and t + 1
    advance(wnext);
    if (T > 0) fetch_row(wcur);
    bool ok = true;
    for (int t = 0; t < T; ++t, advance(wcur), advance(wnext)) {
      const int q0 = pos_q0(wcur);
      // Slot t & 1 was last read in tile t - 2; every compute thread has finished that tile
      // (dK_{t-2}, which needed all of them, precedes dP_{t-1}, which this thread has seen).
      // Stored negated (-LSE log2(e) and -Delta), the addends of the packed FFMA / FADD below.
      float* s_lse2 = s_rows + (t & 1) * 2 * kBlockM;
      float* s_delta = s_lse2 + kBlockM;
      if (h == 0)
        s_lse2[r] = -nxt * kLog2e;
      else
        s_delta[r] = -nxt;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kVecFull + (t & 1)));
      if (!(ok = warp_wait(bar(C::kVecFull + (t & 1)), (t >> 1) & 1, &abort_flag, a.err))) break;
      if (t + 1 < T) fetch_row(wnext);

      if (!(ok = warp_wait(bar(C::kSFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      float p[64];
      {
        // The per-query log-sum-exp values are read from shared memory while the TMEM load of S^T
        // is in flight (the loads are issued before the wait, so their latencies overlap).
        const float4* l4 = reinterpret_cast<const float4*>(s_lse2 + 64 * h);
        float4 lv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) lv[i] = l4[i];
        uint32_t rr[2][32];
        tmem_ld32(tmem + lane_base + C::kColS + 64u * h, rr[0]);
        tmem_ld32(tmem + lane_base + C::kColS + 64u * h + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
        // S^T is in registers: the next tile's S^T may overwrite its columns.
        tc_fence_before();
        warp_arrive(bar(C::kSEmpty));
        // P^T = 2^(scale log2(e) S^T - LSE log2(e)), two queries per packed FFMA.
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
      // Query q0 + 64h + c sees this key iff dmin <= q0 + 64h + c + off - key <= dmax, i.e.
      // c in [vis_lo, vis_hi] - q0 - 64h (queries past the end already have P = 0).
      if (!(q0 >= q_int_lo && q0 <= q_int_hi)) {
        const int base = q0 + 64 * static_cast<int>(h);
        const int lo = vis_lo - base, hi = vis_hi - base;
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = (c >= lo && c <= hi) ? p[c] : 0.f;
      }

      if (!(ok = warp_wait(bar(C::kDPFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      {
        const uint32_t dp_col = tmem + lane_base + C::kColDP + 64u * h;
        uint32_t rr[2][32];
        tmem_ld32(dp_col, rr[0]);
        tmem_ld32(dp_col + 32u, rr[1]);
        tmem_wait_ld_all();
        reg_fence(rr[0]);
        reg_fence(rr[1]);
        // dS^T = P^T (dP^T - Delta), two queries per packed FADD / FMUL; computing it first frees
        // the dP^T registers before P^T is packed.
        const float4* d4 = reinterpret_cast<const float4*>(s_delta + 64 * h);
        uint32_t pk_ds[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = 4 * i;
          const float4 nd = d4[i];  // -Delta of queries c .. c + 3
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
        // dP^T has been read: P^T goes over the first 32 of this half's 64 columns, dS^T over the
        // last 32.
        uint32_t pk_p[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk_p[c] = Elem<F16>::pack(p[2 * c], p[2 * c + 1]);
        tmem_st32(dp_col, pk_p);
        tmem_st32(dp_col + 32u, pk_ds);
      }
      tmem_wait_st();
      warp_arrive(bar(C::kPFull));
    }
    if (ok && warp_wait(bar(C::kDone), 0, &abort_flag, a.err)) {
      tc_fence_after();
      // dK * scale and dV -> bf16, staged in the two Q slots (free: every MMA has completed) and
      // written with tensor stores, one per 64-column chunk (rows past Lk are not written).
      constexpr int kHalf = D / 2;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which == 0 ? C::kColDK : C::kColDV) + kHalf * h;
        const float mul = which == 0 ? a.scale : 1.f;
        const uint32_t stage = sQ0 + which * C::kTileBytes;
        uint32_t rr[kHalf / 32][32];
        if (T > 0) {
#pragma unroll
          for (int c4 = 0; c4 < kHalf / 32; ++c4) tmem_ld32(tmem + lane_base + col + 32u * c4, rr[c4]);
          tmem_wait_ld_all();
        } else {  // no query visits this key block: its gradients are zero
#pragma unroll
          for (int c4 = 0; c4 < kHalf / 32; ++c4)
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[c4][i] = 0u;
        }
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
          tma_store_3d(&tm_dk, sQ0 + hh * C::kChunkBytes, 64 * hh, k0, bhk);
          tma_store_3d(&tm_dv, sQ0 + C::kTileBytes + hh * C::kChunkBytes, 64 * hh, k0, bhk);
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
cudaError_t launch_dkdv_d(const Problem& pb, const void* q, const void* k, const void* v,
                          const void* dO, const float* lse, const float* delta, void* dk, void* dv,
                          cudaStream_t stream) {
  using C = DkdvCfg<D>;
  CUtensorMap tq, tdo, tk, tv, tdk, tdv;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_3d(&tq, q, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tdo, dO, bhq, pb.span.Lq, D, kBlockM, F16) ||
      !make_tmap_3d(&tk, k, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tv, v, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tdk, dk, bhk, pb.span.Lk, D, kBlockN, F16) ||
      !make_tmap_3d(&tdv, dv, bhk, pb.span.Lk, D, kBlockN, F16))
    return cudaErrorInvalidValue;
  auto kern = swa_dkdv_kernel<D, F16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  DkdvArgs a;
  a.lse = lse;
  a.delta = delta;
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.BHK = pb.B * pb.Hkv;
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.G = pb.Hq / pb.Hkv;
  a.span = pb.span;
  a.nkb = (pb.span.Lk + kBlockN - 1) / kBlockN;
  a.scale = pb.scale;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  const unsigned grid = static_cast<unsigned>(a.nkb) * static_cast<unsigned>(a.BHK);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tdo, tk, tv, tdk, tdv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv(const Problem& pb, const void* q, const void* k, const void* v,
                            const void* dO, const float* lse, const float* delta, void* dk,
                            void* dv, cudaStream_t stream) {
  if (pb.D == 256) return launch_dkdv_d256(pb, q, k, v, dO, lse, delta, dk, dv, stream);
  if (pb.D == 64)
    return pb.f16 ? launch_dkdv_d<64, true>(pb, q, k, v, dO, lse, delta, dk, dv, stream)
                  : launch_dkdv_d<64, false>(pb, q, k, v, dO, lse, delta, dk, dv, stream);
  if (pb.D == 128)
    return pb.f16 ? launch_dkdv_d<128, true>(pb, q, k, v, dO, lse, delta, dk, dv, stream)
                  : launch_dkdv_d<128, false>(pb, q, k, v, dO, lse, delta, dk, dv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace swa
