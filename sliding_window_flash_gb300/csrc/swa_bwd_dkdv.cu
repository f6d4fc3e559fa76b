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
// Warp roles (192 threads): warps 0-3 compute (thread r = key row k0 + r = TMEM lane r),
// warp 4 TMA producer (K and V once; Q_t, dO_t through two slots), warp 5 MMA issuer and TMEM
// owner.  P^T and dS^T share one bf16 operand tile in shared memory.  TMEM columns: [0,128) S^T,
// [128,256) dP^T, [256, 256+D) dK, [256+D, 256+2D) dV.
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
  static constexpr int kOpBytes = kBlockN * kBlockM * 2;  // P^T / dS^T operand tile
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;          // 2 slots
  static constexpr int kOffDO = kOffQ + 2 * kTileBytes;     // 2 slots
  static constexpr int kOffOp = kOffDO + 2 * kTileBytes;
  static constexpr int kOffRow = kOffOp + kOpBytes;         // lse2[128], delta[128]
  static constexpr int kOffBar = kOffRow + 2 * kBlockM * 4;
  static constexpr int kKVFull = 0;
  static constexpr int kQFull = 1;       // 2
  static constexpr int kDOFull = 3;      // 2
  static constexpr int kPairEmpty = 5;   // 2
  static constexpr int kSFull = 7;
  static constexpr int kSEmpty = 8;
  static constexpr int kDPFull = 9;
  static constexpr int kDPEmpty = 10;
  static constexpr int kPFull = 11;
  static constexpr int kDSFull = 12;
  static constexpr int kDVDone = 13;
  static constexpr int kDKDone = 14;
  static constexpr int kDrain = 15;
  static constexpr int kNumBars = 16;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 256 + D;
  static constexpr int kThreads = 192;
};

struct DkdvArgs {
  const float* lse;
  const float* delta;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int BHK, Hq, Hkv, G, N, W, nkb;
  float scale, scale_log2;
  unsigned* err;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    swa_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const DkdvArgs a) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  float* s_lse2 = reinterpret_cast<float*>(smem + C::kOffRow);
  float* s_delta = s_lse2 + kBlockM;
  __shared__ int abort_flag;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sV = smem_u32(smem + C::kOffV);
  const uint32_t sQ0 = smem_u32(smem + C::kOffQ);
  const uint32_t sDO0 = smem_u32(smem + C::kOffDO);
  const uint32_t sOp = smem_u32(smem + C::kOffOp);

  // Key blocks with the longest walks (lowest index under a full causal window) go first.
  const int kb = static_cast<int>(blockIdx.x) / a.BHK;
  const int bhk = static_cast<int>(blockIdx.x) % a.BHK;
  const int b = bhk / a.Hkv, hk = bhk % a.Hkv;
  const int k0 = kb * kBlockN;
  const int qb_lo = bwd_first_qblock(k0);
  const int qb_hi = bwd_last_qblock(k0, a.N, a.W);
  const int nq = qb_hi - qb_lo + 1;  // >= 1: the diagonal block always sees the key block
  const int T = a.G * nq;            // (query head, query block) tiles of the walk
  auto tile_q0 = [&](int t) { return (qb_lo + t % nq) * kBlockM; };
  auto tile_bhq = [&](int t) { return b * a.Hq + hk * a.G + t / nq; };

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(C::kKVFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kQFull + s), 1);
      mbar_init(bar(C::kDOFull + s), 1);
      mbar_init(bar(C::kPairEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSEmpty), 128);
    mbar_init(bar(C::kDPFull), 1);
    mbar_init(bar(C::kDPEmpty), 128);
    mbar_init(bar(C::kPFull), 128);
    mbar_init(bar(C::kDSFull), 128);
    mbar_init(bar(C::kDVDone), 1);
    mbar_init(bar(C::kDKDone), 1);
    mbar_init(bar(C::kDrain), 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(C::kKVFull), 2 * C::kTileBytes);
      for (int h = 0; h < C::kChunks; ++h) {
        tma_load_3d(sK + h * C::kChunkBytes, &tm_k, bar(C::kKVFull), 64 * h, k0, bhk);
        tma_load_3d(sV + h * C::kChunkBytes, &tm_v, bar(C::kKVFull), 64 * h, k0, bhk);
      }
      int last_fill[2] = {-1, -1};
      for (int t = 0; t < T; ++t) {
        const int s = t & 1, n = t >> 1;
        if (t >= 2 && !mbar_wait(bar(C::kPairEmpty + s), (n - 1) & 1, &abort_flag, a.err)) break;
        const int q0 = tile_q0(t), bhq = tile_bhq(t);
        const uint32_t sQ = sQ0 + s * C::kTileBytes, sDO = sDO0 + s * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kQFull + s), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(sQ + h * C::kChunkBytes, &tm_q, bar(C::kQFull + s), 64 * h, q0, bhq);
        mbar_arrive_expect_tx(bar(C::kDOFull + s), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(sDO + h * C::kChunkBytes, &tm_do, bar(C::kDOFull + s), 64 * h, q0, bhq);
        last_fill[s] = t;
      }
      drain_wait(bar(C::kKVFull), 0, a.err);
      for (int s = 0; s < 2; ++s) {
        if (last_fill[s] >= 0) {
          drain_wait(bar(C::kQFull + s), (last_fill[s] >> 1) & 1, a.err);
          drain_wait(bar(C::kDOFull + s), (last_fill[s] >> 1) & 1, a.err);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kBlockN, kBlockM, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16(kBlockN, D, false, true);       // dV, dK
      auto issue_s = [&](int t) -> bool {  // S^T = K Q_t^T
        const int s = t & 1;
        if (!mbar_wait(bar(C::kQFull + s), (t >> 1) & 1, &abort_flag, a.err)) return false;
        if (t >= 1 && !mbar_wait(bar(C::kSEmpty), (t - 1) & 1, &abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t sQ = sQ0 + s * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
          umma_ss(tmem + C::kColS, smem_desc_sw128(sK + off, 16, 1024),
                  smem_desc_sw128(sQ + off, 16, 1024), kIdS, ks > 0);
        }
        umma_commit(bar(C::kSFull));
        return true;
      };
      auto issue_dp = [&](int t) -> bool {  // dP^T = V dO_t^T
        const int s = t & 1;
        if (!mbar_wait(bar(C::kDOFull + s), (t >> 1) & 1, &abort_flag, a.err)) return false;
        if (t >= 1 && !mbar_wait(bar(C::kDPEmpty), (t - 1) & 1, &abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t sDO = sDO0 + s * C::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * C::kChunkBytes + (ks & 3) * 32;
          umma_ss(tmem + C::kColDP, smem_desc_sw128(sV + off, 16, 1024),
                  smem_desc_sw128(sDO + off, 16, 1024), kIdS, ks > 0);
        }
        umma_commit(bar(C::kDPFull));
        return true;
      };
      auto issue_acc = [&](int t, int wait_bar, uint32_t b_tile, uint32_t col, int done_bar) -> bool {
        if (!mbar_wait(bar(wait_bar), t & 1, &abort_flag, a.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kBlockM / 16; ++ks) {
          const uint32_t aoff = (ks >> 2) * (kBlockN * 128) + (ks & 3) * 32;
          umma_ss(tmem + col, smem_desc_sw128(sOp + aoff, 16, 1024),
                  smem_desc_sw128(b_tile + ks * 16 * 128, C::kChunkBytes, 1024), kIdAcc,
                  (t > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar(done_bar));
        return true;
      };
      bool ok = mbar_wait(bar(C::kKVFull), 0, &abort_flag, a.err);
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_dp(0);
      for (int t = 0; ok && t < T; ++t) {
        const int s = t & 1;
        // dV += P^T dO_t
        ok = issue_acc(t, C::kPFull, sDO0 + s * C::kTileBytes, C::kColDV, C::kDVDone);
        if (ok && t + 1 < T) ok = issue_s(t + 1);
        // dK += dS^T Q_t, then release the (Q_t, dO_t) slot
        if (ok) ok = issue_acc(t, C::kDSFull, sQ0 + s * C::kTileBytes, C::kColDK, C::kDKDone);
        if (ok) umma_commit(bar(C::kPairEmpty + s));
        if (ok && t + 1 < T) ok = issue_dp(t + 1);
      }
      umma_commit(bar(C::kDrain));
      drain_wait(bar(C::kDrain), 0, a.err);
    }
  } else {
    // ------------------------------------------------------------------ compute (warps 0-3)
    const int r = static_cast<int>(threadIdx.x);
    const int key = k0 + r;
    const uint32_t lane_base = (warp * 32u) << 16;
    const float sl2 = a.scale_log2;
    // This thread's share of the per-query vectors of the next tile (query q0 + r).
    float nxt_lse2 = 0.f, nxt_delta = 0.f;
    auto fetch_row = [&](int t) {
      const int q = tile_q0(t) + r;
      if (q < a.N) {
        const size_t gi = static_cast<size_t>(tile_bhq(t)) * a.N + q;
        nxt_lse2 = a.lse[gi] * kLog2e;
        nxt_delta = a.delta[gi];
      } else {  // queries past the end contribute P = 0
        nxt_lse2 = SWA_POS_INF;
        nxt_delta = 0.f;
      }
    };
    fetch_row(0);
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int q0 = tile_q0(t);
      named_barrier_sync(1, 128);  // every thread is done with the previous tile's vectors
      s_lse2[r] = nxt_lse2;
      s_delta[r] = nxt_delta;
      named_barrier_sync(1, 128);
      if (t + 1 < T) fetch_row(t + 1);

      if (!(ok = warp_wait(bar(C::kSFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      float p[kBlockM];
#pragma unroll
      for (int c4 = 0; c4 < kBlockM / 32; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + C::kColS + 32u * c4, rr);
        tmem_wait_ld(rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) p[32 * c4 + i] = __uint_as_float(rr[i]);
      }
      tc_fence_before();
      mbar_arrive(bar(C::kSEmpty));
      const float4* l4 = reinterpret_cast<const float4*>(s_lse2);
#pragma unroll
      for (int c4 = 0; c4 < kBlockM / 4; ++c4) {
        const float4 l = l4[c4];
        p[4 * c4 + 0] = ex2(fmaf(p[4 * c4 + 0], sl2, -l.x));
        p[4 * c4 + 1] = ex2(fmaf(p[4 * c4 + 1], sl2, -l.y));
        p[4 * c4 + 2] = ex2(fmaf(p[4 * c4 + 2], sl2, -l.z));
        p[4 * c4 + 3] = ex2(fmaf(p[4 * c4 + 3], sl2, -l.w));
      }
      // Query q0 + c sees this key iff 0 <= q0 + c - key < W.
      const bool interior = (q0 >= k0 + kBlockN - 1) && (q0 + kBlockM - 1 - k0 < a.W);
      if (!interior) {
        const int lo = key - q0, hi = key - q0 + a.W - 1;
#pragma unroll
        for (int c = 0; c < kBlockM; ++c) p[c] = (c >= lo && c <= hi) ? p[c] : 0.f;
      }
      uint32_t pk[kBlockM / 2];
#pragma unroll
      for (int c = 0; c < kBlockM / 2; ++c) pk[c] = pack_bf16x2(p[2 * c], p[2 * c + 1]);
      // dK of the previous tile must have consumed the shared operand tile.
      if (t > 0 && !(ok = warp_wait(bar(C::kDKDone), (t - 1) & 1, &abort_flag, a.err))) break;
      store_row_sw128_128(sOp, r, pk);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::kPFull));

      if (!(ok = warp_wait(bar(C::kDPFull), t & 1, &abort_flag, a.err))) break;
      tc_fence_after();
      const float4* d4 = reinterpret_cast<const float4*>(s_delta);
#pragma unroll
      for (int c4 = 0; c4 < kBlockM / 32; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + C::kColDP + 32u * c4, rr);
        tmem_wait_ld(rr);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = 32 * c4 + 4 * i;
          const float4 dl = d4[c >> 2];
          pk[c >> 1] = pack_bf16x2(p[c] * (__uint_as_float(rr[4 * i]) - dl.x),
                                   p[c + 1] * (__uint_as_float(rr[4 * i + 1]) - dl.y));
          pk[(c >> 1) + 1] = pack_bf16x2(p[c + 2] * (__uint_as_float(rr[4 * i + 2]) - dl.z),
                                         p[c + 3] * (__uint_as_float(rr[4 * i + 3]) - dl.w));
        }
      }
      tc_fence_before();
      mbar_arrive(bar(C::kDPEmpty));
      // dV of this tile must have consumed P^T before dS^T replaces it.
      if (!(ok = warp_wait(bar(C::kDVDone), t & 1, &abort_flag, a.err))) break;
      store_row_sw128_128(sOp, r, pk);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::kDSFull));
    }
    if (ok && warp_wait(bar(C::kDKDone), (T - 1) & 1, &abort_flag, a.err)) {
      tc_fence_after();
      const bool in_range = key < a.N;
      const size_t grow = static_cast<size_t>(bhk) * a.N + key;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::kColDK : C::kColDV;
        const float mul = which == 0 ? a.scale : 1.f;
        __nv_bfloat16* dst_row = (which == 0 ? a.dk : a.dv) + grow * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + col + c0, rr);
          tmem_wait_ld(rr);
          uint32_t o16[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o16[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * mul,
                                 __uint_as_float(rr[2 * i + 1]) * mul);
          if (in_range) {
            uint4* dst = reinterpret_cast<uint4*>(dst_row + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(o16[4 * v], o16[4 * v + 1], o16[4 * v + 2], o16[4 * v + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_dkdv_d(const Problem& pb, const void* q, const void* k, const void* v,
                          const void* dO, const float* lse, const float* delta, void* dk, void* dv,
                          cudaStream_t stream) {
  using C = DkdvCfg<D>;
  CUtensorMap tq, tdo, tk, tv;
  const uint64_t bhq = static_cast<uint64_t>(pb.B) * pb.Hq, bhk = static_cast<uint64_t>(pb.B) * pb.Hkv;
  if (!make_tmap_bf16_3d(&tq, q, bhq, pb.N, D, kBlockM) ||
      !make_tmap_bf16_3d(&tdo, dO, bhq, pb.N, D, kBlockM) ||
      !make_tmap_bf16_3d(&tk, k, bhk, pb.N, D, kBlockN) ||
      !make_tmap_bf16_3d(&tv, v, bhk, pb.N, D, kBlockN))
    return cudaErrorInvalidValue;
  auto kern = swa_dkdv_kernel<D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  DkdvArgs a;
  a.lse = lse;
  a.delta = delta;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.BHK = pb.B * pb.Hkv;
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.G = pb.Hq / pb.Hkv;
  a.N = pb.N;
  a.W = pb.W;
  a.nkb = (pb.N + kBlockN - 1) / kBlockN;
  a.scale = pb.scale;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  const unsigned grid = static_cast<unsigned>(a.nkb) * static_cast<unsigned>(a.BHK);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tdo, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv(const Problem& pb, const void* q, const void* k, const void* v,
                            const void* dO, const float* lse, const float* delta, void* dk,
                            void* dv, cudaStream_t stream) {
  if (pb.D == 64) return launch_dkdv_d<64>(pb, q, k, v, dO, lse, delta, dk, dv, stream);
  if (pb.D == 128) return launch_dkdv_d<128>(pb, q, k, v, dO, lse, delta, dk, dv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace swa
