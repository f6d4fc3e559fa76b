// swa_fwd.cu — forward of causal sliding-window attention on sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, query head):
//   O[q0:q0+128] = softmax(scale * Q K^T, window mask) V,  LSE = natural-log row log-sum-exp,
// walking only the key blocks kb_lo..kb_hi that the window reaches ("Off NVIDIA, you fix the
// platform yourself", Lab 28, "What did fixing it take?": skip blocks wholly outside the window,
// mask the cells at its edge; the first block a query tile visits is no longer block zero).
// Only O and LSE are written (mlx-train-perf README, flash-attention section: the saved state is
// the output and the log-sum-exp).
//
// Warp roles (320 threads):
//   warps 0-7  softmax: warp w owns TMEM lanes 32(w%4)..+31 (query rows) and columns
//              [64 h, 64 h + 64) of every score tile, h = w / 4, so each row is split over two
//              threads that swap their partial row max through shared memory every block.  Each
//              masks its half, keeps the running max m and its partial sum l in registers, writes
//              bf16 P back to TMEM (packed pairs), rescales its half of the O row in TMEM when the
//              max grows by more than 2^8, and finally writes its half of O / l (and LSE).
//   warp 8     TMA producer: Q once, then K_j and V_j through two independent shared-memory rings
//              (K is released as soon as S_j is computed, V after P_j V_j).
//   warp 9     MMA issuer (one thread) and TMEM owner: S_j = Q K_j^T into one of two TMEM S buffers
//              (A and B from shared memory); O += P_j V_j with P_j read from TMEM (A operand) and V_j
//              from shared memory.  S_{j+1} is issued before O += P_j V_j so the tensor core computes
//              the next scores while the softmax warps work on this block.  tcgen05.mma operations of
//              one thread run in issue order, which orders every TMEM reuse below.
// TMEM columns: [0,128) S buffer 0, [128,256) S buffer 1, [256, 256+D) O, then two 64-column
// P buffers (128 bf16 per row, two per column).
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"

namespace swa {
namespace {

// Running max is only moved (and O rescaled) when it grows by more than this many powers of 2;
// otherwise P is computed against the stale max, with values up to 2^8 (exact softmax either way).
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = kBlockM * D * 2;  // one 128 x D bf16 tile
  static constexpr int kChunkBytes = kBlockM * 128;   // 128 rows x 64 columns (128-byte rows)
  static constexpr int kChunks = D / 64;
  static constexpr int kKStages = (D == 128) ? 3 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffRed = kOffV + kVStages * kTileBytes;  // [2 slots][2 halves][128] fp32
  static constexpr int kOffBar = kOffRed + 2 * 2 * kBlockM * 4;
  // barrier indices
  static constexpr int kQFull = 0;
  static constexpr int kKFull = 1;
  static constexpr int kKEmpty = kKFull + kKStages;
  static constexpr int kVFull = kKEmpty + kKStages;
  static constexpr int kVEmpty = kVFull + kVStages;
  static constexpr int kSFull = kVEmpty + kVStages;  // 2
  static constexpr int kPFull = kSFull + 2;          // 2
  static constexpr int kPVDone = kPFull + 2;         // 2
  static constexpr int kXch = kPVDone + 2;           // [4 lane quarters][2 slots]
  static constexpr int kOutFull = kXch + 8;  // staged output tile complete (one arrival per warp)
  static constexpr int kDrain = kOutFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + TMEM slot + align
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;  // buffer b at kColS + 128 b
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kColP = 256 + D;  // buffer b at kColP + 64 b
  static constexpr int kThreads = 320;
  static constexpr int kComputeThreads = 256;
};

struct FwdArgs {
  __nv_bfloat16* o;
  float* lse;
  int BH;  // B * Hq
  int Hq, Hkv, G, N, W, nqb;
  float scale_log2;  // scale * log2(e)
  unsigned* err;
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    swa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  __shared__ int abort_flag;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sK0 = smem_u32(smem + C::kOffK);
  const uint32_t sV0 = smem_u32(smem + C::kOffV);
  float* s_red = reinterpret_cast<float*>(smem + C::kOffRed);

  // Heaviest query blocks first (the causal case gives later blocks more key blocks).
  const int qb = a.nqb - 1 - static_cast<int>(blockIdx.x) / a.BH;
  const int bh = static_cast<int>(blockIdx.x) % a.BH;
  const int hq = bh % a.Hq;
  const int bhk = (bh / a.Hq) * a.Hkv + hq / a.G;
  const int q0 = qb * kBlockM;
  const int kb_lo = fwd_first_kblock(q0, a.W);
  const int kb_hi = fwd_last_kblock(q0, a.N);
  const int nkv = kb_hi - kb_lo + 1;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(C::kQFull), 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar(C::kKFull + s), 1);
      mbar_init(bar(C::kKEmpty + s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar(C::kVFull + s), 1);
      mbar_init(bar(C::kVEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kSFull + b), 1);
      mbar_init(bar(C::kPFull + b), C::kComputeThreads / 32);
      mbar_init(bar(C::kPVDone + b), 1);
    }
    for (int x = 0; x < 8; ++x) mbar_init(bar(C::kXch + x), 2);  // the two warps of a lane quarter
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
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(C::kQFull), C::kTileBytes);
      for (int h = 0; h < C::kChunks; ++h)
        tma_load_3d(sQ + h * C::kChunkBytes, &tm_q, bar(C::kQFull), 64 * h, q0, bh);
      int last_k[C::kKStages], last_v[C::kVStages];
      for (int s = 0; s < C::kKStages; ++s) last_k[s] = -1;
      for (int s = 0; s < C::kVStages; ++s) last_v[s] = -1;
      for (int j = 0; j < nkv; ++j) {
        const int k0 = (kb_lo + j) * kBlockN;
        const int sk = j % C::kKStages, nk = j / C::kKStages;
        if (j >= C::kKStages && !mbar_wait(bar(C::kKEmpty + sk), (nk - 1) & 1, &abort_flag, a.err))
          break;
        const uint32_t sK = sK0 + sk * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kKFull + sk), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(sK + h * C::kChunkBytes, &tm_k, bar(C::kKFull + sk), 64 * h, k0, bhk);
        last_k[sk] = j;
        const int sv = j % C::kVStages, nv = j / C::kVStages;
        if (j >= C::kVStages && !mbar_wait(bar(C::kVEmpty + sv), (nv - 1) & 1, &abort_flag, a.err))
          break;
        const uint32_t sV = sV0 + sv * C::kTileBytes;
        mbar_arrive_expect_tx(bar(C::kVFull + sv), C::kTileBytes);
        for (int h = 0; h < C::kChunks; ++h)
          tma_load_3d(sV + h * C::kChunkBytes, &tm_v, bar(C::kVFull + sv), 64 * h, k0, bhk);
        last_v[sv] = j;
      }
      // Never leave a copy in flight: wait for the last fill of every stage.
      drain_wait(bar(C::kQFull), 0, a.err);
      for (int s = 0; s < C::kKStages; ++s)
        if (last_k[s] >= 0) drain_wait(bar(C::kKFull + s), (last_k[s] / C::kKStages) & 1, a.err);
      for (int s = 0; s < C::kVStages; ++s)
        if (last_v[s] >= 0) drain_wait(bar(C::kVFull + s), (last_v[s] / C::kVStages) & 1, a.err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    {  // the whole warp, converged; one elected lane issues
      constexpr uint32_t kIdS = idesc_bf16(kBlockM, kBlockN, false, false);
      constexpr uint32_t kIdO = idesc_bf16(kBlockM, D, false, true);
      auto issue_s = [&](int j) -> bool {
        // S buffer (j & 1) was last read by the softmax warps for block j-2; P_FULL of j-2, which
        // issue_pv(j-2) waited for, already implies that.
        const int s = j % C::kKStages, n = j / C::kKStages, sb = j & 1;
        if (!warp_wait(bar(C::kKFull + s), n & 1, &abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t sK = sK0 + s * C::kTileBytes;
        umma_ss_kmajor_d<D>(tmem + C::kColS + 128u * sb, smem_desc_sw128(sQ, 16, 1024),
                            smem_desc_sw128(sK, 16, 1024), kIdS, 0u);
        umma_commit_w(bar(C::kSFull + sb));
        umma_commit_w(bar(C::kKEmpty + s));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int s = j % C::kVStages, n = j / C::kVStages, pb = j & 1;
        if (!warp_wait(bar(C::kPFull + pb), (j >> 1) & 1, &abort_flag, a.err)) return false;
        if (!warp_wait(bar(C::kVFull + s), n & 1, &abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t sV = sV0 + s * C::kTileBytes;
        umma_ts_mnmajor_x8(tmem + C::kColO, tmem + C::kColP + 64u * pb,
                           smem_desc_sw128(sV, C::kChunkBytes, 1024), kIdO, j > 0 ? 1u : 0u);
        umma_commit_w(bar(C::kPVDone + pb));
        umma_commit_w(bar(C::kVEmpty + s));
        return true;
      };
      bool ok = warp_wait(bar(C::kQFull), 0, &abort_flag, a.err);
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nkv; ++j) {
        if (j + 1 < nkv) ok = issue_s(j + 1);
        if (ok) ok = issue_pv(j);
      }
      // Every issued MMA completes before TMEM is released.
      umma_commit_w(bar(C::kDrain));
      warp_drain_wait(bar(C::kDrain), 0, a.err);
    }
  } else {
    // ------------------------------------------------------------------ softmax (warps 0-7)
    const int r = static_cast<int>(threadIdx.x & 127);  // row within the tile == TMEM lane
    const uint32_t h = warp >> 2;                          // column half of every tile
    const uint32_t quarter = warp & 3u;
    const int row = q0 + r;
    const uint32_t lane_base = (quarter * 32u) << 16;
    const float sl2 = a.scale_log2;
    float m_ref = SWA_NEG_INF;  // reference max (log2 domain) that P and l are taken against
    float l = 0.f;              // partial row sum over this thread's half of the columns
    bool ok = true;
    // Swap a per-row value with the thread that owns the other half of the row.  Slot `n & 1`
    // was last used two exchanges ago, and the partner arrived at the exchange in between only
    // after reading it.
    auto exchange = [&](int n, float v, float* other) -> bool {
      float* red = s_red + (n & 1) * 2 * kBlockM;
      red[h * kBlockM + r] = v;
      __syncwarp();
      const uint32_t xb = bar(C::kXch + quarter * 2 + (n & 1));
      if (lane == 0) mbar_arrive(xb);
      if (!warp_wait(xb, (n >> 1) & 1, &abort_flag, a.err)) return false;
      *other = red[(h ^ 1u) * kBlockM + r];
      return true;
    };
    for (int j = 0; j < nkv; ++j) {
      const int k0 = (kb_lo + j) * kBlockN;
      const int sb = j & 1;
      if (!(ok = warp_wait(bar(C::kSFull + sb), (j >> 1) & 1, &abort_flag, a.err))) break;
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

      // Window mask: the cells of this block visible to row `row` are keys in [row-W+1, row].
      const bool interior = (k0 + kBlockN - 1 <= q0) && (q0 + kBlockM - 1 - k0 < a.W);
      if (!interior) {
        const int hi = row - k0 - 64 * static_cast<int>(h), lo = hi - a.W + 1;
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = (c >= lo && c <= hi) ? x[c] : SWA_NEG_INF;
      }
      // Row max of this half as a tree (eight independent chains), in the log2 domain.
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = x[i];
#pragma unroll
      for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], x[c]);
      float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
      float mx_other;
      if (!(ok = exchange(j, mx, &mx_other))) break;
      mx = fmaxf(mx, mx_other);
      // Both halves of a row see the same maxima, so they take the same decisions below.
      const float m_new = fmaxf(m_ref, mx);
      const bool resc = m_new > m_ref + kRescaleThreshold;
      float factor = 1.f;
      if (resc) {
        factor = ex2(m_ref - m_new);  // 0 when m_ref is -inf
        l *= factor;
        m_ref = m_new;
      }
      const float m_use = (m_ref == SWA_NEG_INF) ? 0.f : m_ref;
      uint32_t pk[32];
      float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        // p = 2^(scale log2(e) S - m): one FFMA and one MUFU.EX2 per score
        const float p0 = ex2(fmaf(x[2 * c], sl2, -m_use)), p1 = ex2(fmaf(x[2 * c + 1], sl2, -m_use));
        rs8[c & 7] += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));

      // P buffer (j & 1) was last read by P_{j-2} V_{j-2}.
      if (j >= 2 && !(ok = warp_wait(bar(C::kPVDone + sb), ((j - 2) >> 1) & 1, &abort_flag, a.err)))
        break;
      // Rescaling O needs P_{j-1} V_{j-1} (and so every earlier one) to have landed.
      if (j >= 1 && __any_sync(0xffffffffu, resc)) {
        if (!(ok = warp_wait(bar(C::kPVDone + (sb ^ 1)), ((j - 1) >> 1) & 1, &abort_flag, a.err)))
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
      // keys [64h, 64h+64) -> packed P columns [32h, 32h+32)
      tmem_st32(tmem + lane_base + C::kColP + 64u * sb + 32u * h, pk);
      tmem_wait_st();
      warp_arrive(bar(C::kPFull + sb));
    }
    float l_other = 0.f;
    if (ok) ok = exchange(nkv, l, &l_other);
    const int last = nkv - 1;
    if (ok && warp_wait(bar(C::kPVDone + (last & 1)), (last >> 1) & 1, &abort_flag, a.err)) {
      tc_fence_after();
      const float l_row = l + l_other;
      const float inv_l = 1.f / l_row;
      const float m_use = (m_ref == SWA_NEG_INF) ? 0.f : m_ref;
      const bool in_range = row < a.N;
      const size_t grow = static_cast<size_t>(bh) * a.N + row;
      if (in_range && h == 0) a.lse[grow] = (m_use + log2f(l_row)) * kLn2;
      // O / l -> bf16, staged in the Q tile (free: every S MMA has completed) in the swizzled layout
      // of the TMA map, then written with one tensor store per 64-column chunk (rows past N are
      // not written).
      constexpr int kHalf = D / 2;
      uint32_t rr[kHalf / 32][32];
#pragma unroll
      for (int c4 = 0; c4 < kHalf / 32; ++c4)
        tmem_ld32(tmem + lane_base + C::kColO + kHalf * h + 32u * c4, rr[c4]);
      tmem_wait_ld_all();
#pragma unroll
      for (int c4 = 0; c4 < kHalf / 32; ++c4) {
        reg_fence(rr[c4]);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(rr[c4][2 * i]) * inv_l,
                              __uint_as_float(rr[c4][2 * i + 1]) * inv_l);
        stage_row32_sw128(sQ, r, kHalf * h + 32u * c4, pk);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kOutFull));
      if (warp == 0 && warp_wait(bar(C::kOutFull), 0, &abort_flag, a.err) && lane == 0) {
        for (int hh = 0; hh < C::kChunks; ++hh) tma_store_3d(&tm_o, sQ + hh * C::kChunkBytes, 64 * hh, q0, bh);
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

template <int D>
cudaError_t launch_fwd_d(const Problem& pb, const void* q, const void* k, const void* v, void* o,
                         float* lse, cudaStream_t stream) {
  using C = FwdCfg<D>;
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_bf16_3d(&tq, q, static_cast<uint64_t>(pb.B) * pb.Hq, pb.N, D, kBlockM) ||
      !make_tmap_bf16_3d(&to, o, static_cast<uint64_t>(pb.B) * pb.Hq, pb.N, D, kBlockM) ||
      !make_tmap_bf16_3d(&tk, k, static_cast<uint64_t>(pb.B) * pb.Hkv, pb.N, D, kBlockN) ||
      !make_tmap_bf16_3d(&tv, v, static_cast<uint64_t>(pb.B) * pb.Hkv, pb.N, D, kBlockN))
    return cudaErrorInvalidValue;
  auto kern = swa_fwd_kernel<D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.BH = pb.B * pb.Hq;
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.G = pb.Hq / pb.Hkv;
  a.N = pb.N;
  a.W = pb.W;
  a.nqb = (pb.N + kBlockM - 1) / kBlockM;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  const unsigned grid = static_cast<unsigned>(a.nqb) * static_cast<unsigned>(a.BH);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Problem& pb, const void* q, const void* k, const void* v, void* o,
                       float* lse, cudaStream_t stream) {
  if (pb.D == 64) return launch_fwd_d<64>(pb, q, k, v, o, lse, stream);
  if (pb.D == 128) return launch_fwd_d<128>(pb, q, k, v, o, lse, stream);
  return cudaErrorInvalidValue;
}

}  // namespace swa
