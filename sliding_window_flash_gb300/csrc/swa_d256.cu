// swa_d256.cu — sliding-window attention with head dimension 256 on sm_103a: the single-CTA
// forward and dQ kernels ("Off NVIDIA, you fix the platform yourself", Lab 28 record, numbers
// entry "Attention backward memory": Gemma 4's sliding layers use 256-wide heads), which run when
// the number of query heads per kv head is odd, and the D = 256 entry points.  An even number of
// query heads per kv head runs the forward and dQ on CTA pairs (swa_d256_fwd_pair.cu,
// swa_d256_dq_pair.cu); dK and dV always run on CTA pairs (swa_d256_dkdv_pair.cu).
//
// The D <= 128 kernels keep whole 128-row operand tiles in shared memory and both dK and dV in
// TMEM.  At D = 256 a 128-row tile is 64 KB and dK + dV alone would fill the 512 TMEM columns, so
// these kernels are built differently:
//   * operands move as half-tiles (128 rows x 128 columns, two 64-column 128B-swizzled chunks,
//     32 KB) through a ring of slots, numbered in the order the MMA warp consumes them; two TMA
//     warps fill alternate items (one warp's copies complete at only ~40 B/clk);
//   * a product over D is two 8-step MMA groups (one per half-tile); a product with N = D is two
//     N = 128 MMAs into the two halves of a 256-column accumulator;
//   * the backward's dK and dV come from separate kernels, each with its 256-column accumulator in
//     TMEM (dV: S^T double-buffered next to it; dK: S^T and dP^T next to it).
// Probabilities and dS go back to TMEM as packed 16-bit pairs over the score columns they came
// from (each half-row thread over the first 32 of its 64 columns); an MMA reading them as the A
// operand is always issued before the MMA that overwrites those columns, and one thread's
// tcgen05.mma operations run in issue order.
//
// Windows, query offsets (Lq <= Lk), masking and the block walks are the D <= 128 kernels' (Span).
#include "swa_kernels.h"
#include "swa_ptx.cuh"
#include "swa_tmap.h"
#include "swa_d256.cuh"

namespace swa {
namespace {

constexpr int kD = 256;
constexpr int kHalfBytes = kBlockM * 128 * 2;  // one half-tile: 128 rows x 128 columns, 16-bit
constexpr int kChunk = kBlockM * 128;          // one 64-column chunk: 128 rows x 128 bytes
constexpr int kFullBytes = 2 * kHalfBytes;     // a whole 128 x 256 tile

// ------------------------------------------------------------------------------------------------
// Half-tile ring.  Item i sits in slot i % kSlots; its producer is warp (i & 1) of the two TMA
// warps.  full[s] completes when an item has landed, empty[s] when the MMA reading it has.
// ------------------------------------------------------------------------------------------------
struct Item {
  const CUtensorMap* map;
  int half;  // column half 0 / 1 (columns 128 half .. +127)
  int row;   // first row (query or key position)
  int bh;    // (batch, head) plane
};

template <int kSlots>
struct Ring {
  uint32_t base;       // shared address of slot 0
  uint32_t full0;      // barrier of slot 0 (full); slot s at +8 s
  uint32_t empty0;     // barrier of slot 0 (empty)
  __device__ uint32_t slot(int i) const { return base + (i % kSlots) * kHalfBytes; }
  __device__ uint32_t full(int i) const { return full0 + 8u * (i % kSlots); }
  __device__ uint32_t empty(int i) const { return empty0 + 8u * (i % kSlots); }
  __device__ uint32_t parity(int i) const { return (i / kSlots) & 1; }
};

// Loads item i (called by its producer lane): waits for the slot's previous item to be consumed.
template <int kSlots>
__device__ __forceinline__ bool ring_load(const Ring<kSlots>& rg, int i, const Item& it,
                                          volatile int* abort_flag, unsigned* err) {
  if (i >= kSlots && !mbar_wait(rg.empty(i), ((i / kSlots) - 1) & 1, abort_flag, err)) return false;
  const uint32_t dst = rg.slot(i);
  mbar_arrive_expect_tx(rg.full(i), kHalfBytes);
  tma_load_3d(dst, it.map, rg.full(i), 128 * it.half, it.row, it.bh);
  tma_load_3d(dst + kChunk, it.map, rg.full(i), 128 * it.half + 64, it.row, it.bh);
  return true;
}

struct Args256 {
  const float* lse;      // backward input
  float* lse_out;        // forward output
  const float* delta;
  uint16_t* dq;          // dQ kernel output (bf16 or fp16 elements)
  int BH, Hq, Hkv, G;    // B * Hq, heads, G = Hq / Hkv
  int nqb, ntiles;       // query blocks per head, B * Hq * nqb
  Span span;
  float scale, scale_log2;  // softmax scale, scale * log2(e)
  unsigned* err;
};

struct QTile {
  int bh, bhk, q0, kb_lo, nkv;
};

// Query tile t: heaviest query blocks first (a causal window gives later blocks more key blocks).
__device__ __forceinline__ QTile qtile(int t, const Args256& a, const Span& sp) {
  QTile f;
  const int qb = a.nqb - 1 - t / a.BH;
  f.bh = t % a.BH;
  f.bhk = (f.bh / a.Hq) * a.Hkv + (f.bh % a.Hq) / a.G;
  f.q0 = qb * kBlockM;
  f.kb_lo = sp.first_kblock(f.q0);
  f.nkv = sp.last_kblock(f.q0) - f.kb_lo + 1;
  return f;
}

// ================================================================================================
// Forward: O = softmax(scale Q K^T, window) V and LSE for one 128-row query tile per iteration.
// Persistent (one CTA per SM).  Warps (384 threads): 0-7 softmax, two threads per row as in the
// D <= 128 forward (warp w: TMEM lanes 32 (w % 4).., score columns [64 h, 64 h + 64), h = w / 4);
// 8 and 11 TMA producers of the K / V ring; 9 MMA issuer and TMEM owner; 10 loads each tile's Q
// and stores its O (staged in the Q buffer once every S of the tile has completed).
// Ring order per tile of n key blocks: K_0, then per block j: K_{j+1} (if any), V_j (two halves
// each) — the order in which S_{j+1} is issued ahead of O += P_j V_j.
// TMEM: [0,128) S / P buffer 0, [128,256) S / P buffer 1, [256,512) O.
// ================================================================================================

struct F256 {
  static constexpr int kSlots = 5;
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kOffQ + kFullBytes;
  static constexpr int kOffRed = kOffRing + kSlots * kHalfBytes;  // [2 slots][2 halves][128] fp32
  static constexpr int kOffBar = kOffRed + 2 * 2 * kBlockM * 4;
  static constexpr int kQFull = 0;
  static constexpr int kFull = 1;
  static constexpr int kEmpty = kFull + kSlots;
  static constexpr int kSFull = kEmpty + kSlots;  // 2
  static constexpr int kPFull = kSFull + 2;       // 2
  static constexpr int kPVDone = kPFull + 2;      // 2
  static constexpr int kXch = kPVDone + 2;        // [4 lane quarters][2 slots]
  static constexpr int kOEmpty = kXch + 8;        // the O accumulator has been read
  static constexpr int kOutFull = kOEmpty + 1;    // staged O tile complete
  static constexpr int kDrain = kOutFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 48;  // + TMEM address,
  // abort flag, producers' last fills
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kColS = 0, kColO = 256;
  static constexpr int kThreads = 384;
};

template <bool F16>
__global__ void __launch_bounds__(384, 1)
    swa_fwd256_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const Args256 a) {
  using C = F256;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (!smem_base_ok(smem, a.err)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);  // raised by a failed wait
  int* s_last = reinterpret_cast<int*>(tmem_slot + 4);        // producers' last fills
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  float* s_red = reinterpret_cast<float*>(smem + C::kOffRed);
  const Ring<C::kSlots> rg{smem_u32(smem + C::kOffRing), bar(C::kFull), bar(C::kEmpty)};
  const int tile_step = static_cast<int>(gridDim.x);
  const Span sp = a.span;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(C::kQFull), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kFull + s), 1);
      mbar_init(bar(C::kEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kSFull + b), 1);
      mbar_init(bar(C::kPFull + b), 8);
      mbar_init(bar(C::kPVDone + b), 1);
    }
    for (int x = 0; x < 8; ++x) mbar_init(bar(C::kXch + x), 2);  // the two warps of a quarter
    mbar_init(bar(C::kOEmpty), 8);
    mbar_init(bar(C::kOutFull), 8);
    mbar_init(bar(C::kDrain), 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8 || warp == 11) {
    // ------------------------------------------------------------ K / V ring (even / odd items)
    const int p = warp == 8 ? 0 : 1;
    int last[C::kSlots];  // lane 0: last item loaded per slot
    for (int s = 0; s < C::kSlots; ++s) last[s] = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int i = 0;
      bool ok = true;
      auto put_block = [&](const CUtensorMap* m, int k0, int bhk) {
        for (int hf = 0; hf < 2; ++hf, ++i) {
          if (!ok || (i & 1) != p) continue;
          ok = ring_load(rg, i, Item{m, hf, k0, bhk}, &abort_flag, a.err);
          if (ok) last[i % C::kSlots] = i;
        }
      };
      for (int t = blockIdx.x; ok && t < a.ntiles; t += tile_step) {
        const QTile f = qtile(t, a, sp);
        put_block(&tm_k, f.kb_lo * kBlockN, f.bhk);
        for (int j = 0; j < f.nkv; ++j) {
          if (j + 1 < f.nkv) put_block(&tm_k, (f.kb_lo + j + 1) * kBlockN, f.bhk);
          put_block(&tm_v, (f.kb_lo + j) * kBlockN, f.bhk);
        }
      }
    }
    d256::drain_ring<C::kSlots>(last, s_last, p, lane, [&](int i) { return rg.full(i); }, a.err);
  } else if (warp == 10) {
    // ------------------------------------------------------------ Q loads, O stores
    auto load_q = [&](int t) {
      const QTile f = qtile(t, a, sp);
      mbar_arrive_expect_tx(bar(C::kQFull), kFullBytes);
      for (int c = 0; c < 4; ++c)
        tma_load_3d(sQ + c * kChunk, &tm_q, bar(C::kQFull), 64 * c, f.q0, f.bh);
    };
    int last_q = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_o);
      if (static_cast<int>(blockIdx.x) < a.ntiles) {
        load_q(blockIdx.x);
        last_q = 0;
      }
    }
    for (int t = blockIdx.x, it = 0; t < a.ntiles; t += tile_step, ++it) {
      if (!warp_wait(bar(C::kOutFull), it & 1, &abort_flag, a.err)) break;
      if (lane == 0) {
        const QTile f = qtile(t, a, sp);
        for (int c = 0; c < 4; ++c) tma_store_3d(&tm_o, sQ + c * kChunk, 64 * c, f.q0, f.bh);
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
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdO = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockM, 128, false, true);
    int i = 0;  // ring items consumed
    // S_gg = Q_lo K_lo^T + Q_hi K_hi^T into S buffer gg & 1.  That buffer last held P_{gg-2},
    // whose P V was issued before this.
    auto issue_s = [&](int gg) -> bool {
      const uint32_t d = tmem + C::kColS + 128u * (gg & 1);
      for (int hf = 0; hf < 2; ++hf, ++i) {
        if (!warp_wait(rg.full(i), rg.parity(i), &abort_flag, a.err)) return false;
        tc_fence_after();
        umma_ss_kmajor_x8(d, smem_desc_sw128(sQ + hf * kHalfBytes, 16, 1024),
                          smem_desc_sw128(rg.slot(i), 16, 1024), kIdS, hf);
        umma_commit_w(rg.empty(i));
      }
      umma_commit_w(bar(C::kSFull + (gg & 1)));
      return true;
    };
    // O[:, 128 hf ..] (+)= P_gg V_hf, P_gg packed over S buffer gg & 1 (two 32-column halves).
    auto issue_pv = [&](int gg, bool first) -> bool {
      const int pb = gg & 1;
      if (!warp_wait(bar(C::kPFull + pb), (gg >> 1) & 1, &abort_flag, a.err)) return false;
      for (int hf = 0; hf < 2; ++hf, ++i) {
        if (!warp_wait(rg.full(i), rg.parity(i), &abort_flag, a.err)) return false;
        tc_fence_after();
        umma_ts_mnmajor_x8_split(tmem + C::kColO + 128u * hf, tmem + C::kColS + 128u * pb,
                                 smem_desc_sw128(rg.slot(i), kChunk, 1024), kIdO,
                                 first ? 0u : 1u);
        umma_commit_w(rg.empty(i));
      }
      umma_commit_w(bar(C::kPVDone + pb));
      return true;
    };
    int g = 0;  // key blocks issued so far by this CTA
    bool ok = true;
    for (int t = blockIdx.x, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const QTile f = qtile(t, a, sp);
      ok = warp_wait(bar(C::kQFull), it & 1, &abort_flag, a.err);
      if (ok) ok = issue_s(g);
      for (int j = 0; ok && j < f.nkv; ++j) {
        if (j + 1 < f.nkv) ok = issue_s(g + j + 1);
        // The first P V of a tile overwrites O: the previous tile's epilogue must have read it.
        if (ok && j == 0 && it > 0)
          ok = warp_wait(bar(C::kOEmpty), (it - 1) & 1, &abort_flag, a.err);
        if (ok) ok = issue_pv(g + j, j == 0);
      }
      g += f.nkv;
    }
    umma_commit_w(bar(C::kDrain));  // every issued MMA completes before TMEM is released
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    static_assert(C::kPFull - C::kSFull == d256::FwdBar::kPFull &&
                      C::kPVDone - C::kSFull == d256::FwdBar::kPVDone &&
                      C::kXch - C::kSFull == d256::FwdBar::kXch &&
                      C::kOEmpty - C::kSFull == d256::FwdBar::kOEmpty &&
                      C::kOutFull - C::kSFull == d256::FwdBar::kOutFull,
                  "softmax barrier layout");
    const d256::FwdSoftmax cx{tmem + C::kColS, sQ,        s_red,      bar(C::kSFull),
                              &abort_flag,     a.err,     a.scale_log2, a.lse_out};
    d256::fwd_softmax<F16, false>(cx, sp, static_cast<int>(blockIdx.x), tile_step, a.ntiles,
                                  [&](int t) { return qtile(t, a, sp); });
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================================================
// dQ: per 128-row query tile, walking the window's key blocks (the forward's walk),
//   S = Q K_j^T,  P = exp(scale S - LSE) (masked),  dP = dO V_j^T,  dS = P (dP - Delta),
//   dQ += dS K_j,  dQ *= scale at the end.
// Persistent.  Warps (384 threads): 0-7 compute (two threads per row), 8 and 11 TMA producers of
// the K / V ring, 9 MMA issuer and TMEM owner, 10 loads each tile's Q and dO (64 KB each, held for
// the whole tile).  dS goes over the dP columns it came from and is the A operand of dQ += dS K_j;
// dP_{j+1} is issued after that MMA, S_{j+1} as soon as the compute warps have read S_j.  K_j is
// streamed twice (for S_j, then again for dQ += dS_j K_j) because the ring holds only three
// half-tiles next to Q and dO.
// Ring order per tile of n key blocks: K_0, V_0, then per block j: K_{j+1} (if any), K_j,
// V_{j+1} (if any).
// TMEM: [0,128) S, [128,256) dP / dS, [256,512) dQ.
// ================================================================================================
struct Q256 {
  static constexpr int kSlots = 3;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kFullBytes;
  static constexpr int kOffRing = kOffDO + kFullBytes;
  static constexpr int kOffBar = kOffRing + kSlots * kHalfBytes;
  static constexpr int kQDFull = 0;
  static constexpr int kQDEmpty = 1;
  static constexpr int kFull = 2;
  static constexpr int kEmpty = kFull + kSlots;
  static constexpr int kSFull = kEmpty + kSlots;
  static constexpr int kSEmpty = kSFull + 1;
  static constexpr int kDPFull = kSEmpty + 1;
  static constexpr int kDSFull = kDPFull + 1;
  static constexpr int kDQDone = kDSFull + 1;   // a tile's last dQ MMA has completed
  static constexpr int kDQEmpty = kDQDone + 1;  // the epilogue has read the dQ accumulator
  static constexpr int kDrain = kDQEmpty + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 48;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;
  static constexpr int kThreads = 384;
};

template <bool F16>
__global__ void __launch_bounds__(384, 1)
    swa_dq256_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Args256 a) {
  using C = Q256;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (!smem_base_ok(smem, a.err)) return;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int& abort_flag = *reinterpret_cast<int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 4);  // producers' last fills
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sDO = smem_u32(smem + C::kOffDO);
  const Ring<C::kSlots> rg{smem_u32(smem + C::kOffRing), bar(C::kFull), bar(C::kEmpty)};
  const int tile_step = static_cast<int>(gridDim.x);
  const Span sp = a.span;

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(C::kQDFull), 1);
    mbar_init(bar(C::kQDEmpty), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kFull + s), 1);
      mbar_init(bar(C::kEmpty + s), 1);
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSEmpty), 8);
    mbar_init(bar(C::kDPFull), 1);
    mbar_init(bar(C::kDSFull), 8);
    mbar_init(bar(C::kDQDone), 1);
    mbar_init(bar(C::kDQEmpty), 8);
    mbar_init(bar(C::kDrain), 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8 || warp == 11) {
    // ------------------------------------------------------------ K / V ring (even / odd items)
    const int p = warp == 8 ? 0 : 1;
    int last[C::kSlots];  // lane 0: last item loaded per slot
    for (int s = 0; s < C::kSlots; ++s) last[s] = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int i = 0;
      bool ok = true;
      auto put_block = [&](const CUtensorMap* m, int k0, int bhk) {
        for (int hf = 0; hf < 2; ++hf, ++i) {
          if (!ok || (i & 1) != p) continue;
          ok = ring_load(rg, i, Item{m, hf, k0, bhk}, &abort_flag, a.err);
          if (ok) last[i % C::kSlots] = i;
        }
      };
      for (int t = blockIdx.x; ok && t < a.ntiles; t += tile_step) {
        const QTile f = qtile(t, a, sp);
        put_block(&tm_k, f.kb_lo * kBlockN, f.bhk);
        put_block(&tm_v, f.kb_lo * kBlockN, f.bhk);
        for (int j = 0; j < f.nkv; ++j) {
          if (j + 1 < f.nkv) put_block(&tm_k, (f.kb_lo + j + 1) * kBlockN, f.bhk);
          put_block(&tm_k, (f.kb_lo + j) * kBlockN, f.bhk);
          if (j + 1 < f.nkv) put_block(&tm_v, (f.kb_lo + j + 1) * kBlockN, f.bhk);
        }
      }
    }
    d256::drain_ring<C::kSlots>(last, s_last, p, lane, [&](int i) { return rg.full(i); }, a.err);
  } else if (warp == 10) {
    // ------------------------------------------------------------ Q and dO of each tile
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      int last = -1;
      for (int t = blockIdx.x, it = 0; t < a.ntiles; t += tile_step, ++it) {
        const QTile f = qtile(t, a, sp);
        // Q / dO of the previous tile are free once its last S and dP have completed.
        if (it >= 1 && !mbar_wait(bar(C::kQDEmpty), (it - 1) & 1, &abort_flag, a.err)) break;
        mbar_arrive_expect_tx(bar(C::kQDFull), 2 * kFullBytes);
        for (int c = 0; c < 4; ++c) {
          tma_load_3d(sQ + c * kChunk, &tm_q, bar(C::kQDFull), 64 * c, f.q0, f.bh);
          tma_load_3d(sDO + c * kChunk, &tm_do, bar(C::kQDFull), 64 * c, f.q0, f.bh);
        }
        last = it;
      }
      if (last >= 0) drain_wait(bar(C::kQDFull), last & 1, a.err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdSq = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockM, kBlockN, false, false);
    constexpr uint32_t kIdDq = idesc_f16kind(Elem<F16>::kMmaFmt, kBlockM, 128, false, true);
    int i = 0;  // ring items consumed
    // X (+)= A_lo B_lo^T + A_hi B_hi^T over D, B from the next two ring items.
    auto product_d = [&](uint32_t d, uint32_t a_tile) -> bool {
      for (int hf = 0; hf < 2; ++hf, ++i) {
        if (!warp_wait(rg.full(i), rg.parity(i), &abort_flag, a.err)) return false;
        tc_fence_after();
        umma_ss_kmajor_x8(d, smem_desc_sw128(a_tile + hf * kHalfBytes, 16, 1024),
                          smem_desc_sw128(rg.slot(i), 16, 1024), kIdSq, hf);
        umma_commit_w(rg.empty(i));
      }
      return true;
    };
    auto issue_s = [&](int gg) -> bool {  // S = Q K_gg^T once S_{gg-1} has been read
      if (gg >= 1 && !warp_wait(bar(C::kSEmpty), (gg - 1) & 1, &abort_flag, a.err)) return false;
      if (!product_d(tmem + C::kColS, sQ)) return false;
      umma_commit_w(bar(C::kSFull));
      return true;
    };
    auto issue_dp = [&](bool tile_last) -> bool {  // dP = dO V^T (after dQ of the previous block)
      if (!product_d(tmem + C::kColDP, sDO)) return false;
      umma_commit_w(bar(C::kDPFull));
      if (tile_last) umma_commit_w(bar(C::kQDEmpty));  // every S and dP of the tile is issued
      return true;
    };
    auto issue_dq = [&](int gg, bool first, bool tile_last) -> bool {  // dQ += dS K_gg
      if (!warp_wait(bar(C::kDSFull), gg & 1, &abort_flag, a.err)) return false;
      for (int hf = 0; hf < 2; ++hf, ++i) {
        if (!warp_wait(rg.full(i), rg.parity(i), &abort_flag, a.err)) return false;
        tc_fence_after();
        umma_ts_mnmajor_x8_split(tmem + C::kColDQ + 128u * hf, tmem + C::kColDP,
                                 smem_desc_sw128(rg.slot(i), kChunk, 1024), kIdDq,
                                 first ? 0u : 1u);
        umma_commit_w(rg.empty(i));
      }
      if (tile_last) umma_commit_w(bar(C::kDQDone));
      return true;
    };
    int g = 0;  // key blocks issued so far by this CTA
    bool ok = true;
    for (int t = blockIdx.x, it = 0; ok && t < a.ntiles; t += tile_step, ++it) {
      const QTile f = qtile(t, a, sp);
      const int n = f.nkv;
      ok = warp_wait(bar(C::kQDFull), it & 1, &abort_flag, a.err);
      if (ok) ok = issue_s(g);
      if (ok) ok = issue_dp(n == 1);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) ok = issue_s(g + j + 1);
        // The first dQ of a tile overwrites the accumulator: the previous tile's epilogue must
        // have read it.
        if (ok && j == 0 && it > 0)
          ok = warp_wait(bar(C::kDQEmpty), (it - 1) & 1, &abort_flag, a.err);
        if (ok) ok = issue_dq(g + j, j == 0, j + 1 == n);
        if (ok && j + 1 < n) ok = issue_dp(j + 2 == n);
      }
      g += n;
    }
    umma_commit_w(bar(C::kDrain));
    warp_drain_wait(bar(C::kDrain), 0, a.err);
  } else {
    // ------------------------------------------------------------ compute (warps 0-7)
    static_assert(C::kSEmpty - C::kSFull == d256::DqBar::kSEmpty &&
                      C::kDPFull - C::kSFull == d256::DqBar::kDPFull &&
                      C::kDSFull - C::kSFull == d256::DqBar::kDSFull &&
                      C::kDQDone - C::kSFull == d256::DqBar::kDQDone &&
                      C::kDQEmpty - C::kSFull == d256::DqBar::kDQEmpty && C::kColDP == 128 &&
                      C::kColDQ == 256,
                  "dQ compute layout");
    d256::dq_compute<F16, false>(a, sp, tmem + C::kColS, bar(C::kSFull), &abort_flag,
                                 static_cast<int>(blockIdx.x), tile_step,
                                 [&](int t) { return qtile(t, a, sp); });
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================================================
// Host launchers
// ================================================================================================
Args256 make_args(const Problem& pb, const float* lse, const float* delta, void* dq,
                  float* lse_out = nullptr) {
  Args256 a;
  a.lse = lse;
  a.lse_out = lse_out;
  a.delta = delta;
  a.dq = static_cast<uint16_t*>(dq);
  a.BH = pb.B * pb.Hq;
  a.Hq = pb.Hq;
  a.Hkv = pb.Hkv;
  a.G = pb.Hq / pb.Hkv;
  a.nqb = (pb.span.Lq + kBlockM - 1) / kBlockM;
  a.ntiles = a.nqb * a.BH;
  a.span = pb.span;
  a.scale = pb.scale;
  a.scale_log2 = pb.scale * kLog2e;
  a.err = pb.err;
  return a;
}

// Maps of the query-shaped (Lq rows) and key-shaped (Lk rows) tensors of one call.
bool qmap(CUtensorMap* m, const void* p, const Problem& pb) {
  return make_tmap_3d(m, p, static_cast<uint64_t>(pb.B) * pb.Hq, pb.span.Lq, kD, kBlockM, pb.f16);
}
bool kmap(CUtensorMap* m, const void* p, const Problem& pb) {
  return make_tmap_3d(m, p, static_cast<uint64_t>(pb.B) * pb.Hkv, pb.span.Lk, kD, kBlockN, pb.f16);
}

template <typename Kern>
cudaError_t set_smem(Kern kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <bool F16>
cudaError_t fwd256(const Problem& pb, const void* q, const void* k, const void* v, void* o,
                   float* lse, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to;
  if (!qmap(&tq, q, pb) || !qmap(&to, o, pb) || !kmap(&tk, k, pb) || !kmap(&tv, v, pb))
    return cudaErrorInvalidValue;
  auto kern = swa_fwd256_kernel<F16>;
  cudaError_t e = set_smem(kern, F256::kSmemBytes);
  if (e != cudaSuccess) return e;
  const Args256 a = make_args(pb, nullptr, nullptr, nullptr, lse);
  const int grid = a.ntiles < sm_count() ? a.ntiles : sm_count();
  kern<<<grid, F256::kThreads, F256::kSmemBytes, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t dq256(const Problem& pb, const void* q, const void* k, const void* v, const void* dO,
                  const float* lse, const float* delta, void* dq, cudaStream_t stream) {
  CUtensorMap tq, tdo, tk, tv;
  if (!qmap(&tq, q, pb) || !qmap(&tdo, dO, pb) || !kmap(&tk, k, pb) || !kmap(&tv, v, pb))
    return cudaErrorInvalidValue;
  auto kern = swa_dq256_kernel<F16>;
  cudaError_t e = set_smem(kern, Q256::kSmemBytes);
  if (e != cudaSuccess) return e;
  const Args256 a = make_args(pb, lse, delta, dq);
  const int grid = a.ntiles < sm_count() ? a.ntiles : sm_count();
  kern<<<grid, Q256::kThreads, Q256::kSmemBytes, stream>>>(tq, tdo, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_d256(const Problem& pb, const void* q, const void* k, const void* v,
                            void* o, float* lse, cudaStream_t stream) {
  if (fwd256_pair_applies(pb)) return launch_fwd256_pair(pb, q, k, v, o, lse, stream);
  return pb.f16 ? fwd256<true>(pb, q, k, v, o, lse, stream)
                : fwd256<false>(pb, q, k, v, o, lse, stream);
}

cudaError_t launch_dq_d256(const Problem& pb, const void* q, const void* k, const void* v,
                           const void* dO, const float* lse, const float* delta, void* dq,
                           cudaStream_t stream) {
  if (dq256_pair_applies(pb)) return launch_dq256_pair(pb, q, k, v, dO, lse, delta, dq, stream);
  return pb.f16 ? dq256<true>(pb, q, k, v, dO, lse, delta, dq, stream)
                : dq256<false>(pb, q, k, v, dO, lse, delta, dq, stream);
}

cudaError_t launch_dkdv_d256(const Problem& pb, const void* q, const void* k, const void* v,
                             const void* dO, const float* lse, const float* delta, void* dk,
                             void* dv, cudaStream_t stream) {
  return launch_dkdv256_pair(pb, q, k, v, dO, lse, delta, dk, dv, stream);
}

}  // namespace swa
