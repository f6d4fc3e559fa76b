// swa_kernels.h — launch interface between the C ABI (swa_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace swa {

// Bits of the per-device error word that kernels set (read and cleared by swa_check_device).
constexpr unsigned kErrWaitTimeout = 1u;  // an mbarrier wait ran out
constexpr unsigned kErrSmemLayout = 2u;   // dynamic shared memory not 1024-byte aligned; the
                                          // kernel returned before any barrier or memory use

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // key rows per tile

// Window geometry.  Queries i in [0, Lq), keys j in [0, Lk), Lq <= Lk; query i sits at key
// position i + off, off = Lk - Lq (the queries are the suffix of the key sequence).  Key j is
// visible to query i iff dmin <= i + off - j <= dmax: [0, W - 1] for a causal sliding window (the
// query itself included), [-(W - 1), W - 1] for a non-causal one.  Every query sees at least the
// key at its own position.  The host and the kernels use these same functions for the block walks.
struct Span {
  int Lq, Lk, off, dmin, dmax;

  // Key blocks a query block [q0, q0 + kBlockM) visits (never empty for q0 < Lq).
  __host__ __device__ int first_kblock(int q0) const {
    const int lo = q0 + off - dmax;
    return lo > 0 ? lo / kBlockN : 0;
  }
  __host__ __device__ int last_kblock(int q0) const {
    const int q_last = (q0 + kBlockM - 1 < Lq - 1) ? q0 + kBlockM - 1 : Lq - 1;
    const int hi = q_last + off - dmin;
    return (hi < Lk - 1 ? hi : Lk - 1) / kBlockN;
  }
  // Query blocks a key block [k0, k0 + kBlockN) is visited by; first > last when none is.
  __host__ __device__ int first_qblock(int k0) const {
    const int lo = k0 + dmin - off;
    return lo > 0 ? lo / kBlockM : 0;
  }
  __host__ __device__ int last_qblock(int k0) const {
    const long long k_last = (k0 + kBlockN - 1 < Lk - 1) ? k0 + kBlockN - 1 : Lk - 1;
    const long long hi = k_last + dmax - off;
    if (hi < 0) return -1;
    return static_cast<int>((hi < Lq - 1 ? hi : Lq - 1) / kBlockM);
  }
  // True when every cell of the (query block q0, key block k0) tile is visible and inside both
  // sequences, so the tile needs no mask.
  __host__ __device__ bool interior(int q0, int k0) const {
    return q0 + off - (k0 + kBlockN - 1) >= dmin && q0 + kBlockM - 1 + off - k0 <= dmax &&
           k0 + kBlockN <= Lk && q0 + kBlockM <= Lq;
  }
};

// Shape and window of one call.  Query tensors (q, o, dO, dq) are contiguous [B, Hq, Lq, D], key
// tensors (k, v, dk, dv) [B, Hkv, Lk, D], LSE and Delta [B, Hq, Lq].
struct Problem {
  int B, Hq, Hkv, D;
  Span span;
  float scale;    // softmax scale
  unsigned* err;  // per-device error word (bounded-wait timeouts)
  int f16 = 0;    // element type of every tensor but LSE / Delta: 0 = bf16, 1 = fp16
};

// Division by a divisor fixed for a launch, without a divide instruction: for 0 <= n < 2^31 and
// 1 <= d < 2^31, n / d = (umulhi(n, m) + n) >> s with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1 (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994; umulhi(n, m) <= n, so the sum does not overflow 32 bits).  Persistent
// kernels split their tile index with it: a runtime division costs a MUFU reciprocal, which queues
// behind the softmax exponentials.
struct FastDiv {
  uint32_t d = 1, m = 1, s = 0;
  FastDiv() = default;
  explicit FastDiv(uint32_t divisor) : d(divisor) {
    s = 0;
    while ((1ull << s) < d) ++s;
    m = static_cast<uint32_t>((((1ull << 32) * ((1ull << s) - d)) / d) + 1);
  }
  __host__ __device__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
    const uint32_t hi = __umulhi(n, m);
#else
    const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(n) * m) >> 32);
#endif
    return (hi + n) >> s;
  }
  __host__ __device__ uint32_t mod(uint32_t n) const { return n - div(n) * d; }
};

// Streaming multiprocessors of the current device (cached per device); persistent kernels launch
// one CTA per SM.
// The cache is filled under a mutex, so host threads calling concurrently see a complete value.
inline int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Clusters of two CTAs of the pair kernel `Kernel` (launched with `threads` threads and `smem` bytes
// of dynamic shared memory) that can be resident at once, cached per device and kernel; half the
// SM count when the occupancy query fails.
template <auto Kernel>
int max_pair_clusters(int threads, int smem) {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return sm_count() / 2;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (sm_count() / 2)));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, Kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = sm_count() / 2;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// Launchers (each returns the launch's cudaError_t).
cudaError_t launch_fwd(const Problem& pb, const void* q, const void* k, const void* v, void* o,
                       float* lse, cudaStream_t stream);
// Forward on CTA pairs (swa_fwd_pair.cu): D = 128 with an even number of query heads per kv
// head; launch_fwd dispatches there when it applies.
bool fwd_pair_applies(const Problem& pb);
cudaError_t launch_fwd_pair(const Problem& pb, const void* q, const void* k, const void* v,
                            void* o, float* lse, cudaStream_t stream);
cudaError_t launch_bwd_delta(const Problem& pb, const void* o, const void* dO, float* delta,
                             cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const Problem& pb, const void* q, const void* k, const void* v,
                            const void* dO, const float* lse, const float* delta, void* dk,
                            void* dv, cudaStream_t stream);
cudaError_t launch_bwd_dq(const Problem& pb, const void* q, const void* k, const void* v,
                          const void* dO, const float* lse, const float* delta, void* dq,
                          cudaStream_t stream);
// dQ on CTA pairs (swa_bwd_dq_pair.cu): D = 128 with an even number of query heads per kv head;
// launch_bwd_dq dispatches there when it applies.
bool dq_pair_applies(const Problem& pb);
cudaError_t launch_dq_pair(const Problem& pb, const void* q, const void* k, const void* v,
                           const void* dO, const float* lse, const float* delta, void* dq,
                           cudaStream_t stream);

// Fused backward (swa_bwd_fused.cu): dK, dV and the dQ partials of every (key block, query tile)
// pair in one kernel.  dQ accumulates in fp32, tile-major: block (bhq, qb) holds query rows
// [128 qb, 128 qb + 128) of plane bhq, as groups of 4 head-dimension columns: column c of block
// row r sits at (c / 4) * 512 + r * 4 + c % 4, so the 4 columns of 32 consecutive rows (one warp's
// vector reduce-add) are 512 contiguous bytes.  Offsets in floats.
__host__ __device__ inline size_t dq_acc_offset(int bhq, int qb, int row, int col, int nqb, int D) {
  return (static_cast<size_t>(bhq) * nqb + qb) * (static_cast<size_t>(kBlockM) * D) +
         static_cast<size_t>(col / 4) * (kBlockM * 4) + row * 4 + col % 4;
}
// Bytes of the accumulator for B x Hq planes of Lq query rows.
inline size_t dq_acc_bytes(int B, int Hq, int Lq, int D) {
  const size_t nqb = static_cast<size_t>((Lq + kBlockM - 1) / kBlockM);
  return static_cast<size_t>(B) * Hq * nqb * kBlockM * D * sizeof(float);
}
cudaError_t launch_bwd_fused(const Problem& pb, const void* q, const void* k, const void* v,
                             const void* dO, const float* lse, const float* delta, float* dq_acc,
                             void* dk, void* dv, cudaStream_t stream);
// Delta as launch_bwd_delta, also zeroing the whole accumulator.
cudaError_t launch_bwd_delta_zero_acc(const Problem& pb, const void* o, const void* dO,
                                      float* delta, float* dq_acc, cudaStream_t stream);
// dq = scale * accumulator, rounded to the element type (rows [0, Lq) of every plane).
cudaError_t launch_dq_from_acc(const Problem& pb, const float* dq_acc, void* dq,
                               cudaStream_t stream);

// Head dimension 256 (swa_d256.cu): the same operations with half-tile streaming; dK and dV come
// from two kernels.  launch_fwd / launch_bwd_dq / launch_bwd_dkdv dispatch here for D = 256.
cudaError_t launch_fwd_d256(const Problem& pb, const void* q, const void* k, const void* v,
                            void* o, float* lse, cudaStream_t stream);
cudaError_t launch_dq_d256(const Problem& pb, const void* q, const void* k, const void* v,
                           const void* dO, const float* lse, const float* delta, void* dq,
                           cudaStream_t stream);
// D = 256 forward on CTA pairs (swa_d256_fwd_pair.cu), for an even number of query heads per kv
// head; launch_fwd_d256 dispatches there when it applies.
bool fwd256_pair_applies(const Problem& pb);
cudaError_t launch_fwd256_pair(const Problem& pb, const void* q, const void* k, const void* v,
                               void* o, float* lse, cudaStream_t stream);
// D = 256 dK and dV on CTA pairs over neighbouring key blocks (swa_d256_dkdv_pair.cu);
// launch_dkdv_d256 dispatches there when it applies.
bool dkdv256_pair_applies(const Problem& pb);
cudaError_t launch_dkdv256_pair(const Problem& pb, const void* q, const void* k, const void* v,
                                const void* dO, const float* lse, const float* delta, void* dk,
                                void* dv, cudaStream_t stream);
// D = 256 dQ on CTA pairs (swa_d256_dq_pair.cu), for an even number of query heads per kv head;
// launch_dq_d256 dispatches there when it applies.
bool dq256_pair_applies(const Problem& pb);
cudaError_t launch_dq256_pair(const Problem& pb, const void* q, const void* k, const void* v,
                              const void* dO, const float* lse, const float* delta, void* dq,
                              cudaStream_t stream);
cudaError_t launch_dkdv_d256(const Problem& pb, const void* q, const void* k, const void* v,
                             const void* dO, const float* lse, const float* delta, void* dk,
                             void* dv, cudaStream_t stream);

// One block whose single bounded wait runs out (the failure path of every kernel's waits).
cudaError_t launch_wait_timeout_selftest(unsigned* err, cudaStream_t stream);

// fp32 tensors around the bf16 kernels: up to four tensors per launch, each a whole number of
// 8-element units (end[t] = units of tensors 0..t, cumulative; unused entries repeat the total).
constexpr int kMaxJobTensors = 4;
struct RoundJob {  // fp32 -> bf16, round to nearest even
  const float* src[kMaxJobTensors];
  uint16_t* dst[kMaxJobTensors];
  uint16_t* lo[kMaxJobTensors];  // if set: the residual x - bf16(x), itself rounded to bf16
  long long end[kMaxJobTensors];
};
struct WidenJob {  // bf16 -> fp32, exact
  const uint16_t* src[kMaxJobTensors];
  float* dst[kMaxJobTensors];
  long long end[kMaxJobTensors];
};
cudaError_t launch_round_bf16(const RoundJob& job, cudaStream_t stream);
cudaError_t launch_widen_bf16(const WidenJob& job, cudaStream_t stream);
// Delta from fp32 O and dO, also writing dO rounded to bf16 (Delta uses the rounded dO).
cudaError_t launch_delta_f32(const Problem& pb, const float* o, const float* dO, float* delta,
                             void* do16, cudaStream_t stream);
// First-order correction of the log-sum-exp for the residuals of a split of q and k into bf16
// high and low parts: lse += scale * (<q_hi, b> + <q_lo, a>) per query row, where a and b are the
// forward's outputs with k_hi and k_lo in place of v (all four [B, Hq, Lq, D] bf16).
cudaError_t launch_lse_correct(const Problem& pb, const void* q_hi, const void* q_lo,
                               const void* a, const void* b, float* lse, cudaStream_t stream);

}  // namespace swa
