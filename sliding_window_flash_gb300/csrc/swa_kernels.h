// swa_kernels.h — launch interface between the C ABI (swa_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace swa {

// Bits of the per-device error word that kernels set (read and cleared by swa_check_device).
constexpr unsigned kErrWaitTimeout = 1u;  // an mbarrier wait ran out
constexpr unsigned kErrSmemLayout = 2u;   // dynamic shared memory not 1024-byte aligned; the
                                          // kernel returned before any barrier or memory use

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // key rows per tile

// Shape and window of one call.  All tensors are contiguous [B, H, N, D].
struct Problem {
  int B, Hq, Hkv, N, D;
  int W;          // window, already clamped to N (W >= N is plain causal)
  float scale;    // softmax scale
  unsigned* err;  // per-device error word (bounded-wait timeouts)
  int f16 = 0;    // element type of every tensor but LSE / Delta: 0 = bf16, 1 = fp16
};

// First and last key block a query block visits, and the same for key blocks, so that the host
// and the kernels agree on the walk.  Window rule: query i sees key j iff 0 <= i - j < W.
__host__ __device__ inline int fwd_first_kblock(int q0, int W) {
  const int lo = q0 - W + 1;
  return lo > 0 ? lo / kBlockN : 0;
}
__host__ __device__ inline int fwd_last_kblock(int q0, int N) {
  const int hi = q0 + kBlockM - 1;
  return (hi < N - 1 ? hi : N - 1) / kBlockN;
}
__host__ __device__ inline int bwd_first_qblock(int k0) { return k0 / kBlockM; }
__host__ __device__ inline int bwd_last_qblock(int k0, int N, int W) {
  const long long hi = static_cast<long long>(k0) + kBlockN - 1 + W - 1;
  return static_cast<int>((hi < N - 1 ? hi : N - 1) / kBlockM);
}

// Streaming multiprocessors of the current device (cached per device); persistent kernels launch
// one CTA per SM.
inline int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Launchers (each returns the launch's cudaError_t).
cudaError_t launch_fwd(const Problem& pb, const void* q, const void* k, const void* v, void* o,
                       float* lse, cudaStream_t stream);
cudaError_t launch_bwd_delta(const Problem& pb, const void* o, const void* dO, float* delta,
                             cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const Problem& pb, const void* q, const void* k, const void* v,
                            const void* dO, const float* lse, const float* delta, void* dk,
                            void* dv, cudaStream_t stream);
cudaError_t launch_bwd_dq(const Problem& pb, const void* q, const void* k, const void* v,
                          const void* dO, const float* lse, const float* delta, void* dq,
                          cudaStream_t stream);

}  // namespace swa
