// swa_bwd_delta.cu — backward preprocess: Delta[i] = sum_d dO[i, d] * O[i, d] (fp32), one value
// per query row of every (batch, query head).  It is the row-sum that turns the softmax Jacobian
// into dS = P * (dP - Delta) in the dK/dV and dQ kernels.
//
// Bandwidth-bound: every row's O and dO are read once (2 * D * 2 bytes) and 4 bytes are written.
// Each lane loads 16 bytes of O and of dO (8 bf16 or fp16), D/8 lanes cover a row, and the partial
// sums are combined with xor-shuffles inside those lanes.  The grid is a whole number of waves
// over the 152 SMs and walks the rows with a grid stride.
#include "swa_kernels.h"
#include "swa_ptx.cuh"

namespace swa {
namespace {

template <int D, bool F16>
__global__ void __launch_bounds__(256) swa_delta_kernel(const uint16_t* __restrict__ o,
                                                        const uint16_t* __restrict__ dO,
                                                        float* __restrict__ delta,
                                                        long long rows) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int sub = lane % kLanesPerRow;
  const long long warp_global =
      (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long warps_total = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long base = warp_global * kRowsPerWarp; base < rows;
       base += warps_total * kRowsPerWarp) {
    const long long row = base + lane / kLanesPerRow;
    float acc = 0.f;
    if (row < rows) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + sub);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(dO + row * D) + sub);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa = Elem<F16>::unpack(av[i]);
        const float2 fb = Elem<F16>::unpack(bv[i]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0 && row < rows) delta[row] = acc;
  }
}

}  // namespace

cudaError_t launch_bwd_delta(const Problem& pb, const void* o, const void* dO, float* delta,
                             cudaStream_t stream) {
  const long long rows = static_cast<long long>(pb.B) * pb.Hq * pb.span.Lq;
  constexpr int kThreads = 256;
  const long long rows_per_block = (kThreads / 32) * (32 / (pb.D / 8));
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = 152ll * 8 * 4;  // 4 waves of 8 resident 256-thread blocks per SM
  if (blocks > cap) blocks = cap;
  const auto* po = static_cast<const uint16_t*>(o);
  const auto* pd = static_cast<const uint16_t*>(dO);
  const dim3 grid(static_cast<unsigned>(blocks));
  if (pb.D == 64 && !pb.f16)
    swa_delta_kernel<64, false><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows);
  else if (pb.D == 64)
    swa_delta_kernel<64, true><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows);
  else if (pb.D == 128 && !pb.f16)
    swa_delta_kernel<128, false><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows);
  else if (pb.D == 128)
    swa_delta_kernel<128, true><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows);
  else if (pb.D == 256 && !pb.f16)
    swa_delta_kernel<256, false><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows);
  else if (pb.D == 256)
    swa_delta_kernel<256, true><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace swa
