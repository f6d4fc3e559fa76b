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

// With dq_acc set (the fused backward), the grid also zeroes the acc_floats floats of the dQ
// accumulator, with 16-byte stores in a grid-stride walk of its own.
template <int D, bool F16>
__global__ void __launch_bounds__(256) swa_delta_kernel(const uint16_t* __restrict__ o,
                                                        const uint16_t* __restrict__ dO,
                                                        float* __restrict__ delta,
                                                        long long rows, float* __restrict__ dq_acc,
                                                        long long acc_floats) {
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
  if (dq_acc != nullptr) {
    const long long n4 = acc_floats / 4;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < n4;
         u += stride)
      reinterpret_cast<float4*>(dq_acc)[u] = z;
  }
}

}  // namespace

namespace {

cudaError_t delta_impl(const Problem& pb, const void* o, const void* dO, float* delta,
                       float* dq_acc, cudaStream_t stream) {
  const long long rows = static_cast<long long>(pb.B) * pb.Hq * pb.span.Lq;
  constexpr int kThreads = 256;
  const long long rows_per_block = (kThreads / 32) * (32 / (pb.D / 8));
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = 152ll * 8 * 4;  // 4 waves of 8 resident 256-thread blocks per SM
  if (blocks > cap) blocks = cap;
  const auto* po = static_cast<const uint16_t*>(o);
  const auto* pd = static_cast<const uint16_t*>(dO);
  const dim3 grid(static_cast<unsigned>(blocks));
  const long long acc_floats =
      dq_acc != nullptr ? static_cast<long long>(dq_acc_bytes(pb.B, pb.Hq, pb.span.Lq, pb.D) / 4) : 0;
  if (pb.D == 64 && !pb.f16)
    swa_delta_kernel<64, false><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows, dq_acc, acc_floats);
  else if (pb.D == 64)
    swa_delta_kernel<64, true><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows, dq_acc, acc_floats);
  else if (pb.D == 128 && !pb.f16)
    swa_delta_kernel<128, false><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows, dq_acc, acc_floats);
  else if (pb.D == 128)
    swa_delta_kernel<128, true><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows, dq_acc, acc_floats);
  else if (pb.D == 256 && !pb.f16 && dq_acc == nullptr)
    swa_delta_kernel<256, false><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows, nullptr, 0);
  else if (pb.D == 256 && dq_acc == nullptr)
    swa_delta_kernel<256, true><<<grid, kThreads, 0, stream>>>(po, pd, delta, rows, nullptr, 0);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_delta(const Problem& pb, const void* o, const void* dO, float* delta,
                             cudaStream_t stream) {
  return delta_impl(pb, o, dO, delta, nullptr, stream);
}

cudaError_t launch_bwd_delta_zero_acc(const Problem& pb, const void* o, const void* dO,
                                      float* delta, float* dq_acc, cudaStream_t stream) {
  if (dq_acc == nullptr) return cudaErrorInvalidValue;
  return delta_impl(pb, o, dO, delta, dq_acc, stream);
}

}  // namespace swa
