// swa_bwd_dq_acc.cu — last step of the fused backward: dQ = scale * (sum of the dQ partials), read
// from the tile-major fp32 accumulator the fused kernel adds into (layout: dq_acc_offset in
// swa_kernels.h) and rounded once to the element type (bf16 or fp16, nearest even).
//
// Bandwidth-bound: 4 bytes read and 2 written per element.  Each thread handles one 16-byte unit of
// output (8 elements of a row): two 16-byte loads from the accumulator (two column groups), one
// 16-byte store; the grid walks the units with a grid stride.
#include "swa_kernels.h"
#include "swa_ptx.cuh"

namespace swa {
namespace {

template <int D, bool F16>
__global__ void __launch_bounds__(256)
    swa_dq_from_acc_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                           long long units, int Lq, int nqb, float scale) {
  constexpr int kUnitsPerRow = D / 8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
       u += stride) {
    const long long row = u / kUnitsPerRow;
    const int d0 = 8 * static_cast<int>(u % kUnitsPerRow);
    const int bhq = static_cast<int>(row / Lq), i = static_cast<int>(row % Lq);
    const float* p = acc + dq_acc_offset(bhq, i / kBlockM, i % kBlockM, d0, nqb, D);
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p + kBlockM * 4));  // columns d0+4..+7
    uint4 o;
    o.x = Elem<F16>::pack(a.x * scale, a.y * scale);
    o.y = Elem<F16>::pack(a.z * scale, a.w * scale);
    o.z = Elem<F16>::pack(b.x * scale, b.y * scale);
    o.w = Elem<F16>::pack(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[u] = o;
  }
}

}  // namespace

cudaError_t launch_dq_from_acc(const Problem& pb, const float* dq_acc, void* dq,
                               cudaStream_t stream) {
  const long long units = static_cast<long long>(pb.B) * pb.Hq * pb.span.Lq * (pb.D / 8);
  if (units == 0) return cudaSuccess;
  constexpr int kThreads = 256;
  long long blocks = (units + kThreads - 1) / kThreads;
  const long long cap = static_cast<long long>(sm_count()) * 8 * 4;
  if (blocks > cap) blocks = cap;
  const int Lq = pb.span.Lq, nqb = (Lq + kBlockM - 1) / kBlockM;
  auto* out = static_cast<uint16_t*>(dq);
  const dim3 grid(static_cast<unsigned>(blocks));
  if (pb.D == 64 && !pb.f16)
    swa_dq_from_acc_kernel<64, false><<<grid, kThreads, 0, stream>>>(dq_acc, out, units, Lq, nqb, pb.scale);
  else if (pb.D == 64)
    swa_dq_from_acc_kernel<64, true><<<grid, kThreads, 0, stream>>>(dq_acc, out, units, Lq, nqb, pb.scale);
  else if (pb.D == 128 && !pb.f16)
    swa_dq_from_acc_kernel<128, false><<<grid, kThreads, 0, stream>>>(dq_acc, out, units, Lq, nqb, pb.scale);
  else if (pb.D == 128)
    swa_dq_from_acc_kernel<128, true><<<grid, kThreads, 0, stream>>>(dq_acc, out, units, Lq, nqb, pb.scale);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace swa
