// swa_f32.cu — fp32 tensors in and out of the bf16 attention kernels.
//
// The tensor cores take bf16 operands, so an fp32 call rounds each input element once to the
// nearest bf16 (ties to even), runs the bf16 kernels on those copies, and widens the bf16 results
// to fp32.  Accumulation, the log-sum-exp and Delta stay fp32 throughout, as in the bf16 path.
// The gradient sweep of "Off NVIDIA, you fix the platform yourself" (Lab 28 record, numbers entry
// "Gradient parity, small shapes") runs fp32 inputs alongside the 16-bit ones.
//
// Three bandwidth-bound kernels, each a grid-stride walk over 8-element units (D is a multiple of
// 8, so a unit never crosses a row):
//   round   up to four fp32 tensors -> bf16 (two 16-byte loads, one 16-byte store per unit);
//   widen   up to four bf16 tensors -> fp32 (one 16-byte load, two 16-byte stores per unit);
//   delta   Delta_i = sum_d bf16(dO_id) * O_id from fp32 O and dO, writing bf16(dO) on the way,
//           so Delta is formed from the same rounded dO that the dP = dO V^T contraction uses
//           (with a one-key window dP - Delta then vanishes exactly, as the exact gradient does).
#include "swa_kernels.h"
#include "swa_ptx.cuh"

namespace swa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int pick(const long long* end, long long u) {
  return u < end[0] ? 0 : u < end[1] ? 1 : u < end[2] ? 2 : 3;
}

__global__ void __launch_bounds__(kThreads) swa_round_bf16_kernel(const RoundJob job) {
  const long long total = job.end[kMaxJobTensors - 1];
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += stride) {
    const int t = pick(job.end, u);
    const long long i = u - (t == 0 ? 0 : job.end[t - 1]);
    const float4* s = reinterpret_cast<const float4*>(job.src[t]) + 2 * i;
    const float4 a = __ldg(s), b = __ldg(s + 1);
    uint4 r;
    r.x = pack_bf16x2(a.x, a.y);
    r.y = pack_bf16x2(a.z, a.w);
    r.z = pack_bf16x2(b.x, b.y);
    r.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(job.dst[t])[i] = r;
  }
}

__global__ void __launch_bounds__(kThreads) swa_widen_bf16_kernel(const WidenJob job) {
  const long long total = job.end[kMaxJobTensors - 1];
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += stride) {
    const int t = pick(job.end, u);
    const long long i = u - (t == 0 ? 0 : job.end[t - 1]);
    const uint4 r = __ldg(reinterpret_cast<const uint4*>(job.src[t]) + i);
    const float2 a = Elem<false>::unpack(r.x), b = Elem<false>::unpack(r.y);
    const float2 c = Elem<false>::unpack(r.z), d = Elem<false>::unpack(r.w);
    float4* o = reinterpret_cast<float4*>(job.dst[t]) + 2 * i;
    o[0] = make_float4(a.x, a.y, b.x, b.y);
    o[1] = make_float4(c.x, c.y, d.x, d.y);
  }
}

// One row per D/8 lanes, as in the bf16 Delta kernel.
template <int D>
__global__ void __launch_bounds__(kThreads)
    swa_delta_f32_kernel(const float* __restrict__ o, const float* __restrict__ dO,
                         float* __restrict__ delta, uint16_t* __restrict__ do16, long long rows) {
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
      const float4* po = reinterpret_cast<const float4*>(o + row * D) + 2 * sub;
      const float4* pd = reinterpret_cast<const float4*>(dO + row * D) + 2 * sub;
      const float4 o0 = __ldg(po), o1 = __ldg(po + 1);
      const float4 d0 = __ldg(pd), d1 = __ldg(pd + 1);
      uint4 r;
      r.x = pack_bf16x2(d0.x, d0.y);
      r.y = pack_bf16x2(d0.z, d0.w);
      r.z = pack_bf16x2(d1.x, d1.y);
      r.w = pack_bf16x2(d1.z, d1.w);
      reinterpret_cast<uint4*>(do16 + row * D)[sub] = r;
      const float ov[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
      const uint32_t rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 g = Elem<false>::unpack(rv[p]);
        acc = fmaf(g.x, ov[2 * p], acc);
        acc = fmaf(g.y, ov[2 * p + 1], acc);
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0 && row < rows) delta[row] = acc;
  }
}

// A whole number of waves of resident 256-thread blocks over the SMs, or fewer when the work is
// smaller.
unsigned grid_for(long long threads_needed) {
  const long long cap = static_cast<long long>(sm_count()) * 8 * 4;
  long long blocks = (threads_needed + kThreads - 1) / kThreads;
  if (blocks > cap) blocks = cap;
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_round_bf16(const RoundJob& job, cudaStream_t stream) {
  const long long total = job.end[kMaxJobTensors - 1];
  if (total == 0) return cudaSuccess;
  swa_round_bf16_kernel<<<grid_for(total), kThreads, 0, stream>>>(job);
  return cudaGetLastError();
}

cudaError_t launch_widen_bf16(const WidenJob& job, cudaStream_t stream) {
  const long long total = job.end[kMaxJobTensors - 1];
  if (total == 0) return cudaSuccess;
  swa_widen_bf16_kernel<<<grid_for(total), kThreads, 0, stream>>>(job);
  return cudaGetLastError();
}

cudaError_t launch_delta_f32(const Problem& pb, const float* o, const float* dO, float* delta,
                             void* do16, cudaStream_t stream) {
  const long long rows = static_cast<long long>(pb.B) * pb.Hq * pb.span.Lq;
  const long long lanes = rows * (pb.D / 8);
  auto* pd = static_cast<uint16_t*>(do16);
  if (pb.D == 64)
    swa_delta_f32_kernel<64><<<grid_for(lanes), kThreads, 0, stream>>>(o, dO, delta, pd, rows);
  else if (pb.D == 128)
    swa_delta_f32_kernel<128><<<grid_for(lanes), kThreads, 0, stream>>>(o, dO, delta, pd, rows);
  else if (pb.D == 256)
    swa_delta_f32_kernel<256><<<grid_for(lanes), kThreads, 0, stream>>>(o, dO, delta, pd, rows);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace swa
