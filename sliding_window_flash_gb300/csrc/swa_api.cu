// swa_api.cu — the C ABI of libswa.so (declared in include/swa_attn.h): argument checks, the
// per-device error word, and the launch sequence of the forward and the backward.
#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "swa_attn.h"
#include "swa_kernels.h"

namespace {

// Set by a kernel whose bounded wait ran out; one copy per device.
__device__ unsigned g_swa_error_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool probed = false;
  bool supported = false;
  unsigned* err = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Capability check and error-word address of the current device (cached).
swa_status current_device(unsigned** err) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SWA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SWA_ERR_CUDA;
    // The kernels are built for sm_103a only (tcgen05, TMEM, TMA).
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_swa_error_word) != cudaSuccess) return SWA_ERR_CUDA;
      st.err = static_cast<unsigned*>(p);
    }
    st.probed = true;
  }
  if (!st.supported) return SWA_ERR_UNSUPPORTED;
  *err = st.err;
  return SWA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

swa_status check_shape(int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < Lq || window < 1) return SWA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return SWA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return SWA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return SWA_ERR_UNSUPPORTED;
  // Index arithmetic: row indices bh*L + i in 32 bits, grids in 31 bits.
  const long long q_rows = static_cast<long long>(B) * Hq * Lq;
  const long long k_rows = static_cast<long long>(B) * Hkv * Lk;
  const long long q_tiles = static_cast<long long>(B) * Hq * ((Lq + swa::kBlockM - 1) / swa::kBlockM);
  const long long k_tiles = static_cast<long long>(B) * Hkv * ((Lk + swa::kBlockN - 1) / swa::kBlockN);
  if (q_rows >= (1ll << 31) || k_rows >= (1ll << 31) || q_tiles >= (1ll << 31) ||
      k_tiles >= (1ll << 31))
    return SWA_ERR_INVALID_ARG;
  return SWA_OK;
}

swa_status check_sizes(int B, int Hq, int Hkv, int N, int D, int window, float scale) {
  return check_shape(B, Hq, Hkv, N, N, D, window, scale);
}

// Lq query rows as the last Lq positions of Lk keys; causal: 0 <= pos - j < W, else |pos - j| < W.
swa::Problem make_problem_ex(int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                             float scale, unsigned* err, int f16) {
  swa::Problem pb;
  pb.B = B;
  pb.Hq = Hq;
  pb.Hkv = Hkv;
  pb.D = D;
  // A window reaching past every key changes nothing; clamping keeps the offsets in range.
  const int W = window < Lk ? window : Lk;
  pb.span.Lq = Lq;
  pb.span.Lk = Lk;
  pb.span.off = Lk - Lq;
  pb.span.dmin = causal ? 0 : -(W - 1);
  pb.span.dmax = W - 1;
  pb.scale = scale;
  pb.err = err;
  pb.f16 = f16;
  return pb;
}

swa::Problem make_problem(int B, int Hq, int Hkv, int N, int D, int window, float scale,
                          unsigned* err, int f16 = 0) {
  return make_problem_ex(B, Hq, Hkv, N, N, D, window, 1, scale, err, f16);
}

// Forward and backward for either element type (f16: 0 = bf16, 1 = fp16), any Lq <= Lk, causal
// or not.
swa_status fwd_impl(int f16, const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                    float scale, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return SWA_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || (f16 != 0 && f16 != 1)) return SWA_ERR_INVALID_ARG;
  swa_status st = check_shape(B, Hq, Hkv, Lq, Lk, D, window, scale);
  if (st != SWA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  const swa::Problem pb = make_problem_ex(B, Hq, Hkv, Lq, Lk, D, window, causal, scale, err, f16);
  if (swa::launch_fwd(pb, q, k, v, o, lse, stream) != cudaSuccess) return SWA_ERR_CUDA;
  return SWA_OK;
}

swa_status bwd_impl(int f16, const void* q, const void* k, const void* v, const void* o,
                    const void* dO, const float* lse, void* dq, void* dk, void* dv, int B, int Hq,
                    int Hkv, int Lq, int Lk, int D, int window, int causal, float scale,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return SWA_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || (f16 != 0 && f16 != 1)) return SWA_ERR_INVALID_ARG;
  swa_status st = check_shape(B, Hq, Hkv, Lq, Lk, D, window, scale);
  if (st != SWA_OK) return st;
  if (!workspace || workspace_bytes < swa_attn_bwd_workspace_bytes(B, Hq, Lq, D))
    return SWA_ERR_WORKSPACE;
  const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  const swa::Problem pb = make_problem_ex(B, Hq, Hkv, Lq, Lk, D, window, causal, scale, err, f16);
  float* delta = static_cast<float*>(workspace);
  if (swa::launch_bwd_delta(pb, o, dO, delta, stream) != cudaSuccess) return SWA_ERR_CUDA;
  if (swa::launch_bwd_dkdv(pb, q, k, v, dO, lse, delta, dk, dv, stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (swa::launch_bwd_dq(pb, q, k, v, dO, lse, delta, dq, stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  return SWA_OK;
}

}  // namespace

extern "C" {

swa_status swa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int N, int D, int window, float scale,
                        cudaStream_t stream) {
  return fwd_impl(0, q, k, v, o, lse, B, Hq, Hkv, N, N, D, window, 1, scale, stream);
}

swa_status swa_attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int N, int D, int window, float scale,
                            cudaStream_t stream) {
  return fwd_impl(1, q, k, v, o, lse, B, Hq, Hkv, N, N, D, window, 1, scale, stream);
}

swa_status swa_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                           float scale, int f16, cudaStream_t stream) {
  return fwd_impl(f16, q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, D, window, causal, scale, stream);
}

size_t swa_attn_bwd_workspace_bytes(int B, int Hq, int N, int D) {
  if (B < 1 || Hq < 1 || N < 1 || (D != 64 && D != 128 && D != 256)) return 0;
  const size_t bytes = static_cast<size_t>(B) * Hq * N * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

swa_status swa_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                        const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                        int N, int D, int window, float scale, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  return bwd_impl(0, q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, N, D, window, 1, scale,
                  workspace, workspace_bytes, stream);
}

swa_status swa_attn_bwd_f16(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                            int Hq, int Hkv, int N, int D, int window, float scale,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return bwd_impl(1, q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, N, D, window, 1, scale,
                  workspace, workspace_bytes, stream);
}

swa_status swa_attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                           int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                           float scale, int f16, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  return bwd_impl(f16, q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lk, D, window, causal,
                  scale, workspace, workspace_bytes, stream);
}

swa_status swa_attn_bwd_preprocess(const void* o, const void* dO, float* delta, int B, int Hq,
                                   int N, int D, cudaStream_t stream) {
  if (!o || !dO || !delta) return SWA_ERR_INVALID_ARG;
  swa_status st = check_sizes(B, Hq, Hq, N, D, 1, 1.f);
  if (st != SWA_OK) return st;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(delta)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  const swa::Problem pb = make_problem(B, Hq, Hq, N, D, 1, 1.f, err);
  return swa::launch_bwd_delta(pb, o, dO, delta, stream) == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

swa_status swa_attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO,
                             const float* lse, const float* delta, void* dk, void* dv, int B,
                             int Hq, int Hkv, int N, int D, int window, float scale,
                             cudaStream_t stream) {
  if (!q || !k || !v || !dO || !lse || !delta || !dk || !dv) return SWA_ERR_INVALID_ARG;
  swa_status st = check_sizes(B, Hq, Hkv, N, D, window, scale);
  if (st != SWA_OK) return st;
  const void* ptrs[] = {q, k, v, dO, lse, delta, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  const swa::Problem pb = make_problem(B, Hq, Hkv, N, D, window, scale, err);
  return swa::launch_bwd_dkdv(pb, q, k, v, dO, lse, delta, dk, dv, stream) == cudaSuccess
             ? SWA_OK
             : SWA_ERR_CUDA;
}

swa_status swa_attn_bwd_dq(const void* q, const void* k, const void* v, const void* dO,
                           const float* lse, const float* delta, void* dq, int B, int Hq, int Hkv,
                           int N, int D, int window, float scale, cudaStream_t stream) {
  if (!q || !k || !v || !dO || !lse || !delta || !dq) return SWA_ERR_INVALID_ARG;
  swa_status st = check_sizes(B, Hq, Hkv, N, D, window, scale);
  if (st != SWA_OK) return st;
  const void* ptrs[] = {q, k, v, dO, lse, delta, dq};
  for (const void* p : ptrs)
    if (!aligned16(p)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  const swa::Problem pb = make_problem(B, Hq, Hkv, N, D, window, scale, err);
  return swa::launch_bwd_dq(pb, q, k, v, dO, lse, delta, dq, stream) == cudaSuccess ? SWA_OK
                                                                                    : SWA_ERR_CUDA;
}

// ---- Fused backward: Delta and the zeroed dQ accumulator, one kernel for dK, dV and the dQ
// partials, then dQ from the accumulator.  Workspace: Delta (256-byte rounded), then the
// accumulator (D <= 128); D = 256 has no fused kernel and runs the split backward on Delta alone.

size_t swa_attn_bwd_fused_workspace_bytes(int B, int Hq, int Lq, int D) {
  if (B < 1 || Hq < 1 || Lq < 1 || (D != 64 && D != 128 && D != 256)) return 0;
  const size_t delta = swa_attn_bwd_workspace_bytes(B, Hq, Lq, D);
  return D == 256 ? delta : delta + swa::dq_acc_bytes(B, Hq, Lq, D);
}

swa_status swa_attn_bwd_fused(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int Lq, int Lk, int D, int window,
                              int causal, float scale, int f16, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return SWA_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || (f16 != 0 && f16 != 1)) return SWA_ERR_INVALID_ARG;
  swa_status st = check_shape(B, Hq, Hkv, Lq, Lk, D, window, scale);
  if (st != SWA_OK) return st;
  if (!workspace || workspace_bytes < swa_attn_bwd_fused_workspace_bytes(B, Hq, Lq, D))
    return SWA_ERR_WORKSPACE;
  if (D == 256)
    return swa_attn_bwd_ex(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lk, D, window, causal,
                           scale, f16, workspace, workspace_bytes, stream);
  const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  const swa::Problem pb = make_problem_ex(B, Hq, Hkv, Lq, Lk, D, window, causal, scale, err, f16);
  float* delta = static_cast<float*>(workspace);
  float* acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        swa_attn_bwd_workspace_bytes(B, Hq, Lq, D));
  if (swa::launch_bwd_delta_zero_acc(pb, o, dO, delta, acc, stream) != cudaSuccess ||
      swa::launch_bwd_fused(pb, q, k, v, dO, lse, delta, acc, dk, dv, stream) != cudaSuccess ||
      swa::launch_dq_from_acc(pb, acc, dq, stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  return SWA_OK;
}

namespace {

// Shared checks of the fused backward's phase entry points (bf16, Lq = Lk = N, causal).
swa_status fused_phase_setup(int B, int Hq, int Hkv, int N, int D, int window, float scale,
                             const void* workspace, size_t workspace_bytes,
                             std::initializer_list<const void*> ptrs, swa::Problem* pb,
                             float** delta, float** acc) {
  for (const void* p : ptrs)
    if (!p) return SWA_ERR_INVALID_ARG;
  swa_status st = check_sizes(B, Hq, Hkv, N, D, window, scale);
  if (st != SWA_OK) return st;
  if (D == 256) return SWA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < swa_attn_bwd_fused_workspace_bytes(B, Hq, N, D))
    return SWA_ERR_WORKSPACE;
  for (const void* p : ptrs)
    if (!aligned16(p)) return SWA_ERR_MISALIGNED;
  if (!aligned16(workspace)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  *pb = make_problem(B, Hq, Hkv, N, D, window, scale, err);
  *delta = static_cast<float*>(const_cast<void*>(workspace));
  *acc = reinterpret_cast<float*>(static_cast<uint8_t*>(const_cast<void*>(workspace)) +
                                  swa_attn_bwd_workspace_bytes(B, Hq, N, D));
  return SWA_OK;
}

}  // namespace

swa_status swa_attn_bwd_fused_preprocess(const void* o, const void* dO, void* workspace,
                                         size_t workspace_bytes, int B, int Hq, int N, int D,
                                         cudaStream_t stream) {
  swa::Problem pb;
  float *delta = nullptr, *acc = nullptr;
  swa_status st = fused_phase_setup(B, Hq, Hq, N, D, 1, 1.f, workspace, workspace_bytes, {o, dO},
                                    &pb, &delta, &acc);
  if (st != SWA_OK) return st;
  return swa::launch_bwd_delta_zero_acc(pb, o, dO, delta, acc, stream) == cudaSuccess
             ? SWA_OK
             : SWA_ERR_CUDA;
}

swa_status swa_attn_bwd_fused_dkdv(const void* q, const void* k, const void* v, const void* dO,
                                   const float* lse, void* dk, void* dv, void* workspace,
                                   size_t workspace_bytes, int B, int Hq, int Hkv, int N, int D,
                                   int window, float scale, cudaStream_t stream) {
  swa::Problem pb;
  float *delta = nullptr, *acc = nullptr;
  swa_status st = fused_phase_setup(B, Hq, Hkv, N, D, window, scale, workspace, workspace_bytes,
                                    {q, k, v, dO, lse, dk, dv}, &pb, &delta, &acc);
  if (st != SWA_OK) return st;
  return swa::launch_bwd_fused(pb, q, k, v, dO, lse, delta, acc, dk, dv, stream) == cudaSuccess
             ? SWA_OK
             : SWA_ERR_CUDA;
}

swa_status swa_attn_bwd_fused_dq(void* dq, const void* workspace, size_t workspace_bytes, int B,
                                 int Hq, int N, int D, float scale, cudaStream_t stream) {
  swa::Problem pb;
  float *delta = nullptr, *acc = nullptr;
  swa_status st = fused_phase_setup(B, Hq, Hq, N, D, 1, scale, workspace, workspace_bytes, {dq},
                                    &pb, &delta, &acc);
  if (st != SWA_OK) return st;
  return swa::launch_dq_from_acc(pb, acc, dq, stream) == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

const char* swa_strerror(swa_status status) {
  switch (status) {
    case SWA_OK: return "SWA_OK";
    case SWA_ERR_INVALID_ARG: return "SWA_ERR_INVALID_ARG: size, window, scale or pointer invalid";
    case SWA_ERR_UNSUPPORTED: return "SWA_ERR_UNSUPPORTED: head dim not in {64,128,256} or device not sm_103";
    case SWA_ERR_MISALIGNED: return "SWA_ERR_MISALIGNED: pointer not 16-byte aligned";
    case SWA_ERR_CUDA: return "SWA_ERR_CUDA: CUDA call or kernel launch failed";
    case SWA_ERR_DEVICE_TIMEOUT: return "SWA_ERR_DEVICE_TIMEOUT: a kernel's bounded wait ran out";
    case SWA_ERR_WORKSPACE: return "SWA_ERR_WORKSPACE: workspace null or too small";
    case SWA_ERR_DEVICE_LAYOUT:
      return "SWA_ERR_DEVICE_LAYOUT: a kernel's shared memory was not 1024-byte aligned";
  }
  return "SWA_ERR_UNKNOWN";
}

swa_status swa_check_device(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SWA_ERR_CUDA;
  unsigned* err = nullptr;
  swa_status st = current_device(&err);
  if (st != SWA_OK) return st;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_swa_error_word, sizeof(word)) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (word != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_swa_error_word, &zero, sizeof(zero)) != cudaSuccess)
      return SWA_ERR_CUDA;
    return (word & swa::kErrSmemLayout) ? SWA_ERR_DEVICE_LAYOUT : SWA_ERR_DEVICE_TIMEOUT;
  }
  return SWA_OK;
}

swa_status swa_selftest_wait_timeout(cudaStream_t stream) {
  unsigned* err = nullptr;
  swa_status st = current_device(&err);
  if (st != SWA_OK) return st;
  return swa::launch_wait_timeout_selftest(err, stream) == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

int swa_version(void) { return 100; }

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// fp32 tensors: rounded to bf16 copies in the caller's workspace, bf16 kernels, widened results.
// ------------------------------------------------------------------------------------------------
namespace {

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets of the workspace regions: bf16 copies of q, k, v, a query-shaped slot (o in the
// forward, dO in the backward), bf16 dq, dk, dv, Delta (fp32), then the forward's log-sum-exp
// correction: the bf16 residuals of q and k and a second query-shaped slot.  In the forward the dq
// slot holds P k_hi, the new slot P k_lo, and Delta's rows the repeated passes' log-sum-exp.
struct F32Layout {
  size_t q16, k16, v16, a16, dq16, dk16, dv16, delta, qlo16, klo16, c16, total;
  long long q_units, k_units;  // 8-element units of a query / key tensor
};

F32Layout f32_layout(int B, int Hq, int Hkv, int Lq, int Lk, int D) {
  F32Layout L;
  const size_t qe = static_cast<size_t>(B) * Hq * Lq * D;
  const size_t ke = static_cast<size_t>(B) * Hkv * Lk * D;
  const size_t qb = round256(qe * 2), kb = round256(ke * 2);
  size_t off = 0;
  L.q16 = off; off += qb;
  L.k16 = off; off += kb;
  L.v16 = off; off += kb;
  L.a16 = off; off += qb;
  L.dq16 = off; off += qb;
  L.dk16 = off; off += kb;
  L.dv16 = off; off += kb;
  L.delta = off; off += round256(static_cast<size_t>(B) * Hq * Lq * sizeof(float));
  L.qlo16 = off; off += qb;
  L.klo16 = off; off += kb;
  L.c16 = off; off += qb;
  L.total = off;
  L.q_units = static_cast<long long>(qe / 8);
  L.k_units = static_cast<long long>(ke / 8);
  return L;
}

swa_status f32_prologue(int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                        float scale, const void* workspace, size_t workspace_bytes,
                        std::initializer_list<const void*> ptrs, swa::Problem* pb) {
  for (const void* p : ptrs)
    if (!p) return SWA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return SWA_ERR_INVALID_ARG;
  swa_status st = check_shape(B, Hq, Hkv, Lq, Lk, D, window, scale);
  if (st != SWA_OK) return st;
  if (!workspace || workspace_bytes < f32_layout(B, Hq, Hkv, Lq, Lk, D).total)
    return SWA_ERR_WORKSPACE;
  for (const void* p : ptrs)
    if (!aligned16(p)) return SWA_ERR_MISALIGNED;
  if (!aligned16(workspace)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  *pb = make_problem_ex(B, Hq, Hkv, Lq, Lk, D, window, causal, scale, err, 0);
  return SWA_OK;
}

// q, k, v rounded to bf16; with `split`, also the bf16 residuals of q and k.
swa::RoundJob round_qkv(const float* q, const float* k, const float* v, uint8_t* ws,
                        const F32Layout& L, bool split = false) {
  swa::RoundJob j{};
  if (split) {
    j.lo[0] = reinterpret_cast<uint16_t*>(ws + L.qlo16);
    j.lo[1] = reinterpret_cast<uint16_t*>(ws + L.klo16);
  }
  j.src[0] = q; j.dst[0] = reinterpret_cast<uint16_t*>(ws + L.q16);
  j.src[1] = k; j.dst[1] = reinterpret_cast<uint16_t*>(ws + L.k16);
  j.src[2] = v; j.dst[2] = reinterpret_cast<uint16_t*>(ws + L.v16);
  j.end[0] = L.q_units;
  j.end[1] = L.q_units + L.k_units;
  j.end[2] = j.end[3] = L.q_units + 2 * L.k_units;
  return j;
}

}  // namespace

extern "C" {

size_t swa_attn_f32_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < Lq || (D != 64 && D != 128 && D != 256))
    return 0;
  return f32_layout(B, Hq, Hkv, Lq, Lk, D).total;
}

swa_status swa_attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                            int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                            float scale, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  swa::Problem pb;
  swa_status st = f32_prologue(B, Hq, Hkv, Lq, Lk, D, window, causal, scale, workspace,
                               workspace_bytes, {q, k, v, o, lse}, &pb);
  if (st != SWA_OK) return st;
  const F32Layout L = f32_layout(B, Hq, Hkv, Lq, Lk, D);
  auto* ws = static_cast<uint8_t*>(workspace);
  if (swa::launch_round_bf16(round_qkv(q, k, v, ws, L, true), stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  // O and LSE from the bf16 operands; then P k_hi and P k_lo (the same scores, so the same P)
  // and the first-order log-sum-exp correction for the residuals of q and k.
  float* lse_rep = reinterpret_cast<float*>(ws + L.delta);
  if (swa::launch_fwd(pb, ws + L.q16, ws + L.k16, ws + L.v16, ws + L.a16, lse, stream) !=
          cudaSuccess ||
      swa::launch_fwd(pb, ws + L.q16, ws + L.k16, ws + L.k16, ws + L.dq16, lse_rep, stream) !=
          cudaSuccess ||
      swa::launch_fwd(pb, ws + L.q16, ws + L.k16, ws + L.klo16, ws + L.c16, lse_rep, stream) !=
          cudaSuccess ||
      swa::launch_lse_correct(pb, ws + L.q16, ws + L.qlo16, ws + L.dq16, ws + L.c16, lse,
                              stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  swa::WidenJob w{};
  w.src[0] = reinterpret_cast<const uint16_t*>(ws + L.a16);
  w.dst[0] = o;
  w.end[0] = w.end[1] = w.end[2] = w.end[3] = L.q_units;
  return swa::launch_widen_bf16(w, stream) == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

swa_status swa_attn_bwd_f32(const float* q, const float* k, const float* v, const float* o,
                            const float* dO, const float* lse, float* dq, float* dk, float* dv,
                            int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                            float scale, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  swa::Problem pb;
  swa_status st = f32_prologue(B, Hq, Hkv, Lq, Lk, D, window, causal, scale, workspace,
                               workspace_bytes, {q, k, v, o, dO, lse, dq, dk, dv}, &pb);
  if (st != SWA_OK) return st;
  const F32Layout L = f32_layout(B, Hq, Hkv, Lq, Lk, D);
  auto* ws = static_cast<uint8_t*>(workspace);
  float* delta = reinterpret_cast<float*>(ws + L.delta);
  if (swa::launch_round_bf16(round_qkv(q, k, v, ws, L), stream) != cudaSuccess) return SWA_ERR_CUDA;
  if (swa::launch_delta_f32(pb, o, dO, delta, ws + L.a16, stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (swa::launch_bwd_dkdv(pb, ws + L.q16, ws + L.k16, ws + L.v16, ws + L.a16, lse, delta,
                           ws + L.dk16, ws + L.dv16, stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (swa::launch_bwd_dq(pb, ws + L.q16, ws + L.k16, ws + L.v16, ws + L.a16, lse, delta,
                         ws + L.dq16, stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  swa::WidenJob w{};
  w.src[0] = reinterpret_cast<const uint16_t*>(ws + L.dq16); w.dst[0] = dq;
  w.src[1] = reinterpret_cast<const uint16_t*>(ws + L.dk16); w.dst[1] = dk;
  w.src[2] = reinterpret_cast<const uint16_t*>(ws + L.dv16); w.dst[2] = dv;
  w.end[0] = L.q_units;
  w.end[1] = L.q_units + L.k_units;
  w.end[2] = w.end[3] = L.q_units + 2 * L.k_units;
  return swa::launch_widen_bf16(w, stream) == cudaSuccess ? SWA_OK : SWA_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Host-resident tensors: forward + backward of one layer, pipelined over (batch, kv head) groups.
// ------------------------------------------------------------------------------------------------
namespace {

constexpr int kMaxHostSlots = 3;  // device buffer sets in flight (one per pipeline stage)

// Streams and events of the host pipeline, created once per device.
struct HostPipe {
  std::mutex enqueue;  // one call at a time enqueues on the shared streams and events
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t fork = nullptr, join_in = nullptr, join_comp = nullptr, join_out = nullptr;
  cudaEvent_t in_fwd[kMaxHostSlots] = {}, in_done[kMaxHostSlots] = {},
              fwd_done[kMaxHostSlots] = {}, dkdv_done[kMaxHostSlots] = {},
              comp_done[kMaxHostSlots] = {}, out_done[kMaxHostSlots] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

swa_status host_pipe(HostPipe** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SWA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    const unsigned sf = cudaStreamNonBlocking;
    const unsigned ef = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&hp.in, sf) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.comp, sf) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.out, sf) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.fork, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.join_in, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.join_comp, ef) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.join_out, ef) == cudaSuccess;
    for (int i = 0; ok && i < kMaxHostSlots; ++i)
      ok = cudaEventCreateWithFlags(&hp.in_fwd[i], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.in_done[i], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.dkdv_done[i], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.fwd_done[i], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.comp_done[i], ef) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.out_done[i], ef) == cudaSuccess;
    if (!ok) return SWA_ERR_CUDA;
    hp.ready = true;
  }
  *out = &hp;
  return SWA_OK;
}

// Byte sizes of one slot's buffers for `units` (batch, kv head) groups of G query heads.
struct HostSlot {
  size_t q, k, lse, total;  // q-shaped, k-shaped, lse-shaped sizes (each rounded to 256 bytes)
};

HostSlot host_slot(int units, int G, int N, int D) {
  HostSlot h;
  h.q = round256(static_cast<size_t>(units) * G * N * D * 2);
  h.k = round256(static_cast<size_t>(units) * N * D * 2);
  h.lse = round256(static_cast<size_t>(units) * G * N * sizeof(float));
  h.total = 4 * h.q + 4 * h.k + 2 * h.lse;  // q, dO, o, dq | k, v, dk, dv | lse, delta
  return h;
}

}  // namespace

extern "C" {

size_t swa_attn_host_workspace_bytes(int B, int Hq, int Hkv, int N, int D, int units_per_chunk) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || Hq % Hkv != 0 || units_per_chunk < 1 ||
      (D != 64 && D != 128 && D != 256))
    return 0;
  const int units = units_per_chunk < B * Hkv ? units_per_chunk : B * Hkv;
  return kMaxHostSlots * host_slot(units, Hq / Hkv, N, D).total;
}

swa_status swa_attn_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO,
                                 void* o, float* lse, void* dq, void* dk, void* dv, int B, int Hq,
                                 int Hkv, int N, int D, int window, float scale,
                                 int units_per_chunk, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
  const void* ptrs[] = {q, k, v, dO, o, lse, dq, dk, dv};
  for (const void* p : ptrs)
    if (!p) return SWA_ERR_INVALID_ARG;
  if (units_per_chunk < 1) return SWA_ERR_INVALID_ARG;
  swa_status st = check_sizes(B, Hq, Hkv, N, D, window, scale);
  if (st != SWA_OK) return st;
  // Three buffer sets let H2D, kernels and D2H each work on its own chunk; two also work (the
  // next chunk's copy-in then waits for an older chunk's copy-out).
  const int G0 = Hq / Hkv, total0 = B * Hkv;
  const size_t slot_bytes =
      host_slot(units_per_chunk < total0 ? units_per_chunk : total0, G0, N, D).total;
  if (!workspace || workspace_bytes < 2 * slot_bytes) return SWA_ERR_WORKSPACE;
  const int nslots = workspace_bytes >= 3 * slot_bytes ? 3 : 2;
  for (const void* p : ptrs)
    if (!aligned16(p)) return SWA_ERR_MISALIGNED;
  if (!aligned16(workspace)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  HostPipe* hp = nullptr;
  if ((st = host_pipe(&hp)) != SWA_OK) return st;

  const int G = Hq / Hkv, total = B * Hkv;
  const int U = units_per_chunk < total ? units_per_chunk : total;
  const HostSlot hs = host_slot(U, G, N, D);
  const size_t q_unit = static_cast<size_t>(G) * N * D * 2, k_unit = static_cast<size_t>(N) * D * 2;
  const size_t l_unit = static_cast<size_t>(G) * N * sizeof(float);
  auto* ws = static_cast<uint8_t*>(workspace);
  auto h2d = [&](void* dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, hp->in) == cudaSuccess;
  };
  auto d2h = [&](void* dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, hp->out) == cudaSuccess;
  };
  auto at = [](const void* base, size_t off) {
    return static_cast<uint8_t*>(const_cast<void*>(base)) + off;
  };

  std::lock_guard<std::mutex> lk(hp->enqueue);
  // Fork: the three streams start after the work already queued on `stream`.
  if (cudaEventRecord(hp->fork, stream) != cudaSuccess ||
      cudaStreamWaitEvent(hp->in, hp->fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->comp, hp->fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->out, hp->fork, 0) != cudaSuccess)
    return SWA_ERR_CUDA;
  // From here on a failure stops enqueueing but still joins the streams back into `stream`.
  swa_status result = SWA_OK;
  const int chunks = (total + U - 1) / U;
  for (int c = 0; c < chunks && result == SWA_OK; ++c) {
    const int u0 = c * U, n = (total - u0) < U ? (total - u0) : U;
    const int slot = c % nslots;
    uint8_t* b = ws + slot * hs.total;
    uint8_t *sq = b, *sdo = b + hs.q, *so = b + 2 * hs.q, *sdq = b + 3 * hs.q;
    uint8_t *sk = b + 4 * hs.q, *sv = sk + hs.k, *sdk = sk + 2 * hs.k, *sdv = sk + 3 * hs.k;
    float* slse = reinterpret_cast<float*>(sk + 4 * hs.k);
    float* sdelta = reinterpret_cast<float*>(sk + 4 * hs.k + hs.lse);
    // inputs of chunk c, once the slot's previous outputs have left
    if (c >= nslots && cudaStreamWaitEvent(hp->in, hp->out_done[slot], 0) != cudaSuccess) {
      result = SWA_ERR_CUDA;
      break;
    }
    // Q, K, V first (the forward needs only those), then dO.
    if (!h2d(sq, at(q, u0 * q_unit), n * q_unit) || !h2d(sk, at(k, u0 * k_unit), n * k_unit) ||
        !h2d(sv, at(v, u0 * k_unit), n * k_unit) ||
        cudaEventRecord(hp->in_fwd[slot], hp->in) != cudaSuccess ||
        !h2d(sdo, at(dO, u0 * q_unit), n * q_unit) ||
        cudaEventRecord(hp->in_done[slot], hp->in) != cudaSuccess) {
      result = SWA_ERR_CUDA;
      break;
    }
    // forward and backward of the chunk's n groups: one problem with B = 1, Hq = n G, Hkv = n.
    // The forward starts while dO is still being copied.
    if (cudaStreamWaitEvent(hp->comp, hp->in_fwd[slot], 0) != cudaSuccess) {
      result = SWA_ERR_CUDA;
      break;
    }
    const swa::Problem pb = make_problem(1, n * G, n, N, D, window, scale, err);
    if (swa::launch_fwd(pb, sq, sk, sv, so, slse, hp->comp) != cudaSuccess ||
        cudaEventRecord(hp->fwd_done[slot], hp->comp) != cudaSuccess ||
        cudaStreamWaitEvent(hp->comp, hp->in_done[slot], 0) != cudaSuccess) {
      result = SWA_ERR_CUDA;
      break;
    }
    if (swa::launch_bwd_delta(pb, so, sdo, sdelta, hp->comp) != cudaSuccess ||
        swa::launch_bwd_dkdv(pb, sq, sk, sv, sdo, slse, sdelta, sdk, sdv, hp->comp) !=
            cudaSuccess ||
        cudaEventRecord(hp->dkdv_done[slot], hp->comp) != cudaSuccess ||
        swa::launch_bwd_dq(pb, sq, sk, sv, sdo, slse, sdelta, sdq, hp->comp) != cudaSuccess ||
        cudaEventRecord(hp->comp_done[slot], hp->comp) != cudaSuccess) {
      result = SWA_ERR_CUDA;
      break;
    }
    // outputs of chunk c: O and LSE as soon as the forward has written them (the backward only
    // reads them), dK and dV once their kernel is done (while dQ is computed), then dQ
    if (cudaStreamWaitEvent(hp->out, hp->fwd_done[slot], 0) != cudaSuccess ||
        !d2h(at(o, u0 * q_unit), so, n * q_unit) || !d2h(at(lse, u0 * l_unit), slse, n * l_unit) ||
        cudaStreamWaitEvent(hp->out, hp->dkdv_done[slot], 0) != cudaSuccess ||
        !d2h(at(dk, u0 * k_unit), sdk, n * k_unit) || !d2h(at(dv, u0 * k_unit), sdv, n * k_unit) ||
        cudaStreamWaitEvent(hp->out, hp->comp_done[slot], 0) != cudaSuccess) {
      result = SWA_ERR_CUDA;
      break;
    }
    if (!d2h(at(dq, u0 * q_unit), sdq, n * q_unit) ||
        cudaEventRecord(hp->out_done[slot], hp->out) != cudaSuccess) {
      result = SWA_ERR_CUDA;
      break;
    }
  }
  // Join: `stream` continues once every copy and kernel above has finished (also after a
  // failure part-way, so no enqueued work outlives the call's ordering on `stream`).
  if (cudaEventRecord(hp->join_comp, hp->comp) != cudaSuccess ||
      cudaEventRecord(hp->join_out, hp->out) != cudaSuccess ||
      cudaEventRecord(hp->join_in, hp->in) != cudaSuccess ||
      cudaStreamWaitEvent(stream, hp->join_in, 0) != cudaSuccess ||
      cudaStreamWaitEvent(stream, hp->join_comp, 0) != cudaSuccess ||
      cudaStreamWaitEvent(stream, hp->join_out, 0) != cudaSuccess)
    return SWA_ERR_CUDA;
  return result;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Backward without caller workspace: the Delta scratch is a fixed device array of this file.
// ------------------------------------------------------------------------------------------------
namespace {

// Delta scratch of swa_attn_bwd_noalloc (one fp32 per query row), shared by every call on a device.
static __device__ __align__(256) float g_swa_noalloc_delta[SWA_NOALLOC_MAX_ROWS];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device (no allocation).
swa_status noalloc_scratch(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SWA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_swa_noalloc_delta) != cudaSuccess || p == nullptr)
      return SWA_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return SWA_OK;
}

}  // namespace

extern "C" swa_status swa_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                           const void* o, const void* dO, const float* lse,
                                           void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                           int N, int D, int window, float scale,
                                           cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return SWA_ERR_INVALID_ARG;
  swa_status st = check_sizes(B, Hq, Hkv, N, D, window, scale);
  if (st != SWA_OK) return st;
  if (static_cast<long long>(B) * Hq * N > SWA_NOALLOC_MAX_ROWS) return SWA_ERR_WORKSPACE;
  const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return SWA_ERR_MISALIGNED;
  unsigned* err = nullptr;
  if ((st = current_device(&err)) != SWA_OK) return st;
  float* delta = nullptr;
  if ((st = noalloc_scratch(&delta)) != SWA_OK) return st;
  const swa::Problem pb = make_problem(B, Hq, Hkv, N, D, window, scale, err);
  if (swa::launch_bwd_delta(pb, o, dO, delta, stream) != cudaSuccess) return SWA_ERR_CUDA;
  if (swa::launch_bwd_dkdv(pb, q, k, v, dO, lse, delta, dk, dv, stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  if (swa::launch_bwd_dq(pb, q, k, v, dO, lse, delta, dq, stream) != cudaSuccess)
    return SWA_ERR_CUDA;
  return SWA_OK;
}
