/*
 * swa_attn.h — C ABI of libswa.so: memory-linear causal sliding-window attention with grouped-query
 * heads, forward and backward, hand-written for NVIDIA GB300 (sm_103a).
 *
 * The operation (per batch b and query head hq, with kv head hk = hq / (Hq / Hkv)):
 *
 *     visible(i, j) <=> 0 <= i - j < window          (each query sees itself and the window-1
 *                                                     keys before it; window >= N is plain causal)
 *     S[i, j] = scale * <Q[i], K[j]>  (visible cells only)
 *     LSE[i]  = ln sum_j exp(S[i, j]),  P = exp(S - LSE),  O = P V
 *
 * This is the attention of "Off NVIDIA, you fix the platform yourself" (Layer2C Lab 28), section
 * "What was broken?": attention scores form a matrix with a row per query and a column per key,
 * and a sliding window of W limits each query to the W most recent positions, itself included.  As in the mlx-train-perf
 * README (flash-attention section) only O and the per-row log-sum-exp are saved by the forward,
 * and the backward recomputes the score tiles it needs; the N x N matrix is never stored.
 *
 * Layout: every tensor is contiguous, row-major.
 *     q, o, dO, dq     bf16  [B, Hq,  N, D]
 *     k, v, dk, dv     bf16  [B, Hkv, N, D]
 *     lse              fp32  [B, Hq,  N]      natural log, over the scaled scores
 * Supported: D in {64, 128, 256}; Hq % Hkv == 0; N >= 1; B >= 1; window >= 1; scale finite and
 * > 0.  D = 256 (the head width of Gemma 4's sliding layers, Lab 28 record, numbers entry
 * "Attention backward memory") runs on kernels that stream half-tiles and compute dK and dV in
 * two passes; results and arguments are the same.
 * All device pointers must be 16-byte aligned.
 *
 * Ownership: the caller allocates every buffer (device memory), including the backward workspace.
 * The library allocates no device memory, keeps no per-call state, and never synchronizes the
 * stream; calls are asynchronous on `stream` (0 = the legacy default stream).
 *
 * Errors: arguments are checked on the host before anything is launched; a bad argument returns
 * its code and launches nothing.  Launch failures return SWA_ERR_CUDA.  The entry points never
 * throw, abort or print.  Every wait inside the kernels is bounded; a kernel whose wait runs out
 * records it in a per-device error word and returns early — read it with swa_check_device().
 */
#ifndef SWA_ATTN_H
#define SWA_ATTN_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SWA_OK = 0,
    SWA_ERR_INVALID_ARG = 1,    /* a size, window or scale outside its domain, or a null pointer  */
    SWA_ERR_UNSUPPORTED = 2,    /* D not in {64, 128, 256}, or no sm_103 device current           */
    SWA_ERR_MISALIGNED = 3,     /* a tensor pointer not 16-byte aligned                          */
    SWA_ERR_CUDA = 4,           /* a CUDA runtime / driver call or a launch failed               */
    SWA_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait ran out (reported by swa_check_device) */
    SWA_ERR_WORKSPACE = 6,      /* backward workspace null or smaller than required              */
    SWA_ERR_DEVICE_LAYOUT = 7   /* a kernel found its shared memory not 1024-byte aligned and did
                                   no work (reported by swa_check_device)                        */
} swa_status;

/*
 * Forward.  Writes o [B,Hq,N,D] bf16 and lse [B,Hq,N] fp32.
 *   q, k, v : inputs (device, bf16, layout above); not modified.
 *   o, lse  : outputs (device); fully overwritten for rows 0..N-1.
 *   window  : W >= 1; values >= N mean full causal attention.
 *   scale   : softmax scale applied to <q, k> (typically 1/sqrt(D)).
 * Saved state for the backward is exactly (o, lse): the lab's windowed forward keeps the per-row
 * log-sum-exp under the window for the backward (Lab 28, "Method and disclosure").
 */
swa_status swa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int Hq, int Hkv, int N, int D, int window, float scale,
                        cudaStream_t stream);

/*
 * Bytes of device workspace swa_attn_bwd needs: one fp32 Delta = rowsum(dO * O) per query row,
 * B*Hq*N*4 bytes (rounded up to 256).  Returns 0 for invalid sizes.
 */
size_t swa_attn_bwd_workspace_bytes(int B, int Hq, int N, int D);

/*
 * Backward of L = sum(dO * O) through the forward above.  Writes dq [B,Hq,N,D], dk and dv
 * [B,Hkv,N,D] (bf16), fully overwritten; dk/dv hold the sum over the G = Hq/Hkv query heads that
 * share each kv head.
 *   q, k, v, o, dO, lse : device inputs; o and lse must be the forward's outputs for (q, k, v).
 *   workspace           : device scratch of at least swa_attn_bwd_workspace_bytes(B,Hq,N,D) bytes,
 *                         16-byte aligned; contents on entry are ignored and left undefined.
 * Three kernels run in order on `stream`: Delta = rowsum(dO * O), the dK/dV kernel (each key block
 * walks only the query blocks inside its window, over every query head of its group) and the dQ
 * kernel (each query block walks only the key blocks inside its window).  The window bookkeeping
 * follows Lab 28's patch ("Method and disclosure"): blocks wholly outside the window are skipped,
 * edge tiles are masked, dQ starts at each query tile's first visited key tile, and dK/dV of key
 * tiles that no query visits are written as zeros.
 */
swa_status swa_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                        const float* lse, void* dq, void* dk, void* dv,
                        int B, int Hq, int Hkv, int N, int D, int window, float scale,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fp16 forms of swa_attn_fwd and swa_attn_bwd: the same arguments, checks, kernels and outputs,
 * with q, k, v, o, dO, dq, dk, dv holding IEEE fp16 instead of bf16 (lse and the workspace stay
 * fp32).  P and dS are rounded to fp16 as tensor-core operands; scores and accumulators stay fp32.
 * The pages' gradient sweep covers fp16 as well as bf16 inputs (Lab 28, "Gradient parity, small
 * shapes").  The caller keeps the values in fp16's range: P is bounded by 2^12 inside the forward,
 * so only the inputs themselves can overflow.
 */
swa_status swa_attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int N, int D, int window, float scale,
                            cudaStream_t stream);
swa_status swa_attn_bwd_f16(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv,
                            int B, int Hq, int Hkv, int N, int D, int window, float scale,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * General forms: queries shorter than keys, non-causal windows, either element type.
 *   q, o, dO, dq : [B, Hq, Lq, D];  k, v, dk, dv : [B, Hkv, Lk, D];  lse : [B, Hq, Lq] fp32.
 *   Lq <= Lk     : the queries are the last Lq positions of the key sequence (query i sits at key
 *                  position i + Lk - Lq); Lq > Lk returns SWA_ERR_INVALID_ARG.
 *   causal       : 1 -> key j visible to query i iff 0 <= i + Lk - Lq - j < window;
 *                  0 -> iff |i + Lk - Lq - j| < window (window >= Lk: full attention).
 *                  Other values return SWA_ERR_INVALID_ARG.
 *   f16          : 0 -> bf16 tensors, 1 -> fp16 tensors; other values SWA_ERR_INVALID_ARG.
 *   workspace    : at least swa_attn_bwd_workspace_bytes(B, Hq, Lq, D) bytes.
 * Key blocks that no query sees (a short query suffix under a narrow window) get dk = dv = 0.
 * The pages' gradient sweep includes query sequences shorter than the key sequence, and both causal
 * and non-causal windows (Lab 28, numbers entry "Gradient parity, small shapes"); neither is
 * defined there further, and
 * the alignment and two-sided window above are this library's reading.  With Lq = Lk, causal = 1
 * these are swa_attn_fwd / swa_attn_bwd (f16 = 1: the _f16 forms).
 */
swa_status swa_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                           float scale, int f16, cudaStream_t stream);
swa_status swa_attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, void* dq, void* dk, void* dv,
                           int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                           float scale, int f16, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * fp32 tensors: the general forms above with q, k, v, o, dO, dq, dk, dv in IEEE fp32.
 * The tensor cores take bf16 operands, so every input element is rounded once to the nearest bf16
 * (ties to even) on the device; scores, accumulators, lse and Delta stay fp32, and the results are
 * widened to fp32.  The forward's lse is then corrected to fp32 accuracy: q and k are also split
 * into bf16 high and low parts, and the first-order change of the log-sum-exp under the scores'
 * missing low-part products, scale (<q_hi, P k_lo> + <q_lo, P k_hi>) per row, is added, with
 * P k_hi and P k_lo taken from two more runs of the forward kernel (v replaced by k_hi, k_lo; the
 * same scores give the same P).  What remains is second order in the rounding, ~1e-5 for
 * unit-scale inputs.  O and the gradients keep bf16 tensor-core operands (as P and dS always
 * are).  In the backward, Delta is formed from fp32 O and the bf16-rounded dO that the dP
 * contraction sees.  The pages' gradient sweep runs fp32 inputs alongside the 16-bit ones (Lab 28,
 * numbers entry "Gradient parity, small shapes").
 *   workspace : device scratch of at least swa_attn_f32_workspace_bytes(B,Hq,Hkv,Lq,Lk,D) bytes,
 *               16-byte aligned, owned by the caller (the bf16 copies, residuals and Delta live
 *               there; it holds nothing between calls).  Too small or NULL: SWA_ERR_WORKSPACE.
 * Shapes, windows, causal and errors as in the general forms; every pointer 16-byte aligned.
 * A forward is six launches (round and split q, k, v; attention three times; lse correction;
 * widen o), a backward five.
 */
size_t swa_attn_f32_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int D);
swa_status swa_attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                            int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                            float scale, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);
swa_status swa_attn_bwd_f32(const float* q, const float* k, const float* v, const float* o,
                            const float* dO, const float* lse, float* dq, float* dk, float* dv,
                            int B, int Hq, int Hkv, int Lq, int Lk, int D, int window, int causal,
                            float scale, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * Forward and backward of one layer whose tensors live in host memory: q, k, v, dO in and
 * o, lse, dq, dk, dv out (host pointers, equal lengths, causal window; layouts as above, bf16).
 * The (batch, kv head) groups are processed in chunks of `units_per_chunk`: chunk c + 1 is copied
 * in while chunk c runs the same kernels as swa_attn_fwd / swa_attn_bwd and chunk c - 1 is copied
 * out (a chunk's forward starts once its q, k, v are in, and its o and lse go back as soon as the
 * forward has written them).  This runs on three library streams forked from `stream` and joined
 * back into it, so the call is asynchronous on `stream` like the others and its results equal
 * theirs bit for bit.  Host
 * buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to overlap.
 *   workspace : device scratch, 16-byte aligned, caller-owned.  swa_attn_host_workspace_bytes
 *               gives three chunks' tensors (copy-in, kernels and copy-out each on their own
 *               chunk); two thirds of it is the minimum (the copy-in of a chunk then also waits
 *               for the copy-out of the chunk two before it).
 * The library creates its three streams and their events once per device and keeps them.
 * Errors as for swa_attn_bwd; units_per_chunk < 1 is SWA_ERR_INVALID_ARG.
 */
size_t swa_attn_host_workspace_bytes(int B, int Hq, int Hkv, int N, int D, int units_per_chunk);
swa_status swa_attn_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO,
                                 void* o, float* lse, void* dq, void* dk, void* dv, int B, int Hq,
                                 int Hkv, int N, int D, int window, float scale,
                                 int units_per_chunk, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * The three phases swa_attn_bwd runs, callable one by one (same arguments, same checks, same
 * kernels), e.g. to time each kernel or to run the dK/dV and dQ phases on two streams once the
 * preprocess has finished.  `delta` is the workspace of swa_attn_bwd (fp32 [B,Hq,N]).
 *   swa_attn_bwd_preprocess : delta = rowsum(dO * O) per query row.
 *   swa_attn_bwd_dkdv       : dk, dv, walking for each key block only the query blocks inside its
 *                             window, summed over the query heads of its kv group; needs delta.
 *   swa_attn_bwd_dq         : dq, walking for each query block only the key blocks inside its
 *                             window; needs delta.
 */
swa_status swa_attn_bwd_preprocess(const void* o, const void* dO, float* delta,
                                   int B, int Hq, int N, int D, cudaStream_t stream);
swa_status swa_attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO,
                             const float* lse, const float* delta, void* dk, void* dv,
                             int B, int Hq, int Hkv, int N, int D, int window, float scale,
                             cudaStream_t stream);
swa_status swa_attn_bwd_dq(const void* q, const void* k, const void* v, const void* dO,
                           const float* lse, const float* delta, void* dq,
                           int B, int Hq, int Hkv, int N, int D, int window, float scale,
                           cudaStream_t stream);

/*
 * Fused backward: the same gradients as swa_attn_bwd_ex, with one kernel for dK, dV and dQ.  Per
 * (key block, query tile) pair it runs the backward's five contractions once each (the split
 * backward's dQ kernel recomputes S and dP), following the window walk of "Off NVIDIA, you fix the
 * platform yourself" (Lab 28, "What did fixing it take?", "Method and disclosure": tiles outside the
 * window skipped, edge tiles masked, dK / dV of key tiles no query visits written as zeros).  dK and
 * dV accumulate on chip over each kv group as in the split path; every query tile's dQ gets one fp32
 * partial per key block of its window, added into an fp32 accumulator in the workspace with vector
 * reduce-adds at the L2, then scaled and rounded once by a small kernel.  Launches: Delta (also
 * zeroing the accumulator), the fused kernel, the dQ rounding.
 *   Speed: on GB300 the split backward is faster.  The accumulator's reduce-adds (a 64 KB fp32
 *   partial per 128 x 128 tile pair) are bounded by the L2's reduction throughput, which costs more
 *   than the split path's recomputation of S and dP; the fused form is kept for callers who want
 *   one pass over the key blocks.
 *   Determinism: dK and dV equal the split path's bit for bit; the order of the fp32 additions into
 *   dQ's accumulator varies between runs, so dQ can differ in the last bits from run to run (the
 *   split swa_attn_bwd / swa_attn_bwd_ex is the bit-reproducible path).
 *   workspace : device scratch of at least swa_attn_bwd_fused_workspace_bytes(B,Hq,Lq,D) bytes,
 *               16-byte aligned, owned by the caller: Delta (fp32 [B,Hq,Lq], rounded up to 256
 *               bytes), then the accumulator (B*Hq*ceil(Lq/128)*128*D fp32).  Nothing is kept
 *               between calls.  Too small or NULL: SWA_ERR_WORKSPACE.
 *   D = 256 has no fused kernel: the call runs the split backward (the size function then returns
 *   the Delta bytes alone).
 * Shapes, windows, causal, f16 and errors as in swa_attn_bwd_ex.
 */
size_t swa_attn_bwd_fused_workspace_bytes(int B, int Hq, int Lq, int D);
swa_status swa_attn_bwd_fused(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int Lq, int Lk, int D, int window,
                              int causal, float scale, int f16, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * The three phases swa_attn_bwd_fused runs, one by one (bf16, Lq = Lk = N, causal, D in {64, 128};
 * D = 256: SWA_ERR_UNSUPPORTED), e.g. to time each kernel.  `workspace` is swa_attn_bwd_fused's.
 *   swa_attn_bwd_fused_preprocess : Delta, and the accumulator zeroed.
 *   swa_attn_bwd_fused_dkdv       : dk, dv, and every dQ partial added into the accumulator.
 *   swa_attn_bwd_fused_dq         : dq = scale * accumulator, rounded to bf16.
 */
swa_status swa_attn_bwd_fused_preprocess(const void* o, const void* dO, void* workspace,
                                         size_t workspace_bytes, int B, int Hq, int N, int D,
                                         cudaStream_t stream);
swa_status swa_attn_bwd_fused_dkdv(const void* q, const void* k, const void* v, const void* dO,
                                   const float* lse, void* dk, void* dv, void* workspace,
                                   size_t workspace_bytes, int B, int Hq, int Hkv, int N, int D,
                                   int window, float scale, cudaStream_t stream);
swa_status swa_attn_bwd_fused_dq(void* dq, const void* workspace, size_t workspace_bytes, int B,
                                 int Hq, int N, int D, float scale, cudaStream_t stream);

/*
 * Backward without any caller-provided workspace and without allocating: the same computation and
 * kernels as swa_attn_bwd, but the per-row Delta scratch lives in a fixed array of device memory
 * that is part of the library image (SWA_NOALLOC_MAX_ROWS fp32 values, 16 MiB; every GPU that loads
 * the library keeps that array until the process exits).  The pages this library follows have no
 * counterpart of this entry point.
 *
 * It is for callers that cannot obtain scratch device memory: code whose device memory is owned
 * and planned by a host framework's allocator (which a side cudaMalloc would bypass), code that
 * must not allocate once its steady state has begun (an allocation can synchronize the device or
 * fail under memory pressure mid-run), and plain C callers that only hold the tensors' pointers.
 * The caller still passes every input and output buffer.
 *
 *   Limit: B*Hq*N <= SWA_NOALLOC_MAX_ROWS, else SWA_ERR_WORKSPACE and nothing is launched.
 *   Set-up: the first call on each device, with that device current, looks up the array's device
 *           address (no allocation); make that first call before any stream capture.
 *   Sharing: every call on a device uses the same array, and it keeps the last call's contents.
 *           Each call fully rewrites the rows it reads before reading them, so nothing has to start
 *           at zero; but calls whose kernels overlap on the GPU (other streams, other threads) race
 *           on the array and give wrong results.  Serialize them.
 * Other arguments, checks and errors are those of swa_attn_bwd.
 */
#define SWA_NOALLOC_MAX_ROWS (1 << 22)
swa_status swa_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                int B, int Hq, int Hkv, int N, int D, int window, float scale,
                                cudaStream_t stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* swa_strerror(swa_status status);

/*
 * Synchronizes `stream`, then reads and clears the current device's error word, which a kernel
 * sets when one of its bounded waits runs out (or when it finds its dynamic shared memory not
 * 1024-byte aligned, which the 128-byte-swizzled tiles need; it then returns without work).
 * Returns SWA_ERR_DEVICE_LAYOUT or SWA_ERR_DEVICE_TIMEOUT if the word was set, SWA_ERR_CUDA if
 * the synchronize failed, else SWA_OK.
 */
swa_status swa_check_device(cudaStream_t stream);

/*
 * Self-test of the failure path: launches on `stream` one block that waits, with the kernels'
 * own bounded wait, on a barrier nothing arrives on.  After about a second the wait runs out,
 * sets the error word and the block exits, so a following swa_check_device returns
 * SWA_ERR_DEVICE_TIMEOUT and the context stays usable.  Returns SWA_OK once launched.
 */
swa_status swa_selftest_wait_timeout(cudaStream_t stream);

/* Library ABI version (major*100 + minor). */
int swa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWA_ATTN_H */
