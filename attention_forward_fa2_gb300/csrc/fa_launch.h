// fa_launch.h -- host-side launch interface between the C-ABI layer and the
// kernel translation units (one per head dimension, compiled in parallel).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "fa_bwd_kernel.cuh"
#include "fa_fwd_kernel.cuh"

namespace fa {

struct LaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  FwdParams p;
  dim3 grid;
  cudaStream_t stream;
};

// Key/value tile width of the key-split form and of the default config.
constexpr int kBC = 128;

// Raises a kernel's dynamic shared-memory limit once per device (the
// attribute persists; setting it on every launch costs host time).
// `done` is one bit per device ordinal < 64, owned by the calling kernel.
inline cudaError_t set_smem_once(const void* kern, int smem, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <int D, int BC, int STAGES, bool VARLEN, bool CAUSAL, bool QUAD = false>
cudaError_t launch_fwd(const LaunchArgs& a);

// Defined in the translation unit that owns the kernel.
#define FA_DEFINE_LAUNCH(D, BC, STAGES, VARLEN, CAUSAL)                                       \
  template <>                                                                                 \
  cudaError_t launch_fwd<D, BC, STAGES, VARLEN, CAUSAL>(const LaunchArgs& a) {                \
    auto* kern = &fa_fwd_kernel<D, BC, STAGES, VARLEN, CAUSAL>;                               \
    constexpr int smem = SmemLayout<D, BC, STAGES>::kAlloc;                                   \
    static std::atomic<unsigned long long> done{0};                                          \
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, done);          \
    if (e != cudaSuccess) return e;                                                           \
    kern<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);          \
    return cudaGetLastError();                                                                \
  }

// The quad-shuffle softmax form (128-key tiles, no mask).
#define FA_DEFINE_LAUNCH_QUAD(D, STAGES, VARLEN)                                              \
  template <>                                                                                 \
  cudaError_t launch_fwd<D, 128, STAGES, VARLEN, false, true>(const LaunchArgs& a) {          \
    auto* kern = &fa_fwd_kernel<D, 128, STAGES, VARLEN, false, false, true>;                  \
    constexpr int smem = SmemLayout<D, 128, STAGES>::kAlloc;                                  \
    static std::atomic<unsigned long long> done{0};                                          \
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, done);          \
    if (e != cudaSuccess) return e;                                                           \
    kern<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);          \
    return cudaGetLastError();                                                                \
  }

// Key-split form (dense tensors only): the unit also carries a key split.
template <int D, int STAGES, bool CAUSAL>
cudaError_t launch_fwd_split(const LaunchArgs& a);

#define FA_DEFINE_LAUNCH_SPLIT(D, STAGES, CAUSAL)                                              \
  template <>                                                                                 \
  cudaError_t launch_fwd_split<D, STAGES, CAUSAL>(const LaunchArgs& a) {                      \
    auto* kern = &fa_fwd_kernel<D, kBC, STAGES, false, CAUSAL, true>;                         \
    constexpr int smem = SmemLayout<D, kBC, STAGES>::kAlloc;                                  \
    static std::atomic<unsigned long long> done{0};                                          \
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, done);          \
    if (e != cudaSuccess) return e;                                                           \
    kern<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);          \
    return cudaGetLastError();                                                                \
  }

// Backward pass (fa_bwd_kernel.cuh): preprocessing, the key-block kernel and
// the dQ conversion, enqueued in that order on a.stream.
struct BwdLaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  BwdParams p;
  dim3 grid;
  cudaStream_t stream;
};

// VARLEN: packed [total, heads, d] tensors with cu_seqlens in a.p (3-D maps).
template <int D, bool CAUSAL, bool VARLEN>
cudaError_t launch_bwd(const BwdLaunchArgs& a);

// FP8 path (fa_fp8.cu; the variable-length kernels in fa_fp8_varlen.cu).
struct Fp8QuantParams {
  const __nv_bfloat16 *q, *k, *v;  // bf16 inputs, [B, Nq, H, D] and [B, Nk, Hk, D]
                                   // (variable length: packed [total_q, H, D] / [total_k, Hk, D])
  uint8_t *q8, *k8;                // e4m3 codes, same layouts
  uint8_t* vt8;                    // e4m3 codes of V, [B, Hk, D, nk_pad]
                                   // (variable length: [Hk, D, kp_total], sequence b from
                                   // column fp8_vt_col0(cu_k[b], b))
  float *q_scale, *k_scale, *v_scale;
  int B, Nq, Nk, H, Hk, D, nk_pad;  // variable length: Nq / Nk are the maximum lengths
  const int *cu_q, *cu_k;           // variable length: int32 [B + 1] (null when dense)
  int total_q, total_k;             // variable length: packed rows of q / k
  long long kp_total;               // variable length: columns of vt8
};
constexpr int kFp8Stages = 4;  // K/V ring slots of the FP8 kernels
cudaError_t launch_fp8_quantize(const Fp8QuantParams& p, cudaStream_t stream);
cudaError_t launch_fwd_fp8(bool causal, const LaunchArgs& a);
cudaError_t launch_fwd_fp8_varlen(bool causal, const LaunchArgs& a);
int fp8_smem_bytes();

// Host-side argument check of the key-split form (the checks fa_fwd_splitkv
// makes before sizing its workspace): FA_OK, 1 for a problem with nothing to
// do, or a negative FA_ERR_* code.
int check_split_problem(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Nq,
                        int Nk, int H, int Hk, int d, float scale, int flags);

// Merge of the key splits (fa_combine.cuh); D in {64, 128}.
cudaError_t launch_combine(int D, const float* ws_o, const float* ws_lse, int S, long long rows, int H,
                           int Nq, __nv_bfloat16* o, float* lse, cudaStream_t stream);

}  // namespace fa
