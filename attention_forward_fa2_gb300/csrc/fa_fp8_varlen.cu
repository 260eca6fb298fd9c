// Kernel instantiations of the variable-length FP8 forward (packed e4m3 Q and
// K rows, per-sequence transposed V columns; see fa_fp8.cu for the layouts).
#include "fa_launch.h"

namespace fa {
namespace {

template <bool CAUSAL>
cudaError_t launch_impl(const LaunchArgs& a) {
  auto* kern = &fa_fwd_kernel<128, 128, kFp8Stages, true, CAUSAL, false, false, true>;
  constexpr int smem = SmemLayout<128, 128, kFp8Stages, 1>::kAlloc;
  static std::atomic<unsigned long long> done{0};
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, done);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8_varlen(bool causal, const LaunchArgs& a) {
  return causal ? launch_impl<true>(a) : launch_impl<false>(a);
}

}  // namespace fa
