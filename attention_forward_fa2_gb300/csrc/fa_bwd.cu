// Instantiations and launchers of the backward pass (d_head = 128).
#include "fa_launch.h"

namespace fa {

namespace {
constexpr int kBwdStages = 2;

template <int D, bool CAUSAL>
cudaError_t launch_bwd_impl(const BwdLaunchArgs& a) {
  const long long prep_rows = static_cast<long long>(a.p.B) * a.p.H * a.p.nq_pad;
  const long long dq_rows = static_cast<long long>(a.p.B) * a.p.H * a.p.Nq;
  cudaError_t e;
  if (prep_rows > 0) {
    fa_bwd_prep_kernel<D><<<static_cast<unsigned>((prep_rows + 7) / 8), 256, 0, a.stream>>>(a.p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto* kern = &fa_bwd_kernel<D, kBwdStages, CAUSAL>;
  constexpr int smem = BwdSmem<D, kBwdStages>::kAlloc;
  static std::atomic<unsigned long long> done{0};
  e = set_smem_once(reinterpret_cast<const void*>(kern), smem, done);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dq_rows > 0) fa_bwd_dq_kernel<D><<<static_cast<unsigned>((dq_rows + 7) / 8), 256, 0, a.stream>>>(a.p);
  return cudaGetLastError();
}
}  // namespace

template <>
cudaError_t launch_bwd<128, false>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<128, false>(a);
}
template <>
cudaError_t launch_bwd<128, true>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<128, true>(a);
}

}  // namespace fa
