// Instantiations and launchers of the backward pass (d_head = 64 and 128;
// dense and packed variable-length tensors; causal or not).
#include "fa_launch.h"

namespace fa {

namespace {
// Q/dO ring depth: two 64 KB slots fit beside K, V and dS^T for d = 128; the
// d = 64 slots are half the size, so four fit.
template <int D>
constexpr int kBwdStages = D == 128 ? 2 : 4;

template <int D, bool CAUSAL, bool VARLEN>
cudaError_t launch_bwd_impl(const BwdLaunchArgs& a) {
  const long long prep_rows = static_cast<long long>(a.p.B) * a.p.H * a.p.nq_pad;
  const long long dq_rows = static_cast<long long>(a.p.B) * a.p.H * a.p.Nq;
  cudaError_t e;
  if (prep_rows > 0) {
    fa_bwd_prep_kernel<D, VARLEN><<<static_cast<unsigned>((prep_rows + 7) / 8), 256, 0, a.stream>>>(a.p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto* kern = &fa_bwd_kernel<D, kBwdStages<D>, CAUSAL, VARLEN>;
  constexpr int smem = BwdSmem<D, kBwdStages<D>>::kAlloc;
  static std::atomic<unsigned long long> done{0};
  e = set_smem_once(reinterpret_cast<const void*>(kern), smem, done);
  if (e != cudaSuccess) return e;
  if (a.grid.x > 0) {  // packed sequences may have no keys at all: dQ = 0 from the two row passes
    kern<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (dq_rows > 0) fa_bwd_dq_kernel<D, VARLEN><<<static_cast<unsigned>((dq_rows + 7) / 8), 256, 0, a.stream>>>(a.p);
  return cudaGetLastError();
}
}  // namespace

template <>
cudaError_t launch_bwd<128, false, false>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<128, false, false>(a);
}
template <>
cudaError_t launch_bwd<128, false, true>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<128, false, true>(a);
}
template <>
cudaError_t launch_bwd<128, true, false>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<128, true, false>(a);
}
template <>
cudaError_t launch_bwd<128, true, true>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<128, true, true>(a);
}
template <>
cudaError_t launch_bwd<64, false, false>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<64, false, false>(a);
}
template <>
cudaError_t launch_bwd<64, false, true>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<64, false, true>(a);
}
template <>
cudaError_t launch_bwd<64, true, false>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<64, true, false>(a);
}
template <>
cudaError_t launch_bwd<64, true, true>(const BwdLaunchArgs& a) {
  return launch_bwd_impl<64, true, true>(a);
}

}  // namespace fa
