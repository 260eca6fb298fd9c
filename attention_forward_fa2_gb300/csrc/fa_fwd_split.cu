// Kernel instantiations for the key-split form (dense tensors), and the
// combine kernel launcher.
#include "fa_combine.cuh"
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH_SPLIT(128, 2, false)
FA_DEFINE_LAUNCH_SPLIT(128, 2, true)
FA_DEFINE_LAUNCH_SPLIT(64, 3, false)
FA_DEFINE_LAUNCH_SPLIT(64, 3, true)

cudaError_t launch_combine(int D, const float* ws_o, const float* ws_lse, int S, long long rows, int H,
                           int Nq, __nv_bfloat16* o, float* lse, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
  if (D == 128)
    splitkv_combine_kernel<128><<<blocks, 128, 0, stream>>>(ws_o, ws_lse, S, rows, H, Nq, o, lse);
  else
    splitkv_combine_kernel<64><<<blocks, 128, 0, stream>>>(ws_o, ws_lse, S, rows, H, Nq, o, lse);
  return cudaGetLastError();
}
}  // namespace fa
