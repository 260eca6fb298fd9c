// fa_combine.cuh -- merge of key-split partial results.
//
// Each split s of a query row produced a normalised output O_s and its
// log-sum-exp LSE_s over its own keys.  The two-block merge of
// "GPU 内核与 FlashAttention" §11.2, applied to any number of blocks and to the
// outputs as well, gives the exact result over all keys:
//     M = max_s LSE_s,  w_s = e^(LSE_s - M),  l = sum_s w_s,
//     LSE = M + log l,  O = sum_s (w_s / l) O_s.
// A row whose splits all saw no key gets O = 0 and LSE = -inf.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace fa {

// One warp per query row; lane c owns output columns [c * D/32, (c+1) * D/32).
// ws_o: [S, rows, D] fp32, ws_lse: [S, rows] fp32 with rows = B * H * Nq ordered
// (b, h, i); o: [B, Nq, H, D] bf16; lse: [B, H, Nq] fp32.
template <int D>
__global__ void __launch_bounds__(128) splitkv_combine_kernel(const float* __restrict__ ws_o,
                                                             const float* __restrict__ ws_lse, int S,
                                                             long long rows, int H, int Nq,
                                                             __nv_bfloat16* __restrict__ o,
                                                             float* __restrict__ lse) {
  constexpr int kPer = D / 32;
  const long long r = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float m = -INFINITY;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, ws_lse[static_cast<size_t>(s) * rows + r]);
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, w));
  const long long bh = r / Nq;
  const int i = static_cast<int>(r % Nq);
  const int h = static_cast<int>(bh % H);
  const long long b = bh / H;
  __nv_bfloat16* const orow = o + ((b * Nq + i) * H + h) * D + lane * kPer;
  if (m == -INFINITY) {
#pragma unroll
    for (int c = 0; c < kPer; ++c) orow[c] = __float2bfloat16(0.f);
    if (lane == 0) lse[r] = -INFINITY;
    return;
  }
  float acc[kPer];
#pragma unroll
  for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
  float l = 0.f;
  for (int s = 0; s < S; ++s) {
    const float ls = ws_lse[static_cast<size_t>(s) * rows + r];
    const float wgt = ptx::ex2((ls - m) * 1.4426950408889634f);  // e^(LSE_s - M); 0 for -inf
    l += wgt;
    const float* src = ws_o + (static_cast<size_t>(s) * rows + r) * D + lane * kPer;
#pragma unroll
    for (int c = 0; c < kPer; ++c) acc[c] = fmaf(wgt, src[c], acc[c]);
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int c = 0; c < kPer; c += 2) {
    const uint32_t pk = ptx::pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
    *reinterpret_cast<uint32_t*>(orow + c) = pk;
  }
  if (lane == 0) lse[r] = m + logf(l);
}

}  // namespace fa
