// FP8 (e4m3) forward: block quantisation of bf16 Q, K, V and the
// kind::f8f6f4 instantiations of the forward kernel.
//
// Block quantisation ("GPU 内核与 FlashAttention" §15.5): each block of
// values shares one fp32 scale s = amax / 448 (448 is the largest finite
// e4m3 value), and a value x is stored as the e4m3 code nearest to x / s
// (round to nearest even, saturating).  Blocks: 128 query rows of one head for
// Q, 128 keys of one key/value head for K, one whole key/value head for V.
// V is written transposed, [B, Hk, d, nk_pad] with nk_pad = Nk rounded up to
// 16 (zero padding), so that it is a K-major operand of O += P V.
#include <cuda_bf16.h>

#include "fa_launch.h"

namespace fa {
namespace {

constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ float block_amax(float v) {
  // v: this thread's partial maximum; returns the block maximum (256 threads).
  __shared__ float red[8];
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) r = fmaxf(r, red[i]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ float scale_of(float amax) { return amax > 0.f ? amax / kE4M3Max : 1.f; }

// One block per scale: blockIdx.x < nq -> a 128-row block of Q, then K blocks,
// then one block per key/value head for V.
template <int D>
__global__ void __launch_bounds__(256) fp8_scales_kernel(Fp8QuantParams p) {
  const int qb = (p.Nq + kBR - 1) / kBR, kb = (p.Nk + kBR - 1) / kBR;
  const long long nq = static_cast<long long>(p.B) * p.H * qb;
  const long long nk = static_cast<long long>(p.B) * p.Hk * kb;
  long long id = blockIdx.x;
  float m = 0.f;
  float* out;
  if (id < nq) {
    const int blk = static_cast<int>(id % qb);
    const long long bh = id / qb;
    const int h = static_cast<int>(bh % p.H), b = static_cast<int>(bh / p.H);
    const int r0 = blk * kBR, r1 = min(p.Nq, r0 + kBR);
    for (int e = threadIdx.x; e < (r1 - r0) * D; e += blockDim.x) {
      const int r = r0 + e / D, c = e % D;
      m = fmaxf(m, fabsf(__bfloat162float(p.q[((static_cast<size_t>(b) * p.Nq + r) * p.H + h) * D + c])));
    }
    out = p.q_scale + id;
  } else if (id < nq + nk) {
    id -= nq;
    const int blk = static_cast<int>(id % kb);
    const long long bh = id / kb;
    const int h = static_cast<int>(bh % p.Hk), b = static_cast<int>(bh / p.Hk);
    const int r0 = blk * kBR, r1 = min(p.Nk, r0 + kBR);
    for (int e = threadIdx.x; e < (r1 - r0) * D; e += blockDim.x) {
      const int r = r0 + e / D, c = e % D;
      m = fmaxf(m, fabsf(__bfloat162float(p.k[((static_cast<size_t>(b) * p.Nk + r) * p.Hk + h) * D + c])));
    }
    out = p.k_scale + id;
  } else {
    id -= nq + nk;
    const int h = static_cast<int>(id % p.Hk), b = static_cast<int>(id / p.Hk);
    for (long long e = threadIdx.x; e < static_cast<long long>(p.Nk) * D; e += blockDim.x) {
      const long long r = e / D;
      const int c = static_cast<int>(e % D);
      m = fmaxf(m, fabsf(__bfloat162float(p.v[((static_cast<size_t>(b) * p.Nk + r) * p.Hk + h) * D + c])));
    }
    out = p.v_scale + id;
  }
  m = block_amax(m);
  if (threadIdx.x == 0) *out = scale_of(m);
}

__device__ __forceinline__ uint32_t to_e4m3x2(float lo, float hi) { return ptx::pack_e4m3x2(lo, hi); }

// Q and K codes, same layout as the bf16 input; 8 elements per thread.
template <int D>
__global__ void __launch_bounds__(256) fp8_quant_qk_kernel(Fp8QuantParams p) {
  const long long nq8 = static_cast<long long>(p.B) * p.Nq * p.H * D / 8;
  const long long nk8 = static_cast<long long>(p.B) * p.Nk * p.Hk * D / 8;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nq8 + nk8) return;
  const bool isq = i < nq8;
  const long long e = (isq ? i : i - nq8) * 8;  // first element
  const int Hx = isq ? p.H : p.Hk, Nx = isq ? p.Nq : p.Nk;
  const long long row = e / D;                  // (b * N + n) * Hx + h
  const int h = static_cast<int>(row % Hx);
  const long long bn = row / Hx;
  const int n = static_cast<int>(bn % Nx), b = static_cast<int>(bn / Nx);
  const int blocks = (Nx + kBR - 1) / kBR;
  const float s = isq ? p.q_scale[(static_cast<size_t>(b) * p.H + h) * blocks + n / kBR]
                      : p.k_scale[(static_cast<size_t>(b) * p.Hk + h) * blocks + n / kBR];
  const __nv_bfloat16* src = (isq ? p.q : p.k) + e;
  uint8_t* dst = (isq ? p.q8 : p.k8) + e;
  uint32_t w[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = __bfloat162float(src[4 * half + k]) / s;
    w[half] = to_e4m3x2(x[0], x[1]) | (to_e4m3x2(x[2], x[3]) << 16);
  }
  *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
}

// V codes, transposed: one block per (b, hk, 64 keys); a 64 x D tile goes
// through shared memory so that both the reads (rows of d) and the writes
// (rows of keys) are contiguous.
template <int D>
__global__ void __launch_bounds__(256) fp8_quant_vt_kernel(Fp8QuantParams p) {
  __shared__ uint8_t tile[D][64 + 4];
  const int kt = blockIdx.x;  // 64-key tile
  const int bh = blockIdx.y;  // b * Hk + hk
  const int h = bh % p.Hk, b = bh / p.Hk;
  const float s = p.v_scale[bh];
  for (int e = threadIdx.x; e < 64 * D; e += blockDim.x) {
    const int r = e / D, c = e % D;
    const int key = kt * 64 + r;
    float x = 0.f;
    if (key < p.Nk) x = __bfloat162float(p.v[((static_cast<size_t>(b) * p.Nk + key) * p.Hk + h) * D + c]) / s;
    tile[c][r] = static_cast<uint8_t>(to_e4m3x2(x, 0.f) & 0xffu);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 64 * D; e += blockDim.x) {
    const int c = e / 64, r = e % 64;
    const int key = kt * 64 + r;
    if (key < p.nk_pad) p.vt8[(static_cast<size_t>(bh) * D + c) * p.nk_pad + key] = tile[c][r];
  }
}

constexpr int kFp8Stages = 4;

template <bool CAUSAL>
cudaError_t launch_fwd_fp8_impl(const LaunchArgs& a) {
  auto* kern = &fa_fwd_kernel<128, 128, kFp8Stages, false, CAUSAL, false, false, true>;
  constexpr int smem = SmemLayout<128, 128, kFp8Stages, 1>::kAlloc;
  static std::atomic<unsigned long long> done{0};
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, done);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantParams& p, cudaStream_t stream) {
  if (p.D != 128) return cudaErrorInvalidValue;
  const long long qb = (p.Nq + kBR - 1) / kBR, kb = (p.Nk + kBR - 1) / kBR;
  const long long nscales = static_cast<long long>(p.B) * p.H * qb + static_cast<long long>(p.B) * p.Hk * kb +
                            static_cast<long long>(p.B) * p.Hk;
  fp8_scales_kernel<128><<<static_cast<unsigned>(nscales), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long n8 = (static_cast<long long>(p.B) * p.Nq * p.H + static_cast<long long>(p.B) * p.Nk * p.Hk) * 128 / 8;
  if (n8 > 0) {
    fp8_quant_qk_kernel<128><<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int kt = (p.nk_pad + 63) / 64;
  if (kt > 0) {
    fp8_quant_vt_kernel<128><<<dim3(static_cast<unsigned>(kt), static_cast<unsigned>(p.B * p.Hk)), 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_fwd_fp8(bool causal, const LaunchArgs& a) {
  return causal ? launch_fwd_fp8_impl<true>(a) : launch_fwd_fp8_impl<false>(a);
}

int fp8_smem_bytes() { return SmemLayout<128, 128, kFp8Stages, 1>::kAlloc; }

}  // namespace fa
