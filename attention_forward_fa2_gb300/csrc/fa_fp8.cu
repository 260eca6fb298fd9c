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
//
// Variable-length batches: Q and K codes keep the packed row layout, and the
// blocks restart at every sequence (block j of sequence b covers its rows
// 128j .. 128j + 127; scales [B, H, ceil(max_q / 128)] and [B, Hk,
// ceil(max_k / 128)], scale 1 for blocks past a sequence's end; V scales
// [B, Hk]).  The transposed V codes are [Hk, d, kp_total]: sequence b owns
// columns [fp8_vt_col0(cu_k[b], b), fp8_vt_col0(cu_k[b + 1], b + 1)), its keys
// first and zeros after them, so each sequence starts on a 16-byte boundary
// (the TMA rule for the innermost coordinate) and every column is written.
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

// e4m3 codes of x / s for the bf16 values x of a block sharing the scale s > 0.
// The quotient is the fp32 division's (x / s rounded to nearest) at two packed
// multiplies and two packed FMAs per pair instead of two divisions: with
// rs = RN(1 / s), q = RN(x rs) lies within an ulp of x / s, the residual
// x - q s is exact in one FMA, and q + (x - q s) rs rounded once is the
// correctly rounded quotient (Markstein, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  The
// theorem wants x and the residual above the subnormal range: for scales below
// 2^-60, x and s are first multiplied by 2^64 (exact, same quotient); for larger
// scales a subnormal x has |x / s| < 2^-66, whose code is zero either way.  The
// quotient takes the sign of x, as the division's does, also when it is zero.
// An infinite scale (an infinite input) gives quotients 0 as the division does.
struct BlockQuantizer {
  uint64_t k2, rs2, nsk2;
  __device__ explicit BlockQuantizer(float s) {
    const float k = s < 0x1p-60f ? 0x1p64f : 1.f;
    const float sk = s * k;
    const float rs = __frcp_rn(sk);
    const float nsk = isinf(sk) ? 0.f : -sk;
    k2 = ptx::f2_pack(k, k);
    rs2 = ptx::f2_pack(rs, rs);
    nsk2 = ptx::f2_pack(nsk, nsk);
  }
  // Codes of the low and high bf16 halves of w (low code in the low byte).
  __device__ __forceinline__ uint32_t codes2(uint32_t w) const {
    const uint64_t x = ptx::f2_mul(ptx::f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)), k2);
    const uint64_t q = ptx::f2_mul(x, rs2);
    const uint64_t r = ptx::f2_fma(q, nsk2, x);
    constexpr uint64_t kSign = 0x8000000080000000ull;
    const uint64_t qq = (ptx::f2_fma(r, rs2, q) & ~kSign) | (x & kSign);
    float lo, hi;
    ptx::f2_unpack(qq, lo, hi);
    return ptx::pack_e4m3x2(lo, hi);
  }
};

__device__ __forceinline__ float amax8(uint4 u) {
  // Largest magnitude of eight bf16 values (the sign bit cleared).
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, __uint_as_float((w[i] << 16) & 0x7fffffffu));
    m = fmaxf(m, __uint_as_float(w[i] & 0x7fff0000u));
  }
  return m;
}

// One block per 128-row block of Q (blockIdx.x < nq) or of K.  A block's rows
// are read once into registers (eight 16-byte chunks per thread: 128 rows x
// 256 bytes), reduced to the block maximum, and written as codes with the
// block's scale.  K blocks also reduce the same rows of V and fold them into
// the per-head V maximum (non-negative floats order like their bit patterns,
// so an integer atomicMax on the bits is exact and order-independent).
// Rows of sequence b in the packed tensors (variable length; an inconsistent
// entry counts as empty, so nothing outside the tensors is touched) or of
// batch b (dense).
template <bool VARLEN>
__device__ __forceinline__ void fp8_seq(const int* cu, int max_len, int total, int b, int& row0, int& len) {
  if constexpr (VARLEN) {
    row0 = cu[b];
    len = cu[b + 1] - row0;
    if (len < 0 || len > max_len || row0 < 0 || row0 > total - len) len = 0;
  } else {
    row0 = b * max_len;
    len = max_len;
  }
}

template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) fp8_quant_qk_kernel(Fp8QuantParams p, unsigned int* v_amax_bits) {
  static_assert(D == 128, "16 chunks of 16 bytes per row");
  const int qb = (p.Nq + kBR - 1) / kBR, kb = (p.Nk + kBR - 1) / kBR;
  const long long nq = static_cast<long long>(p.B) * p.H * qb;
  long long id = blockIdx.x;
  const bool isq = id < nq;
  if (!isq) id -= nq;
  const int blocks = isq ? qb : kb;
  const int Hx = isq ? p.H : p.Hk;
  // Heads vary fastest over consecutive blocks: blocks resident together read
  // the same rows of every head, i.e. whole contiguous rows of the tensor,
  // rather than slices of one head a row stride apart.
  const int h = static_cast<int>(id % Hx);
  const long long rest = id / Hx;
  const int blk = static_cast<int>(rest % blocks), b = static_cast<int>(rest / blocks);
  const long long bh = static_cast<long long>(b) * Hx + h;
  int seq0, len;
  fp8_seq<VARLEN>(isq ? p.cu_q : p.cu_k, isq ? p.Nq : p.Nk, isq ? p.total_q : p.total_k, b, seq0, len);
  const int r0 = blk * kBR, rows = min(len - r0, kBR);  // <= 0: a block past the sequence (scale 1)
  const __nv_bfloat16* src = isq ? p.q : p.k;
  uint8_t* dst = isq ? p.q8 : p.k8;
  uint4 x[8];
  float m = 0.f, mv = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = threadIdx.x + 256 * i;  // chunk index in the block: row e / 16, chunk e % 16
    const int r = e >> 4, c = e & 15;
    x[i] = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) {
      const size_t off = ((static_cast<size_t>(seq0) + r0 + r) * Hx + h) * D + c * 8;
      x[i] = *reinterpret_cast<const uint4*>(src + off);
      m = fmaxf(m, amax8(x[i]));
      if (!isq) mv = fmaxf(mv, amax8(*reinterpret_cast<const uint4*>(p.v + off)));
    }
  }
  m = block_amax(m);
  const float s = scale_of(m);
  const BlockQuantizer qz(s);
  if (threadIdx.x == 0) (isq ? p.q_scale : p.k_scale)[bh * blocks + blk] = s;
  if (!isq) {
    mv = block_amax(mv);
    if (threadIdx.x == 0) atomicMax(v_amax_bits + bh, __float_as_uint(mv));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = threadIdx.x + 256 * i;
    const int r = e >> 4, c = e & 15;
    if (r < rows) {
      const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
      uint32_t o[2];
#pragma unroll
      for (int half = 0; half < 2; ++half) o[half] = qz.codes2(w[2 * half]) | (qz.codes2(w[2 * half + 1]) << 16);
      const size_t off = ((static_cast<size_t>(seq0) + r0 + r) * Hx + h) * D + c * 8;
      *reinterpret_cast<uint2*>(dst + off) = make_uint2(o[0], o[1]);
    }
  }
}

// The per-head V scales from the reduced maxima (after the transposed codes are written).
__global__ void fp8_v_scale_kernel(Fp8QuantParams p, const unsigned int* v_amax_bits) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < p.B * p.Hk) p.v_scale[i] = scale_of(__uint_as_float(v_amax_bits[i]));
}

// V codes, transposed: one block per (b, 64-key tile, hk), hk fastest (as in
// the kernel above, resident blocks read contiguous rows).  Thread
// (chunk, kg) = (tid % 16, tid / 16) loads 8 features of keys 4kg .. 4kg+3
// (16-byte loads; a warp reads two whole 256-byte key rows per instruction),
// converts them and regroups the bytes into one 32-bit word per feature (four
// consecutive keys).  The words go through shared memory in feature-major
// rows of 17 words (conflict-free for both phases) and leave as coalesced
// 4-byte stores of the transposed rows.
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) fp8_quant_vt_kernel(Fp8QuantParams p, const unsigned int* v_amax_bits,
                                                           int ktiles) {
  static_assert(D == 128, "16 chunks of 8 features per key");
  constexpr int kRowWords = 17;  // 16 words of 4 keys, one word of padding
  __shared__ uint32_t tile[D * kRowWords];
  const int h = static_cast<int>(blockIdx.x % p.Hk);
  const long long rest = blockIdx.x / p.Hk;
  const int kt = static_cast<int>(rest % ktiles);  // 64-key tile
  const int b = static_cast<int>(rest / ktiles);
  const int bh = b * p.Hk + h;
  const BlockQuantizer qz(scale_of(__uint_as_float(v_amax_bits[bh])));
  int seq0, len;
  fp8_seq<VARLEN>(p.cu_k, p.Nk, p.total_k, b, seq0, len);
  // Columns this sequence owns (keys, then zeros).
  long long col0 = 0;
  int span = p.nk_pad;
  if constexpr (VARLEN) {
    col0 = fp8_vt_col0(p.cu_k[b], b);
    const long long end = min(fp8_vt_col0(p.cu_k[b + 1], b + 1), p.kp_total);
    span = col0 >= 0 && end > col0 ? static_cast<int>(min(end - col0, 64LL * ktiles)) : 0;
  }
  if (kt * 64 >= span) return;
  const int chunk = threadIdx.x & 15, kg = threadIdx.x >> 4;
  uint32_t q2[4][4];  // [key][feature pair]: e4m3 codes of features 2i (low byte) and 2i+1
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int key = kt * 64 + 4 * kg + k;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (key < len)
      u = *reinterpret_cast<const uint4*>(p.v + ((static_cast<size_t>(seq0) + key) * p.Hk + h) * D + chunk * 8);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      q2[k][i] = qz.codes2(w[i]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t01 = __byte_perm(q2[0][i], q2[1][i], 0x5410);  // k0.f0 k0.f1 k1.f0 k1.f1
    const uint32_t t23 = __byte_perm(q2[2][i], q2[3][i], 0x5410);
    tile[(chunk * 8 + 2 * i) * kRowWords + kg] = __byte_perm(t01, t23, 0x6420);      // feature 2i, keys 0..3
    tile[(chunk * 8 + 2 * i + 1) * kRowWords + kg] = __byte_perm(t01, t23, 0x7531);  // feature 2i+1
  }
  __syncthreads();
#pragma unroll
  for (int e = threadIdx.x; e < D * 16; e += 256) {
    const int c = e >> 4, wd = e & 15;
    const int key0 = kt * 64 + 4 * wd;
    // Spans are multiples of 16 keys: a word is wholly inside or outside.
    if (key0 < span) {
      const size_t row = VARLEN ? static_cast<size_t>(h) * D + c : static_cast<size_t>(bh) * D + c;
      const size_t pitch = VARLEN ? static_cast<size_t>(p.kp_total) : static_cast<size_t>(p.nk_pad);
      *reinterpret_cast<uint32_t*>(p.vt8 + row * pitch + col0 + key0) = tile[c * kRowWords + wd];
    }
  }
}

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
  // v_scale holds the bit patterns of the per-head V maxima until the last
  // kernel turns them into scales (it is the only scratch the call needs).
  unsigned int* const v_amax_bits = reinterpret_cast<unsigned int*>(p.v_scale);
  const long long bhk = static_cast<long long>(p.B) * p.Hk;
  cudaError_t e = cudaMemsetAsync(v_amax_bits, 0, static_cast<size_t>(bhk) * sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;
  const bool varlen = p.cu_q != nullptr;
  const long long qb = (p.Nq + kBR - 1) / kBR, kb = (p.Nk + kBR - 1) / kBR;
  const long long nblocks = static_cast<long long>(p.B) * p.H * qb + bhk * kb;
  if (nblocks > 0) {
    if (varlen)
      fp8_quant_qk_kernel<128, true><<<static_cast<unsigned>(nblocks), 256, 0, stream>>>(p, v_amax_bits);
    else
      fp8_quant_qk_kernel<128, false><<<static_cast<unsigned>(nblocks), 256, 0, stream>>>(p, v_amax_bits);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // Variable length: a sequence's span is at most its length + 31 columns.
  const int kt = varlen ? (p.Nk + 31 + 63) / 64 : (p.nk_pad + 63) / 64;
  if (kt > 0 && bhk > 0) {
    const long long nvt = bhk * kt;
    if (nvt > 0x7fffffffLL) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(nvt));
    if (varlen)
      fp8_quant_vt_kernel<128, true><<<grid, 256, 0, stream>>>(p, v_amax_bits, kt);
    else
      fp8_quant_vt_kernel<128, false><<<grid, 256, 0, stream>>>(p, v_amax_bits, kt);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  fp8_v_scale_kernel<<<static_cast<unsigned>((bhk + 255) / 256), 256, 0, stream>>>(p, v_amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(bool causal, const LaunchArgs& a) {
  return causal ? launch_fwd_fp8_impl<true>(a) : launch_fwd_fp8_impl<false>(a);
}

int fp8_smem_bytes() { return SmemLayout<128, 128, kFp8Stages, 1>::kAlloc; }

}  // namespace fa
