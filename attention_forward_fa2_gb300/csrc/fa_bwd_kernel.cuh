// fa_bwd_kernel.cuh -- FlashAttention-2 backward pass for sm_103a (GB300).
//
// What it computes ("GPU 内核与 FlashAttention" §13): given the forward's
// inputs, its output O and per-row log-sum-exp L, and dO = d(loss)/dO,
//     P   = exp(scale * Q K^T - L)        (recomputed, never stored)
//     dV  = P^T dO
//     dP  = dO V^T
//     D_i = do_i . o_i                    (§13.1: equals sum_j P_ij dP_ij)
//     dS  = P o (dP - D)
//     dQ  = scale * dS K,   dK = scale * dS^T Q
// following the blockwise order of §13.2 (FA2's Algorithm 2): a preprocessing
// kernel computes D (and clears the dQ accumulator), then the main kernel runs
// with the key/value block outermost -- each work unit owns one block of 128
// keys of one (batch, key/value head), keeps dK and dV on chip for the whole
// unit, loops over every query block of every query head that reads this
// key/value head (grouped heads are summed here, §14.2), and adds its share
// of dQ into an fp32 accumulator in global memory (§14.3: dQ is the one
// shared write, accumulated with atomic adds; here reductions straight from
// registers, performed at L2).  A last kernel scales the accumulator into
// bf16 dQ.
//
// Head dimension 64 or 128.  For d = 64 the K tile keeps a second, zeroed
// 64-feature panel so that dQ^T = K^T dS^T stays an M = 128 product (its rows
// 64-127 are zero and never drained).  Packed variable-length sequences
// (VARLEN, "Flash Attention实现深度解析" §3.1 layout) use the forward's tile
// rule: a tile that would run past its sequence's end is shifted back to end
// there, keys of a shifted tile that belong to the previous block are masked,
// and the preprocessing pass lays out the scaled LSE, D and the dQ
// accumulator in tile order, so that the repeated query rows of a shifted
// tile carry LSE = +inf (P = dS = 0) and drop out.
//
// Main kernel, per step (one block of 128 queries of one head):
//   S^T  = K Q^T        M=128 keys, N=128 queries, K=d    tensor memory S
//   dP^T = V dO^T       M=128 keys, N=128                 tensor memory dP
//   P^T  = 2^(S^T * scale * log2 e - L * log2 e)           softmax warps, bf16 over S
//   dS^T = P^T o (dP^T - D)                                bf16, to shared memory
//   dV  += P^T dO       M=128 keys, N=d, K=128             P^T from tensor memory
//   dK  += dS^T Q       M=128 keys, N=d, K=128             both from shared memory
//   dQ^T = K^T dS^T     M=d, N=128 queries, K=128 keys     both from shared memory,
//                                                          result over dP
// Every product is N = 128 (the full tensor rate; N = 64 products are bound by
// shared-memory operand reads) and a step issues 40 MMAs for 21 MFLOP.
// Computing dQ transposed keeps every MMA at M = 128 and makes each TMEM lane a
// feature index: for each query the 32 lanes of a drain warp hold 32
// consecutive features, one 128-byte line of the [B, H, queries, d]
// accumulator, so one reduction instruction per query adds a whole line and
// nothing is staged in shared memory.
// Tensor memory (512 columns): S [0,128) dP [128,256) dV [256,384)
// dK [384,512); dQ^T(g) reuses dP's columns once the softmax warps have read
// dP(g).  The single MMA thread issues, per step g:
//   dV(g) | S(g+1) | dK(g) dQ^T(g) | dP(g+1)   (dP(g+1) after the drain read dQ^T(g))
// Softmax warpgroup c reads columns [64c, 64c + 64) of S and dP and writes
// its packed bf16 P^T words over the first 32 of S's, 32 columns at a time;
// dS^T goes to shared memory only (the one copy both dK and dQ^T read).
//
// Roles (512 threads):
//   warps 0-7   softmax: P, dS (warps 0-3 query columns 0-63, 4-7 columns 64-127)
//   warps 8-11  dQ drain (TMEM -> registers -> L2 reductions) and the dK/dV epilogue
//               (152 registers: all 128 accumulator columns are held at once, so
//               the tensor memory is released before the reductions are issued)
//   warp 12     MMA issue (one thread) + TMEM allocation
//   warp 13     TMA loads (one thread)
//   warps 14-15 idle
// Every wait is bounded (ptx.cuh mbar_wait); on a timeout the kernel records
// the site, stops every role, drains its own copies and MMAs and frees TMEM.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "fa_fwd_kernel.cuh"
#include "ptx.cuh"

namespace fa {

constexpr int kBwdBK = 128;  // keys per work unit (M of the key-row products)
constexpr int kBwdBQ = 128;  // queries per step

struct BwdParams {
  int B, Nq, Nk, H, Hk, group;  // variable-length form: Nq / Nk are the maximum lengths
  int causal;           // bottom-right aligned: query i sees keys j <= i + len_k - len_q (per sequence)
  int nq_pad;           // Nq rounded up to kBwdBQ (row stride of lse2 / delta / dq_acc)
  int num_kb;           // key blocks per head
  int num_units;        // B * Hk * num_kb
  int units_per_item;   // 2 when causal (a balanced pair of key blocks)
  int num_items;
  const __nv_bfloat16* o;     // [B, Nq, H, d]  (preprocessing)
  const __nv_bfloat16* dout;  // [B, Nq, H, d]  (preprocessing)
  const float* lse;           // [B, H, Nq] natural log, from the forward
  const int* cu_q;            // variable-length form: int32 [B + 1] packed row offsets
  const int* cu_k;
  // The next three are in tile order: entry qb * 128 + c belongs to column c
  // of query tile qb as the main kernel loads it (the same as query row
  // qb * 128 + c, except for a variable-length sequence's last tile, which is
  // shifted back to end at the sequence end; its columns that repeat the
  // previous tile's rows carry lse2 = +inf, so they take no part).
  float* lse2;                // [B, H, nq_pad]  L * log2(e); +inf where no gradient flows
  float* delta;               // [B, H, nq_pad]  D_i (0 where no gradient flows)
  float* dq_acc;              // [B, H, nq_pad, d] fp32
  __nv_bfloat16* dq;          // [B, Nq, H, d]
  __nv_bfloat16* dk;          // [B, Nk, Hk, d]
  __nv_bfloat16* dv;          // [B, Nk, Hk, d]
  float scale;
  float scale_log2;           // scale * log2(e)
  unsigned long long timeout_ns;
  int* status;
};

// ------------------------------------------------------------ preprocessing
// Query rows of a sequence: its packed start and length (dense: 0 and Nq).
template <bool VARLEN>
__device__ __forceinline__ void bwd_seq_q(const BwdParams& p, int b, int& start, int& len) {
  start = 0;
  len = p.Nq;
  if constexpr (VARLEN) {
    start = p.cu_q[b];
    len = p.cu_q[b + 1] - start;
    if (len < 0 || len > p.Nq || start < 0) len = 0;  // reported by the main kernel
  }
}

// One warp per (b, h, tile entry t < nq_pad): D_i = sum_c do_ic o_ic in fp32,
// lse2_i for the query row i that column t % 128 of tile t / 128 holds, and a
// zeroed row of the dQ accumulator.  Entries that hold no row of their own
// (padding, or the repeated rows of a shifted last tile) and rows without
// keys (L = -inf) get lse2 = +inf and D = 0, so their P and dS are exactly 0.
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const BwdParams p) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(p.B) * p.H * p.nq_pad;
  if (row >= rows) return;
  const int t = static_cast<int>(row % p.nq_pad);
  const long long bh = row / p.nq_pad;
  const int h = static_cast<int>(bh % p.H);
  const int b = static_cast<int>(bh / p.H);
  constexpr int kPer = D / 32;  // elements per lane
  int q_start, len_q;
  bwd_seq_q<VARLEN>(p, b, q_start, len_q);
  const int qb = t / kBwdBQ, c = t % kBwdBQ;
  const RowWindow qw = make_window<VARLEN>(q_start, q_start + len_q, q_start + qb * kBwdBQ, kBwdBQ);
  float acc = 0.f;
  float l2 = INFINITY;
  if (qb * kBwdBQ < len_q && c >= qw.lo && c < qw.hi) {
    const int i = qw.load_row - q_start + c;  // query row within the sequence
    const size_t prow = VARLEN ? static_cast<size_t>(qw.load_row + c) : static_cast<size_t>(b) * p.Nq + i;
    const size_t off = (prow * p.H + h) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      acc += __bfloat162float(p.dout[off + e]) * __bfloat162float(p.o[off + e]);
    const float L = p.lse[static_cast<size_t>(bh) * p.Nq + i];
    if (L > -INFINITY) l2 = L * 1.44269504088896340736f;
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) {
    p.delta[row] = acc;
    p.lse2[row] = l2;
  }
  float* const dst = p.dq_acc + static_cast<size_t>(row) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) dst[e] = 0.f;
}

// dq[b, i, h, :] = bf16(scale * dq_acc[b, h, t(i), :]) with t(i) the tile
// entry that holds query row i; one warp per row.
template <int D, bool VARLEN>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdParams p) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(p.B) * p.H * p.Nq;
  if (row >= rows) return;
  const int i = static_cast<int>(row % p.Nq);
  const long long bh = row / p.Nq;
  const int h = static_cast<int>(bh % p.H);
  const int b = static_cast<int>(bh / p.H);
  constexpr int kPer = D / 32;
  int q_start, len_q;
  bwd_seq_q<VARLEN>(p, b, q_start, len_q);
  if (i >= len_q) return;
  const int qb = i / kBwdBQ;
  const RowWindow qw = make_window<VARLEN>(q_start, q_start + len_q, q_start + qb * kBwdBQ, kBwdBQ);
  const int t = qb * kBwdBQ + (q_start + i - qw.load_row);
  const size_t prow = VARLEN ? static_cast<size_t>(q_start + i) : static_cast<size_t>(b) * p.Nq + i;
  const float* src = p.dq_acc + (static_cast<size_t>(bh) * p.nq_pad + t) * D + lane * kPer;
  __nv_bfloat16* dst = p.dq + (prow * p.H + h) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; e += 2) {
    const float x0 = src[e] * p.scale, x1 = src[e + 1] * p.scale;
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(x0, x1);
  }
}

// ---------------------------------------------------------------- main kernel
template <int D, int STAGES>
struct BwdSmem {
  static constexpr int kKVBytes = kBwdBK * D * 2;        // one K or V block as loaded
  // K's shared tile always spans 128 features (two 64-feature panels): for
  // d = 64 the second panel stays zero, so that dQ^T = K^T dS^T keeps M = 128
  // (rows 64-127 of that product are zero and never drained).
  static constexpr int kKBytes = kBwdBK * 128 * 2;
  static constexpr int kKVPanel = kBwdBK * 128;          // 64 features x 128 rows
  static constexpr int kQBytes = kBwdBQ * D * 2;         // one Q or dO block
  static constexpr int kQPanel = kBwdBQ * 128;           // 64 features x 128 queries
  static constexpr int kSlotBytes = 2 * kQBytes;         // Q then dO
  static constexpr int kDSPanel = kBwdBK * 128;          // dS^T: 64 queries x 128 keys
  static constexpr int kDSBytes = kBwdBK * kBwdBQ * 2;   // two query panels
  static constexpr int kLDBytes = 2 * kBwdBQ * 4;        // scaled LSE then D of a query block
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKBytes;
  static constexpr int kOffQ = kOffV + kKVBytes;
  static constexpr int kOffDS = kOffQ + STAGES * kSlotBytes;
  static constexpr int kOffLD = kOffDS + kDSBytes;       // one kLDBytes block per Q/dO slot
  static constexpr int kOffBar = kOffLD + STAGES * kLDBytes;
  static constexpr int kBarKVFull = 0;
  static constexpr int kBarKVEmpty = 1;
  static constexpr int kBarQFull = 2;
  static constexpr int kBarQEmpty = kBarQFull + STAGES;
  static constexpr int kBarSFull = kBarQEmpty + STAGES;
  static constexpr int kBarDPFull = kBarSFull + 1;
  static constexpr int kBarPFull = kBarDPFull + 1;
  static constexpr int kBarDSFull = kBarPFull + 1;
  static constexpr int kBarDQFull = kBarDSFull + 1;
  static constexpr int kBarDQEmpty = kBarDQFull + 1;
  static constexpr int kBarAccFull = kBarDQEmpty + 1;
  static constexpr int kBarAccEmpty = kBarAccFull + 1;
  static constexpr int kBarTeardown = kBarAccEmpty + 1;
  static constexpr int kNumBars = kBarTeardown + 1;
  static constexpr int kOffTmem = kOffBar + ((kNumBars * 8 + 15) / 16) * 16;
  static constexpr int kOffAbort = kOffTmem + 16;
  static constexpr int kBytes = kOffAbort + 16;
  // Up to 1 KiB of slack aligns the tiles when the dynamic window does not
  // start on a 1 KiB boundary; the budget leaves less than that, so the
  // kernel checks at run time that its aligned layout fits (it does when the
  // window starts 1 KiB-aligned, as it does with no static shared memory).
  static constexpr int kAlloc = kBytes + 1024 <= 232448 ? kBytes + 1024 : 232448;
  static_assert(kOffV % 1024 == 0 && kOffQ % 1024 == 0 && kOffDS % 1024 == 0,
                "swizzled tiles need 1 KiB alignment");
  static_assert(kBytes <= 232448, "shared memory budget exceeded");
};

// One work unit: key block kb of key/value head hk in batch b, and the query
// blocks [qb0, qb0 + nqb) of each of the group's query heads.  Rows are
// sequence rows (packed rows = start + row in the variable-length form).
struct BwdUnit {
  int b, hk, kb;
  int q_start, len_q;  // the sequence's queries (dense: 0, Nq)
  int k_start, len_k;  // its keys
  int off;             // causal: query i sees keys j <= i + off
  RowWindow kw;        // the key tile as loaded (shifted back to end at the sequence end
                       // in the variable-length form; keys [lo, hi) of it are this block's)
  int qb0;             // first query block that sees any key of this block
  int nqb;             // query blocks per head
  int nsteps;          // group * nqb
};

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ BwdUnit bwd_decode(const BwdParams& p, int u) {
  BwdUnit w;
  int kb = u % p.num_kb;
  if constexpr (CAUSAL) {
    // Heaviest key blocks (the first ones: every query sees them) paired with
    // the lightest, as consecutive units of one item.
    const int pi = kb >> 1;
    kb = (kb & 1) ? p.num_kb - 1 - pi : pi;
  }
  const int r = u / p.num_kb;
  w.kb = kb;
  w.hk = r % p.Hk;
  w.b = r / p.Hk;
  w.q_start = 0;
  w.len_q = p.Nq;
  w.k_start = 0;
  w.len_k = p.Nk;
  if constexpr (VARLEN) {
    w.q_start = p.cu_q[w.b];
    w.len_q = p.cu_q[w.b + 1] - w.q_start;
    w.k_start = p.cu_k[w.b];
    w.len_k = p.cu_k[w.b + 1] - w.k_start;
    if (w.len_q < 0 || w.len_k < 0 || w.len_q > p.Nq || w.len_k > p.Nk || w.q_start < 0 || w.k_start < 0) {
      if (kb == 0 && w.hk == 0 && (threadIdx.x & 31) == 0 && threadIdx.x < 32)
        record_error(p.status, kErrBadSeqlens, 0);
      w.len_q = 0;
      w.len_k = 0;
    }
  }
  w.off = w.len_k - w.len_q;
  w.kw = make_window<VARLEN>(w.k_start, w.k_start + w.len_k, w.k_start + kb * kBwdBK, kBwdBK);
  const int num_qb = (w.len_q + kBwdBQ - 1) / kBwdBQ;
  w.qb0 = 0;
  if constexpr (CAUSAL) {
    // Query i sees key j iff j <= i + off: the first query of interest is
    // kb * 128 - off (never past the last query: every key j < len_k is seen
    // by query len_q - 1).
    const int first = kb * kBwdBK - w.off;
    w.qb0 = first <= 0 ? 0 : first / kBwdBQ;
  }
  w.nqb = kb * kBwdBK < w.len_k ? num_qb - w.qb0 : 0;
  w.nsteps = w.nqb > 0 ? p.group * w.nqb : 0;
  return w;
}

#define FA_BWD_FOR_EACH_UNIT(u)                                                      \
  for (int it_ = blockIdx.x; it_ < p.num_items && ok; it_ += gridDim.x)               \
    for (int sub_ = 0, u = it_ * p.units_per_item;                                     \
         sub_ < p.units_per_item && u < p.num_units && ok; ++sub_, ++u)

// Wait-site identifiers recorded with a timeout.
enum BwdSite : int {
  kBSiteLoadKV = 101, kBSiteLoadQ = 102, kBSiteMmaKV = 103, kBSiteMmaQ = 104, kBSiteMmaP = 105,
  kBSiteMmaDS = 106, kBSiteMmaDQ = 107, kBSiteMmaAcc = 108, kBSiteSoftS = 109, kBSiteSoftDP = 110,
  kBSiteSoftDQ = 111, kBSiteSoftQ = 112, kBSiteDrainDQ = 113, kBSiteDrainAcc = 114, kBSiteTeardown = 115,
  kBSiteSmemWindow = 116
};

// Register split (setmaxnreg): softmax warpgroups 128, the drain warpgroup
// 168 (all 128 accumulator columns in registers), MMA / load warpgroup 88.
struct BwdRegSplit {
  static constexpr int kSoftmax = 128;  // the launch allocation (__launch_bounds__(512, 1))
  static constexpr int kDrain = 152;
  static constexpr int kOther = 104;
  static_assert(2 * 128 * kSoftmax + 128 * kDrain + 128 * kOther <= 65536,
                "register split exceeds the launch allocation");
};

template <int D, int STAGES, bool CAUSAL, bool VARLEN = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  static_assert(D == 64 || D == 128, "backward kernel: d = 64 or 128");
  static_assert(STAGES >= 2, "backward ring depth");
  using L = BwdSmem<D, STAGES>;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
  constexpr int kDPanels = D / 64;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw_base);
  if ((base - raw_base) + static_cast<uint32_t>(L::kBytes) > static_cast<uint32_t>(L::kAlloc)) {
    // The aligned layout would run past the allocation (uniform over the CTA,
    // decided before any barrier or tensor-memory use).
    if (threadIdx.x == 0) record_error(p.status, kErrUnsupported, kBSiteSmemWindow);
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bar0 = base + L::kOffBar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* const s_tmem = reinterpret_cast<volatile uint32_t*>(gbase + L::kOffTmem);
  volatile int* const s_abort = reinterpret_cast<volatile int*>(gbase + L::kOffAbort);
  const uint64_t tmo = p.timeout_ns;

  if (warp == 13 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_do);
  }
  if (threadIdx.x == 0) {
    *s_abort = 0;
    ptx::mbar_init(bar(L::kBarKVFull), 1);
    ptx::mbar_init(bar(L::kBarKVEmpty), 1);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(L::kBarQFull + s), 1);
      ptx::mbar_init(bar(L::kBarQEmpty + s), 1);
    }
    ptx::mbar_init(bar(L::kBarSFull), 1);
    ptx::mbar_init(bar(L::kBarDPFull), 1);
    ptx::mbar_init(bar(L::kBarPFull), 256);
    ptx::mbar_init(bar(L::kBarDSFull), 256);
    ptx::mbar_init(bar(L::kBarDQFull), 1);
    ptx::mbar_init(bar(L::kBarDQEmpty), 128);
    ptx::mbar_init(bar(L::kBarAccFull), 1);
    ptx::mbar_init(bar(L::kBarAccEmpty), 128);
    ptx::mbar_init(bar(L::kBarTeardown), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 12) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(s_tmem)), 512);
    ptx::tmem_relinquish();
  }
  if constexpr (D < 128) {
    // The K panels beyond d are never loaded: zero them once, visible to the
    // tensor core (async proxy) before any MMA reads them.
    for (uint32_t i = threadIdx.x; i < (L::kKBytes - L::kKVBytes) / 16; i += blockDim.x)
      ptx::st_shared_v4(base + L::kOffK + L::kKVBytes + 16 * i, 0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // Handshake barriers are single: each one's next completion needs an action
  // of its own waiter first (S(g+1) is issued after P(g) is seen, dP(g+1)
  // after the drain has read dQ^T(g), which follows dS(g), and so on).
  if (warp >= 12) {
    ptx::setmaxnreg_dec<BwdRegSplit::kOther>();
    if (warp == 13 && lane == 0) {
      // ============================================================ TMA loads
      uint32_t g = 0, uc = 0;
      bool ok = true;
#pragma unroll 1
      FA_BWD_FOR_EACH_UNIT(u) {
        const BwdUnit w = bwd_decode<CAUSAL, VARLEN>(p, u);
        if (w.nsteps == 0) continue;
        if (uc > 0 && !ptx::mbar_wait(bar(L::kBarKVEmpty), (uc - 1) & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kBSiteLoadKV);
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(bar(L::kBarKVFull), 2 * L::kKVBytes);  // K and V, D features each
#pragma unroll
        for (int pn = 0; pn < kDPanels; ++pn) {
          if constexpr (VARLEN) {
            // Packed rows; a tile shifted back below row 0 is zero-filled there.
            ptx::tma_load_3d(base + L::kOffK + pn * L::kKVPanel, &tm_k, bar(L::kBarKVFull), pn * 64, w.hk,
                             w.kw.load_row);
            ptx::tma_load_3d(base + L::kOffV + pn * L::kKVPanel, &tm_v, bar(L::kBarKVFull), pn * 64, w.hk,
                             w.kw.load_row);
          } else {
            ptx::tma_load_4d(base + L::kOffK + pn * L::kKVPanel, &tm_k, bar(L::kBarKVFull), pn * 64, w.hk,
                             w.kb * kBwdBK, w.b);
            ptx::tma_load_4d(base + L::kOffV + pn * L::kKVPanel, &tm_v, bar(L::kBarKVFull), pn * 64, w.hk,
                             w.kb * kBwdBK, w.b);
          }
        }
        ++uc;
#pragma unroll 1
        for (int i = 0; i < w.nsteps && ok; ++i, ++g) {
          const uint32_t slot = g % STAGES;
          if (g >= STAGES && !ptx::mbar_wait(bar(L::kBarQEmpty + slot), ((g / STAGES) - 1) & 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kBSiteLoadQ);
            ok = false;
            break;
          }
          const int h = w.hk * p.group + i / w.nqb;
          const int qb = w.qb0 + i % w.nqb;
          const uint32_t fb = bar(L::kBarQFull + slot);
          ptx::mbar_arrive_expect_tx(fb, L::kSlotBytes + L::kLDBytes);
          const uint32_t sq = base + L::kOffQ + slot * L::kSlotBytes;
#pragma unroll
          for (int pn = 0; pn < kDPanels; ++pn) {
            if constexpr (VARLEN) {
              const int qrow = make_window<true>(w.q_start, w.q_start + w.len_q, w.q_start + qb * kBwdBQ, kBwdBQ).load_row;
              ptx::tma_load_3d(sq + pn * L::kQPanel, &tm_q, fb, pn * 64, h, qrow);
              ptx::tma_load_3d(sq + L::kQBytes + pn * L::kQPanel, &tm_do, fb, pn * 64, h, qrow);
            } else {
              ptx::tma_load_4d(sq + pn * L::kQPanel, &tm_q, fb, pn * 64, h, qb * kBwdBQ, w.b);
              ptx::tma_load_4d(sq + L::kQBytes + pn * L::kQPanel, &tm_do, fb, pn * 64, h, qb * kBwdBQ, w.b);
            }
          }
          // The block's scaled LSE and D rows (512 bytes each, 512-byte aligned:
          // nq_pad is a multiple of the block) for the softmax warps.
          const size_t ro = (static_cast<size_t>(w.b) * p.H + h) * p.nq_pad + static_cast<size_t>(qb) * kBwdBQ;
          const uint32_t sld = base + L::kOffLD + slot * L::kLDBytes;
          ptx::bulk_load(sld, p.lse2 + ro, kBwdBQ * 4, fb);
          ptx::bulk_load(sld + kBwdBQ * 4, p.delta + ro, kBwdBQ * 4, fb);
        }
      }
      // Drain: every issued copy must land before the CTA exits.
      if (uc > 0) ptx::mbar_wait_drain(bar(L::kBarKVFull), (uc - 1) & 1u, tmo);
      for (uint32_t s = 0; s < STAGES; ++s) {
        if (g > s) {
          const uint32_t rounds = (g - 1 - s) / STAGES + 1;
          ptx::mbar_wait_drain(bar(L::kBarQFull + s), (rounds - 1) & 1u, tmo);
        }
      }
    } else if (warp == 12 && lane == 0) {
      // ============================================================ MMA issue
      constexpr uint32_t id_s = ptx::idesc_bf16_f32(128, kBwdBQ, 0, 0);   // K Q^T, V dO^T
      constexpr uint32_t id_acc = ptx::idesc_bf16_f32(128, D, 0, 1);      // P^T dO, dS^T Q
      constexpr uint32_t id_dq = ptx::idesc_bf16_f32(128, kBwdBQ, 1, 1);  // K^T dS^T (K padded to 128 rows)
      uint32_t g = 0, uc = 0;
      bool ok = true;
      auto wait = [&](uint32_t b, uint32_t par, int site) -> bool {
        if (ptx::mbar_wait(b, par, s_abort, tmo)) return true;
        record_error(p.status, kErrTimeout, site);
        ok = false;
        return false;
      };
      // Shared-memory descriptors advance by byte offset / 16 in their low
      // word (the address field cannot carry below 256 KiB), so each MMA
      // costs the issuing thread an add instead of a descriptor build.
      const uint64_t kdesc = ptx::sw128_desc(base + L::kOffK, 16, 1024);
      const uint64_t vdesc = ptx::sw128_desc(base + L::kOffV, 16, 1024);
      const uint64_t kdesc_mn = ptx::sw128_desc(base + L::kOffK, L::kKVPanel, 1024);
      const uint64_t dsdesc_mn = ptx::sw128_desc(base + L::kOffDS, L::kDSPanel, 1024);
      const uint64_t dsdesc_k = ptx::sw128_desc(base + L::kOffDS, 16, 1024);
      auto issue_s = [&](uint32_t t) {
        const uint64_t qdesc = ptx::sw128_desc(base + L::kOffQ + (t % STAGES) * L::kSlotBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oa = (kk / 4) * L::kKVPanel + (kk % 4) * 32;
          const uint32_t ob = (kk / 4) * L::kQPanel + (kk % 4) * 32;
          ptx::mma_ss(tmem + kColS, kdesc + (oa >> 4), qdesc + (ob >> 4), id_s, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bar(L::kBarSFull));
      };
      auto issue_dp = [&](uint32_t t) {
        const uint64_t dodesc =
            ptx::sw128_desc(base + L::kOffQ + (t % STAGES) * L::kSlotBytes + L::kQBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oa = (kk / 4) * L::kKVPanel + (kk % 4) * 32;
          const uint32_t ob = (kk / 4) * L::kQPanel + (kk % 4) * 32;
          ptx::mma_ss(tmem + kColDP, vdesc + (oa >> 4), dodesc + (ob >> 4), id_s, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bar(L::kBarDPFull));
      };
#pragma unroll 1
      FA_BWD_FOR_EACH_UNIT(u) {
        const BwdUnit w = bwd_decode<CAUSAL, VARLEN>(p, u);
        if (w.nsteps == 0) continue;
        if (!wait(bar(L::kBarKVFull), uc & 1u, kBSiteMmaKV)) break;
        ptx::tc_fence_after();
        if (!wait(bar(L::kBarQFull + g % STAGES), (g / STAGES) & 1u, kBSiteMmaQ)) break;
        ptx::tc_fence_after();
        issue_s(g);
        // dP's columns last held dQ^T(g - 1) (the previous unit's last step).
        if (g > 0 && !wait(bar(L::kBarDQEmpty), (g - 1) & 1u, kBSiteMmaDQ)) break;
        ptx::tc_fence_after();
        issue_dp(g);
#pragma unroll 1
        for (int i = 0; i < w.nsteps && ok; ++i, ++g) {
          const uint32_t slot = g % STAGES;
          const uint32_t sq = base + L::kOffQ + slot * L::kSlotBytes;
          const uint32_t sdo = sq + L::kQBytes;
          // dV += P^T dO (P^T of warpgroup c at columns 64c .. 64c + 31).
          if (!wait(bar(L::kBarPFull), g & 1u, kBSiteMmaP)) break;
          if (i == 0 && uc > 0 && !wait(bar(L::kBarAccEmpty), (uc - 1) & 1u, kBSiteMmaAcc)) break;
          ptx::tc_fence_after();
          const uint64_t dodesc_mn = ptx::sw128_desc(sdo, L::kQPanel, 1024);
#pragma unroll
          for (int kk = 0; kk < kBwdBQ / 16; ++kk)
            ptx::mma_ts(tmem + kColDV, tmem + kColS + (kk >> 2) * 64 + (kk & 3) * 8, dodesc_mn + kk * 128, id_acc,
                        (i > 0 || kk > 0) ? 1u : 0u);
          // S(g + 1) over P(g) (read by the dV just issued, which runs first).
          if (i + 1 < w.nsteps) {
            if (!wait(bar(L::kBarQFull + (g + 1) % STAGES), ((g + 1) / STAGES) & 1u, kBSiteMmaQ)) break;
            ptx::tc_fence_after();
            issue_s(g + 1);
          }
          // dK += dS^T Q, then dQ^T = K^T dS^T over dP.  Both read dS^T from shared
          // memory: as dK's A operand it is K-major (key rows, queries along the
          // 128-byte rows), as dQ^T's B operand MN-major.
          if (!wait(bar(L::kBarDSFull), g & 1u, kBSiteMmaDS)) break;
          ptx::tc_fence_after();
          const uint64_t qdesc_mn = ptx::sw128_desc(sq, L::kQPanel, 1024);
#pragma unroll
          for (int kk = 0; kk < kBwdBQ / 16; ++kk) {
            const uint32_t oa = (kk / 4) * L::kDSPanel + (kk % 4) * 32;
            ptx::mma_ss(tmem + kColDK, dsdesc_k + (oa >> 4), qdesc_mn + kk * 128, id_acc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(bar(L::kBarQEmpty + slot));  // Q(g) and dO(g) read
#pragma unroll
          for (int kk = 0; kk < kBwdBK / 16; ++kk)
            ptx::mma_ss(tmem + kColDP, kdesc_mn + kk * 128, dsdesc_mn + kk * 128, id_dq, kk > 0 ? 1u : 0u);
          ptx::mma_commit(bar(L::kBarDQFull));
          // dP(g + 1) once the drain has read dQ^T(g) out of those columns.
          if (i + 1 < w.nsteps) {
            if (!wait(bar(L::kBarDQEmpty), g & 1u, kBSiteMmaDQ)) break;
            ptx::tc_fence_after();
            issue_dp(g + 1);
          }
        }
        if (!ok) break;
        ptx::mma_commit(bar(L::kBarAccFull));
        ptx::mma_commit(bar(L::kBarKVEmpty));
        ++uc;
      }
      ptx::mma_commit(bar(L::kBarTeardown));
      if (!ptx::mbar_wait_drain(bar(L::kBarTeardown), 0, tmo)) record_error(p.status, kErrTimeout, kBSiteTeardown);
    }
  } else if (warp < 8) {
    // (softmax warpgroups keep the launch allocation, BwdRegSplit::kSoftmax)
    // ================================================================ softmax
    const int c = warp >> 2;                    // query columns [64c, 64c + 64)
    const int r = ((warp & 3) << 5) + lane;     // key row of the block
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tSc = tmem + lane_off + kColS + c * 64;
    const uint32_t tDc = tmem + lane_off + kColDP + c * 64;  // dP^T columns of this warpgroup
    const float c2 = p.scale_log2;
    uint32_t g = 0;
    bool ok = true;
#pragma unroll 1
    FA_BWD_FOR_EACH_UNIT(u) {
      const BwdUnit w = bwd_decode<CAUSAL, VARLEN>(p, u);
      if (w.nsteps == 0) continue;
      const int kj = w.kw.load_row - w.k_start + r;        // this thread's key (sequence index)
      const bool key_ok = r >= w.kw.lo && r < w.kw.hi;  // a key of this block
#pragma unroll 1
      for (int i = 0; i < w.nsteps && ok; ++i, ++g) {
        const int h = w.hk * p.group + i / w.nqb;
        const int qb = w.qb0 + i % w.nqb;
        // First query (sequence index) of this warpgroup's columns of the tile as loaded.
        const int q0 = make_window<VARLEN>(w.q_start, w.q_start + w.len_q, w.q_start + qb * kBwdBQ, kBwdBQ).load_row -
                       w.q_start + c * 64;
        // Scaled LSE and D of this warpgroup's 64 queries, staged with Q(g)
        // (shared-memory broadcasts instead of dependent global loads).
        const uint32_t slot = g % STAGES;
        const float4* l2g = reinterpret_cast<const float4*>(gbase + L::kOffLD + slot * L::kLDBytes) + c * 16;
        const float4* dlg = l2g + kBwdBQ / 4;
        if (!ptx::mbar_wait_warp(bar(L::kBarSFull), g & 1u, s_abort, tmo) ||
            !ptx::mbar_wait_warp(bar(L::kBarQFull + slot), (g / STAGES) & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kBSiteSoftS);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // P^T = 2^(S^T c2 - L log2 e), 32 columns at a time; keys outside the block and
        // (causal) keys after a query's limit get 0; the bf16 pairs of half hh
        // go to columns 16 hh .. 16 hh + 15 (already read).  The packed pairs
        // stay in registers for dS: S(g + 1) overwrites these columns as soon
        // as dV(g) has read them.
        uint32_t pk[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t sr[32];
          ptx::tmem_ld32(tSc + hh * 32, sr);
          ptx::tmem_wait_ld();
          const int lim = CAUSAL ? kj - w.off - (q0 + hh * 32) : -1;  // column k masked when k < lim
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            const float4 l = l2g[hh * 8 + k4];
#pragma unroll
            for (int k = 4 * k4; k < 4 * k4 + 4; k += 2) {
              const float la = (k & 3) == 0 ? l.x : l.z, lb = (k & 3) == 0 ? l.y : l.w;
              float x0, x1;
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])),
                                         ptx::f2_pack(c2, c2), ptx::f2_pack(-la, -lb)),
                             x0, x1);
              float e0 = ptx::ex2(x0), e1 = ptx::ex2(x1);
              if (!key_ok || (CAUSAL && k < lim)) e0 = 0.f;
              if (!key_ok || (CAUSAL && k + 1 < lim)) e1 = 0.f;
              pk[16 * hh + k / 2] = ptx::pack_bf16x2(e0, e1);
            }
          }
          ptx::tmem_st16(tSc + hh * 16, &pk[16 * hh]);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarPFull));
        // dS^T = P^T o (dP^T - D), from the bf16 P^T pairs held above.
        if (!ptx::mbar_wait_warp(bar(L::kBarDPFull), g & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kBSiteSoftDP);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // The previous step's dQ^T MMA must have read the shared dS^T buffer.
        if (g > 0 && !ptx::mbar_wait_warp(bar(L::kBarDQFull), (g - 1) & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kBSiteSoftDQ);
          ok = false;
          break;
        }
        // Row r of panel c (64 queries) of the shared dS^T: 128 bytes, 128-byte swizzle.
        const uint32_t row_addr = base + L::kOffDS + c * L::kDSPanel + r * 128;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t dr[32], ds[16];
          ptx::tmem_ld32(tDc + hh * 32, dr);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            const float4 dl = dlg[hh * 8 + k4];
#pragma unroll
            for (int k = 4 * k4; k < 4 * k4 + 4; k += 2) {
              const float da = (k & 3) == 0 ? dl.x : dl.z, db = (k & 3) == 0 ? dl.y : dl.w;
              const uint32_t pw = pk[16 * hh + k / 2];
              const float p0 = __uint_as_float(pw << 16), p1 = __uint_as_float(pw & 0xffff0000u);
              ds[k / 2] = ptx::pack_bf16x2(p0 * (__uint_as_float(dr[k]) - da), p1 * (__uint_as_float(dr[k + 1]) - db));
            }
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = 4 * hh + q4;
            ptx::st_shared_v4(row_addr + ((chunk ^ (r & 7)) << 4), ds[4 * q4], ds[4 * q4 + 1], ds[4 * q4 + 2],
                              ds[4 * q4 + 3]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();  // the dP loads above precede dQ^T overwriting those columns
        ptx::mbar_arrive(bar(L::kBarDSFull));
      }
    }
  } else {
    ptx::setmaxnreg_inc<BwdRegSplit::kDrain>();
    // ======================================== dQ drain and the dK / dV epilogue
    const int wq = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(wq << 5) << 16;
    uint32_t g = 0, uc = 0;
    bool ok = true;
#pragma unroll 1
    FA_BWD_FOR_EACH_UNIT(u) {
      const BwdUnit w = bwd_decode<CAUSAL, VARLEN>(p, u);
      const int kr = (wq << 5) + lane;  // this thread's key row of the tile
      const bool key_ok = kr >= w.kw.lo && kr < w.kw.hi;
      const size_t prow = VARLEN ? static_cast<size_t>(w.kw.load_row + kr)
                                 : static_cast<size_t>(w.b) * p.Nk + w.kw.load_row + kr;
      const size_t krow = (prow * p.Hk + w.hk) * D;
      if (w.nsteps == 0) {
        // No query sees these keys: dK = dV = 0.
        if (key_ok) {
          for (int e = 0; e < D; e += 8) {
            ptx::st_global_v4(p.dk + krow + e, 0u, 0u, 0u, 0u);
            ptx::st_global_v4(p.dv + krow + e, 0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
#pragma unroll 1
      for (int i = 0; i < w.nsteps && ok; ++i, ++g) {
        const int h = w.hk * p.group + i / w.nqb;
        const int qb = w.qb0 + i % w.nqb;
        if (!ptx::mbar_wait_warp(bar(L::kBarDQFull), g & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kBSiteDrainDQ);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if ((wq << 5) < D) {
          uint32_t v[128];
#pragma unroll
          for (int q32 = 0; q32 < 4; ++q32) ptx::tmem_ld32(tmem + lane_off + kColDP + q32 * 32, v + 32 * q32);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::kBarDQEmpty));
          // Query q of the block: the warp's 32 features are one 128-byte line.
          float* const dst = p.dq_acc +
                             (static_cast<size_t>(w.b * p.H + h) * p.nq_pad + static_cast<size_t>(qb) * kBwdBQ) * D +
                             (wq << 5) + lane;
#pragma unroll
          for (int q = 0; q < kBwdBQ; ++q) ptx::red_add(dst + static_cast<size_t>(q) * D, __uint_as_float(v[q]));
        } else {
          // Lanes (features) at or beyond d hold the zero rows of the padded product.
          ptx::mbar_arrive(bar(L::kBarDQEmpty));
        }
      }
      if (!ok) break;
      // Unit done: dK (times the scale) and dV to bf16, one key row per thread.
      if (!ptx::mbar_wait_warp(bar(L::kBarAccFull), uc & 1u, s_abort, tmo)) {
        record_error(p.status, kErrTimeout, kBSiteDrainAcc);
        ok = false;
        break;
      }
      ptx::tc_fence_after();
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? kColDV : kColDK;
        const float mul = which == 0 ? 1.f : p.scale;
        __nv_bfloat16* const dst = which == 0 ? p.dv : p.dk;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t a[32];
          ptx::tmem_ld32(tmem + lane_off + col + c4 * 32, a);
          ptx::tmem_wait_ld();
          if (key_ok) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t wv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                wv[e] = ptx::pack_bf16x2(__uint_as_float(a[8 * q4 + 2 * e]) * mul,
                                         __uint_as_float(a[8 * q4 + 2 * e + 1]) * mul);
              ptx::st_global_v4(dst + krow + c4 * 32 + q4 * 8, wv[0], wv[1], wv[2], wv[3]);
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::kBarAccEmpty));
      ++uc;
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
