// fa_fwd_kernel.cuh -- FlashAttention-2 forward for sm_103a (GB300).
//
// What it computes ("GPU 内核与 FlashAttention" §10-§14): for every batch b,
// head h and query row i,
//     O[b,i,h,:] = softmax_j(scale * q_i . k_j) V[b,:,h,:]
//     LSE[b,h,i] = log sum_j exp(scale * q_i . k_j)          (natural log)
// tile by tile with the online-softmax recurrence (§11.3): running row max m,
// running sum l, rescale of the unnormalised output, one division by l at the
// end and only the log-sum-exp kept per row (§14.1).  The N x N score matrix
// never reaches global memory.
//
// Work split (§14.2, loop order with the query block outermost): one CTA owns
// two 128-row query tiles of one (b, h) and streams all key/value tiles of
// that head.  Roles inside the CTA (§15.2-§15.4, re-expressed for tcgen05):
//   warps 0-3   softmax warpgroup for query tile 0 (one thread per row)
//   warps 4-7   softmax warpgroup for query tile 1
//   warps 8-11  correction warpgroup: rescales O in TMEM, then the epilogue
//   warp 12     MMA issue (one thread) + TMEM allocation
//   warp 13     TMA loads (one thread)
//   warps 14-15 idle (they only complete the register hand-off warpgroup)
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   S_t  = columns [t*BC, t*BC + BC)         fp32 scores of tile t
//   P_t  = columns [t*BC + BC/2, t*BC + BC)  bf16 probabilities, packed in pairs
//   O_t  = columns [2*BC + t*D, 2*BC + t*D + D)  fp32 output accumulator
// Two query tiles alternate on the tensor core: while one softmax warpgroup
// exponentiates its S, the tensor core runs the other tile's GEMMs
// ("GPU 内核与 FlashAttention" §15.3 ping-pong).  Within a tile, the MMA for
// P(j-1) V(j-1) is issued before S(j) = Q K(j)^T; tcgen05.mma operations from
// one thread execute in issue order, so S(j) may overwrite the columns that
// held P(j-1).
//
// Scale folding ("Flash Attention 2 Chapter6", Kernel 6): p = 2^(s * c - m * c)
// with c = scale * log2(e), one FFMA feeding the ex2 unit per score.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace fa {

constexpr int kBR = 128;       // query rows per tile (tcgen05 M)
constexpr int kQT = 2;         // query tiles per CTA
constexpr int kThreads = 512;  // 16 warps
constexpr int kPanel = 64;     // bf16 columns per 128-byte swizzle row

// Register split after setmaxnreg (must sum to 65536 over 512 threads).
constexpr int kRegSoftmax = 176;
constexpr int kRegCorrection = 96;
constexpr int kRegOther = 64;
static_assert(2 * 128 * kRegSoftmax + 128 * kRegCorrection + 128 * kRegOther <= 65536,
              "register split exceeds the launch allocation");

// Where a wait gave up (recorded with FA_ERR_TIMEOUT).
enum WaitSite : int {
  kSiteLoadKV = 1,
  kSiteMmaQ = 2,
  kSiteMmaK = 3,
  kSiteMmaV = 4,
  kSiteMmaP = 5,
  kSiteMmaO = 6,
  kSiteSoftS = 7,
  kSiteCorrAlpha = 8,
  kSiteCorrFinal = 9,
  kSiteTeardown = 10,
};

struct FwdParams {
  int B, Nq, Nk, H;            // variable-length form: Nq / Nk are the maximum lengths
  int num_mblocks;             // ceil(Nq / (kBR * kQT))
  const int* cu_q;             // variable-length form: int32 [B + 1]
  const int* cu_k;
  float* lse;                  // [B, H, Nq] fp32
  __nv_bfloat16* o;            // output base (row stores of partial tiles)
  float scale;                 // softmax scale (natural units)
  float scale_log2;            // scale * log2(e)
  float rescale_threshold;     // log2 units; the O rescale is skipped while the max grows less
  unsigned long long timeout_ns;
  int* status;                 // [4]: code, block, warp, site
};

// Error codes shared with the C-ABI header.
constexpr int kErrTimeout = -5;
constexpr int kErrBadSeqlens = -7;

__device__ __forceinline__ void record_error(int* status, int code, int site) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    status[2] = threadIdx.x >> 5;
    status[3] = site;
  }
}

template <int D, int BC, int STAGES>
struct SmemLayout {
  static constexpr int kQTileBytes = kBR * D * 2;
  static constexpr int kQPanelBytes = kBR * 128;
  static constexpr int kKVTileBytes = BC * D * 2;
  static constexpr int kKVPanelBytes = BC * 128;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQT * kQTileBytes;
  static constexpr int kOffBar = kOffKV + STAGES * kKVTileBytes;
  // barriers (8 bytes each)
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKVFull = 1;
  static constexpr int kBarKVEmpty = kBarKVFull + STAGES;
  static constexpr int kBarSFull = kBarKVEmpty + STAGES;
  static constexpr int kBarPFull = kBarSFull + kQT;
  static constexpr int kBarAlpha = kBarPFull + kQT;
  static constexpr int kBarOReady = kBarAlpha + kQT;
  static constexpr int kBarOFinal = kBarOReady + kQT;
  static constexpr int kBarTeardown = kBarOFinal + kQT;
  static constexpr int kNumBars = kBarTeardown + 1;
  static constexpr int kOffAlpha = kOffBar + ((kNumBars * 8 + 15) / 16) * 16;
  static constexpr int kOffInvL = kOffAlpha + kQT * kBR * 4;
  static constexpr int kOffTmem = kOffInvL + kQT * kBR * 4;
  static constexpr int kOffAbort = kOffTmem + 16;
  static constexpr int kBytes = kOffAbort + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kOffKV % 1024 == 0 && kKVTileBytes % 1024 == 0, "swizzled tiles need 1 KiB alignment");
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
};

// Geometry of one 128-row tile along the sequence axis.  `load_row` is the
// first row the TMA box reads; rows [lo, hi) of the box are valid.  In the
// variable-length form a tile that would run past the end of its sequence is
// shifted back so that it ends exactly at the end, never touching memory past
// the last row of the packed tensor (rows before the sequence are masked).
struct RowWindow {
  int load_row;
  int lo, hi;
};

template <bool VARLEN>
__device__ __forceinline__ RowWindow make_window(int seq_start, int seq_end, int row0, int rows) {
  RowWindow w;
  if (!VARLEN || row0 + rows <= seq_end) {
    w.load_row = row0;
    w.lo = 0;
    w.hi = min(rows, seq_end - row0);
  } else {
    w.load_row = seq_end - rows;
    w.lo = row0 - w.load_row;
    w.hi = rows;
  }
  return w;
}

template <int D, int BC, int STAGES, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
  using L = SmemLayout<D, BC, STAGES>;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BC == 64 || BC == 128, "key tile");
  static_assert(2 * BC + 2 * D <= 512, "TMEM columns");
  constexpr int kTmemCols = 512;
  constexpr int kDPanels = D / kPanel;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int mb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;

  // ------------------------------------------------ work unit and sequence
  int q_start = 0, q_end = p.Nq, k_start = 0, k_end = p.Nk;
  if constexpr (VARLEN) {
    q_start = p.cu_q[b];
    q_end = p.cu_q[b + 1];
    k_start = p.cu_k[b];
    k_end = p.cu_k[b + 1];
    const int len_q = q_end - q_start, len_k = k_end - k_start;
    if (len_q < 0 || len_k < 0 || len_q > p.Nq || len_k > p.Nk || q_start < 0 || k_start < 0) {
      if (threadIdx.x == 0 && mb == 0 && h == 0) record_error(p.status, kErrBadSeqlens, 0);
      return;
    }
  }
  const int q_row0 = q_start + mb * (kBR * kQT);
  if (q_row0 >= q_end) return;  // past the end of this sequence
  const int nkv = (k_end - k_start + BC - 1) / BC;
  const int lse_base = (b * p.H + h) * p.Nq;

  if (nkv == 0) {
    // No keys: o = 0 and LSE = -inf (log of an empty sum).
    const int rows = min(kBR * kQT, q_end - q_row0);
    const size_t rs = static_cast<size_t>(p.H) * D;
    for (int e = threadIdx.x; e < rows * D; e += kThreads) {
      const int r = e / D, c = e % D;
      p.o[static_cast<size_t>(q_row0 + r) * rs + static_cast<size_t>(h) * D + c] = __float2bfloat16(0.f);
    }
    for (int r = threadIdx.x; r < rows; r += kThreads)
      p.lse[lse_base + (q_row0 - q_start) + r] = -INFINITY;
    return;
  }

  bool tile_active[kQT];
  RowWindow qwin[kQT];
#pragma unroll
  for (int t = 0; t < kQT; ++t) {
    const int r0 = q_row0 + t * kBR;
    tile_active[t] = r0 < q_end;
    qwin[t] = make_window<VARLEN>(q_start, q_end, r0, kBR);
  }

  const uint32_t bar0 = base + L::kOffBar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  float* const s_alpha = reinterpret_cast<float*>(gbase + L::kOffAlpha);
  float* const s_invl = reinterpret_cast<float*>(gbase + L::kOffInvL);
  volatile uint32_t* const s_tmem = reinterpret_cast<volatile uint32_t*>(gbase + L::kOffTmem);
  volatile int* const s_abort = reinterpret_cast<volatile int*>(gbase + L::kOffAbort);
  const uint64_t tmo = p.timeout_ns;

  // ------------------------------------------------------------------ setup
  if (warp == 13 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_o);
  }
  if (threadIdx.x == 0) {
    *s_abort = 0;
    ptx::mbar_init(bar(L::kBarQFull), 1);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(L::kBarKVFull + s), 1);
      ptx::mbar_init(bar(L::kBarKVEmpty + s), 1);
    }
    for (int t = 0; t < kQT; ++t) {
      ptx::mbar_init(bar(L::kBarSFull + t), 1);
      ptx::mbar_init(bar(L::kBarPFull + t), kBR);
      ptx::mbar_init(bar(L::kBarAlpha + t), kBR);
      ptx::mbar_init(bar(L::kBarOReady + t), kBR);
      ptx::mbar_init(bar(L::kBarOFinal + t), 1);
    }
    ptx::mbar_init(bar(L::kBarTeardown), 1);
    ptx::fence_mbar_init();
  }
  if (warp == 12) {
    ptx::tmem_alloc(base + L::kOffTmem, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp >= 12) {
    ptx::setmaxnreg_dec<kRegOther>();
    if (warp == 13 && lane == 0) {
      // =========================================================== TMA loads
      uint32_t q_bytes = 0;
#pragma unroll
      for (int t = 0; t < kQT; ++t) q_bytes += tile_active[t] ? L::kQTileBytes : 0;
      ptx::mbar_arrive_expect_tx(bar(L::kBarQFull), q_bytes);
#pragma unroll
      for (int t = 0; t < kQT; ++t) {
        if (!tile_active[t]) continue;
#pragma unroll
        for (int pnl = 0; pnl < kDPanels; ++pnl) {
          const uint32_t dst = base + L::kOffQ + t * L::kQTileBytes + pnl * L::kQPanelBytes;
          if constexpr (VARLEN)
            ptx::tma_load_3d(dst, &tm_q, bar(L::kBarQFull), pnl * kPanel, h, qwin[t].load_row);
          else
            ptx::tma_load_4d(dst, &tm_q, bar(L::kBarQFull), pnl * kPanel, h, qwin[t].load_row, b);
        }
      }
      int issued = 0;  // ring positions handed to the TMA unit so far
      bool ok = true;
#pragma unroll 1
      for (int j = 0; j < nkv && ok; ++j) {
        const RowWindow kw = make_window<VARLEN>(k_start, k_end, k_start + j * BC, BC);
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const int tpos = 2 * j + which;
          const int slot = tpos % STAGES;
          const uint32_t round = static_cast<uint32_t>(tpos / STAGES);
          if (!ptx::mbar_wait(bar(L::kBarKVEmpty + slot), (round & 1u) ^ 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kSiteLoadKV);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(bar(L::kBarKVFull + slot), L::kKVTileBytes);
          issued = tpos + 1;
          const void* tm = which == 0 ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
#pragma unroll
          for (int pnl = 0; pnl < kDPanels; ++pnl) {
            const uint32_t dst = base + L::kOffKV + slot * L::kKVTileBytes + pnl * L::kKVPanelBytes;
            if constexpr (VARLEN)
              ptx::tma_load_3d(dst, tm, bar(L::kBarKVFull + slot), pnl * kPanel, h, kw.load_row);
            else
              ptx::tma_load_4d(dst, tm, bar(L::kBarKVFull + slot), pnl * kPanel, h, kw.load_row, b);
          }
        }
      }
      // Teardown: never leave a TMA write to shared memory in flight.  Slot s
      // last received ring position s + STAGES * (rounds - 1).
      ptx::mbar_wait_drain(bar(L::kBarQFull), 0, tmo);
      for (int s = 0; s < STAGES; ++s) {
        if (issued > s) {
          const int rounds = (issued - 1 - s) / STAGES + 1;
          ptx::mbar_wait_drain(bar(L::kBarKVFull + s), static_cast<uint32_t>(rounds - 1) & 1u, tmo);
        }
      }
    } else if (warp == 12 && lane == 0) {
      // ========================================================== MMA issue
      constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(kBR, BC, 0, 0);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(kBR, D, 0, 1);
      bool ok = ptx::mbar_wait(bar(L::kBarQFull), 0, s_abort, tmo);
      if (!ok) record_error(p.status, kErrTimeout, kSiteMmaQ);
      ptx::tc_fence_after();
#pragma unroll 1
      for (int j = 0; j <= nkv && ok; ++j) {
        const int posK = 2 * j, posV = 2 * (j - 1) + 1;
        const int slotK = posK % STAGES, slotV = (posV + STAGES) % STAGES;
        if (j < nkv) {
          if (!ptx::mbar_wait(bar(L::kBarKVFull + slotK), static_cast<uint32_t>(posK / STAGES) & 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kSiteMmaK);
            ok = false;
            break;
          }
        }
        if (j >= 1) {
          if (!ptx::mbar_wait(bar(L::kBarKVFull + slotV), static_cast<uint32_t>(posV / STAGES) & 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kSiteMmaV);
            ok = false;
            break;
          }
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int t = 0; t < kQT; ++t) {
          if (!tile_active[t]) continue;
          const uint32_t tS = tmem + static_cast<uint32_t>(t * BC);
          const uint32_t tP = tS + BC / 2;
          const uint32_t tO = tmem + static_cast<uint32_t>(2 * BC + t * D);
          if (j >= 1) {
            // O_t += P_t(j-1) V(j-1)
            if (!ptx::mbar_wait(bar(L::kBarPFull + t), static_cast<uint32_t>(j - 1) & 1u, s_abort, tmo)) {
              record_error(p.status, kErrTimeout, kSiteMmaP);
              ok = false;
              break;
            }
            if (j >= 2 && !ptx::mbar_wait(bar(L::kBarOReady + t), static_cast<uint32_t>(j - 2) & 1u, s_abort, tmo)) {
              record_error(p.status, kErrTimeout, kSiteMmaO);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t v_base = base + L::kOffKV + slotV * L::kKVTileBytes;
#pragma unroll
            for (int kk = 0; kk < BC / 16; ++kk) {
              // V is MN-major: 16 keys = two 8-row swizzle atoms = 2048 bytes;
              // the two 64-column halves of d sit one panel (BC * 128 bytes) apart.
              const uint64_t bdesc = ptx::sw128_desc(v_base + kk * 2048, L::kKVPanelBytes, 1024);
              ptx::mma_ts(tO, tP + kk * 8, bdesc, idesc_pv, (j - 1 > 0 || kk > 0) ? 1u : 0u);
            }
            if (j == nkv) ptx::mma_commit(bar(L::kBarOFinal + t));
          }
          if (j < nkv) {
            // S_t = Q_t K(j)^T
            const uint32_t q_base = base + L::kOffQ + t * L::kQTileBytes;
            const uint32_t k_base = base + L::kOffKV + slotK * L::kKVTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              // K-major, 128-byte swizzle: 16 columns = 32 bytes inside a panel.
              const uint32_t off_q = (kk / 4) * L::kQPanelBytes + (kk % 4) * 32;
              const uint32_t off_k = (kk / 4) * L::kKVPanelBytes + (kk % 4) * 32;
              const uint64_t adesc = ptx::sw128_desc(q_base + off_q, 16, 1024);
              const uint64_t bdesc = ptx::sw128_desc(k_base + off_k, 16, 1024);
              ptx::mma_ss(tS, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(bar(L::kBarSFull + t));
          }
        }
        if (!ok) break;
        if (j < nkv) ptx::mma_commit(bar(L::kBarKVEmpty + slotK));
        if (j >= 1) ptx::mma_commit(bar(L::kBarKVEmpty + slotV));
      }
      // Teardown: all MMAs must be complete before TMEM is released.
      ptx::mma_commit(bar(L::kBarTeardown));
      if (!ptx::mbar_wait_drain(bar(L::kBarTeardown), 0, tmo)) record_error(p.status, kErrTimeout, kSiteTeardown);
    }
  } else if (warp < 8) {
    ptx::setmaxnreg_inc<kRegSoftmax>();
    // ================================================================ softmax
    const int t = warp >> 2;
    const int row = ((warp & 3) << 5) + lane;
    const RowWindow qw = t == 0 ? qwin[0] : qwin[1];  // no dynamic indexing of local arrays
    const bool active = t == 0 ? tile_active[0] : tile_active[1];
    if (active) {
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
      const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(t * BC);
      const uint32_t tP = tS + BC / 2;
      const float c2 = p.scale_log2;
      float m_ref = -INFINITY;
      float l = 0.f;
      bool ok = true;
#pragma unroll 1
      for (int j = 0; j < nkv; ++j) {
        if (!ptx::mbar_wait_warp(bar(L::kBarSFull + t), static_cast<uint32_t>(j) & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kSiteSoftS);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        uint32_t sr[BC];
#pragma unroll
        for (int c = 0; c < BC / 32; ++c)
          ptx::tmem_ld32(tS + c * 32, &sr[c * 32]);
        ptx::tmem_wait_ld();
        float s[BC];
#pragma unroll
        for (int c = 0; c < BC; ++c) s[c] = __uint_as_float(sr[c]);
        const RowWindow kw = make_window<VARLEN>(k_start, k_end, k_start + j * BC, BC);
        if (kw.lo != 0 || kw.hi != BC) {
#pragma unroll
          for (int c = 0; c < BC; ++c)
            if (c < kw.lo || c >= kw.hi) s[c] = -INFINITY;
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < BC; c += 4) {
          mx0 = fmaxf(mx0, s[c]);
          mx1 = fmaxf(mx1, s[c + 1]);
          mx2 = fmaxf(mx2, s[c + 2]);
          mx3 = fmaxf(mx3, s[c + 3]);
        }
        const float bm = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        // Move the reference max only when the block max exceeds it by more
        // than the threshold (log2 units): the merge identity of §11.2 holds
        // for any common reference value, so results stay exact.
        float m_new = m_ref;
        if (bm > m_ref && (m_ref == -INFINITY || (bm - m_ref) * c2 > p.rescale_threshold)) m_new = bm;
        const float alpha = (m_new == m_ref) ? 1.f : ptx::ex2((m_ref - m_new) * c2);
        if (j >= 1) {
          s_alpha[t * kBR + row] = alpha;
          ptx::mbar_arrive(bar(L::kBarAlpha + t));
        }
        m_ref = m_new;
        const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref * c2;
        float sum0 = 0.f, sum1 = 0.f;
        uint32_t pk[BC / 2];
#pragma unroll
        for (int c = 0; c < BC; c += 2) {
          const float e0 = ptx::ex2(fmaf(s[c], c2, neg));
          const float e1 = ptx::ex2(fmaf(s[c + 1], c2, neg));
          sum0 += e0;
          sum1 += e1;
          pk[c / 2] = ptx::pack_bf16x2(e0, e1);
        }
        l = l * alpha + (sum0 + sum1);
#pragma unroll
        for (int c = 0; c < BC / 2; c += 16) ptx::tmem_st16(tP + c, &pk[c]);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarPFull + t));
      }
      if (ok) {
        // Final message for the epilogue: 1 / l, and the row's log-sum-exp.
        const bool has = l > 0.f;
        s_invl[t * kBR + row] = has ? 1.f / l : 0.f;
        const int r_in_seq = qw.load_row - q_start + row;
        if (row >= qw.lo && row < qw.hi) {
          const float lse = has ? (m_ref * p.scale + log2f(l) * 0.69314718055994530942f) : -INFINITY;
          p.lse[lse_base + r_in_seq] = lse;
        }
        ptx::mbar_arrive(bar(L::kBarAlpha + t));
      }
    }
  } else {
    ptx::setmaxnreg_dec<kRegCorrection>();
    // ============================================================= correction
    const int wq = warp & 3;
    const int row = (wq << 5) + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq << 5) << 16;
    bool ok = true;
#pragma unroll 1
    for (int j = 1; j < nkv && ok; ++j) {
#pragma unroll
      for (int t = 0; t < kQT; ++t) {
        if (!tile_active[t]) continue;
        if (!ptx::mbar_wait_warp(bar(L::kBarAlpha + t), static_cast<uint32_t>(j - 1) & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kSiteCorrAlpha);
          ok = false;
          break;
        }
        const float a = s_alpha[t * kBR + row];
        if (__any_sync(0xffffffffu, a != 1.f)) {
          ptx::tc_fence_after();
          const uint32_t tO = tmem + lane_off + static_cast<uint32_t>(2 * BC + t * D);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            ptx::tmem_ld32(tO + c * 32, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * a);
            ptx::tmem_st32(tO + c * 32, r);
          }
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarOReady + t));
      }
    }
    // ============================================================== epilogue
    bool stored = false;
#pragma unroll
    for (int t = 0; t < kQT; ++t) {
      if (!ok || !tile_active[t]) continue;
      if (!ptx::mbar_wait_warp(bar(L::kBarAlpha + t), static_cast<uint32_t>(nkv - 1) & 1u, s_abort, tmo) ||
          !ptx::mbar_wait_warp(bar(L::kBarOFinal + t), 0, s_abort, tmo)) {
        record_error(p.status, kErrTimeout, kSiteCorrFinal);
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const float inv_l = s_invl[t * kBR + row];
      const uint32_t tO = tmem + lane_off + static_cast<uint32_t>(2 * BC + t * D);
      const RowWindow& qw = qwin[t];
      const bool warp_full = (wq << 5) >= qw.lo;  // every row of this warp is valid
      const bool use_tma = !VARLEN || warp_full;
      const bool row_ok = row >= qw.lo && row < qw.hi;
      // The query tile's shared memory is free once its last S MMA is done,
      // which the O-final commit guarantees; reuse it as the staging buffer.
      const uint32_t stage = base + L::kOffQ + t * L::kQTileBytes;
      // Row pointer for the direct-store path (only formed for valid rows).
      __nv_bfloat16* const grow =
          row_ok ? p.o + (static_cast<size_t>(qw.load_row + row) * p.H + h) * D : p.o;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(tO + c * 32, r);
        ptx::tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = ptx::pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
        if (use_tma) {
          const int pnl = (c * 32) / kPanel;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int chunk = ((c * 32) % kPanel) / 8 + q4;
            const uint32_t addr = stage + pnl * L::kQPanelBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
            ptx::st_shared_v4(addr, w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
          }
        } else if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            ptx::st_global_v4(grow + c * 32 + q4 * 8, w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
        }
      }
      if (use_tma) {
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int pnl = 0; pnl < kDPanels; ++pnl) {
            const uint32_t src = stage + pnl * L::kQPanelBytes + (wq << 5) * 128;
            if constexpr (VARLEN)
              ptx::tma_store_3d(&tm_o, src, pnl * kPanel, h, qw.load_row + (wq << 5));
            else
              ptx::tma_store_4d(&tm_o, src, pnl * kPanel, h, qw.load_row + (wq << 5), b);
          }
          ptx::bulk_commit_group();
          stored = true;
        }
      }
    }
    if (lane == 0 && stored) ptx::bulk_wait_group_read_0();
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();  // single-lane roles rejoin their warp before the CTA barrier
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
