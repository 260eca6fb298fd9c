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
// Work split (§14.2, loop order with the query block outermost): a work unit
// is two 128-row query tiles of one (b, h) against all key/value tiles of that
// head (B_r = 256; with qtiles = 1 a unit is one tile, B_r = 128, and the
// second softmax warpgroup idles).  Dense problems run a persistent grid: each
// CTA walks the items blockIdx.x, blockIdx.x + gridDim.x, ...  Packed
// variable-length batches launch one CTA per item, and a running CTA takes over
// the items of CTAs not yet started (cluster launch control); its load thread
// hands the item sequence to the other roles through a shared-memory ring.
// Units are numbered with the query block fastest, so the CTAs that run at the
// same time share the K/V of a few heads in L2.
// Roles inside the CTA (§15.2-§15.4, re-expressed for tcgen05):
//   warps 0-3   softmax warpgroup for query tile 0 (one thread per row)
//   warps 4-7   softmax warpgroup for query tile 1
//   warps 8-11  correction/epilogue warpgroup: final correction of O by 1/l,
//               bf16 conversion, TMA store -- overlapping the next unit
//   warp 12     MMA issue (one thread) + TMEM allocation
//   warp 13     TMA loads (one thread)
//   warps 14-15 idle (they only complete the register hand-off warpgroup)
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   S_t  = columns [t*BC, t*BC + BC)         fp32 scores of tile t
//   P_t  = columns [t*BC + BC/2, t*BC + BC)  bf16 probabilities, packed in pairs
//   O_t  = columns [2*BC + t*D, 2*BC + t*D + D)  fp32 output accumulator
// Key/value ring: slot g holds K(j) and V(j-1), the two tiles step j of a unit
// consumes (S(j) = Q K(j)^T and O += P(j-1) V(j-1)); one barrier fills it and
// one MMA commit releases it.  The ring runs on across units.
// Two query tiles alternate on the tensor core: while one softmax warpgroup
// exponentiates its S, the tensor core runs the other tile's GEMMs
// ("GPU 内核与 FlashAttention" §15.3 ping-pong).  Within a tile, the MMA for
// P(j-1) V(j-1) is issued before S(j) = Q K(j)^T; tcgen05.mma operations from
// one thread execute in issue order, so S(j) may overwrite the columns that
// held P(j-1).
//
// Rescale of O when a row maximum grows ("Flash Attention 2 Chapter6",
// scale_l_O): the reference maximum only moves when a block maximum exceeds it
// by more than a threshold, so rescales are rare after the first blocks; the
// softmax warp that owns the rows applies it in TMEM itself (its TMEM lane
// quarter holds exactly its rows of O), after S(j) completed, which implies
// that P(j-1) V(j-1) has completed.  The block maximum itself is computed only
// when needed: the exponentials are first taken against the current reference,
// and a block sum of at most 2^threshold proves that no exponent exceeded the
// threshold, i.e. that the maximum rule would leave the reference in place.
//
// Causal masking ("GPU 内核与 FlashAttention" §14.4): key tiles entirely above
// the diagonal are skipped (each query tile runs only the key tiles its rows
// can see), only tiles that cross the diagonal are masked element-wise, and the
// heaviest query blocks are scheduled first.  With different query and key
// lengths the mask is aligned bottom-right: query i sees keys j <= i + Nk - Nq.
// Grouped key/value heads (§14.2, MQA/GQA): query head h reads key/value head
// h / G; K and V are never replicated in memory.
//
// Split keys (SPLIT): for short query sets a unit covers only a range of key
// tiles; its normalised fp32 output and log-sum-exp go to a workspace, and a
// second kernel merges the splits with the two-block merge of §11.2
// (LSE = log sum_s e^LSE_s, O = sum_s e^(LSE_s - LSE) O_s), which is exact.
//
// Scale folding ("Flash Attention 2 Chapter6", Kernel 6): p = 2^(s * c - m * c)
// with c = scale * log2(e), one FFMA feeding the ex2 unit per score.
//
// FP8 ("GPU 内核与 FlashAttention" §15.5, block quantization): Q, K and V arrive
// as e4m3 codes with one fp32 scale per 128 query rows, per 128 keys and per
// key/value head; V is stored transposed ([B, Hk, d, keys]) so that both
// operands of every product are K-major.  S = Q K^T runs as kind::f8f6f4 MMAs
// (32 elements per instruction), the scales fold into the exp2 coefficient of
// each key tile (the row maximum is then kept in scaled log2 units), P is
// rounded to e4m3 (four per TMEM column) for O += P V, and the V scale joins
// the final 1/l.  Variable-length FP8 batches keep every tile at a multiple of
// 128 rows from its sequence's start (no shifted last tile), so that a tile is
// exactly one quantisation block; rows read past a sequence's end belong to
// the next sequence or to the TMA zero fill and are masked (keys) or never
// stored (queries).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace fa {

constexpr int kBR = 128;       // query rows per tile (tcgen05 M)
constexpr int kQT = 2;         // query tiles per work unit
constexpr int kThreads = 512;  // 16 warps
constexpr int kPanel = 64;     // bf16 columns per 128-byte swizzle row

// Register split after setmaxnreg (must sum to 65536 over 512 threads).  The
// MMA-issue/load warps get more than the correction warps: with fewer they
// spill in the issue loop, whose instruction slots the softmax warps of the
// same scheduler compete for.
template <bool VARLEN>
struct RegSplit {
  static constexpr int kSoftmax = 176;
  static constexpr int kCorrection = 64;
  static constexpr int kOther = 96;
  static_assert(2 * 128 * kSoftmax + 128 * kCorrection + 128 * kOther <= 65536,
                "register split exceeds the launch allocation");
};

// Where a wait gave up (recorded with FA_ERR_TIMEOUT).
enum WaitSite : int {
  kSiteLoadKV = 1,
  kSiteMmaQ = 2,
  kSiteMmaK = 3,
  kSiteLoadQ = 4,
  kSiteMmaP = 5,
  kSiteMmaOEmpty = 6,
  kSiteSoftS = 7,
  kSiteCorrFinal = 9,
  kSiteTeardown = 10,
  kSiteItem = 11,
  kSiteSoftFinal = 12,
};

// Work items reach the roles through a ring of kItemSlots entries in shared
// memory: the load thread writes item n (the x index of a CTA whose work this
// CTA took over, or -1 at the end) and every consumer -- the MMA thread, the
// eight softmax warps and the four epilogue warps -- releases the slot.
constexpr int kItemSlots = 4;
constexpr int kItemConsumers = 1 + 8 + 4;

// Phase clocks: per-CTA cycle counts of where each role spends its time,
// compiled in only when FA_PHASE_CLOCKS is 1 (a separate build of the
// library; the default build has none of this code).  Each role keeps a few
// accumulators in registers: `lap(i)` adds the cycles since the previous lap
// to slot i, so a role's time is partitioned into its waits and its work; the
// accumulators are stored once, at the end, to
//   phase[blockIdx.x * kPhaseWords + role base + slot]  (unsigned 64-bit).
#ifndef FA_PHASE_CLOCKS
#define FA_PHASE_CLOCKS 0
#endif

constexpr int kPhaseWords = 48;   // per CTA
constexpr int kPhaseRole = 8;     // slots per role
enum PhaseBase : int {
  kPhMma = 0,        // wait Q-full, wait K/V-full, wait P-full, wait O-empty, issue, steps, units
  kPhLoad = 8,       // wait Q-empty, wait K/V-empty, issue, ring slots
  kPhSoft0 = 16,     // tile 0 (warp 0, lane 0): wait S-full, store P and publish, steps, maximum
                     // recomputed, final, load S, exponentials
  kPhSoft1 = 24,     // tile 1 (warp 4, lane 0): same slots
  kPhEpi = 32,       // warp 8, lane 0: wait l and O, read O, staging wait, store, tiles
  kPhTimer = 40,     // %globaltimer (ns) at thread 0's start and end
};
enum PhaseSlot : int {
  kPhMmaWaitQ = 0, kPhMmaWaitKV = 1, kPhMmaWaitP = 2, kPhMmaWaitO = 3, kPhMmaIssue = 4, kPhMmaSteps = 5,
  kPhMmaUnits = 6,
  kPhLoadWaitQ = 0, kPhLoadWaitKV = 1, kPhLoadIssue = 2, kPhLoadSlots = 3,
  kPhSoftWait = 0, kPhSoftWork = 1, kPhSoftSteps = 2, kPhSoftSlow = 3, kPhSoftFinal = 4, kPhSoftLoad = 5,
  kPhSoftExp = 6,
  kPhEpiWait = 0, kPhEpiRead = 1, kPhEpiStage = 2, kPhEpiStore = 3, kPhEpiTiles = 4,
};

// Event trace (phase-clock builds): clock64 stamps of every hand-off of the
// first kTraceUnits work units of CTA 0, at phase[trace_off + (unit *
// kTraceSteps + step) * kTraceEvents + event], when the buffer has room.
constexpr int kTraceUnits = 3;
constexpr int kTraceSteps = 40;
constexpr int kTraceEvents = 32;
constexpr int kTraceWords = kTraceUnits * kTraceSteps * kTraceEvents;
enum TraceEvent : int {
  kTrMmaKV = 0,        // MMA thread: K/V slot of step j full
  kTrMmaP0 = 1,        // MMA thread: P of tile 0 / 1 observed (step j covers P(j-1))
  kTrMmaPV0 = 3,       // MMA thread: P V of tile 0 / 1 issued
  kTrMmaS0 = 5,        // MMA thread: S of tile 0 / 1 issued and committed
  kTrMmaOEmpty = 7,    // MMA thread: O-empty of tile 0 observed (first P V of the unit)
  kTrSoftS0 = 8,       // softmax tile 0 / 1 (warp 0 / 4, lane 0): S(j) observed
  kTrSoftP0 = 10,      // softmax tile 0 / 1: P(j) published
  kTrSoftLoad0 = 12,   // softmax tile 0: S(j) in registers
  kTrSoftExp0 = 13,    // softmax tile 0: exponentials done
  kTrEpiO0 = 14,       // epilogue (step 0 row): O of tile 0 / 1 final observed;
                       // (step 1 row): O of tile 0 / 1 read, O-empty signalled;
                       // (step 2 row): the staging wait of tile 0 / 1 done
  kTrLoadKV = 16,      // load thread: K/V slot of step j free, its copies issued
  kTrLoadQ = 17,       // load thread (step 0 row): Q-empty observed, Q copies issued
  kTrMmaQ = 18,        // MMA thread (step 0 row): Q-full observed
  kTrMmaQEmpty = 19,   // MMA thread: Q-empty committed (row of the step that commits it)
  kTrMmaWaitQ = 20,    // MMA thread (step 0 row): starts waiting for Q-full
  kTrMmaWaitKV = 21,   // MMA thread: starts waiting for the K/V slot of step j
  kTrMmaStepEnd = 22,  // MMA thread: step j's last commit issued
  kTrMmaDecoded = 23,  // MMA thread (step 0 row): unit decoded
  kTrSoftWarpP = 24,   // softmax warp w (0-7, lane 0): P(j) published (24 + w)
};

__device__ __forceinline__ void trace_event(unsigned long long* phase, int trace_off, int unit, int step, int ev) {
#if FA_PHASE_CLOCKS
  if (phase != nullptr && trace_off > 0 && blockIdx.x == 0 && unit < kTraceUnits && step < kTraceSteps)
    phase[trace_off + (unit * kTraceSteps + step) * kTraceEvents + ev] = static_cast<unsigned long long>(clock64());
#else
  (void)phase;
  (void)trace_off;
  (void)unit;
  (void)step;
  (void)ev;
#endif
}
#define FA_TRACE(unit, step, ev) trace_event(p.phase, p.trace_off, (unit), (step), (ev))

struct PhaseClock {
#if FA_PHASE_CLOCKS
  unsigned long long acc[kPhaseRole];
  long long t;
  __device__ __forceinline__ void start() {
#pragma unroll
    for (int i = 0; i < kPhaseRole; ++i) acc[i] = 0;
    t = clock64();
  }
  __device__ __forceinline__ void lap(int i) {
    const long long n = clock64();
    acc[i] += static_cast<unsigned long long>(n - t);
    t = n;
  }
  __device__ __forceinline__ void count(int i, int n = 1) { acc[i] += static_cast<unsigned long long>(n); }
  __device__ __forceinline__ void store(unsigned long long* phase, int base) const {
    if (phase == nullptr) return;
#pragma unroll
    for (int i = 0; i < kPhaseRole; ++i) phase[static_cast<size_t>(blockIdx.x) * kPhaseWords + base + i] = acc[i];
  }
#else
  __device__ __forceinline__ void start() {}
  __device__ __forceinline__ void lap(int) {}
  __device__ __forceinline__ void count(int, int = 1) {}
  __device__ __forceinline__ void store(unsigned long long*, int) const {}
#endif
};

struct FwdParams {
  int B, Nq, Nk, H;            // variable-length form: Nq / Nk are the maximum lengths
  int group;                   // query heads per key/value head (H / Hk)
  int causal;                  // 1: causal mask, bottom-right aligned
  int qtiles;                  // query tiles per unit: 1 (B_r = 128) or 2 (B_r = 256)
  int num_mblocks;             // ceil(Nq / (kBR * qtiles))
  int num_units;               // B * H * num_mblocks
  int units_per_item;          // units a CTA takes at a time (2 when causal: a balanced pair)
  int num_items;               // ceil(num_units / units_per_item)
  int num_splits;              // key splits per query block (1 unless split)
  int split_tiles;             // key tiles per split
  float* ws_o;                 // split: [num_splits, B, H, Nq, D] fp32 partial outputs
  float* ws_lse;               // split: [num_splits, B, H, Nq] fp32 partial log-sum-exp
  const int* cu_q;             // variable-length form: int32 [B + 1]
  const int* cu_k;
  float* lse;                  // [B, H, Nq] fp32
  __nv_bfloat16* o;            // output base (row stores of partial tiles)
  float scale;                 // softmax scale (natural units)
  float scale_log2;            // scale * log2(e)
  float rescale_threshold;     // log2 units; the O rescale is skipped while the max grows less
  const float* q_scale;        // FP8: [B, H, q_blocks] dequantisation scales of 128 query rows
  const float* k_scale;        // FP8: [B, Hk, k_blocks] of 128 keys
  const float* v_scale;        // FP8: [B, Hk] of a key/value head
  int q_blocks, k_blocks;
  int total_q, total_k;        // variable-length form: packed rows (sequences past them are rejected)
  unsigned long long timeout_ns;
  int* status;                 // [4]: code, block, warp, site
  unsigned long long* phase;   // phase clocks, [grid][kPhaseWords] (FA_PHASE_CLOCKS builds only; else null)
  int trace_off;               // word offset of the event trace in `phase` (0: no trace)
};

// Error codes shared with the C-ABI header.
constexpr int kErrUnsupported = -2;
constexpr int kErrTimeout = -5;
constexpr int kErrBadSeqlens = -7;

__device__ __forceinline__ void record_error(int* status, int code, int site) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = blockIdx.x;
    status[2] = threadIdx.x >> 5;
    status[3] = site;
  }
}

template <int D, int BC, int STAGES, int ESZ = 2>
struct SmemLayout {
  static constexpr int kQTileBytes = kBR * D * ESZ;
  static constexpr int kQPanelBytes = kBR * 128;
  static constexpr int kKVTileBytes = BC * D * ESZ;
  static constexpr int kKVPanelBytes = BC * 128;
  static constexpr int kSlotBytes = 2 * kKVTileBytes;  // K(j) then V(j-1)
  static constexpr int kStageWarpBytes = 32 * D * 2;   // 32 output rows per epilogue warp
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQT * kQTileBytes;
  static constexpr int kOffStage = kOffKV + STAGES * kSlotBytes;
  static constexpr int kOffBar = kOffStage + 4 * kStageWarpBytes;
  // barriers (8 bytes each)
  static constexpr int kBarQFull = 0;
  static constexpr int kBarQEmpty = 1;
  static constexpr int kBarKVFull = 2;
  static constexpr int kBarKVEmpty = kBarKVFull + STAGES;
  static constexpr int kBarSFull = kBarKVEmpty + STAGES;
  static constexpr int kBarPFull = kBarSFull + kQT;
  static constexpr int kBarLReady = kBarPFull + kQT;
  static constexpr int kBarOFinal = kBarLReady + kQT;
  static constexpr int kBarOEmpty = kBarOFinal + kQT;
  static constexpr int kBarTeardown = kBarOEmpty + kQT;
  static constexpr int kBarItemFull = kBarTeardown + 1;
  static constexpr int kBarItemEmpty = kBarItemFull + kItemSlots;
  static constexpr int kBarClc = kBarItemEmpty + kItemSlots;  // cancel response landed
  static constexpr int kNumBars = kBarClc + 1;
  static constexpr int kOffInvL = kOffBar + ((kNumBars * 8 + 15) / 16) * 16;
  static constexpr int kOffTmem = kOffInvL + kQT * kBR * 4;
  static constexpr int kOffAbort = kOffTmem + 16;
  static constexpr int kOffItems = kOffAbort + 16;  // kItemSlots ints
  static constexpr int kOffClc = kOffItems + 16;    // 16-byte cancel response (16-byte aligned)
  static constexpr int kBytes = kOffClc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kOffKV % 1024 == 0 && kKVTileBytes % 1024 == 0 && kOffStage % 1024 == 0 &&
                    kStageWarpBytes % 1024 == 0,
                "swizzled tiles need 1 KiB alignment");
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
};

// First column of sequence b in the variable-length FP8 V^T codes: its packed
// key offset rounded up to 16 plus 16 per earlier sequence.  Sequence b then
// starts 16-byte aligned and its keys, rounded up to 16, end at or before the
// start of sequence b + 1 (ceil((x + n) / 16) >= ceil(x / 16) + ceil(n / 16) - 1).
__host__ __device__ __forceinline__ long long fp8_vt_col0(long long cu_b, int b) {
  return (cu_b + 15) / 16 * 16 + 16LL * b;
}

// Geometry of one 128-row tile along the sequence axis.  `load_row` is the
// first row the TMA box reads; rows [lo, hi) of the box are valid.  In the
// variable-length form (SHIFT) a tile that would run past the end of its
// sequence is shifted back so that it ends exactly at the end, never touching
// memory past the last row of the packed tensor (rows before the sequence are
// masked).
struct RowWindow {
  int load_row;
  int lo, hi;
};

template <bool SHIFT>
__device__ __forceinline__ RowWindow make_window(int seq_start, int seq_end, int row0, int rows) {
  RowWindow w;
  if (!SHIFT || row0 + rows <= seq_end) {
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

// One work unit: query block mb (two 128-row tiles) of head h in batch b.
struct Unit {
  int b, h, hk;                        // batch, query head, key/value head
  int q_start, q_end, k_start, k_end;  // row ranges of the sequence (packed rows if variable length)
  int q_row0;                          // first query row of the unit
  int off;                             // causal: query i sees keys j <= i + off
  int nkv;                             // key/value steps of the unit (max over its tiles)
  int j0;                              // first key tile of the unit (split)
  int split;                           // split index
  int nkv_all;                         // key tiles of the whole sequence
  int lse_base;                        // (b * H + h) * Nq
  bool run;                            // some tile of the unit has rows and visible keys
  bool nokeys;                         // query rows but no keys at all (variable length only)
  bool active[kQT];                    // tile t has rows and runs nt[t] > 0 key steps
  bool zero[kQT];                      // tile t has rows but sees no key: o = 0, LSE = -inf
  int nt[kQT];                         // key/value tiles tile t needs
  RowWindow qwin[kQT];
};

// Every role decodes the same unit identically (pure function of u and params).
// SHIFT: variable-length tiles at a sequence's end are shifted back (make_window).
template <int BC, bool VARLEN, bool CAUSAL, bool SPLIT, bool SHIFT = VARLEN>
__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int u) {
  Unit w;
  w.split = 0;
  if constexpr (SPLIT) {
    w.split = u % p.num_splits;
    u /= p.num_splits;
  }
  int mb = u % p.num_mblocks;
  if constexpr (CAUSAL) {
    // Zigzag order within a head: last, first, second last, second, ... so that
    // the two units of an item (the heaviest left with the lightest left) carry
    // the same work and the persistent round-robin stays balanced.
    const int pi = mb >> 1;
    mb = (mb & 1) ? pi : p.num_mblocks - 1 - pi;
  }
  const int r = u / p.num_mblocks;
  w.h = r % p.H;
  w.b = r / p.H;
  w.hk = w.h / p.group;
  w.q_start = 0;
  w.q_end = p.Nq;
  w.k_start = 0;
  w.k_end = p.Nk;
  bool bad = false;
  if constexpr (VARLEN) {
    w.q_start = p.cu_q[w.b];
    w.q_end = p.cu_q[w.b + 1];
    w.k_start = p.cu_k[w.b];
    w.k_end = p.cu_k[w.b + 1];
    const int len_q = w.q_end - w.q_start, len_k = w.k_end - w.k_start;
    bad = len_q < 0 || len_k < 0 || len_q > p.Nq || len_k > p.Nk || w.q_start < 0 || w.k_start < 0 ||
          w.q_start > p.total_q - len_q || w.k_start > p.total_k - len_k;
  }
  w.q_row0 = w.q_start + mb * (kBR * p.qtiles);
  w.off = (w.k_end - w.k_start) - (w.q_end - w.q_start);
  const int nkv_all = bad ? 0 : (w.k_end - w.k_start + BC - 1) / BC;
  w.nkv_all = nkv_all;
  w.j0 = SPLIT ? w.split * p.split_tiles : 0;
  const int nkv_here = SPLIT ? max(0, min(p.split_tiles, nkv_all - w.j0)) : nkv_all;
  w.lse_base = (w.b * p.H + w.h) * p.Nq;
  const bool has_rows = !bad && w.q_row0 < w.q_end;
  w.nkv = 0;
#pragma unroll
  for (int t = 0; t < kQT; ++t) {
    const int r0 = w.q_row0 + t * kBR;
    w.qwin[t] = make_window<SHIFT>(w.q_start, w.q_end, r0, kBR);
    const bool rows = has_rows && t < p.qtiles && r0 < w.q_end;
    int n = nkv_here;
    if (CAUSAL && rows) {
      // Last valid row of the tile, in sequence coordinates, and the last key it sees.
      const int i_last = w.qwin[t].load_row - w.q_start + w.qwin[t].hi - 1;
      const int key_last = i_last + w.off;
      n = key_last < 0 ? 0 : min(nkv_here, key_last / BC + 1 - w.j0);
      n = max(n, 0);
    }
    w.nt[t] = rows ? n : 0;
    w.active[t] = rows && n > 0;
    w.zero[t] = rows && n == 0 && (nkv_all > 0 || SPLIT);
    w.nkv = max(w.nkv, w.nt[t]);
  }
  w.run = w.active[0] || w.active[1];
  w.nokeys = has_rows && nkv_all == 0 && !SPLIT;
  if (bad && mb == 0 && w.h == 0) {
    if ((threadIdx.x & 31) == 0 && threadIdx.x < 32) record_error(p.status, kErrBadSeqlens, 0);
  }
  return w;
}

// Next entry of this CTA's work-item sequence (consumer side of the item
// ring): the item, -1 at the end, -2 if a wait gave up.  `n` counts the items
// read so far; `warp`: the whole warp reads and lane 0 releases the slot,
// else a single thread does both.
// The grid has one CTA per work item; a CTA starts with item blockIdx.x and
// its load thread takes over the items of CTAs that have not started yet
// (cluster launch control), so items are handed out in launch order to
// whichever SM is free: CTAs never drift apart over unequal work (variable
// lengths), which keeps the K/V of the heads in flight together in L2.
__device__ __forceinline__ int item_next(uint32_t bar_full, uint32_t bar_empty, const volatile int* items,
                                         volatile int* abort, uint64_t tmo, int* status, uint32_t& n, bool warp) {
  const uint32_t slot = n % kItemSlots;
  const uint32_t parity = (n / kItemSlots) & 1u;
  const bool got = warp ? ptx::mbar_wait_warp(bar_full + 8u * slot, parity, abort, tmo)
                        : ptx::mbar_wait(bar_full + 8u * slot, parity, abort, tmo);
  if (!got) {
    if (!warp || (threadIdx.x & 31) == 0) record_error(status, kErrTimeout, kSiteItem);
    return -2;
  }
  const int item = items[slot];
  if (warp) __syncwarp();
  if (!warp || (threadIdx.x & 31) == 0) ptx::mbar_arrive(bar_empty + 8u * slot);
  ++n;
  return item;
}

// Walk over the work units of this CTA: each item is units_per_item
// consecutive units.  Every role reads the same item sequence, so all roles
// see the same unit sequence.
// Dynamic (kDynamic: the item ring) or static (items blockIdx.x,
// blockIdx.x + gridDim.x, ... on a grid of one CTA per SM) item sequence.
#define FA_NEXT_ITEM(prev)                                                                        \
  (kDynamic ? item_next(bar(L::kBarItemFull), bar(L::kBarItemEmpty), s_items, s_abort, tmo, p.status, \
                        item_n_, warp != 12)                                                      \
            : ((prev) < 0 ? static_cast<int>(blockIdx.x) : (prev) + static_cast<int>(gridDim.x)))
#define FA_FOR_EACH_UNIT(u)                                                                       \
  for (int it_ = FA_NEXT_ITEM(-1); it_ >= 0 && it_ < p.num_items && ok; it_ = FA_NEXT_ITEM(it_))  \
    for (int sub_ = 0, u = it_ * p.units_per_item;                                                  \
         sub_ < p.units_per_item && u < p.num_units && ok; ++sub_, ++u)

template <int D, int BC, int STAGES, bool VARLEN, bool CAUSAL, bool SPLIT = false, bool QUAD = false,
          bool FP8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
  using L = SmemLayout<D, BC, STAGES, FP8 ? 1 : 2>;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!FP8 || (D == 128 && BC == 128 && !SPLIT && !QUAD), "FP8: d 128, 128-key tiles");
  // Variable-length tiles: shifted at a sequence's end, except FP8 ones (which
  // must coincide with quantisation blocks).
  constexpr bool kShift = VARLEN && !FP8;
  // Packed variable-length batches hand out work items dynamically (units of
  // unequal work); dense problems, whose units are all alike, walk a static
  // round-robin over a grid of one CTA per SM.
  constexpr bool kDynamic = VARLEN;
  static_assert(BC == 64 || BC == 128, "key tile");
  static_assert(2 * BC + 2 * D <= 512, "TMEM columns");
  static_assert(!QUAD || (BC == 128 && !CAUSAL && !SPLIT), "quad reduction: 128-key tiles, no mask or split");
  constexpr int kTmemCols = 512;
  // 128-byte swizzle panels along d: 64 bf16 or 128 e4m3 elements each.
  constexpr int kPanelElems = FP8 ? 128 : kPanel;
  constexpr int kDPanels = D / kPanelElems;  // input (Q, K, V) panels
  constexpr int kOutPanels = D / kPanel;     // bf16 output panels

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = base + L::kOffBar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  float* const s_invl = reinterpret_cast<float*>(gbase + L::kOffInvL);
  volatile uint32_t* const s_tmem = reinterpret_cast<volatile uint32_t*>(gbase + L::kOffTmem);
  volatile int* const s_abort = reinterpret_cast<volatile int*>(gbase + L::kOffAbort);
  volatile int* const s_items = reinterpret_cast<volatile int*>(gbase + L::kOffItems);
  const uint64_t tmo = p.timeout_ns;
  // Items read from the work-item ring (the MMA thread reads alone, the
  // softmax and epilogue warps read warp-wide; the load thread writes it).
  uint32_t item_n_ = 0;

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
    ptx::mbar_init(bar(L::kBarQEmpty), 1);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(L::kBarKVFull + s), 1);
      ptx::mbar_init(bar(L::kBarKVEmpty + s), 1);
    }
    for (int t = 0; t < kQT; ++t) {
      ptx::mbar_init(bar(L::kBarSFull + t), 1);
      ptx::mbar_init(bar(L::kBarPFull + t), kBR);   // P(j) written, O rescaled
      ptx::mbar_init(bar(L::kBarLReady + t), kBR);  // final 1/l of every row
      ptx::mbar_init(bar(L::kBarOFinal + t), 1);    // last P V of the unit done
      ptx::mbar_init(bar(L::kBarOEmpty + t), kBR);  // epilogue finished reading O_t
    }
    ptx::mbar_init(bar(L::kBarTeardown), 1);
    for (int i = 0; i < kItemSlots; ++i) {
      ptx::mbar_init(bar(L::kBarItemFull + i), 1);
      ptx::mbar_init(bar(L::kBarItemEmpty + i), kItemConsumers);
    }
    ptx::mbar_init(bar(L::kBarClc), 1);
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
#if FA_PHASE_CLOCKS
  if (threadIdx.x == 0 && p.phase) p.phase[static_cast<size_t>(blockIdx.x) * kPhaseWords + kPhTimer] = ptx::globaltimer_ns();
#endif

  if (warp >= 12) {
    ptx::setmaxnreg_dec<RegSplit<VARLEN>::kOther>();
    if (warp == 13 && lane == 0) {
      // =========================================================== TMA loads
      uint32_t qcount = 0;  // units whose Q was loaded
      uint32_t g = 0;       // ring slots handed to the TMA unit so far
      int tr_unit = 0;      // units loaded (event trace)
      bool ok = true;
      PhaseClock ph;
      ph.start();
      // Dynamic schedule: the load thread produces the work-item ring, this
      // CTA's own item first, then the items of CTAs whose launch the hardware
      // cancelled on request.  The request for the next item is issued when an
      // item starts, so its answer is back by the time the item's loads are
      // all issued.  Static schedule: items blockIdx.x + k * gridDim.x.
      uint32_t n_pub = 0, n_clc = 0;
      bool clc_pending = false;
      auto publish = [&](int item) -> bool {
        const uint32_t slot = n_pub % kItemSlots;
        if (!ptx::mbar_wait(bar(L::kBarItemEmpty + slot), ((n_pub / kItemSlots) & 1u) ^ 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kSiteItem);
          return false;
        }
        s_items[slot] = item;
        ptx::mbar_arrive(bar(L::kBarItemFull + slot));
        ++n_pub;
        return true;
      };
      auto request = [&]() {
        ptx::fence_proxy_async_smem();  // the previous answer was read before it is overwritten
        ptx::mbar_arrive_expect_tx(bar(L::kBarClc), 16);
        ptx::clc_try_cancel(base + L::kOffClc, bar(L::kBarClc));
        clc_pending = true;
      };
      int cur = blockIdx.x;
      if constexpr (kDynamic) {
        ok = publish(cur);
        if (ok) request();
      }
#pragma unroll 1
      while (ok && cur >= 0 && cur < p.num_items) {
#pragma unroll 1
        for (int sub_ = 0, u = cur * p.units_per_item; sub_ < p.units_per_item && u < p.num_units && ok;
             ++sub_, ++u) {
          const Unit w = decode_unit<BC, VARLEN, CAUSAL, SPLIT, kShift>(p, u);
          if (!w.run) continue;
          // Q of this unit, once the previous unit's S MMAs no longer read it.
          ph.lap(kPhLoadIssue);
          if (!ptx::mbar_wait(bar(L::kBarQEmpty), (qcount & 1u) ^ 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kSiteLoadQ);
            ok = false;
            break;
          }
          ph.lap(kPhLoadWaitQ);
          uint32_t q_bytes = 0;
#pragma unroll
          for (int t = 0; t < kQT; ++t) q_bytes += w.active[t] ? L::kQTileBytes : 0;
          ptx::mbar_arrive_expect_tx(bar(L::kBarQFull), q_bytes);
          ++qcount;
#pragma unroll
          for (int t = 0; t < kQT; ++t) {
            if (!w.active[t]) continue;
#pragma unroll
            for (int pnl = 0; pnl < kDPanels; ++pnl) {
              const uint32_t dst = base + L::kOffQ + t * L::kQTileBytes + pnl * L::kQPanelBytes;
              if constexpr (VARLEN)
                ptx::tma_load_3d(dst, &tm_q, bar(L::kBarQFull), pnl * kPanelElems, w.h, w.qwin[t].load_row);
              else
                ptx::tma_load_4d(dst, &tm_q, bar(L::kBarQFull), pnl * kPanelElems, w.h, w.qwin[t].load_row, w.b);
            }
          }
          FA_TRACE(tr_unit, 0, kTrLoadQ);
#pragma unroll 1
          for (int j = 0; j <= w.nkv; ++j) {
            const uint32_t slot = g % STAGES;
            ph.lap(kPhLoadIssue);
            if (!ptx::mbar_wait(bar(L::kBarKVEmpty + slot), ((g / STAGES) & 1u) ^ 1u, s_abort, tmo)) {
              record_error(p.status, kErrTimeout, kSiteLoadKV);
              ok = false;
              break;
            }
            ph.lap(kPhLoadWaitKV);
            ph.count(kPhLoadSlots);
            FA_TRACE(tr_unit, j, kTrLoadKV);
            const uint32_t bytes = (j < w.nkv ? L::kKVTileBytes : 0) + (j >= 1 ? L::kKVTileBytes : 0);
            ptx::mbar_arrive_expect_tx(bar(L::kBarKVFull + slot), bytes);
            ++g;
            const uint32_t sbase = base + L::kOffKV + slot * L::kSlotBytes;
            if (j < w.nkv) {
              const RowWindow kw = make_window<kShift>(w.k_start, w.k_end, w.k_start + (w.j0 + j) * BC, BC);
#pragma unroll
              for (int pnl = 0; pnl < kDPanels; ++pnl) {
                const uint32_t dst = sbase + pnl * L::kKVPanelBytes;
                if constexpr (VARLEN)
                  ptx::tma_load_3d(dst, &tm_k, bar(L::kBarKVFull + slot), pnl * kPanelElems, w.hk, kw.load_row);
                else
                  ptx::tma_load_4d(dst, &tm_k, bar(L::kBarKVFull + slot), pnl * kPanelElems, w.hk, kw.load_row, w.b);
              }
            }
            if (j >= 1) {
              const RowWindow vw = make_window<kShift>(w.k_start, w.k_end, w.k_start + (w.j0 + j - 1) * BC, BC);
              if constexpr (FP8 && VARLEN) {
                // V^T tile: d rows x 128 keys (one box, keys innermost) from the sequence's columns.
                const int col = static_cast<int>(fp8_vt_col0(w.k_start, w.b)) + (vw.load_row - w.k_start);
                ptx::tma_load_3d(sbase + L::kKVTileBytes, &tm_v, bar(L::kBarKVFull + slot), col, 0, w.hk);
              } else if constexpr (FP8) {
                ptx::tma_load_4d(sbase + L::kKVTileBytes, &tm_v, bar(L::kBarKVFull + slot), vw.load_row, 0, w.hk, w.b);
              } else {
#pragma unroll
                for (int pnl = 0; pnl < kDPanels; ++pnl) {
                  const uint32_t dst = sbase + L::kKVTileBytes + pnl * L::kKVPanelBytes;
                  if constexpr (VARLEN)
                    ptx::tma_load_3d(dst, &tm_v, bar(L::kBarKVFull + slot), pnl * kPanel, w.hk, vw.load_row);
                  else
                    ptx::tma_load_4d(dst, &tm_v, bar(L::kBarKVFull + slot), pnl * kPanel, w.hk, vw.load_row, w.b);
                }
              }
            }
          }
          ++tr_unit;
        }
        if (!ok) break;
        if constexpr (kDynamic) {
          // The next item: the cancelled CTA's index, or -1 when none is left.
          if (!ptx::mbar_wait(bar(L::kBarClc), n_clc & 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kSiteItem);
            ok = false;
            break;
          }
          ++n_clc;
          clc_pending = false;
          cur = ptx::clc_cancelled_x(base + L::kOffClc);
          if (!publish(cur)) {
            ok = false;
            break;
          }
          if (cur >= 0) request();
        } else {
          cur += gridDim.x;
        }
      }
      ph.lap(kPhLoadIssue);
      ph.store(p.phase, kPhLoad);
      // An answer still in flight is written by the async proxy: wait for it.
      if (clc_pending) ptx::mbar_wait_drain(bar(L::kBarClc), n_clc & 1u, tmo);
      // Teardown: never leave a TMA write to shared memory in flight.  Slot s
      // last received ring index s + STAGES * (rounds - 1).
      if (qcount > 0) ptx::mbar_wait_drain(bar(L::kBarQFull), (qcount - 1) & 1u, tmo);
      for (uint32_t s = 0; s < STAGES; ++s) {
        if (g > s) {
          const uint32_t rounds = (g - 1 - s) / STAGES + 1;
          ptx::mbar_wait_drain(bar(L::kBarKVFull + s), (rounds - 1) & 1u, tmo);
        }
      }
    } else if (warp == 12 && lane == 0) {
      // ========================================================== MMA issue
      constexpr uint32_t idesc_qk = FP8 ? ptx::idesc_e4m3_f32(kBR, BC) : ptx::idesc_bf16_f32(kBR, BC, 0, 0);
      constexpr uint32_t idesc_pv = FP8 ? ptx::idesc_e4m3_f32(kBR, D) : ptx::idesc_bf16_f32(kBR, D, 0, 1);
      uint32_t qcount = 0, g = 0;
      uint32_t pc[kQT] = {0, 0};  // P-full completions consumed, per tile
      uint32_t uc[kQT] = {0, 0};  // units with the tile active, per tile
      int tr_unit = 0;            // units issued (event trace)
      bool ok = true;
      PhaseClock ph;
      ph.start();
#pragma unroll 1
      FA_FOR_EACH_UNIT(u) {
        const Unit w = decode_unit<BC, VARLEN, CAUSAL, SPLIT, kShift>(p, u);
        if (!w.run) continue;
        FA_TRACE(tr_unit, 0, kTrMmaDecoded);
        ph.lap(kPhMmaIssue);
        FA_TRACE(tr_unit, 0, kTrMmaWaitQ);
        if (!ptx::mbar_wait(bar(L::kBarQFull), qcount & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kSiteMmaQ);
          ok = false;
          break;
        }
        ph.lap(kPhMmaWaitQ);
        ph.count(kPhMmaUnits);
        FA_TRACE(tr_unit, 0, kTrMmaQ);
        ++qcount;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int j = 0; j <= w.nkv && ok; ++j) {
          const uint32_t slot = g % STAGES;
          ph.lap(kPhMmaIssue);
          FA_TRACE(tr_unit, j, kTrMmaWaitKV);
          if (!ptx::mbar_wait(bar(L::kBarKVFull + slot), (g / STAGES) & 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kSiteMmaK);
            ok = false;
            break;
          }
          ph.lap(kPhMmaWaitKV);
          ph.count(kPhMmaSteps);
          FA_TRACE(tr_unit, j, kTrMmaKV);
          ptx::tc_fence_after();
          const uint32_t k_base = base + L::kOffKV + slot * L::kSlotBytes;
          const uint32_t v_base = k_base + L::kKVTileBytes;
#pragma unroll
          for (int t = 0; t < kQT; ++t) {
            if (!w.active[t]) continue;
            const int nt = t == 0 ? w.nt[0] : w.nt[1];
            const uint32_t tS = tmem + static_cast<uint32_t>(t * BC);
            const uint32_t tP = tS + BC / 2;
            const uint32_t tO = tmem + static_cast<uint32_t>(2 * BC + t * D);
            if (j >= 1 && j <= nt) {
              // O_t += P_t(j-1) V(j-1), once P is written and O rescaled.
              ph.lap(kPhMmaIssue);
              if (!ptx::mbar_wait(bar(L::kBarPFull + t), pc[t] & 1u, s_abort, tmo)) {
                record_error(p.status, kErrTimeout, kSiteMmaP);
                ok = false;
                break;
              }
              ph.lap(kPhMmaWaitP);
              FA_TRACE(tr_unit, j, kTrMmaP0 + t);
              ++pc[t];
              // The first P V of a unit overwrites O_t: the epilogue of the
              // previous unit must have finished reading it.
              if (j == 1 && !ptx::mbar_wait(bar(L::kBarOEmpty + t), (uc[t] & 1u) ^ 1u, s_abort, tmo)) {
                record_error(p.status, kErrTimeout, kSiteMmaOEmpty);
                ok = false;
                break;
              }
              ph.lap(kPhMmaWaitO);
              if (j == 1 && t == 0) FA_TRACE(tr_unit, j, kTrMmaOEmpty);
              ptx::tc_fence_after();
              // Descriptors advance by byte offset / 16 in their low word (the
              // address field cannot carry: shared addresses stay below 256 KiB);
              // building each one from scratch per MMA costs the issuing
              // thread instruction slots it shares with two softmax warps.
              if constexpr (FP8) {
                // P: 32 e4m3 per step = 8 TMEM columns; V^T is K-major (keys
                // along the 128-byte rows): 32 keys = 32 bytes.
                const uint64_t vdesc = ptx::sw128_desc(v_base, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < BC / 32; ++kk)
                  ptx::mma_ts_f8(tO, tP + kk * 8, vdesc + static_cast<uint64_t>(kk * 2), idesc_pv,
                                 (j - 1 > 0 || kk > 0) ? 1u : 0u);
              } else {
                // V is MN-major: 16 keys = two 8-row swizzle atoms = 2048 bytes;
                // the two 64-column halves of d sit one panel (BC * 128 bytes) apart.
                const uint64_t vdesc = ptx::sw128_desc(v_base, L::kKVPanelBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < BC / 16; ++kk)
                  ptx::mma_ts(tO, tP + kk * 8, vdesc + static_cast<uint64_t>(kk * 128), idesc_pv,
                              (j - 1 > 0 || kk > 0) ? 1u : 0u);
              }
              if (j == nt) ptx::mma_commit(bar(L::kBarOFinal + t));
              FA_TRACE(tr_unit, j, kTrMmaPV0 + t);
            }
            if (j < nt) {
              // S_t = Q_t K(j)^T
              const uint32_t q_base = base + L::kOffQ + t * L::kQTileBytes;
              const uint64_t qdesc = ptx::sw128_desc(q_base, 16, 1024);
              const uint64_t kdesc = ptx::sw128_desc(k_base, 16, 1024);
              if constexpr (FP8) {
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk)  // 32 e4m3 = 32 bytes inside the single 128-byte panel
                  ptx::mma_ss_f8(tS, qdesc + static_cast<uint64_t>(kk * 2), kdesc + static_cast<uint64_t>(kk * 2),
                                 idesc_qk, kk > 0 ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  // K-major, 128-byte swizzle: 16 columns = 32 bytes inside a panel.
                  const uint32_t off_q = (kk / 4) * L::kQPanelBytes + (kk % 4) * 32;
                  const uint32_t off_k = (kk / 4) * L::kKVPanelBytes + (kk % 4) * 32;
                  ptx::mma_ss(tS, qdesc + static_cast<uint64_t>(off_q >> 4), kdesc + static_cast<uint64_t>(off_k >> 4),
                              idesc_qk, kk > 0 ? 1u : 0u);
                }
              }
              ptx::mma_commit(bar(L::kBarSFull + t));
              FA_TRACE(tr_unit, j, kTrMmaS0 + t);
            }
          }
          if (!ok) break;
          // Q of this unit is free once its last S MMAs complete.
          if (j == w.nkv - 1) {
            ptx::mma_commit(bar(L::kBarQEmpty));
            FA_TRACE(tr_unit, j, kTrMmaQEmpty);
          }
          ptx::mma_commit(bar(L::kBarKVEmpty + slot));  // K(j) and V(j-1) no longer needed
          FA_TRACE(tr_unit, j, kTrMmaStepEnd);
          ++g;
        }
#pragma unroll
        for (int t = 0; t < kQT; ++t) uc[t] += w.active[t] ? 1u : 0u;
        ++tr_unit;
      }
      ph.lap(kPhMmaIssue);
      ph.store(p.phase, kPhMma);
      // Teardown: all MMAs must be complete before TMEM is released.
      ptx::mma_commit(bar(L::kBarTeardown));
      if (!ptx::mbar_wait_drain(bar(L::kBarTeardown), 0, tmo)) record_error(p.status, kErrTimeout, kSiteTeardown);
    }
  } else if (warp < 8) {
    ptx::setmaxnreg_inc<RegSplit<VARLEN>::kSoftmax>();
    // ================================================================ softmax
    const int t = warp >> 2;
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(t * BC);
    const uint32_t tP = tS + BC / 2;
    const float c2 = p.scale_log2;
    // Largest block sum for which every p of the block is below 2^T (T the
    // rescale threshold), with a margin for the rounding of the exponent.
    const float accept_sum = exp2f(p.rescale_threshold) * 0.9990234375f;
    // Bits 0-30: S-full completions consumed; bit 31: parity of the units
    // this tile has finished (the epilogue's O-empty count).
    uint32_t sc = 0;
    int tr_unit = 0;  // units processed (event trace)
    const bool tr_lead = lane == 0 && (warp & 3) == 0;
    bool ok = true;
    // Before a unit's final message the epilogue must have taken the previous
    // one (1 / l is one shared word per row, L-ready one barrier phase per
    // unit).  With two or more key tiles the MMA thread's O-empty wait before
    // the unit's first P V already orders the two; a unit of one key tile
    // could otherwise finish while the epilogue still waits for the last.
    auto wait_epilogue = [&]() -> bool {
      if (!ptx::mbar_wait_warp(bar(L::kBarOEmpty + t), (sc >> 31) ^ 1u, s_abort, tmo)) {
        if (lane == 0) record_error(p.status, kErrTimeout, kSiteSoftFinal);
        return false;
      }
      return true;
    };
    PhaseClock ph;
    ph.start();
#pragma unroll 1
    FA_FOR_EACH_UNIT(u) {
      const Unit w = decode_unit<BC, VARLEN, CAUSAL, SPLIT, kShift>(p, u);
      const bool active = t == 0 ? w.active[0] : w.active[1];
      if (!active) continue;
      const RowWindow qw = t == 0 ? w.qwin[0] : w.qwin[1];
      const int nt = t == 0 ? w.nt[0] : w.nt[1];
      // Causal: this row sees sequence keys <= i_row + off.
      const int key_lim = (qw.load_row - w.q_start + row) + w.off;
      const int first_row_lim = (qw.load_row - w.q_start + qw.lo) + w.off;
      // Only the last key tile (ragged end, shifted variable-length window) and,
      // when causal, the tiles from the first one crossing the diagonal need masks.
      int j_mask = w.nkv_all - 1;
      if constexpr (CAUSAL) j_mask = min(j_mask, first_row_lim + 1 < 0 ? 0 : (first_row_lim + 1) / BC);
      if constexpr (QUAD) {
        // Row max and row sum reduced with warp shuffles: the 16-lane TMEM
        // shapes spread each row over the four threads of a quad.  Thread
        // (qr, qc) = (lane / 4, lane % 4) owns rows 8r + qr (r = 0..3) of the
        // warp's 32 rows and, of each 8-column group g, columns 8g + 2qc and
        // 8g + 2qc + 1 (32 of the 128 columns of every row).
        const int qr = lane >> 2, qc = lane & 3;
        const uint32_t tSw = tmem + lane_off + static_cast<uint32_t>(t * BC);
        const uint32_t tPw = tSw + BC / 2;
        const uint32_t tOw = tmem + lane_off + static_cast<uint32_t>(2 * BC + t * D);
        float m_q[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float l_q[4] = {0.f, 0.f, 0.f, 0.f};  // this thread's share of each row sum
#pragma unroll 1
        for (int j = 0; j < nt; ++j) {
          ph.lap(kPhSoftWork);
          if (!ptx::mbar_wait_warp(bar(L::kBarSFull + t), sc & 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kSiteSoftS);
            ok = false;
            break;
          }
          ph.lap(kPhSoftWait);
          ph.count(kPhSoftSteps);
          ++sc;
          ptx::tc_fence_after();
          uint32_t raw[4][32];
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ch = 0; ch < 2; ++ch)
              ptx::tmem_ld16x256_x8(tSw + (static_cast<uint32_t>(16 * h) << 16) + ch * 64, raw[2 * h + ch]);
          ptx::tmem_wait_ld();
          // s[r][k]: row 8r + qr, column 8 * (k / 2) + 2 * qc + k % 2.
          float s[4][32];
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ch = 0; ch < 2; ++ch)
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                const int k = 2 * (8 * ch + g);
                s[2 * h][k] = __uint_as_float(raw[2 * h + ch][4 * g]);
                s[2 * h][k + 1] = __uint_as_float(raw[2 * h + ch][4 * g + 1]);
                s[2 * h + 1][k] = __uint_as_float(raw[2 * h + ch][4 * g + 2]);
                s[2 * h + 1][k + 1] = __uint_as_float(raw[2 * h + ch][4 * g + 3]);
              }
          if (w.j0 + j >= j_mask) {
            const RowWindow kw = make_window<kShift>(w.k_start, w.k_end, w.k_start + (w.j0 + j) * BC, BC);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const int col = 8 * (k >> 1) + 2 * qc + (k & 1);
                if (col < kw.lo || col >= kw.hi) s[r][k] = -INFINITY;
              }
          }
          float alpha[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            float mx0 = ptx::fmax3(s[r][0], s[r][1], s[r][2]);
            float mx1 = ptx::fmax3(s[r][3], s[r][4], s[r][5]);
#pragma unroll
            for (int k = 6; k < 30; k += 4) {
              mx0 = ptx::fmax3(mx0, s[r][k], s[r][k + 1]);
              mx1 = ptx::fmax3(mx1, s[r][k + 2], s[r][k + 3]);
            }
            float bm = ptx::fmax3(mx0, mx1, fmaxf(s[r][30], s[r][31]));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
            float m_new = m_q[r];
            if (bm > m_q[r] && (m_q[r] == -INFINITY || (bm - m_q[r]) * c2 > p.rescale_threshold)) m_new = bm;
            alpha[r] = (m_new == m_q[r]) ? 1.f : ptx::ex2((m_q[r] - m_new) * c2);
            m_q[r] = m_new;
          }
          const uint64_t c2x2 = ptx::f2_pack(c2, c2);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[32];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int r = 2 * h + rr;
              const float neg = (m_q[r] == -INFINITY) ? 0.f : -m_q[r] * c2;
              const uint64_t negx2 = ptx::f2_pack(neg, neg);
              uint64_t acc[2] = {0, 0};
#pragma unroll
              for (int g = 0; g < 16; ++g) {
                float x0, x1;
                ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[r][2 * g], s[r][2 * g + 1]), c2x2, negx2), x0, x1);
                const float e0 = ptx::ex2(x0), e1 = ptx::ex2(x1);
                acc[g & 1] = ptx::f2_add(acc[g & 1], ptx::f2_pack(e0, e1));
                pk[2 * g + rr] = ptx::pack_bf16x2(e0, e1);
              }
              float a0, a1, a2, a3;
              ptx::f2_unpack(acc[0], a0, a1);
              ptx::f2_unpack(acc[1], a2, a3);
              l_q[r] = l_q[r] * alpha[r] + ((a0 + a1) + (a2 + a3));
            }
            ptx::tmem_st16x128_x16(tPw + (static_cast<uint32_t>(16 * h) << 16), pk);
          }
          const bool any_rescale = alpha[0] != 1.f || alpha[1] != 1.f || alpha[2] != 1.f || alpha[3] != 1.f;
          if (j >= 1 && __any_sync(0xffffffffu, any_rescale)) {
            // Same correction as the one-row-per-thread form, in the quad layout.
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int ch = 0; ch < D / 64; ++ch) {
                uint32_t r[32];
                const uint32_t a = tOw + (static_cast<uint32_t>(16 * h) << 16) + ch * 64;
                ptx::tmem_ld16x256_x8(a, r);
                ptx::tmem_wait_ld();
                const uint64_t ax = ptx::f2_pack(alpha[2 * h], alpha[2 * h]);
                const uint64_t bx = ptx::f2_pack(alpha[2 * h + 1], alpha[2 * h + 1]);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  float x0, x1, y0, y1;
                  ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1])), ax), x0, x1);
                  ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3])), bx), y0, y1);
                  r[4 * g] = __float_as_uint(x0);
                  r[4 * g + 1] = __float_as_uint(x1);
                  r[4 * g + 2] = __float_as_uint(y0);
                  r[4 * g + 3] = __float_as_uint(y1);
                }
                ptx::tmem_st16x256_x8(a, r);
              }
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::kBarPFull + t));
        }
        if (!ok || (nt == 1 && !(ok = wait_epilogue()))) break;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float l = l_q[r] + __shfl_xor_sync(0xffffffffu, l_q[r], 1);
          l += __shfl_xor_sync(0xffffffffu, l, 2);
          const int row_r = ((warp & 3) << 5) + 8 * r + qr;
          if (qc == 0) {
            const bool has = l > 0.f;
            s_invl[t * kBR + row_r] = has ? 1.f / l : 0.f;
            if (row_r >= qw.lo && row_r < qw.hi) {
              const float lse = has ? (m_q[r] * p.scale + log2f(l) * 0.69314718055994530942f) : -INFINITY;
              p.lse[w.lse_base + (qw.load_row - w.q_start + row_r)] = lse;
            }
          }
        }
      } else {
        float m_ref = -INFINITY;  // FP8: in scaled log2 units
        float l = 0.f;
        // FP8: dequantisation scales of this query tile and key/value head.
        float cq = 0.f, vsc = 1.f;
        if constexpr (FP8) {
          cq = c2 * p.q_scale[(w.b * p.H + w.h) * p.q_blocks + (qw.load_row - w.q_start) / kBR];
          vsc = p.v_scale[w.b * (p.H / p.group) + w.hk];
        }
  #pragma unroll 1
        for (int j = 0; j < nt; ++j) {
          // FP8: exp2 coefficient of this key tile (query and key scales folded in).
          const float c2j = FP8 ? cq * p.k_scale[(w.b * (p.H / p.group) + w.hk) * p.k_blocks + w.j0 + j] : c2;
          ph.lap(kPhSoftWork);
          if (!ptx::mbar_wait_warp(bar(L::kBarSFull + t), sc & 1u, s_abort, tmo)) {
            record_error(p.status, kErrTimeout, kSiteSoftS);
            ok = false;
            break;
          }
          ph.lap(kPhSoftWait);
          ph.count(kPhSoftSteps);
          if (tr_lead) FA_TRACE(tr_unit, j, kTrSoftS0 + t);
          ++sc;
          ptx::tc_fence_after();
          // S row of this thread, with the keys outside the row's window at -inf.
          float s[BC];
          auto load_scores = [&]() {
            uint32_t sr[BC];
  #pragma unroll
            for (int c = 0; c < BC / 32; ++c) ptx::tmem_ld32(tS + c * 32, &sr[c * 32]);
            ptx::tmem_wait_ld();
  #pragma unroll
            for (int c = 0; c < BC; ++c) s[c] = __uint_as_float(sr[c]);
            if (w.j0 + j >= j_mask) {
              const RowWindow kw = make_window<kShift>(w.k_start, w.k_end, w.k_start + (w.j0 + j) * BC, BC);
              if (kw.lo != 0 || kw.hi != BC) {
                // Keys outside [lo, hi) of this tile: past the end, or (variable
                // length) before the sequence start / already seen by the previous tile.
  #pragma unroll
                for (int c = 0; c < BC; ++c)
                  if (c < kw.lo || c >= kw.hi) s[c] = -INFINITY;
              }
              const int kbase = kw.load_row - w.k_start;  // sequence index of column 0
              if (CAUSAL && kbase + BC - 1 > first_row_lim) {
                // The tile crosses the diagonal: mask keys above this row's limit.
                const int lim = key_lim - kbase;
  #pragma unroll
                for (int c = 0; c < BC; ++c)
                  if (c > lim) s[c] = -INFINITY;
              }
            }
          };
          // p = 2^(s*c - m*c): one packed FFMA per two scores, then ex2 each;
          // row sum in four packed accumulators (fixed order); P packed as bf16
          // pairs (FP8: e4m3, four per word).
          uint32_t pk[FP8 ? BC / 4 : BC / 2];
          auto exp_range = [&](int c0, int c1, float ng, uint64_t (&acc)[4]) {
            const uint64_t c2x2 = ptx::f2_pack(c2j, c2j);
            const uint64_t negx2 = ptx::f2_pack(ng, ng);
  #pragma unroll
            for (int c = c0; c < c1; c += 2) {
              float x0, x1;
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[c], s[c + 1]), c2x2, negx2), x0, x1);
              const float e0 = ptx::ex2(x0), e1 = ptx::ex2(x1);
              acc[(c >> 1) & 3] = ptx::f2_add(acc[(c >> 1) & 3], ptx::f2_pack(e0, e1));
              if constexpr (FP8) {
                const uint32_t h = ptx::pack_e4m3x2(e0, e1);
                if ((c >> 1) & 1)
                  pk[c >> 2] |= h << 16;
                else
                  pk[c >> 2] = h;
              } else {
                pk[c >> 1] = ptx::pack_bf16x2(e0, e1);
              }
            }
          };
          auto sum_acc = [&](const uint64_t (&acc)[4]) -> float {
            float a0, a1, a2, a3, a4, a5, a6, a7;
            ptx::f2_unpack(acc[0], a0, a1);
            ptx::f2_unpack(acc[1], a2, a3);
            ptx::f2_unpack(acc[2], a4, a5);
            ptx::f2_unpack(acc[3], a6, a7);
            return ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
          };
          auto exponentiate = [&](float ng) -> float {
            uint64_t acc[4] = {0, 0, 0, 0};
            exp_range(0, BC, ng, acc);
            return sum_acc(acc);
          };
          // The reference maximum m only moves when a block maximum exceeds it
          // by more than the threshold T (log2 units); the merge identity of
          // §11.2 holds for any common reference value, so results stay exact.
          // Speculation: exponentiate against the current m first.  A block sum
          // of at most 2^T (1 - 2^-10) bounds every p below 2^T, which is exactly
          // the case where the maximum rule would leave m in place, so the row
          // maximum is needed only when the sum says otherwise (rare once m has
          // settled), or for a row that has seen no key yet.  Either way the
          // result is the one the maximum rule gives.
          float alpha = 1.f, lblk = 0.f;
          bool slow = __all_sync(0xffffffffu, m_ref == -INFINITY);
          const float ng_ref = m_ref == -INFINITY ? 0.f : (FP8 ? -m_ref : -m_ref * c2);
          if (!FP8 && !slow && w.j0 + j < j_mask) {
            // Unmasked tile, speculative path: the second half of the scores
            // is loaded while the first half is exponentiated (the sums keep
            // the order of the single pass, so results are identical).
            // Measured on the page workload: 1.474 -> 1.453 ms; the FP8 form
            // (2 % slower with it) keeps the single load.
            uint32_t sr[BC];
  #pragma unroll
            for (int c = 0; c < BC / 64; ++c) ptx::tmem_ld32(tS + c * 32, &sr[c * 32]);
            ptx::tmem_wait_ld();
  #pragma unroll
            for (int c = BC / 64; c < BC / 32; ++c) ptx::tmem_ld32(tS + c * 32, &sr[c * 32]);
  #pragma unroll
            for (int c = 0; c < BC / 2; ++c) s[c] = __uint_as_float(sr[c]);
            ph.lap(kPhSoftLoad);
            if (tr_lead && t == 0) FA_TRACE(tr_unit, j, kTrSoftLoad0);
            uint64_t acc[4] = {0, 0, 0, 0};
            exp_range(0, BC / 2, ng_ref, acc);
            ptx::tmem_wait_ld();
  #pragma unroll
            for (int c = BC / 2; c < BC; ++c) s[c] = __uint_as_float(sr[c]);
            exp_range(BC / 2, BC, ng_ref, acc);
            lblk = sum_acc(acc);
            slow = __any_sync(0xffffffffu, m_ref == -INFINITY || !(lblk <= accept_sum));
            if (slow) load_scores();  // the scores were consumed
          } else {
            load_scores();
            ph.lap(kPhSoftLoad);
            if (tr_lead && t == 0) FA_TRACE(tr_unit, j, kTrSoftLoad0);
            if (!slow) {
              lblk = exponentiate(ng_ref);
              slow = __any_sync(0xffffffffu, m_ref == -INFINITY || !(lblk <= accept_sum));
              if (slow) load_scores();  // the scores were consumed
            }
          }
          if (slow) {
            ph.count(kPhSoftSlow);
            // Row max: four independent chains of three-input maxima.
            float mx[4] = {s[0], s[1], s[2], s[3]};
  #pragma unroll
            for (int c = 4; c < BC; c += 8) {
              mx[0] = ptx::fmax3(mx[0], s[c], s[c + 1]);
              mx[1] = ptx::fmax3(mx[1], s[c + 2], s[c + 3]);
              if (c + 4 < BC) {
                mx[2] = ptx::fmax3(mx[2], s[c + 4], s[c + 5]);
                mx[3] = ptx::fmax3(mx[3], s[c + 6], s[c + 7]);
              }
            }
            const float bm = fmaxf(ptx::fmax3(mx[0], mx[1], mx[2]), mx[3]);
            float m_new = m_ref, neg;
            if constexpr (FP8) {
              // Maximum compared in scaled log2 units (the coefficient changes per key tile).
              const float bms = bm * c2j;
              if (bms > m_ref && (m_ref == -INFINITY || bms - m_ref > p.rescale_threshold)) m_new = bms;
              alpha = (m_new == m_ref) ? 1.f : ptx::ex2(m_ref - m_new);
              m_ref = m_new;
              neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
            } else {
              if (bm > m_ref && (m_ref == -INFINITY || (bm - m_ref) * c2 > p.rescale_threshold)) m_new = bm;
              alpha = (m_new == m_ref) ? 1.f : ptx::ex2((m_ref - m_new) * c2);
              m_ref = m_new;
              neg = (m_ref == -INFINITY) ? 0.f : -m_ref * c2;
            }
            lblk = exponentiate(neg);
          }
          ph.lap(kPhSoftExp);
          if (tr_lead && t == 0) FA_TRACE(tr_unit, j, kTrSoftExp0);
  #pragma unroll
          for (int c0 = 0; c0 < BC; c0 += 32) {
            if constexpr (FP8)
              ptx::tmem_st8(tP + c0 / 4, &pk[c0 / 4]);
            else
              ptx::tmem_st16(tP + c0 / 2, &pk[c0 / 2]);
          }
          l = l * alpha + lblk;
          if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
            // Correction of the unnormalised output: O_t rows of this warp hold
            // the sum over steps < j referenced to the old maximum.  Done after
            // the exponentials (the scores are dead by then); it only has to
            // land before P(j) is published.
            const uint32_t tO = tmem + lane_off + static_cast<uint32_t>(2 * BC + t * D);
            const uint64_t ax2 = ptx::f2_pack(alpha, alpha);
  #pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              ptx::tmem_ld32(tO + c * 32, r);
              ptx::tmem_wait_ld();
  #pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float x0, x1;
                ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), ax2), x0, x1);
                r[e] = __float_as_uint(x0);
                r[e + 1] = __float_as_uint(x1);
              }
              ptx::tmem_st32(tO + c * 32, r);
            }
          }
          ptx::tmem_wait_st();  // P stores (and any O rescale) have landed
          ptx::tc_fence_before();
          if (tr_lead) FA_TRACE(tr_unit, j, kTrSoftP0 + t);
          if (lane == 0) FA_TRACE(tr_unit, j, kTrSoftWarpP + warp);
          ptx::mbar_arrive(bar(L::kBarPFull + t));
        }
        if (!ok) break;
        ph.lap(kPhSoftWork);
        if (nt == 1 && !(ok = wait_epilogue())) break;
        // Final message for the epilogue: 1 / l, and the row's log-sum-exp.
        const bool has = l > 0.f;
        s_invl[t * kBR + row] = has ? vsc / l : 0.f;
        if (row >= qw.lo && row < qw.hi) {
          const float lse = !has ? -INFINITY
                            : FP8 ? (m_ref + log2f(l)) * 0.69314718055994530942f
                                  : (m_ref * p.scale + log2f(l) * 0.69314718055994530942f);
          const int i_seq = qw.load_row - w.q_start + row;
          if constexpr (SPLIT)
            p.ws_lse[static_cast<size_t>(w.split) * p.B * p.H * p.Nq + w.lse_base + i_seq] = lse;
          else
            p.lse[w.lse_base + i_seq] = lse;
        }
      }
      ptx::mbar_arrive(bar(L::kBarLReady + t));
      ph.lap(kPhSoftFinal);
      sc ^= 0x80000000u;
      ++tr_unit;
    }
    if (lane == 0 && (warp & 3) == 0) ph.store(p.phase, t == 0 ? kPhSoft0 : kPhSoft1);
  } else {
    ptx::setmaxnreg_dec<RegSplit<VARLEN>::kCorrection>();
    // ================================================= correction + epilogue
    const int wq = warp & 3;
    const int row = (wq << 5) + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq << 5) << 16;
    // This warp's 32 output rows are staged here for the TMA store.
    const uint32_t stage = base + L::kOffStage + wq * L::kStageWarpBytes;
    uint32_t uc[kQT] = {0, 0};
    int tr_unit = 0;       // units processed (event trace)
    bool pending = false;  // a TMA store from the staging area may still be reading it
    bool ok = true;
    PhaseClock ph;
    ph.start();
#pragma unroll 1
    FA_FOR_EACH_UNIT(u) {
      const Unit w = decode_unit<BC, VARLEN, CAUSAL, SPLIT, kShift>(p, u);
      if (w.nokeys) {
        // No keys: o = 0 and LSE = -inf (log of an empty sum).
        const int rows = min(kBR * p.qtiles, w.q_end - w.q_row0);
        const size_t rs = static_cast<size_t>(p.H) * D;
        for (int e = threadIdx.x - 256; e < rows * D; e += 128) {
          const int r = e / D, c = e % D;
          p.o[static_cast<size_t>(w.q_row0 + r) * rs + static_cast<size_t>(w.h) * D + c] = __float2bfloat16(0.f);
        }
        for (int r = threadIdx.x - 256; r < rows; r += 128)
          p.lse[w.lse_base + (w.q_row0 - w.q_start) + r] = -INFINITY;
        continue;
      }
#pragma unroll
      for (int t = 0; t < kQT; ++t) {
        if (SPLIT && w.zero[t]) {
          // No visible key in this split: partial o = 0, partial LSE = -inf.
          const RowWindow zw = w.qwin[t];
          const size_t sbase = static_cast<size_t>(w.split) * p.B * p.H * p.Nq + w.lse_base;
          for (int e = threadIdx.x - 256; e < kBR * D; e += 128) {
            const int r = e / D, c = e % D;
            if (r >= zw.lo && r < zw.hi)
              p.ws_o[(sbase + (zw.load_row - w.q_start + r)) * D + c] = 0.f;
          }
          for (int r = threadIdx.x - 256; r < kBR; r += 128)
            if (r >= zw.lo && r < zw.hi) p.ws_lse[sbase + (zw.load_row - w.q_start + r)] = -INFINITY;
        } else if (w.zero[t]) {
          // Causal rows that see no key: o = 0 and LSE = -inf.
          const RowWindow zw = w.qwin[t];
          const size_t rs = static_cast<size_t>(p.H) * D;
          for (int e = threadIdx.x - 256; e < kBR * D; e += 128) {
            const int r = e / D, c = e % D;
            if (r >= zw.lo && r < zw.hi)
              p.o[static_cast<size_t>(zw.load_row + r) * rs + static_cast<size_t>(w.h) * D + c] = __float2bfloat16(0.f);
          }
          for (int r = threadIdx.x - 256; r < kBR; r += 128)
            if (r >= zw.lo && r < zw.hi) p.lse[w.lse_base + (zw.load_row - w.q_start + r)] = -INFINITY;
        }
        if (!w.active[t]) continue;
        ph.lap(kPhEpiStore);
        if (!ptx::mbar_wait_warp(bar(L::kBarLReady + t), uc[t] & 1u, s_abort, tmo) ||
            !ptx::mbar_wait_warp(bar(L::kBarOFinal + t), uc[t] & 1u, s_abort, tmo)) {
          record_error(p.status, kErrTimeout, kSiteCorrFinal);
          ok = false;
          break;
        }
        ph.lap(kPhEpiWait);
        ph.count(kPhEpiTiles);
        if (lane == 0 && warp == 8) FA_TRACE(tr_unit, 0, kTrEpiO0 + t);
        ++uc[t];
        ptx::tc_fence_after();
        const float inv_l = s_invl[t * kBR + row];
        const uint32_t tO = tmem + lane_off + static_cast<uint32_t>(2 * BC + t * D);
        const RowWindow qw = w.qwin[t];
        const bool warp_full = (wq << 5) >= qw.lo && (wq << 5) + 32 <= qw.hi;  // every row of this warp is valid
        const bool use_tma = !SPLIT && (!VARLEN || warp_full);
        const bool row_ok = row >= qw.lo && row < qw.hi;
        // Row pointer for the direct-store path (only formed for valid rows).
        __nv_bfloat16* const grow =
            row_ok ? p.o + (static_cast<size_t>(qw.load_row + row) * p.H + w.h) * D : p.o;
        float* const srow =
            SPLIT && row_ok ? p.ws_o + (static_cast<size_t>(w.split) * p.B * p.H * p.Nq + w.lse_base +
                                        (qw.load_row - w.q_start + row)) * D
                            : nullptr;
        if (use_tma && pending) {
          // The previous store from this warp's staging area must have read it.
          if (lane == 0) ptx::bulk_wait_group_read_0();
          __syncwarp();
          pending = false;
        }
        ph.lap(kPhEpiStage);
        if (lane == 0 && warp == 8) FA_TRACE(tr_unit, 2, kTrEpiO0 + t);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          ptx::tmem_ld32(tO + c * 32, r);
          ptx::tmem_wait_ld();
          if constexpr (SPLIT) {
            // Partial output of this key split, normalised by its own l, in fp32.
            if (row_ok) {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                ptx::st_global_v4(srow + c * 32 + q4 * 4,
                                  __float_as_uint(__uint_as_float(r[4 * q4]) * inv_l),
                                  __float_as_uint(__uint_as_float(r[4 * q4 + 1]) * inv_l),
                                  __float_as_uint(__uint_as_float(r[4 * q4 + 2]) * inv_l),
                                  __float_as_uint(__uint_as_float(r[4 * q4 + 3]) * inv_l));
            }
            continue;
          }
          uint32_t wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            wv[e] = ptx::pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
          if (use_tma) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              // 16-byte chunk (4c + q4) of the row: panel / chunk in panel, swizzled.
              const int c16 = 4 * c + q4;
              const int pnl = c16 / 8, chunk = c16 % 8;
              const uint32_t addr = stage + pnl * 4096 + lane * 128 + ((chunk ^ (lane & 7)) << 4);
              ptx::st_shared_v4(addr, wv[4 * q4], wv[4 * q4 + 1], wv[4 * q4 + 2], wv[4 * q4 + 3]);
            }
          } else if (row_ok) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              ptx::st_global_v4(grow + c * 32 + q4 * 8, wv[4 * q4], wv[4 * q4 + 1], wv[4 * q4 + 2], wv[4 * q4 + 3]);
          }
        }
        // O_t has been read: the next unit's first P V may overwrite it.
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarOEmpty + t));
        ph.lap(kPhEpiRead);
        if (lane == 0 && warp == 8) FA_TRACE(tr_unit, 1, kTrEpiO0 + t);
        if (use_tma) {
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int pnl = 0; pnl < kOutPanels; ++pnl) {
              if constexpr (VARLEN)
                ptx::tma_store_3d(&tm_o, stage + pnl * 4096, pnl * kPanel, w.h, qw.load_row + (wq << 5));
              else
                ptx::tma_store_4d(&tm_o, stage + pnl * 4096, pnl * kPanel, w.h, qw.load_row + (wq << 5), w.b);
            }
            ptx::bulk_commit_group();
          }
          pending = true;
        }
      }
      ++tr_unit;
    }
    if (lane == 0 && pending) ptx::bulk_wait_group_read_0();
    ph.lap(kPhEpiStore);
    if (lane == 0 && warp == 8) ph.store(p.phase, kPhEpi);
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();  // single-lane roles rejoin their warp before the CTA barrier
  ptx::tc_fence_before();
  __syncthreads();
#if FA_PHASE_CLOCKS
  if (threadIdx.x == 0 && p.phase)
    p.phase[static_cast<size_t>(blockIdx.x) * kPhaseWords + kPhTimer + 1] = ptx::globaltimer_ns();
#endif
  if (warp == 12) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
