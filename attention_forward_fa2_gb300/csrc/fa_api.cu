// fa_api.cu -- the C ABI declared in include/fa.h: argument validation, TMA
// tensor-map encoding, configuration selection / autotuning, launch and the
// device status word.
//
// The host entry mirrors the one on "Flash Attention实现深度解析" §3.1 (the
// forward returns the output and a per-row log-sum-exp shaped [batch, heads,
// max_seqlen_q]; packed tensors plus cu_seqlens describe variable lengths),
// but the caller owns every buffer: nothing is allocated per call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "fa.h"
#include "fa_launch.h"

namespace {

constexpr int kMaxDevices = 64;

// First device-side error since the last fa_check_status(): code, flat block
// index, warp, wait site.  One copy per device (module global).
__device__ int g_status[4];

thread_local int t_last_cuda_error = 0;

std::mutex g_mu;
unsigned long long g_timeout_ns = 1000000000ull;

// Phase-clock buffer of the instrumented build (FA_PHASE_CLOCKS=1): device
// words, kPhaseWords per CTA; null = not attached.
unsigned long long* g_phase_buf = nullptr;
long long g_phase_words = 0;

// Tile configuration ("Flash Attention 2 Chapter6", Kernel 7 searches B_r, B_c
// and the pipeline depth per shape).
struct Config {
  int bc;           // B_c: keys per K/V tile, 64 or 128
  int qtiles;       // query tiles of 128 rows per work unit: B_r = 128 * qtiles
  int stages;       // K/V ring slots
  float threshold;  // O-rescale threshold, log2 units
  int quad;         // 1: row max / sum over the four threads of a quad (warp shuffles)
};
constexpr Config kSpecBase{128, 2, 4, 8.f, 0};  // fields a spec leaves out
bool g_forced = false;
Config g_forced_cfg = kSpecBase;
std::map<std::tuple<int, int, int>, Config> g_tuned;  // (d, N bucket, varlen) -> config

struct DeviceState {
  bool init = false;
  bool supported = false;
  int* status = nullptr;  // device address of g_status on this device
  int num_sms = 0;
};
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return FA_ERR_CUDA;
}

// Per-device setup, once, with that device current: check the architecture
// and resolve the address of the status word on this device.
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    t_last_cuda_error = static_cast<int>(e);
    return FA_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.init) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    st.supported = (major == 10 && minor == 3);
    if ((e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (st.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_status)) != cudaSuccess) return cuda_fail(e);
      st.status = static_cast<int*>(p);
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cuda_fail(e == cudaSuccess ? cudaErrorNotSupported : e);
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.init = true;
  }
  if (!st.supported) return FA_ERR_UNSUPPORTED;
  *out = &st;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Forward grid.  Packed variable-length batches launch one CTA per work item
// and the running CTAs take over the items of CTAs not yet started (cluster
// launch control: a dynamic schedule for units of unequal work); dense
// problems launch one CTA per SM (at most the item count), each walking the
// items blockIdx.x + k * gridDim.x.
dim3 grid_for(int num_items, bool dynamic, int num_sms) {
  return dim3(static_cast<unsigned>(dynamic || num_items < num_sms ? num_items : num_sms), 1, 1);
}

// Attaches the phase-clock buffer to a forward launch whose grid is set
// (instrumented build only; the default build always leaves it null).
int attach_phase(fa::LaunchArgs& a) {
  a.p.phase = nullptr;
  a.p.trace_off = 0;
#if FA_PHASE_CLOCKS
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_phase_buf != nullptr) {
    const long long need = static_cast<long long>(a.grid.x) * fa::kPhaseWords;
    if (need > g_phase_words) return FA_ERR_INVALID_ARG;
    a.p.phase = g_phase_buf;
    // The event trace of CTA 0 follows the per-CTA words when there is room.
    if (need + fa::kTraceWords <= g_phase_words && need <= 0x7fffffffLL - fa::kTraceWords)
      a.p.trace_off = static_cast<int>(need);
  }
#endif
  return FA_OK;
}

// Tiled tensor map (bf16 with 128-byte swizzle unless told otherwise).
// dims/strides are innermost first; strides are in bytes for dims 1..rank-1.
int encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
           const cuuint64_t* strides, const cuuint32_t* box,
           CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
           CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = static_cast<int>(r);
    return FA_ERR_INVALID_ARG;
  }
  return FA_OK;
}

int n_bucket(int N) {
  int b = 0;
  while ((1 << b) < N && b < 30) ++b;
  return b;
}

Config pick_config(int d, int N, int varlen) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_forced) return g_forced_cfg;
  auto it = g_tuned.find(std::make_tuple(d, n_bucket(N), varlen));
  if (it != g_tuned.end()) return it->second;
  return Config{128, 2, d == 128 ? 2 : 3, 8.f, 0};
}

bool parse_config(const char* spec, Config* out) {
  Config c = kSpecBase;
  std::string s(spec);
  size_t pos = 0;
  while (pos < s.size()) {
    size_t end = s.find(',', pos);
    if (end == std::string::npos) end = s.size();
    std::string item = s.substr(pos, end - pos);
    size_t eq = item.find('=');
    if (eq == std::string::npos) return false;
    std::string key = item.substr(0, eq), val = item.substr(eq + 1);
    char* e = nullptr;
    if (key == "stages") {
      long v = std::strtol(val.c_str(), &e, 10);
      if (val.empty() || *e || v < 2 || v > 4) return false;
      c.stages = static_cast<int>(v);
    } else if (key == "bc") {
      long v = std::strtol(val.c_str(), &e, 10);
      if (val.empty() || *e || (v != 64 && v != 128)) return false;
      c.bc = static_cast<int>(v);
    } else if (key == "br") {
      long v = std::strtol(val.c_str(), &e, 10);
      if (val.empty() || *e || (v != 128 && v != 256)) return false;
      c.qtiles = static_cast<int>(v / 128);
    } else if (key == "reduce") {
      if (val == "thread")
        c.quad = 0;
      else if (val == "quad")
        c.quad = 1;
      else
        return false;
    } else if (key == "threshold") {
      double v = std::strtod(val.c_str(), &e);
      if (*e || !std::isfinite(v) || v < 0 || v > 64) return false;
      c.threshold = static_cast<float>(v);
    } else {
      return false;
    }
    pos = end + 1;
  }
  *out = c;
  return true;
}

// The config a call actually runs.  Each ring slot holds one K tile and one V
// tile: with d = 128 and 128-key tiles only two slots fit next to the query
// tiles.  The causal kernels are built with 128-key tiles only.
// The quad-shuffle form is built for 128-key tiles without mask, with the
// default ring depth only.
Config resolve(Config c, int d, bool causal) {
  if (causal) c.bc = 128;
  if (causal || c.bc != 128) c.quad = 0;
  if (d == 128 && c.bc == 128) c.stages = 2;
  if (c.quad && d == 64) c.stages = 3;
  return c;
}

template <int D, int BC, bool VARLEN, bool CAUSAL>
cudaError_t dispatch_stages(int stages, const fa::LaunchArgs& a) {
  switch (stages) {
    case 2: return fa::launch_fwd<D, BC, 2, VARLEN, CAUSAL>(a);
    case 3: return fa::launch_fwd<D, BC, 3, VARLEN, CAUSAL>(a);
    default: return fa::launch_fwd<D, BC, 4, VARLEN, CAUSAL>(a);
  }
}

// Expects a resolved config.
template <bool VARLEN, bool CAUSAL>
cudaError_t dispatch(int d, const Config& c, const fa::LaunchArgs& a) {
  if constexpr (CAUSAL) {
    if (d == 128) return fa::launch_fwd<128, 128, 2, VARLEN, true>(a);
    return dispatch_stages<64, 128, VARLEN, true>(c.stages, a);
  } else {
    if (c.quad) {
      if (d == 128) return fa::launch_fwd<128, 128, 2, VARLEN, false, true>(a);
      return fa::launch_fwd<64, 128, 3, VARLEN, false, true>(a);
    }
    if (d == 128) {
      if (c.bc == 128) return fa::launch_fwd<128, 128, 2, VARLEN, false>(a);
      return dispatch_stages<128, 64, VARLEN, false>(c.stages, a);
    }
    if (c.bc == 128) return dispatch_stages<64, 128, VARLEN, false>(c.stages, a);
    return dispatch_stages<64, 64, VARLEN, false>(c.stages, a);
  }
}

struct Problem {
  const void *q, *k, *v;
  void* o;
  float* lse;
  int B, Nq, Nk, H, Hk, d;
  float scale;
  const int *cu_q, *cu_k;
  int flags;
  cudaStream_t stream;
};

// Validates a problem; returns FA_OK, a negative error, or 1 for "nothing to do".
int validate(const Problem& P) {
  if (P.B < 0 || P.Nq < 0 || P.Nk < 0 || P.H < 0 || P.Hk < 0) return FA_ERR_INVALID_ARG;
  if ((P.flags & ~FA_FLAG_CAUSAL) != 0) return FA_ERR_INVALID_ARG;
  if (P.H > 0 && (P.Hk == 0 || P.H % P.Hk != 0)) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(P.scale) && P.scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (P.d != 64 && P.d != 128) return FA_ERR_UNSUPPORTED;
  const bool varlen = P.cu_q != nullptr;
  if ((P.cu_q == nullptr) != (P.cu_k == nullptr)) return FA_ERR_INVALID_ARG;
  if (P.B == 0 || P.Nq == 0 || P.H == 0) return 1;
  if (!P.q || !P.k || !P.v || !P.o || !P.lse) return FA_ERR_INVALID_ARG;
  if (!varlen && P.Nk == 0) return FA_ERR_INVALID_ARG;
  if (!aligned16(P.q) || !aligned16(P.k) || !aligned16(P.v) || !aligned16(P.o)) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(P.lse) & 3u) != 0) return FA_ERR_ALIGN;
  if (varlen && ((reinterpret_cast<uintptr_t>(P.cu_q) & 3u) || (reinterpret_cast<uintptr_t>(P.cu_k) & 3u)))
    return FA_ERR_ALIGN;
  // Launch-grid limits (grid.y = H, grid.z = B) and 32-bit index ranges.
  if (P.H > 65535 || P.B > 65535) return FA_ERR_INVALID_ARG;
  const long long rows_q = static_cast<long long>(P.B) * P.Nq;
  const long long rows_k = static_cast<long long>(P.B) * P.Nk;
  if (rows_q > 0x7fffffffLL || rows_k > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(P.B) * P.H * P.Nq > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Encodes the tensor maps and fills the kernel parameters shared by every
// form (grid left to the caller).  Expects a validated, non-empty problem and
// a resolved config.
int prepare(const Problem& P, const Config& cfg, DeviceState* st, fa::LaunchArgs& a) {
  const bool varlen = P.cu_q != nullptr;
  const int D = P.d;
  std::memset(&a, 0, sizeof(a));
  const cuuint64_t esz = 2;
  if (!varlen) {
    cuuint64_t dq[4] = {(cuuint64_t)D, (cuuint64_t)P.H, (cuuint64_t)P.Nq, (cuuint64_t)P.B};
    cuuint64_t sq[3] = {D * esz, (cuuint64_t)P.H * D * esz, (cuuint64_t)P.Nq * P.H * D * esz};
    cuuint64_t dk[4] = {(cuuint64_t)D, (cuuint64_t)P.Hk, (cuuint64_t)P.Nk, (cuuint64_t)P.B};
    cuuint64_t sk[3] = {D * esz, (cuuint64_t)P.Hk * D * esz, (cuuint64_t)P.Nk * P.Hk * D * esz};
    cuuint32_t box_q[4] = {64, 1, (cuuint32_t)fa::kBR, 1};
    cuuint32_t box_k[4] = {64, 1, (cuuint32_t)cfg.bc, 1};
    cuuint32_t box_o[4] = {64, 1, 32, 1};
    int e;
    if ((e = encode(&a.tm_q, P.q, 4, dq, sq, box_q)) != FA_OK) return e;
    if ((e = encode(&a.tm_k, P.k, 4, dk, sk, box_k)) != FA_OK) return e;
    if ((e = encode(&a.tm_v, P.v, 4, dk, sk, box_k)) != FA_OK) return e;
    if ((e = encode(&a.tm_o, P.o, 4, dq, sq, box_o)) != FA_OK) return e;
  } else {
    // Packed rows: the row extent is an upper bound (every length <= the
    // maximum); the kernel never addresses rows at or past a sequence's end.
    cuuint64_t dq[3] = {(cuuint64_t)D, (cuuint64_t)P.H, (cuuint64_t)P.B * P.Nq};
    cuuint64_t dk[3] = {(cuuint64_t)D, (cuuint64_t)P.Hk, (cuuint64_t)(P.B * (long long)P.Nk > 0 ? P.B * (long long)P.Nk : 1)};
    cuuint64_t sr[2] = {D * esz, (cuuint64_t)P.H * D * esz};
    cuuint64_t srk[2] = {D * esz, (cuuint64_t)P.Hk * D * esz};
    cuuint32_t box_q[3] = {64, 1, (cuuint32_t)fa::kBR};
    cuuint32_t box_k[3] = {64, 1, (cuuint32_t)cfg.bc};
    cuuint32_t box_o[3] = {64, 1, 32};
    int e;
    if ((e = encode(&a.tm_q, P.q, 3, dq, sr, box_q)) != FA_OK) return e;
    if ((e = encode(&a.tm_k, P.k, 3, dk, srk, box_k)) != FA_OK) return e;
    if ((e = encode(&a.tm_v, P.v, 3, dk, srk, box_k)) != FA_OK) return e;
    if ((e = encode(&a.tm_o, P.o, 3, dq, sr, box_o)) != FA_OK) return e;
  }
  fa::FwdParams& p = a.p;
  p.B = P.B;
  p.Nq = P.Nq;
  p.Nk = P.Nk;
  p.H = P.H;
  p.group = P.H / P.Hk;
  p.causal = (P.flags & FA_FLAG_CAUSAL) ? 1 : 0;
  p.qtiles = cfg.qtiles;
  p.num_mblocks = (P.Nq + fa::kBR * cfg.qtiles - 1) / (fa::kBR * cfg.qtiles);
  const long long units = static_cast<long long>(P.B) * P.H * p.num_mblocks;
  if (units > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.num_units = static_cast<int>(units);
  p.units_per_item = p.causal ? 2 : 1;
  p.num_items = static_cast<int>((units + p.units_per_item - 1) / p.units_per_item);
  p.cu_q = P.cu_q;
  p.cu_k = P.cu_k;
  p.lse = P.lse;
  p.o = static_cast<__nv_bfloat16*>(P.o);
  p.scale = P.scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(P.scale) * 1.4426950408889634);
  p.rescale_threshold = cfg.threshold;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    p.timeout_ns = g_timeout_ns;
  }
  p.status = st->status;
  p.num_splits = 1;
  p.split_tiles = 0;
  p.total_q = p.total_k = 0x7fffffff;  // packed row counts are not passed to the bf16 forms
  a.stream = P.stream;
  return FA_OK;
}

int run(const Problem& P, const Config& cfg_in) {
  const int rc = validate(P);
  if (rc != FA_OK) return rc == 1 ? FA_OK : rc;
  DeviceState* st = nullptr;
  const int drc = device_state(&st);
  if (drc != FA_OK) return drc;
  const bool varlen = P.cu_q != nullptr;
  const int D = P.d;
  const Config cfg = resolve(cfg_in, D, (P.flags & FA_FLAG_CAUSAL) != 0);
  fa::LaunchArgs a;
  const int prc = prepare(P, cfg, st, a);
  if (prc != FA_OK) return prc;
  fa::FwdParams& p = a.p;
  // Persistent grid: one CTA per SM (each walks items blockIdx.x + k * gridDim.x).
  a.grid = grid_for(p.num_items, varlen, st->num_sms);
  const int arc = attach_phase(a);
  if (arc != FA_OK) return arc;

  cudaError_t e;
  if (p.causal)
    e = varlen ? dispatch<true, true>(D, cfg, a) : dispatch<false, true>(D, cfg, a);
  else
    e = varlen ? dispatch<true, false>(D, cfg, a) : dispatch<false, false>(D, cfg, a);
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

constexpr int kMaxSplits = 128;

// Key tiles per split for a requested number of splits (<= 0: choose one).
// Chooses enough splits to give every SM a unit, at least two key tiles per
// split, at most kMaxSplits.
int split_tiles_for(int B, int Nq, int Nk, int H, int num_sms, int requested) {
  const int nkv = (Nk + fa::kBC - 1) / fa::kBC;
  if (nkv <= 0) return 1;
  int splits = requested;
  if (splits <= 0) {
    const long long units = static_cast<long long>(B) * H * ((Nq + fa::kBR * fa::kQT - 1) / (fa::kBR * fa::kQT));
    splits = units >= num_sms ? 1 : static_cast<int>(num_sms / units);
    splits = std::min(splits, (nkv + 1) / 2);
  }
  splits = std::max(1, std::min(std::min(splits, nkv), kMaxSplits));
  return (nkv + splits - 1) / splits;
}

int splits_for_tiles(int Nk, int tiles) {
  const int nkv = (Nk + fa::kBC - 1) / fa::kBC;
  return nkv <= 0 ? 1 : (nkv + tiles - 1) / tiles;
}

size_t split_workspace_bytes(int B, int Nq, int H, int d, int splits) {
  const size_t rows = static_cast<size_t>(B) * H * Nq;
  return static_cast<size_t>(splits) * rows * (static_cast<size_t>(d) + 1) * sizeof(float);
}

// The key-split form: partial results into ws (fp32, [S, rows, d] then
// [S, rows]), then the combine kernel.  Dense tensors only.
int run_split(const Problem& P, const Config& cfg, int requested_splits, void* ws, size_t ws_bytes) {
  if (P.cu_q != nullptr || P.cu_k != nullptr) return FA_ERR_INVALID_ARG;
  const int rc = validate(P);
  if (rc != FA_OK) return rc == 1 ? FA_OK : rc;
  DeviceState* st = nullptr;
  const int drc = device_state(&st);
  if (drc != FA_OK) return drc;
  const int tiles = split_tiles_for(P.B, P.Nq, P.Nk, P.H, st->num_sms, requested_splits);
  const int splits = splits_for_tiles(P.Nk, tiles);
  const size_t need = split_workspace_bytes(P.B, P.Nq, P.H, P.d, splits);
  if (ws == nullptr || ws_bytes < need || !aligned16(ws)) return FA_ERR_INVALID_ARG;
  // The split kernels use 128-key tiles and 256-row units (the split count
  // above assumes both); only the rescale threshold follows the config.
  Config scfg{128, 2, P.d == 128 ? 2 : 3, cfg.threshold, 0};
  fa::LaunchArgs a;
  const int prc = prepare(P, scfg, st, a);
  if (prc != FA_OK) return prc;
  fa::FwdParams& p = a.p;
  const long long units = static_cast<long long>(p.num_units) * splits;
  if (units > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.num_splits = splits;
  p.split_tiles = tiles;
  p.num_units = static_cast<int>(units);
  p.units_per_item = 1;
  p.num_items = p.num_units;
  const size_t rows = static_cast<size_t>(P.B) * P.H * P.Nq;
  p.ws_o = static_cast<float*>(ws);
  p.ws_lse = p.ws_o + static_cast<size_t>(splits) * rows * P.d;
  a.grid = grid_for(p.num_items, false, st->num_sms);
  const int arc = attach_phase(a);
  if (arc != FA_OK) return arc;
  cudaError_t e;
  if (P.d == 128)
    e = p.causal ? fa::launch_fwd_split<128, 2, true>(a) : fa::launch_fwd_split<128, 2, false>(a);
  else
    e = p.causal ? fa::launch_fwd_split<64, 3, true>(a) : fa::launch_fwd_split<64, 3, false>(a);
  if (e != cudaSuccess) return cuda_fail(e);
  e = fa::launch_combine(P.d, p.ws_o, p.ws_lse, splits, static_cast<long long>(rows), P.H, P.Nq,
                         static_cast<__nv_bfloat16*>(P.o), P.lse, P.stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

// ---------------------------------------------------------------- backward
int bwd_nq_pad(int Nq) { return (Nq + fa::kBwdBQ - 1) / fa::kBwdBQ * fa::kBwdBQ; }

// Workspace: dq_acc fp32 [B, H, nq_pad, d], then lse2 and delta fp32 [B, H, nq_pad].
size_t bwd_workspace_bytes(int B, int Nq, int H, int d) {
  const size_t rows = static_cast<size_t>(B) * H * bwd_nq_pad(Nq);
  return rows * (static_cast<size_t>(d) + 2) * sizeof(float);
}

struct BwdProblem {
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  const int *cu_q, *cu_k;  // variable-length form (both or neither)
  int B, Nq, Nk, H, Hk, d;
  float scale;
  int flags;
  void* ws;
  long long ws_bytes;
  cudaStream_t stream;
};

int run_bwd(const BwdProblem& P) {
  if (P.B < 0 || P.Nq < 0 || P.Nk < 0 || P.H < 0 || P.Hk < 0) return FA_ERR_INVALID_ARG;
  if ((P.flags & ~FA_FLAG_CAUSAL) != 0) return FA_ERR_INVALID_ARG;
  if (P.H > 0 && (P.Hk == 0 || P.H % P.Hk != 0)) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(P.scale) && P.scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (P.d != 64 && P.d != 128) return FA_ERR_UNSUPPORTED;
  const bool varlen = P.cu_q != nullptr;
  if ((P.cu_q == nullptr) != (P.cu_k == nullptr)) return FA_ERR_INVALID_ARG;
  if (varlen && ((reinterpret_cast<uintptr_t>(P.cu_q) & 3u) || (reinterpret_cast<uintptr_t>(P.cu_k) & 3u)))
    return FA_ERR_ALIGN;
  if (P.B == 0 || P.H == 0) return FA_OK;
  // Dense queries need keys (as the forward); packed sequences without keys
  // are allowed and get dQ = 0.
  if (!varlen && P.Nk == 0) return P.Nq == 0 ? FA_OK : FA_ERR_INVALID_ARG;
  if (varlen && P.Nq == 0 && P.Nk == 0) return FA_OK;
  if (!P.k || !P.v || !P.dk || !P.dv || !P.ws) return FA_ERR_INVALID_ARG;
  if (P.Nq > 0 && (!P.q || !P.o || !P.dout || !P.lse || !P.dq)) return FA_ERR_INVALID_ARG;
  for (const void* ptr : {P.q, P.k, P.v, P.o, P.dout, static_cast<const void*>(P.dq), static_cast<const void*>(P.dk),
                          static_cast<const void*>(P.dv), static_cast<const void*>(P.ws)})
    if (ptr && !aligned16(ptr)) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(P.lse) & 3u) != 0) return FA_ERR_ALIGN;
  if (P.H > 65535 || P.B > 65535) return FA_ERR_INVALID_ARG;
  const long long rows_pad = static_cast<long long>(P.B) * P.H * bwd_nq_pad(P.Nq);
  if (rows_pad > 0x7fffffffLL || static_cast<long long>(P.B) * P.Nk > 0x7fffffffLL ||
      static_cast<long long>(P.B) * P.Nq > 0x7fffffffLL)
    return FA_ERR_INVALID_ARG;
  if (P.ws_bytes < 0 || static_cast<size_t>(P.ws_bytes) < bwd_workspace_bytes(P.B, P.Nq, P.H, P.d))
    return FA_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  const int drc = device_state(&st);
  if (drc != FA_OK) return drc;

  const int D = P.d;
  const cuuint64_t esz = 2;
  fa::BwdLaunchArgs a;
  std::memset(&a, 0, sizeof(a));
  fa::BwdParams& p = a.p;
  p.B = P.B;
  p.Nq = P.Nq;
  p.Nk = P.Nk;
  p.H = P.H;
  p.Hk = P.Hk;
  p.group = P.H / P.Hk;
  p.causal = (P.flags & FA_FLAG_CAUSAL) ? 1 : 0;
  p.nq_pad = bwd_nq_pad(P.Nq);
  p.num_kb = (P.Nk + fa::kBwdBK - 1) / fa::kBwdBK;
  const long long units = static_cast<long long>(P.B) * P.Hk * p.num_kb;
  if (units > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.num_units = static_cast<int>(units);
  p.units_per_item = p.causal ? 2 : 1;
  p.num_items = (p.num_units + p.units_per_item - 1) / p.units_per_item;
  p.o = static_cast<const __nv_bfloat16*>(P.o);
  p.dout = static_cast<const __nv_bfloat16*>(P.dout);
  p.lse = P.lse;
  p.dq_acc = static_cast<float*>(P.ws);
  p.lse2 = p.dq_acc + static_cast<size_t>(rows_pad) * D;
  p.delta = p.lse2 + rows_pad;
  p.dq = static_cast<__nv_bfloat16*>(P.dq);
  p.dk = static_cast<__nv_bfloat16*>(P.dk);
  p.dv = static_cast<__nv_bfloat16*>(P.dv);
  p.scale = P.scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(P.scale) * 1.4426950408889634);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    p.timeout_ns = g_timeout_ns;
  }
  p.status = st->status;

  // Query-side maps: at least one row even when Nq = 0 (the kernel then loads
  // nothing; the map only has to be valid).
  const void* qptr = P.Nq > 0 ? P.q : P.k;
  const void* doptr = P.Nq > 0 ? P.dout : P.k;
  const int nq_map = P.Nq > 0 ? P.Nq : 1;
  const int nk_map = P.Nk > 0 ? P.Nk : 1;
  const void* kptr = P.Nk > 0 ? P.k : qptr;
  const void* vptr = P.Nk > 0 ? P.v : qptr;
  const int hq_map = P.Nq > 0 ? P.H : P.Hk;
  const int hk_map = P.Nk > 0 ? P.Hk : hq_map;
  int e;
  if (!varlen) {
    cuuint64_t dq4[4] = {(cuuint64_t)D, (cuuint64_t)hq_map, (cuuint64_t)nq_map, (cuuint64_t)P.B};
    cuuint64_t sq4[3] = {D * esz, (cuuint64_t)hq_map * D * esz, (cuuint64_t)nq_map * hq_map * D * esz};
    cuuint64_t dk4[4] = {(cuuint64_t)D, (cuuint64_t)hk_map, (cuuint64_t)nk_map, (cuuint64_t)P.B};
    cuuint64_t sk4[3] = {D * esz, (cuuint64_t)hk_map * D * esz, (cuuint64_t)nk_map * hk_map * D * esz};
    cuuint32_t box_q[4] = {64, 1, (cuuint32_t)fa::kBwdBQ, 1};
    cuuint32_t box_k[4] = {64, 1, (cuuint32_t)fa::kBwdBK, 1};
    if ((e = encode(&a.tm_q, qptr, 4, dq4, sq4, box_q)) != FA_OK) return e;
    if ((e = encode(&a.tm_do, doptr, 4, dq4, sq4, box_q)) != FA_OK) return e;
    if ((e = encode(&a.tm_k, kptr, 4, dk4, sk4, box_k)) != FA_OK) return e;
    if ((e = encode(&a.tm_v, vptr, 4, dk4, sk4, box_k)) != FA_OK) return e;
  } else {
    // Packed rows; the row extent is an upper bound (every length is at most
    // the maximum), and the kernel never addresses a row past its sequence's
    // end (a sequence's last tile is shifted back instead).
    cuuint64_t dq3[3] = {(cuuint64_t)D, (cuuint64_t)hq_map, (cuuint64_t)P.B * nq_map};
    cuuint64_t sq3[2] = {D * esz, (cuuint64_t)hq_map * D * esz};
    cuuint64_t dk3[3] = {(cuuint64_t)D, (cuuint64_t)hk_map, (cuuint64_t)P.B * nk_map};
    cuuint64_t sk3[2] = {D * esz, (cuuint64_t)hk_map * D * esz};
    cuuint32_t box_q[3] = {64, 1, (cuuint32_t)fa::kBwdBQ};
    cuuint32_t box_k[3] = {64, 1, (cuuint32_t)fa::kBwdBK};
    if ((e = encode(&a.tm_q, qptr, 3, dq3, sq3, box_q)) != FA_OK) return e;
    if ((e = encode(&a.tm_do, doptr, 3, dq3, sq3, box_q)) != FA_OK) return e;
    if ((e = encode(&a.tm_k, kptr, 3, dk3, sk3, box_k)) != FA_OK) return e;
    if ((e = encode(&a.tm_v, vptr, 3, dk3, sk3, box_k)) != FA_OK) return e;
  }
  p.cu_q = P.cu_q;
  p.cu_k = P.cu_k;
  a.grid = dim3(static_cast<unsigned>(p.num_items < st->num_sms ? p.num_items : st->num_sms), 1, 1);
  a.stream = P.stream;
  cudaError_t ce;
  if (D == 128)
    ce = varlen ? (p.causal ? fa::launch_bwd<128, true, true>(a) : fa::launch_bwd<128, false, true>(a))
                : (p.causal ? fa::launch_bwd<128, true, false>(a) : fa::launch_bwd<128, false, false>(a));
  else
    ce = varlen ? (p.causal ? fa::launch_bwd<64, true, true>(a) : fa::launch_bwd<64, false, true>(a))
                : (p.causal ? fa::launch_bwd<64, true, false>(a) : fa::launch_bwd<64, false, false>(a));
  if (ce != cudaSuccess) return cuda_fail(ce);
  return FA_OK;
}

// ------------------------------------------------------------------ FP8
int fp8_nk_pad(int Nk) { return (Nk + 15) / 16 * 16; }

int fp8_check_shape(int B, int Nq, int Nk, int H, int Hk, int d) {
  if (B < 0 || Nq < 0 || Nk < 0 || H < 0 || Hk < 0) return FA_ERR_INVALID_ARG;
  if (H > 0 && (Hk == 0 || H % Hk != 0)) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Nq * H > 0x7fffffffLL || static_cast<long long>(B) * Nk * Hk > 0x7fffffffLL)
    return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Variable-length FP8: columns of the transposed V codes (the start column of
// a sequence b = B past the last one).
long long fp8_vt_cols(int B, int total_k) { return fa::fp8_vt_col0(total_k, B); }

int fp8_check_varlen(int B, int total_q, int total_k, int max_q, int max_k, int H, int Hk, int d) {
  const int rc = fp8_check_shape(B, max_q, max_k, H, Hk, d);
  if (rc != FA_OK) return rc;
  if (total_q < 0 || total_k < 0) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(total_q) * H > 0x7fffffffLL || static_cast<long long>(total_k) * Hk > 0x7fffffffLL)
    return FA_ERR_INVALID_ARG;
  if (fp8_vt_cols(B, total_k) > 0x7fffffffLL - 256) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

bool misaligned4(const void* a, const void* b, const void* c) {
  return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(c)) & 3u) != 0;
}

__global__ void wait_timeout_kernel(unsigned long long timeout_ns, int* status) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  const uint32_t b = fa::ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::ptx::mbar_init(b, 1);
    fa::ptx::fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the wait must give up after timeout_ns.
  if (threadIdx.x == 0) {
    if (!fa::ptx::mbar_wait(b, 0, &abort_flag, timeout_ns)) fa::record_error(status, fa::kErrTimeout, 99);
  }
  __syncthreads();
}

}  // namespace

namespace fa {
// Argument check of the key-split form, shared with the allocation-free entry
// so that both return the same code for the same arguments.
int check_split_problem(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Nq,
                        int Nk, int H, int Hk, int d, float scale, int flags) {
  Problem P{q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, nullptr, nullptr, flags, nullptr};
  return validate(P);
}
}  // namespace fa

extern "C" {

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Nq,
              int Nk, int H, int Hk, int d, float scale, const int* cu_seqlens_q,
              const int* cu_seqlens_k, int flags, void* stream) {
  Problem P{q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, cu_seqlens_q, cu_seqlens_k, flags,
            static_cast<cudaStream_t>(stream)};
  return run(P, pick_config(d, Nk, cu_seqlens_q != nullptr));
}

int fa_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Nq,
              int Nk, int H, int d, float scale, const int* cu_seqlens_q,
              const int* cu_seqlens_k, void* stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, Nq, Nk, H, H, d, scale, cu_seqlens_q, cu_seqlens_k, 0, stream);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int N, int H,
           int d, float scale, const int* cu_seqlens, void* stream) {
  return fa_fwd_qk(q, k, v, o, lse, B, N, N, H, d, scale, cu_seqlens, cu_seqlens, stream);
}

int fa_check_status(void* stream, int* info) {
  DeviceState* st = nullptr;
  const int drc = device_state(&st);
  if (drc != FA_OK) return drc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int h[4] = {0, 0, 0, 0};
  if ((e = cudaMemcpy(h, st->status, sizeof(h), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  const int zero[4] = {0, 0, 0, 0};
  if ((e = cudaMemcpy(st->status, zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess) return cuda_fail(e);
  if (info) {
    info[0] = h[1];
    info[1] = h[2];
    info[2] = h[3];
  }
  return h[0];
}

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or device (needs d in {64,128} and sm_103)";
    case FA_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA error (see fa_last_cuda_error)";
    case FA_ERR_TIMEOUT: return "device-side wait timed out";
    case FA_ERR_NO_DEVICE: return "no CUDA device";
    case FA_ERR_BAD_SEQLENS: return "cu_seqlens inconsistent with the maximum sequence length";
    case FA_ERR_SCRATCH_LIMIT: return "problem needs more than the library's fixed 16 MiB scratch";
    default: return "unknown error";
  }
}

int fa_last_cuda_error(void) { return t_last_cuda_error; }

int fa_set_timeout_ns(unsigned long long ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timeout_ns = ns == 0 ? 1000000000ull : ns;
  return FA_OK;
}

int fa_set_config(const char* spec) {
  if (spec == nullptr || spec[0] == '\0') {
    std::lock_guard<std::mutex> lk(g_mu);
    g_forced = false;
    return FA_OK;
  }
  Config c;
  if (!parse_config(spec, &c)) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_forced = true;
  g_forced_cfg = c;
  return FA_OK;
}

int fa_get_config(int d, int N, int varlen, char* buf, int len) {
  if (!buf || len <= 0) return FA_ERR_INVALID_ARG;
  const Config c = resolve(pick_config(d, N, varlen ? 1 : 0), d, false);
  std::snprintf(buf, static_cast<size_t>(len), "br=%d,bc=%d,stages=%d,threshold=%g,reduce=%s",
                128 * c.qtiles, c.bc, c.stages, c.threshold, c.quad ? "quad" : "thread");
  return FA_OK;
}

int fa_autotune(const void* q, const void* k, const void* v, void* o, float* lse, int B, int N,
                int H, int d, float scale, const int* cu_seqlens, void* stream) {
  Problem P{q, k, v, o, lse, B, N, N, H, H, d, scale, cu_seqlens, cu_seqlens, 0,
            static_cast<cudaStream_t>(stream)};
  const int rc = validate(P);
  if (rc != FA_OK) return rc == 1 ? FA_OK : rc;
  cudaEvent_t e0, e1;
  cudaError_t ce;
  if ((ce = cudaEventCreate(&e0)) != cudaSuccess) return cuda_fail(ce);
  if ((ce = cudaEventCreate(&e1)) != cudaSuccess) {
    cudaEventDestroy(e0);
    return cuda_fail(ce);
  }
  // The search space: B_r in {256, 128}, B_c in {128, 64}, every ring depth
  // that fits, rescale threshold 8 or 0 (rescale whenever the max grows), and
  // the row reduction (one thread per row, or a quad of threads with warp
  // shuffles; the latter built for 128-key tiles at the default depth).
  // Configs that do not fit shared memory or tensor memory are never built.
  Config cands[52];
  int n_cands = 0;
  for (int qt = 2; qt >= 1; --qt)
    for (int bc = 128; bc >= 64; bc /= 2)
      for (int st = 2; st <= 4; ++st) {
        if (d == 128 && bc == 128 && st > 2) continue;
        for (float th : {8.f, 0.f}) cands[n_cands++] = Config{bc, qt, st, th, 0};
      }
  for (float th : {8.f, 0.f}) cands[n_cands++] = Config{128, 2, d == 128 ? 2 : 3, th, 1};
  Config best = pick_config(d, N, cu_seqlens ? 1 : 0);
  float best_ms = 1e30f;
  int result = FA_OK;
  for (int ci = 0; ci < n_cands; ++ci) {
    const Config& c = cands[ci];
    int r = run(P, c);  // warm-up
    if (r != FA_OK) { result = r; break; }
    float ms_min = 1e30f;
    for (int rep = 0; rep < 3; ++rep) {
      cudaEventRecord(e0, P.stream);
      r = run(P, c);
      cudaEventRecord(e1, P.stream);
      if (r != FA_OK) break;
      if ((ce = cudaEventSynchronize(e1)) != cudaSuccess) { r = cuda_fail(ce); break; }
      float ms = 0.f;
      cudaEventElapsedTime(&ms, e0, e1);
      if (ms < ms_min) ms_min = ms;
    }
    if (r != FA_OK) { result = r; break; }
    if (ms_min < best_ms) {
      best_ms = ms_min;
      best = c;
    }
  }
  if (result == FA_OK) {
    {
      std::lock_guard<std::mutex> lk(g_mu);
      g_tuned[std::make_tuple(d, n_bucket(N), cu_seqlens ? 1 : 0)] = best;
    }
    result = run(P, best);
    if (result == FA_OK && (ce = cudaStreamSynchronize(P.stream)) != cudaSuccess) result = cuda_fail(ce);
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return result;
}

int fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  const int drc = device_state(&st);
  if (drc != FA_OK) return drc;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns, st->status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return FA_OK;
}

long long fa_bwd_workspace_bytes(int B, int Nq, int H, int d) {
  if (B < 0 || Nq < 0 || H < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return static_cast<long long>(bwd_workspace_bytes(B, Nq, H, d));
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, int B, int Nq, int Nk, int H, int Hk, int d, float scale, int flags,
           void* workspace, long long workspace_bytes, void* stream) {
  BwdProblem P{q, k, v, o, dout, lse, dq, dk, dv, nullptr, nullptr, B, Nq, Nk, H, Hk, d, scale, flags, workspace,
               workspace_bytes, static_cast<cudaStream_t>(stream)};
  return run_bwd(P);
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                  int max_seqlen_q, int max_seqlen_k, int H, int Hk, int d, float scale, int flags,
                  void* workspace, long long workspace_bytes, void* stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  BwdProblem P{q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B, max_seqlen_q, max_seqlen_k,
               H, Hk, d, scale, flags, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  return run_bwd(P);
}

int fa_fp8_sizes(int B, int Nq, int Nk, int H, int Hk, int d, long long* sizes) {
  if (!sizes) return FA_ERR_INVALID_ARG;
  const int rc = fp8_check_shape(B, Nq, Nk, H, Hk, d);
  if (rc != FA_OK) return rc;
  const long long qb = (Nq + fa::kBR - 1) / fa::kBR, kb = (Nk + fa::kBR - 1) / fa::kBR;
  sizes[0] = static_cast<long long>(B) * Nq * H * d;
  sizes[1] = static_cast<long long>(B) * Nk * Hk * d;
  sizes[2] = static_cast<long long>(B) * Hk * d * fp8_nk_pad(Nk);
  sizes[3] = static_cast<long long>(B) * H * qb;
  sizes[4] = static_cast<long long>(B) * Hk * kb;
  sizes[5] = static_cast<long long>(B) * Hk;
  return FA_OK;
}

int fa_quantize_fp8(const void* q, const void* k, const void* v, int B, int Nq, int Nk, int H, int Hk, int d,
                    void* q8, void* k8, void* vt8, float* q_scale, float* k_scale, float* v_scale, void* stream) {
  int rc = fp8_check_shape(B, Nq, Nk, H, Hk, d);
  if (rc != FA_OK) return rc;
  if (B == 0 || H == 0 || (Nq == 0 && Nk == 0)) return FA_OK;
  if ((Nq > 0 && (!q || !q8 || !q_scale)) || (Nk > 0 && (!k || !v || !k8 || !vt8 || !k_scale)) || !v_scale)
    return FA_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, static_cast<const void*>(q8), static_cast<const void*>(k8), static_cast<const void*>(vt8)})
    if (ptr && !aligned16(ptr)) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return FA_ERR_ALIGN;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != FA_OK) return rc;
  fa::Fp8QuantParams p{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                       static_cast<const __nv_bfloat16*>(v), static_cast<uint8_t*>(q8), static_cast<uint8_t*>(k8),
                       static_cast<uint8_t*>(vt8), q_scale, k_scale, v_scale, B, Nq, Nk, H, Hk, d, fp8_nk_pad(Nk),
                       nullptr, nullptr, 0, 0, 0};
  const cudaError_t e = fa::launch_fp8_quantize(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int Nq, int Nk, int H, int Hk, int d, float scale,
               int flags, void* stream) {
  int rc = fp8_check_shape(B, Nq, Nk, H, Hk, d);
  if (rc != FA_OK) return rc;
  Problem P{q8, k8, vt8, o, lse, B, Nq, Nk, H, Hk, d, scale, nullptr, nullptr, flags,
            static_cast<cudaStream_t>(stream)};
  rc = validate(P);
  if (rc != FA_OK) return rc == 1 ? FA_OK : rc;
  if (!q_scale || !k_scale || !v_scale) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return FA_ERR_ALIGN;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != FA_OK) return rc;
  fa::LaunchArgs a;
  // Parameters and the bf16 output map as for the bf16 forward (128-key
  // tiles, 256-row units), then the e4m3 input maps.
  const Config cfg{128, 2, 2, 8.f, 0};
  if ((rc = prepare(P, cfg, st, a)) != FA_OK) return rc;
  const int nkp = fp8_nk_pad(Nk);
  cuuint64_t dq[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)Nq, (cuuint64_t)B};
  cuuint64_t sq[3] = {(cuuint64_t)d, (cuuint64_t)H * d, (cuuint64_t)Nq * H * d};
  cuuint64_t dk[4] = {(cuuint64_t)d, (cuuint64_t)Hk, (cuuint64_t)Nk, (cuuint64_t)B};
  cuuint64_t sk[3] = {(cuuint64_t)d, (cuuint64_t)Hk * d, (cuuint64_t)Nk * Hk * d};
  cuuint64_t dv[4] = {(cuuint64_t)nkp, (cuuint64_t)d, (cuuint64_t)Hk, (cuuint64_t)B};
  cuuint64_t sv[3] = {(cuuint64_t)nkp, (cuuint64_t)d * nkp, (cuuint64_t)Hk * d * nkp};
  cuuint32_t box_q[4] = {128, 1, (cuuint32_t)fa::kBR, 1};
  cuuint32_t box_k[4] = {128, 1, (cuuint32_t)fa::kBC, 1};
  cuuint32_t box_v[4] = {(cuuint32_t)fa::kBC, 128, 1, 1};
  if ((rc = encode(&a.tm_q, q8, 4, dq, sq, box_q, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != FA_OK) return rc;
  if ((rc = encode(&a.tm_k, k8, 4, dk, sk, box_k, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != FA_OK) return rc;
  if ((rc = encode(&a.tm_v, vt8, 4, dv, sv, box_v, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != FA_OK) return rc;
  a.p.q_scale = q_scale;
  a.p.k_scale = k_scale;
  a.p.v_scale = v_scale;
  a.p.q_blocks = (Nq + fa::kBR - 1) / fa::kBR;
  a.p.k_blocks = (Nk + fa::kBR - 1) / fa::kBR;
  a.grid = grid_for(a.p.num_items, false, st->num_sms);
  if ((rc = attach_phase(a)) != FA_OK) return rc;
  const cudaError_t e = fa::launch_fwd_fp8((flags & FA_FLAG_CAUSAL) != 0, a);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_fp8_varlen_sizes(int B, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H, int Hk,
                        int d, long long* sizes) {
  if (!sizes) return FA_ERR_INVALID_ARG;
  const int rc = fp8_check_varlen(B, total_q, total_k, max_seqlen_q, max_seqlen_k, H, Hk, d);
  if (rc != FA_OK) return rc;
  const long long qb = (max_seqlen_q + fa::kBR - 1) / fa::kBR, kb = (max_seqlen_k + fa::kBR - 1) / fa::kBR;
  sizes[0] = static_cast<long long>(total_q) * H * d;
  sizes[1] = static_cast<long long>(total_k) * Hk * d;
  sizes[2] = static_cast<long long>(Hk) * d * fp8_vt_cols(B, total_k);
  sizes[3] = static_cast<long long>(B) * H * qb;
  sizes[4] = static_cast<long long>(B) * Hk * kb;
  sizes[5] = static_cast<long long>(B) * Hk;
  return FA_OK;
}

int fa_quantize_fp8_varlen(const void* q, const void* k, const void* v, const int* cu_seqlens_q,
                           const int* cu_seqlens_k, int B, int total_q, int total_k, int max_seqlen_q,
                           int max_seqlen_k, int H, int Hk, int d, void* q8, void* k8, void* vt8, float* q_scale,
                           float* k_scale, float* v_scale, void* stream) {
  int rc = fp8_check_varlen(B, total_q, total_k, max_seqlen_q, max_seqlen_k, H, Hk, d);
  if (rc != FA_OK) return rc;
  if (B == 0 || H == 0) return FA_OK;
  if (!cu_seqlens_q || !cu_seqlens_k || !vt8 || !v_scale) return FA_ERR_INVALID_ARG;
  if ((total_q > 0 && (!q || !q8)) || (max_seqlen_q > 0 && !q_scale) || (total_k > 0 && (!k || !v || !k8)) ||
      (max_seqlen_k > 0 && !k_scale))
    return FA_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, static_cast<const void*>(q8), static_cast<const void*>(k8), static_cast<const void*>(vt8)})
    if (ptr && !aligned16(ptr)) return FA_ERR_ALIGN;
  if (misaligned4(q_scale, k_scale, v_scale) || misaligned4(cu_seqlens_q, cu_seqlens_k, nullptr)) return FA_ERR_ALIGN;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != FA_OK) return rc;
  fa::Fp8QuantParams p{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                       static_cast<const __nv_bfloat16*>(v), static_cast<uint8_t*>(q8), static_cast<uint8_t*>(k8),
                       static_cast<uint8_t*>(vt8), q_scale, k_scale, v_scale, B, max_seqlen_q, max_seqlen_k, H, Hk,
                       d, 0, cu_seqlens_q, cu_seqlens_k, total_q, total_k, fp8_vt_cols(B, total_k)};
  const cudaError_t e = fa::launch_fp8_quantize(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_fwd_fp8_varlen(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
                      const float* v_scale, void* o, float* lse, const int* cu_seqlens_q, const int* cu_seqlens_k,
                      int B, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H, int Hk, int d,
                      float scale, int flags, void* stream) {
  int rc = fp8_check_varlen(B, total_q, total_k, max_seqlen_q, max_seqlen_k, H, Hk, d);
  if (rc != FA_OK) return rc;
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  Problem P{q8, k8, vt8, o, lse, B, max_seqlen_q, max_seqlen_k, H, Hk, d, scale, cu_seqlens_q, cu_seqlens_k, flags,
            static_cast<cudaStream_t>(stream)};
  rc = validate(P);
  if (rc != FA_OK) return rc == 1 ? FA_OK : rc;
  if (total_q == 0) return FA_OK;  // no query rows
  if (!q_scale || !k_scale || !v_scale) return FA_ERR_INVALID_ARG;
  if (misaligned4(q_scale, k_scale, v_scale)) return FA_ERR_ALIGN;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != FA_OK) return rc;
  fa::LaunchArgs a;
  const Config cfg{128, 2, 2, 8.f, 0};
  if ((rc = prepare(P, cfg, st, a)) != FA_OK) return rc;
  // e4m3 maps over the packed rows (exact extents: a tile that runs past the
  // last sequence reads the TMA zero fill) and over the V^T columns.
  const long long kp = fp8_vt_cols(B, total_k);
  const cuuint64_t tk = total_k > 0 ? (cuuint64_t)total_k : 1;  // no key is read when total_k == 0
  cuuint64_t dq[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)total_q};
  cuuint64_t sq[2] = {(cuuint64_t)d, (cuuint64_t)H * d};
  cuuint64_t dk[3] = {(cuuint64_t)d, (cuuint64_t)Hk, tk};
  cuuint64_t sk[2] = {(cuuint64_t)d, (cuuint64_t)Hk * d};
  cuuint64_t dv[3] = {(cuuint64_t)kp, (cuuint64_t)d, (cuuint64_t)Hk};
  cuuint64_t sv[2] = {(cuuint64_t)kp, (cuuint64_t)d * kp};
  cuuint32_t box_q[3] = {128, 1, (cuuint32_t)fa::kBR};
  cuuint32_t box_k[3] = {128, 1, (cuuint32_t)fa::kBC};
  cuuint32_t box_v[3] = {(cuuint32_t)fa::kBC, 128, 1};
  if ((rc = encode(&a.tm_q, q8, 3, dq, sq, box_q, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != FA_OK) return rc;
  if ((rc = encode(&a.tm_k, k8, 3, dk, sk, box_k, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != FA_OK) return rc;
  if ((rc = encode(&a.tm_v, vt8, 3, dv, sv, box_v, CU_TENSOR_MAP_DATA_TYPE_UINT8)) != FA_OK) return rc;
  a.p.q_scale = q_scale;
  a.p.k_scale = k_scale;
  a.p.v_scale = v_scale;
  a.p.q_blocks = (max_seqlen_q + fa::kBR - 1) / fa::kBR;
  a.p.k_blocks = (max_seqlen_k + fa::kBR - 1) / fa::kBR;
  a.p.total_q = total_q;
  a.p.total_k = total_k;
  a.grid = grid_for(a.p.num_items, true, st->num_sms);
  const int arc = attach_phase(a);
  if (arc != FA_OK) return arc;
  const cudaError_t e = fa::launch_fwd_fp8_varlen((flags & FA_FLAG_CAUSAL) != 0, a);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

int fa_splitkv_num_splits(int B, int Nq, int Nk, int H, int d, int requested) {
  if (B < 0 || Nq < 0 || Nk < 0 || H < 0 || (d != 64 && d != 128)) return FA_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  const int drc = device_state(&st);
  if (drc != FA_OK) return drc;
  return splits_for_tiles(Nk, split_tiles_for(B, Nq, Nk, H, st->num_sms, requested));
}

long long fa_splitkv_workspace_bytes(int B, int Nq, int H, int d, int num_splits) {
  if (B < 0 || Nq < 0 || H < 0 || (d != 64 && d != 128) || num_splits < 1 || num_splits > kMaxSplits)
    return FA_ERR_INVALID_ARG;
  return static_cast<long long>(split_workspace_bytes(B, Nq, H, d, num_splits));
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Nq,
                   int Nk, int H, int Hk, int d, float scale, int flags, int num_splits,
                   void* workspace, unsigned long long workspace_bytes, void* stream) {
  Problem P{q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, nullptr, nullptr, flags,
            static_cast<cudaStream_t>(stream)};
  return run_split(P, pick_config(d, Nk, 0), num_splits, workspace, static_cast<size_t>(workspace_bytes));
}

int fa_set_phase_buffer(unsigned long long* buf, long long words) {
#if FA_PHASE_CLOCKS
  if (buf != nullptr && (words < fa::kPhaseWords || (reinterpret_cast<uintptr_t>(buf) & 7u) != 0))
    return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_phase_buf = buf;
  g_phase_words = buf ? words : 0;
  return fa::kPhaseWords;
#else
  (void)buf;
  (void)words;
  return FA_ERR_UNSUPPORTED;
#endif
}

int fa_version(void) { return 100; }

}  // extern "C"
