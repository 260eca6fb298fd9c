// fa_static_scratch.cu -- key-split forward whose scratch lives in a fixed,
// library-owned device array, for callers that cannot allocate device memory.
//
// Who needs it: code that must not call cudaMalloc (or any allocator) at the
// point where attention runs -- for example a runtime that reserves all of its
// device memory at start-up and forbids later allocations, a real-time path
// where an allocation's latency or failure is unacceptable, or plain C callers
// that link only this library and have no memory pool of their own.  fa_fwd_splitkv
// needs a caller-provided workspace; this entry point uses the array below
// instead, so the caller passes only its inputs and outputs.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds its kScratchBytes until the process exits.  All calls on a
// device share it, so calls that overlap on that GPU (two streams, or two host
// threads) race on it and must be serialised by the caller.  Nothing in it
// needs to start at zero: every entry the merge kernel reads is written by the
// same call, so the contents a previous call left behind are never used.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_launch.h"

namespace {

// 16 MiB: B * H * Nq * num_splits * (d + 1) * 4 bytes must fit.
constexpr unsigned long long kScratchBytes = 16ull << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_split_scratch[kScratchBytes / sizeof(float)];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};  // device address of g_split_scratch, per device

// Host code must not pass g_split_scratch itself to a kernel (on the host it
// names a host-side stand-in, not device memory): the device address is looked
// up once per device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_NO_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_split_scratch);
    if (e != cudaSuccess || ptr == nullptr) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                           int Nq, int Nk, int H, int Hk, int d, float scale, int flags,
                           int num_splits, void* stream) {
  // The same argument checks, in the same order, as fa_fwd_splitkv: both
  // entries return the same code for the same arguments.
  const int vrc = fa::check_split_problem(q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, flags);
  if (vrc == 1) return FA_OK;  // nothing to do
  if (vrc != FA_OK) return vrc;
  // The scratch address is the current device's: a stream of another device
  // would run the kernels against memory that is not theirs.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (st != nullptr && st != cudaStreamLegacy && st != cudaStreamPerThread) {
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return FA_ERR_NO_DEVICE;
    if (cudaStreamGetDevice(st, &sdev) != cudaSuccess) return FA_ERR_INVALID_ARG;
    if (sdev != cur) return FA_ERR_INVALID_ARG;
  }
  const int splits = fa_splitkv_num_splits(B, Nq, Nk, H, d, num_splits);
  if (splits < 0) return splits;
  const long long need = fa_splitkv_workspace_bytes(B, Nq, H, d, splits);
  if (need < 0) return static_cast<int>(need);
  if (static_cast<unsigned long long>(need) > kScratchBytes) return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != FA_OK) return rc;
  return fa_fwd_splitkv(q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, flags, splits, scratch,
                        kScratchBytes, stream);
}

}  // extern "C"
