// mla_decode_noalloc: the rebuilt-cache decode step without a caller-supplied
// workspace, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running under a host framework
// that owns all device memory and allows no allocation of its own (plugins of
// inference servers, runtimes with a fixed memory budget), or latency-critical
// loops that cannot afford the implicit device synchronisation an allocation
// may cause.  This entry point gives them the decode step with its scratch
// (intermediate activations, split-KV partials, the status word) in a
// file-scope device array of fixed size instead of a workspace argument.
//
// The array is a static __device__ variable of this library: every GPU that
// loads the library holds its kNoAllocScratchBytes until the process exits.
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress once per device (the first
// call on each device does it, with that device current).
#include "common.cuh"
#include "../../include/mla.h"

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_noalloc(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int P,
                                  void* k_cache, void* v_cache, int cap, void* out, void* stream) {
  const size_t need = mla_workspace_size(MLA_MODE_DECODE, B, P, cap);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;  // batch too large for the fixed scratch
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MLA_OK) return rc;
  // Same checks, kernels and results as mla_decode; the status word at the
  // start of the scratch is cleared by it on every call, and every other
  // scratch region is written before it is read.
  return mla_decode(w, params, x, B, P, k_cache, v_cache, cap, out, scratch, kNoAllocScratchBytes, stream);
}
