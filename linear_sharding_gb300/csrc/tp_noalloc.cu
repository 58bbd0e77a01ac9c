// tp_noalloc.cu - tp_mlp_forward_noalloc: the MLP forward pass with its
// scratch in a fixed, statically allocated device array, for callers that
// must not allocate device memory during a call.
//
// The scratch lives in this file's module as a file-scope __device__ array.
// In host code its name is only a host-side stand-in, not a device address,
// so the address is taken once per device with cudaGetSymbolAddress (with
// that device current) and handed to the kernels as their workspace.
#include <mutex>

#include "tp_internal.h"

namespace {

// Largest scratch one call may use: 16 MiB, enough for the memory-bound
// decode shapes (M <= 16 tokens) of an H = 8192, F = 28672, T = 8 MLP.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_tp_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch[kMaxDevices];

// Device address of the scratch on the current device, looked up on the
// first call on that device.
tp_status_t scratch_address(int dev, void **out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tp_noalloc_scratch) != cudaSuccess || !p) return TP_ERR_CUDA;
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return TP_OK;
}

}  // namespace

extern "C" TP_API tp_status_t tp_mlp_forward_noalloc(tp_shards_t s, const void *X, int64_t M,
                                                     tp_act_t act, float *Z, void *stream) {
  if (!s || M < 0) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TP_ERR_CUDA;
  // A handle made on this device means the library's per-device state exists,
  // so neither the size query nor the forward pass below allocates.
  if (!tp::handle_ready_on_current_device(s)) return TP_ERR_ARG;
  // The AUTO plan, or, where its workspace exceeds the scratch (it grows with the SM count's
  // split-K choice), the same pass refitted to the scratch.
  const size_t need = tp::mlp_workspace_within(s, M, kNoAllocScratchBytes);
  if (need == 0) return TP_ERR_ARG;
  if (need > kNoAllocScratchBytes) return TP_ERR_WORKSPACE;
  void *scratch = nullptr;
  const tp_status_t st = scratch_address(dev, &scratch);
  if (st != TP_OK) return st;
  return tp::mlp_forward_within(s, X, M, act, Z, scratch, kNoAllocScratchBytes, static_cast<cudaStream_t>(stream));
}
