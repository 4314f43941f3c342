// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass with a library-owned
// scratch array instead of a caller workspace, for callers that have input
// and output buffers but no way to allocate device memory (see include/fa.h).
// The array is a file-scope __device__ variable.  CUDA reserves it on a
// device when this module is loaded there; with lazy module loading (CUDA's
// default) that is the first cudaGetSymbolAddress of it on that device, made
// by the first fa_bwd_noalloc call there, which can therefore take device
// memory and synchronise.  Later calls run exactly fa_bwd on the array.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fa.h"

namespace {

// The scratch: device memory reserved when this module is loaded on a GPU and
// held until the process exits.  In host code this name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

bool ok_ptr(const void* p) {
  return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) fa_status fa_bwd_noalloc(
    const void* Q, const void* K, const void* V, const void* O, const void* dO,
    const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
    float scale, int causal, fa_dtype dt, void* stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0)  // a shape fa_bwd rejects: return its status, launch nothing
    return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal,
                  dt, nullptr, 0, stream);
  if (need > FA_BWD_NOALLOC_SCRATCH_BYTES) return FA_ERR_INVALID_ARG;
  if (!ok_ptr(Q) || !ok_ptr(K) || !ok_ptr(V) || !ok_ptr(O) || !ok_ptr(dO) ||
      !ok_ptr(LSE) || !ok_ptr(dQ) || !ok_ptr(dK) || !ok_ptr(dV))
    return FA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {  // first call on this device: load, resolve, keep
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p)
        return FA_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal, dt,
                scratch, FA_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
