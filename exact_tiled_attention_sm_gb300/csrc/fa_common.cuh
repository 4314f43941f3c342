// fa_common.cuh -- definitions shared by every kernel translation unit.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Device status word of this translation unit: 0, or FA_ERR_TIMEOUT in the
// low byte with the id of the wait site that gave up in bits 8..15.  Each
// kernel .cu file has its own copy (no relocatable device code), read and
// cleared through that file's status reader.
static __device__ unsigned int g_fa_device_status = 0;

// Default limit of every bounded wait inside a kernel: far above any wait a
// correct launch makes on the sizes this library accepts.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Suspend-time hint of one polling step of a bounded wait: long next to a
// pipeline step, short next to the wait's time limit.
constexpr uint32_t kWaitSleepNs = 20000;

constexpr int kTile = 128;  // rows of a query block and of a key block

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: the attribute belongs to the device's context, so
// a process that launches on several GPUs needs it on each.  `done` keeps one
// bit per device ordinal below 64 (higher ordinals set it on every call).
template <typename Kern>
cudaError_t smem_limit_once(Kern kernel, int bytes,
                            std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launches `kernel` as a programmatic dependent of the launch before it on
// `stream`: its CTAs may start once every CTA of that launch has signalled
// (griddep_launch_dependents) or exited, so its launch and set-up overlap the
// other's last CTAs.  The kernel must call griddep_wait before it touches
// anything the earlier launch writes; everything older than that launch is
// complete when it starts.
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
  const cudaError_t last = cudaGetLastError();  // read and clear, as after <<<>>>
  return e != cudaSuccess ? e : last;
}

}  // namespace fa

// Defines `unsigned int NAME(cudaStream_t)` that synchronises the stream,
// returns this file's status word and clears it.  Returns 0xFFFFFFFF if the
// CUDA calls fail.
#define FA_DEFINE_STATUS_READER(NAME)                                          \
  unsigned int NAME(cudaStream_t stream) {                                     \
    unsigned int v = 0, zero = 0;                                              \
    if (cudaStreamSynchronize(stream) != cudaSuccess) return 0xFFFFFFFFu;      \
    if (cudaMemcpyFromSymbol(&v, fa::g_fa_device_status, sizeof(v)) !=        \
        cudaSuccess)                                                           \
      return 0xFFFFFFFFu;                                                      \
    if (v != 0 && cudaMemcpyToSymbol(fa::g_fa_device_status, &zero,            \
                                     sizeof(zero)) != cudaSuccess)             \
      return 0xFFFFFFFFu;                                                      \
    return v;                                                                  \
  }
