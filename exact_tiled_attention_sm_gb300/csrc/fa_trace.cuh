// fa_trace.cuh -- per-CTA timing of the persistent kernels, for measuring
// how evenly the schedulers spread the work.  Compiled only into the trace
// build of the library (FA_CTA_TRACE defined, libfa_trace.so); in the product
// library every macro below expands to nothing.
//
// Each CTA records the global timer (ns) once after its set-up (barriers
// initialised, TMEM allocated) and once after its last work item (every role
// finished, before TMEM is released).  From these the host computes each
// CTA's busy time and the spread between the first and the last CTA to
// finish.  The array is per translation unit (no relocatable device code), so
// each kernel file defines its own array and exported reader.
#pragma once

#ifdef FA_CTA_TRACE
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace fa {
constexpr int kTraceMaxCtas = 1024;  // CTAs past this are not recorded
}  // namespace fa

// Defines the trace array ARR of this file and the exported host reader
// `int READER(unsigned long long* out, int ctas)`, which synchronises the
// device, copies 2 * ctas words (start, end of CTA 0, of CTA 1, ...; 0 for a
// CTA that did not run) and clears them; it returns 0, or -1 on a CUDA error
// or ctas outside 1..kTraceMaxCtas.
#define FA_TRACE_DEFINE(ARR, READER)                                          \
  static __device__ unsigned long long ARR[2 * fa::kTraceMaxCtas];            \
  extern "C" __attribute__((visibility("default"))) int READER(              \
      unsigned long long* out, int ctas) {                                    \
    if (!out || ctas < 1 || ctas > fa::kTraceMaxCtas) return -1;              \
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;                    \
    if (cudaMemcpyFromSymbol(out, ARR, 2 * sizeof(unsigned long long) * ctas) \
        != cudaSuccess)                                                       \
      return -1;                                                              \
    static unsigned long long zero[2 * fa::kTraceMaxCtas];                    \
    return cudaMemcpyToSymbol(ARR, zero, sizeof(zero)) == cudaSuccess ? 0 : -1; \
  }

// Thread 0 of the CTA records the start (after the set-up __syncthreads) or
// the end (after the final __syncthreads).
#define FA_TRACE_MARK(ARR, WHICH)                                   \
  do {                                                              \
    if (threadIdx.x == 0 && blockIdx.x < (unsigned)fa::kTraceMaxCtas) \
      ARR[2 * blockIdx.x + (WHICH)] = fa::globaltimer_ns();         \
  } while (0)

#else
#define FA_TRACE_DEFINE(ARR, READER)
#define FA_TRACE_MARK(ARR, WHICH) \
  do {                            \
  } while (0)
#endif
