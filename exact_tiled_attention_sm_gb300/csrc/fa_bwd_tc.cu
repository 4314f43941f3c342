// fa_bwd_tc.cu -- bf16 exact attention backward on sm_103a tensor cores.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

cudaError_t launch_bwd_tc(const AttnShape&, const TileMaps&, const float*,
                          const float*, float*, void*, void*, int, uint64_t,
                          cudaStream_t) {
  return cudaErrorNotSupported;
}

FA_DEFINE_STATUS_READER(read_status_bwd_tc)

}  // namespace fa
