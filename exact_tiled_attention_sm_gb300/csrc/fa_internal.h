// fa_internal.h -- launchers shared between the C-ABI layer (fa_api.cu) and
// the kernel translation units.  Host-only declarations.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Dropout parameters as the kernels take them: the byte threshold t (keep
// iff the random byte is >= t) in all four bytes, t4 = 0 meaning no dropout;
// the factor 256/(256 - t) of a kept entry; the Philox key (seed low word,
// seed high word); and 256 - t in all four bytes, whole (c4) and without
// each byte's top bit (c7), for the carry-based byte compare (t >= 1).
struct DropSpec {
  uint32_t t4 = 0;
  float keep_scale = 1.f;
  uint32_t k0 = 0, k1 = 0;
  uint32_t c4 = 0, c7 = 0;
};

struct AttnShape {
  int B, H, N, d;
  float scale;
  int causal;
  int window = 0;  // > 0: causal sliding window of this many keys
  DropSpec drop{};
  int fp8 = 0;           // Q, K, V are E4M3; `scale` includes their factors
  float v_descale = 1.f; // fp8: the factor of V
};

// TMA descriptors (built by fa_api.cu): the bf16 [B*H, N, d] tensors with
// 64-column x 128-row boxes, and the fp32 dQ accumulator [B*H, N, d] with
// 32-column x 128-row boxes (the backward's bulk reductions); all with the
// 128-byte swizzle.
struct TileMaps {
  CUtensorMap q, k, v, o, dO, dq_acc, dk, dv;
};

// fa_fwd_tc.cu -- bf16 forward on tcgen05/TMEM.
cudaError_t launch_fwd_tc(const AttnShape& s, const TileMaps& maps, void* O,
                          float* LSE, int num_sms, uint64_t wait_limit_ns,
                          cudaStream_t stream);
unsigned int read_status_fwd_tc(cudaStream_t stream);

// fa_fwd256_tc.cu -- bf16 forward for d = 256 (one query block per item).
cudaError_t launch_fwd256_tc(const AttnShape& s, const TileMaps& maps, void* O,
                             float* LSE, int num_sms, uint64_t wait_limit_ns,
                             cudaStream_t stream);
unsigned int read_status_fwd256_tc(cudaStream_t stream);

// fa_bwd_tc.cu -- bf16 backward on tcgen05/TMEM.
cudaError_t launch_bwd_tc(const AttnShape& s, const TileMaps& maps,
                          const float* LSE, const float* Dvec, float* dQacc,
                          void* dK, void* dV, int num_sms,
                          uint64_t wait_limit_ns, cudaStream_t stream);
unsigned int read_status_bwd_tc(cudaStream_t stream);

// fa_bwd64_tc.cu -- bf16 backward for d = 64 without dropout (dQ with TMEM
// columns and a shared-memory staging ring of its own); the maps and the
// zeroed accumulator (maps.dq_acc) are fa_bwd_tc's.
cudaError_t launch_bwd64_tc(const AttnShape& s, const TileMaps& maps,
                            const float* LSE, const float* Dvec, void* dK,
                            void* dV, int num_sms, uint64_t wait_limit_ns,
                            cudaStream_t stream);
unsigned int read_status_bwd64_tc(cudaStream_t stream);

// fa_bwd256_tc.cu -- bf16 backward for d = 256 on tcgen05/TMEM.  maps.q and
// maps.dO must have 64-row boxes (64 queries per block), maps.k 128-row ones;
// V is read directly (into TMEM); dQacc is the fp32 accumulator, zeroed.
cudaError_t launch_bwd256_tc(const AttnShape& s, const TileMaps& maps,
                             const float* LSE, const float* Dvec, const void* V,
                             float* dQacc, void* dK, void* dV, int num_sms,
                             uint64_t wait_limit_ns, cudaStream_t stream);
unsigned int read_status_bwd256_tc(cudaStream_t stream);

// fa_simt.cu -- fp32 forward/backward on the CUDA cores, and the backward's
// pre/post passes for both dtypes.
cudaError_t launch_fwd_f32(const AttnShape& s, const float* Q, const float* K,
                           const float* V, float* O, float* LSE,
                           cudaStream_t stream);
cudaError_t launch_bwd_f32(const AttnShape& s, const float* Q, const float* K,
                           const float* V, const float* dO, const float* LSE,
                           const float* Dvec, float* dQ, float* dK, float* dV,
                           cudaStream_t stream);
// D = rowsum(dO * O) (fp32), and dQacc zeroed when non-null.
cudaError_t launch_bwd_pre(const AttnShape& s, const void* O, const void* dO,
                           int is_bf16, float* Dvec, float* dQacc,
                           cudaStream_t stream);
// keep[bh][r][k] = 1 if dropout keeps (r, k), else 0 (bytes, B*H*N*N).
cudaError_t launch_dropout_mask(const AttnShape& s, uint8_t* keep,
                                cudaStream_t stream);
// dQ (bf16) = dQacc.
cudaError_t launch_dq_convert(const AttnShape& s, const float* dQacc, void* dQ,
                              cudaStream_t stream);
cudaError_t launch_selftest_timeout(uint64_t limit_ns, cudaStream_t stream);
unsigned int read_status_simt(cudaStream_t stream);

}  // namespace fa
