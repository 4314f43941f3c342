// fa_simt.cu -- CUDA-core kernels: the fp32 forward and backward (fp32
// inputs and arithmetic, expf/logf), the backward's pre pass (D = rowsum(dO*O),
// dQ accumulator cleared) and post pass (dQ accumulator -> bf16), and the
// bounded-wait self test.
//
// fp32 forward: the same online-softmax recurrence as the tensor-core path
// ("LLM Architecture Refresh [3]", section 4), on 32x32 tiles: a CTA of four
// warps owns 32 query rows; for every key block each warp takes 8 rows, lane
// k scores key k, and the row max and row sum are warp-shuffle reductions.
// Causal key blocks after the query block are skipped.
//
// Dropout in the fp32 kernels: each thread holds single (query, key) entries
// and draws each one's keep decision with its own Philox call (keep_one).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "ptx.cuh"

namespace fa {
namespace simt {

constexpr int kRows = 32;   // query rows per CTA
constexpr int kKeys = 32;   // keys per block

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Loads rows [r0, r0+32) of one head into shared memory (as fp32) with row
// stride `ld`, zero-filling rows >= N.
template <int D, typename T>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* src,
                                          int r0, int N) {
  for (int i = threadIdx.x; i < kRows * D; i += blockDim.x) {
    const int r = i / D, c = i % D;
    dst[r * ld + c] = (r0 + r < N) ? to_f(src[(size_t)(r0 + r) * D + c]) : 0.f;
  }
}

template <int D>
__global__ void __launch_bounds__(128)
    fwd_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                   const float* __restrict__ V, float* __restrict__ O,
                   float* __restrict__ LSE, int N, float scale, int causal,
                   int window, const DropSpec drop) {
  constexpr int LD = D + 1;  // padded: lane k reads row k without conflicts
  extern __shared__ float sm[];
  float* sQ = sm;                  // [kRows][D]
  float* sK = sQ + kRows * D;      // [kKeys][LD]
  float* sV = sK + kKeys * LD;     // [kKeys][D]
  const int bh = blockIdx.y;
  const int r0 = blockIdx.x * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t head = (size_t)bh * N * D;
  load_rows<D>(sQ, D, Q + head, r0, N);

  float m[8], l[8], o[8][D / 32];
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) o[rr][c] = 0.f;
  }
  const int last_row = min(r0 + kRows, N) - 1;
  const int n_kb = causal ? (last_row / kKeys + 1) : (N + kKeys - 1) / kKeys;
  for (int kb = 0; kb < n_kb; ++kb) {
    __syncthreads();
    load_rows<D>(sK, LD, K + head, kb * kKeys, N);
    load_rows<D>(sV, D, V + head, kb * kKeys, N);
    __syncthreads();
    const int key = kb * kKeys + lane;
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const int lr = warp * 8 + rr;
      const int row = r0 + lr;
      float s = 0.f;
#pragma unroll 16
      for (int c = 0; c < D; ++c) s = fmaf(sQ[lr * D + c], sK[lane * LD + c], s);
      s *= scale;
      if (key >= N || (causal && key > row) || (window > 0 && row - key >= window))
        s = -INFINITY;
      const float m_new = fmaxf(m[rr], warp_max(s));
      const float corr = (m_new == -INFINITY) ? 1.f : expf(m[rr] - m_new);
      const float pr = (s == -INFINITY) ? 0.f : expf(s - m_new);
      l[rr] = l[rr] * corr + warp_sum(pr);  // the undropped row sum
      m[rr] = m_new;
      const float pv = (drop.t4 == 0 || keep_one(drop, bh, row, key)) ? pr : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float acc = 0.f;
#pragma unroll 8
        for (int k = 0; k < kKeys; ++k)
          acc = fmaf(__shfl_sync(0xffffffffu, pv, k), sV[k * D + c * 32 + lane], acc);
        o[rr][c] = o[rr][c] * corr + acc;
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int row = r0 + warp * 8 + rr;
    if (row >= N) continue;
    const float inv = drop.keep_scale / l[rr];
#pragma unroll
    for (int c = 0; c < D / 32; ++c)
      O[head + (size_t)row * D + c * 32 + lane] = o[rr][c] * inv;
    if (lane == 0) LSE[(size_t)bh * N + row] = m[rr] + logf(l[rr]);
  }
}

// dK, dV for 32 keys per CTA (8 per warp); lane = query within a 32-query
// block.  P is recomputed from LSE: p = exp(scale*<q,k> - LSE)
// ("FlashAttention from scratch", follow-up on the backward pass).  T: the
// tensors' type (fp32, or bf16 where no tensor-core backward exists);
// arithmetic in fp32 either way.
template <int D, typename T>
__global__ void __launch_bounds__(128)
    bwd_f32_dkdv_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                        const T* __restrict__ V, const T* __restrict__ dO,
                        const float* __restrict__ LSE, const float* __restrict__ Dv,
                        T* __restrict__ dK, T* __restrict__ dV, int N,
                        float scale, int causal, int window, const DropSpec drop) {
  constexpr int LD = D + 1;
  extern __shared__ float sm[];
  float* sQ = sm;                  // [kRows][LD]
  float* sdO = sQ + kRows * LD;    // [kRows][LD]
  float* sK = sdO + kRows * LD;    // [kKeys][D]
  float* sV = sK + kKeys * D;      // [kKeys][D]
  const int bh = blockIdx.y;
  const int k0 = blockIdx.x * kKeys;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t head = (size_t)bh * N * D;
  load_rows<D>(sK, D, K + head, k0, N);
  load_rows<D>(sV, D, V + head, k0, N);
  float ak[8][D / 32], av[8][D / 32];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int c = 0; c < D / 32; ++c) ak[i][c] = av[i][c] = 0.f;
  const int qb0 = causal ? k0 / kRows : 0;
  const int n_qb = (N + kRows - 1) / kRows;
  for (int qb = qb0; qb < n_qb; ++qb) {
    __syncthreads();
    load_rows<D>(sQ, LD, Q + head, qb * kRows, N);
    load_rows<D>(sdO, LD, dO + head, qb * kRows, N);
    __syncthreads();
    const int qrow = qb * kRows + lane;
    const bool qvalid = qrow < N;
    const float lse = qvalid ? LSE[(size_t)bh * N + qrow] : 0.f;
    const float Dq = qvalid ? Dv[(size_t)bh * N + qrow] : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int lk = warp * 8 + i;
      const int key = k0 + lk;
      float s = 0.f, dp = 0.f;
#pragma unroll 16
      for (int c = 0; c < D; ++c) {
        s = fmaf(sQ[lane * LD + c], sK[lk * D + c], s);
        dp = fmaf(sdO[lane * LD + c], sV[lk * D + c], dp);
      }
      const bool vis = qvalid && key < N && !(causal && key > qrow) &&
                       !(window > 0 && qrow - key >= window);
      const float pr = vis ? expf(s * scale - lse) : 0.f;
      // dropout: P o M for dV (the factor applied at the end), P (M dP - D)
      const bool kept = drop.t4 == 0 || keep_one(drop, bh, qrow, key);
      const float pv = kept ? pr : 0.f;
      const float ds = pr * ((kept ? dp * drop.keep_scale : 0.f) - Dq);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float a1 = 0.f, a2 = 0.f;
#pragma unroll 8
        for (int q = 0; q < kRows; ++q) {
          a1 = fmaf(__shfl_sync(0xffffffffu, pv, q), sdO[q * LD + c * 32 + lane], a1);
          a2 = fmaf(__shfl_sync(0xffffffffu, ds, q), sQ[q * LD + c * 32 + lane], a2);
        }
        av[i][c] += a1;
        ak[i][c] += a2;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int key = k0 + warp * 8 + i;
    if (key >= N) continue;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      dV[head + (size_t)key * D + c * 32 + lane] = from_f<T>(av[i][c] * drop.keep_scale);
      dK[head + (size_t)key * D + c * 32 + lane] = from_f<T>(ak[i][c] * scale);
    }
  }
}

// dQ for 32 query rows per CTA: dQ_r = scale * sum_k dS_rk k_k.
template <int D, typename T>
__global__ void __launch_bounds__(128)
    bwd_f32_dq_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                      const T* __restrict__ V, const T* __restrict__ dO,
                      const float* __restrict__ LSE, const float* __restrict__ Dv,
                      T* __restrict__ dQ, int N, float scale, int causal,
                      int window, const DropSpec drop) {
  constexpr int LD = D + 1;
  extern __shared__ float sm[];
  float* sQ = sm;                  // [kRows][D]
  float* sdO = sQ + kRows * D;     // [kRows][D]
  float* sK = sdO + kRows * D;     // [kKeys][LD]
  float* sV = sK + kKeys * LD;     // [kKeys][LD]
  const int bh = blockIdx.y;
  const int r0 = blockIdx.x * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t head = (size_t)bh * N * D;
  load_rows<D>(sQ, D, Q + head, r0, N);
  load_rows<D>(sdO, D, dO + head, r0, N);
  float acc[8][D / 32];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[i][c] = 0.f;
  const int last_row = min(r0 + kRows, N) - 1;
  const int n_kb = causal ? (last_row / kKeys + 1) : (N + kKeys - 1) / kKeys;
  for (int kb = 0; kb < n_kb; ++kb) {
    __syncthreads();
    load_rows<D>(sK, LD, K + head, kb * kKeys, N);
    load_rows<D>(sV, LD, V + head, kb * kKeys, N);
    __syncthreads();
    const int key = kb * kKeys + lane;
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const int lr = warp * 8 + rr;
      const int row = r0 + lr;
      const bool rvalid = row < N;
      const float lse = rvalid ? LSE[(size_t)bh * N + row] : 0.f;
      const float Dq = rvalid ? Dv[(size_t)bh * N + row] : 0.f;
      float s = 0.f, dp = 0.f;
#pragma unroll 16
      for (int c = 0; c < D; ++c) {
        s = fmaf(sQ[lr * D + c], sK[lane * LD + c], s);
        dp = fmaf(sdO[lr * D + c], sV[lane * LD + c], dp);
      }
      const bool vis = rvalid && key < N && !(causal && key > row) &&
                       !(window > 0 && row - key >= window);
      const float pr = vis ? expf(s * scale - lse) : 0.f;
      const bool kept = drop.t4 == 0 || keep_one(drop, bh, row, key);
      const float ds = pr * ((kept ? dp * drop.keep_scale : 0.f) - Dq);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float a = 0.f;
#pragma unroll 8
        for (int k = 0; k < kKeys; ++k)
          a = fmaf(__shfl_sync(0xffffffffu, ds, k), sK[k * LD + c * 32 + lane], a);
        acc[rr][c] += a;
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int row = r0 + warp * 8 + rr;
    if (row >= N) continue;
#pragma unroll
    for (int c = 0; c < D / 32; ++c)
      dQ[head + (size_t)row * D + c * 32 + lane] = from_f<T>(acc[rr][c] * scale);
  }
}

// One warp per row: D_r = sum_c dO_rc O_rc in fp32; zeroes the row of the
// fp32 dQ accumulator when one is given.
template <int D, typename T>
__global__ void __launch_bounds__(256)
    bwd_pre_kernel(const T* __restrict__ O, const T* __restrict__ dO,
                   float* __restrict__ Dv, float* __restrict__ dQacc,
                   long long rows) {
  // the backward kernel after this launch reads D and the zeroed
  // accumulator only after its griddep_wait, which waits for all of this grid
  griddep_launch_dependents();
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float acc = 0.f;
#pragma unroll
  for (int c = lane; c < D; c += 32)
    acc = fmaf((float)O[row * D + c], (float)dO[row * D + c], acc);
  acc = warp_sum(acc);
  if (lane == 0) Dv[row] = acc;
  if (dQacc) {
#pragma unroll
    for (int c = lane; c < D; c += 32) dQacc[row * D + c] = 0.f;
  }
}

// keep[bh][r][k] = 1 when dropout keeps (r, k), else 0: one thread per 4 x 4
// patch (one Philox call), patches of one row of patches along x, heads
// along z.
__global__ void __launch_bounds__(128)
    dropout_mask_kernel(uint8_t* __restrict__ keep, int BH, int N, const DropSpec d) {
  const int np = (N + 3) / 4;
  const int kp = blockIdx.x * blockDim.x + threadIdx.x;
  const int rp = blockIdx.y;
  if (kp >= np) return;
  for (int bh = blockIdx.z; bh < BH; bh += gridDim.z) {
    const Philox4 o = philox4x32_10((uint32_t)kp, (uint32_t)rp, (uint32_t)bh, 0u,
                                    d.k0, d.k1);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int r = 4 * rp + w;
      if (r >= N) break;
      const uint32_t kb = keep_bytes(o.x[w], d.t4) & 0x01010101u;
      uint8_t* dst = keep + ((size_t)bh * N + r) * N + 4 * (size_t)kp;
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (4 * kp + b < N) dst[b] = (uint8_t)((kb >> (8 * b)) & 1u);
    }
  }
}

__global__ void __launch_bounds__(256)
    dq_convert_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                      long long n4) {
  griddep_wait();  // the backward kernel launched before has finished dQacc
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 v = src[i];
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    dst[i] = o;
  }
}

// One thread waits on a barrier that nothing completes; the bounded wait
// gives up after `limit_ns`, records FA_ERR_TIMEOUT and the kernel exits.
__global__ void selftest_timeout_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    wait_one(smem_u32(&bar), 0, &abort_flag, limit_ns, 0x7F);
  __syncthreads();
}

}  // namespace simt


template <int D>
static cudaError_t fwd_f32_launch(const AttnShape& s, const float* Q,
                                  const float* K, const float* V, float* O,
                                  float* LSE, cudaStream_t stream) {
  constexpr int bytes =
      (simt::kRows * D + simt::kKeys * (D + 1) + simt::kKeys * D) * 4;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t attr = smem_limit_once(simt::fwd_f32_kernel<D>, bytes, attr_done);
  if (attr != cudaSuccess) return attr;
  dim3 grid((s.N + simt::kRows - 1) / simt::kRows, s.B * s.H);
  simt::fwd_f32_kernel<D><<<grid, 128, bytes, stream>>>(
      Q, K, V, O, LSE, s.N, s.scale, s.causal, s.window, s.drop);
  return cudaGetLastError();
}

template <int D, typename T>
static cudaError_t bwd_f32_launch(const AttnShape& s, const T* Q, const T* K,
                                  const T* V, const T* dO, const float* LSE,
                                  const float* Dvec, T* dQ, T* dK, T* dV,
                                  cudaStream_t stream) {
  constexpr int bytes = (2 * simt::kRows * (D + 1) + 2 * simt::kKeys * D) * 4;
  static std::atomic<unsigned long long> done1{0}, done2{0};
  const cudaError_t a1 = smem_limit_once(simt::bwd_f32_dkdv_kernel<D, T>, bytes, done1);
  if (a1 != cudaSuccess) return a1;
  const cudaError_t a2 = smem_limit_once(simt::bwd_f32_dq_kernel<D, T>, bytes, done2);
  if (a2 != cudaSuccess) return a2;
  dim3 grid((s.N + simt::kRows - 1) / simt::kRows, s.B * s.H);
  simt::bwd_f32_dkdv_kernel<D, T><<<grid, 128, bytes, stream>>>(
      Q, K, V, dO, LSE, Dvec, dK, dV, s.N, s.scale, s.causal, s.window, s.drop);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  simt::bwd_f32_dq_kernel<D, T><<<grid, 128, bytes, stream>>>(
      Q, K, V, dO, LSE, Dvec, dQ, s.N, s.scale, s.causal, s.window, s.drop);
  return cudaGetLastError();
}

cudaError_t launch_fwd_f32(const AttnShape& s, const float* Q, const float* K,
                           const float* V, float* O, float* LSE,
                           cudaStream_t stream) {
  if (s.d == 64) return fwd_f32_launch<64>(s, Q, K, V, O, LSE, stream);
  if (s.d == 256) return fwd_f32_launch<256>(s, Q, K, V, O, LSE, stream);
  return fwd_f32_launch<128>(s, Q, K, V, O, LSE, stream);
}

cudaError_t launch_bwd_f32(const AttnShape& s, const float* Q, const float* K,
                           const float* V, const float* dO, const float* LSE,
                           const float* Dvec, float* dQ, float* dK, float* dV,
                           cudaStream_t stream) {
  if (s.d == 64)
    return bwd_f32_launch<64>(s, Q, K, V, dO, LSE, Dvec, dQ, dK, dV, stream);
  if (s.d == 256)
    return bwd_f32_launch<256>(s, Q, K, V, dO, LSE, Dvec, dQ, dK, dV, stream);
  return bwd_f32_launch<128>(s, Q, K, V, dO, LSE, Dvec, dQ, dK, dV, stream);
}

cudaError_t launch_bwd_pre(const AttnShape& s, const void* O, const void* dO,
                           int is_bf16, float* Dvec, float* dQacc,
                           cudaStream_t stream) {
  const long long rows = (long long)s.B * s.H * s.N;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  if (is_bf16) {
    auto o = reinterpret_cast<const __nv_bfloat16*>(O);
    auto g = reinterpret_cast<const __nv_bfloat16*>(dO);
    if (s.d == 64)
      simt::bwd_pre_kernel<64, __nv_bfloat16><<<grid, 256, 0, stream>>>(o, g, Dvec, dQacc, rows);
    else if (s.d == 256)
      simt::bwd_pre_kernel<256, __nv_bfloat16><<<grid, 256, 0, stream>>>(o, g, Dvec, dQacc, rows);
    else
      simt::bwd_pre_kernel<128, __nv_bfloat16><<<grid, 256, 0, stream>>>(o, g, Dvec, dQacc, rows);
  } else {
    auto o = reinterpret_cast<const float*>(O);
    auto g = reinterpret_cast<const float*>(dO);
    if (s.d == 64)
      simt::bwd_pre_kernel<64, float><<<grid, 256, 0, stream>>>(o, g, Dvec, dQacc, rows);
    else if (s.d == 256)
      simt::bwd_pre_kernel<256, float><<<grid, 256, 0, stream>>>(o, g, Dvec, dQacc, rows);
    else
      simt::bwd_pre_kernel<128, float><<<grid, 256, 0, stream>>>(o, g, Dvec, dQacc, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_dropout_mask(const AttnShape& s, uint8_t* keep,
                                cudaStream_t stream) {
  const int np = (s.N + 3) / 4;
  const int BH = s.B * s.H;
  dim3 grid((unsigned)((np + 127) / 128), (unsigned)np,
            (unsigned)(BH < 65535 ? BH : 65535));
  simt::dropout_mask_kernel<<<grid, 128, 0, stream>>>(keep, BH, s.N, s.drop);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const AttnShape& s, const float* dQacc, void* dQ,
                              cudaStream_t stream) {
  const long long n4 = (long long)s.B * s.H * s.N * s.d / 4;
  long long blocks = (n4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  return launch_after(simt::dq_convert_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                      reinterpret_cast<const float4*>(dQacc), reinterpret_cast<uint2*>(dQ), n4);
}

cudaError_t launch_selftest_timeout(uint64_t limit_ns, cudaStream_t stream) {
  simt::selftest_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

FA_DEFINE_STATUS_READER(read_status_simt)

}  // namespace fa
