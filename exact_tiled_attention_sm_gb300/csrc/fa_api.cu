// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA
// descriptors, kernel selection and launch.  No device memory is allocated
// here; every tensor and the backward workspace belong to the caller.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_common.cuh"
#include "fa_internal.h"
#include "fa_sched.cuh"

#define FA_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int checked = 0;  // 0 unknown, 1 ok
  int sm_major = 0, sm_minor = 0, num_sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

fa_status current_device(int* dev, DeviceInfo* info) {
  if (cudaGetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[*dev];
  if (!d.checked) {
    if (cudaDeviceGetAttribute(&d.sm_major, cudaDevAttrComputeCapabilityMajor,
                               *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_minor, cudaDevAttrComputeCapabilityMinor,
                               *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount,
                               *dev) != cudaSuccess)
      return FA_ERR_CUDA;
    d.checked = 1;
  }
  *info = d;
  return FA_OK;
}

fa_status get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return FA_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                       cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return FA_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return FA_OK;
}

// [B*H, N, d] bf16 tensor; boxes of 64 columns x `rows` rows (128, or 64 for
// the d = 256 backward's query blocks) x 1 head, 128-byte swizzle,
// out-of-range rows read as zero.
fa_status make_map(CUtensorMap* m, const void* base, int BH, int N, int d,
                   int rows = 128) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// [B*H, N, d] 8-bit tensor; boxes of 128 columns (bytes) x 128 rows x 1
// head, 128-byte swizzle, out-of-range rows read as zero.
fa_status make_map_u8(CUtensorMap* m, const void* base, int BH, int N, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)N * d};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// fp32 [B*H, N, d] dQ accumulator; boxes of 32 columns x 128 rows x 1 head,
// 128-byte swizzle; used only as the target of bulk reduce-adds.
fa_status make_map_f32(CUtensorMap* m, const void* base, int BH, int N, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool aligned16(const void* p) {
  return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

fa_status check_shape(int B, int H, int N, int d, float scale, int dt) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (dt != FA_BF16 && dt != FA_F32) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  const long long elems = (long long)B * H * N * d;
  if (elems >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if ((long long)B * H >= (1ll << 31) / 128) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

fa_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Dropout threshold t = round(256 p), ties to even; -1 when p is NaN,
// negative, or rounds to 256 or more.
int threshold_of(float p) {
  if (!(p >= 0.f) || !std::isfinite(p)) return -1;
  const double t = std::nearbyint(256.0 * (double)p);
  return t <= 255.0 ? (int)t : -1;
}

fa::DropSpec drop_spec(int t, unsigned long long seed) {
  fa::DropSpec d;
  if (t > 0) {
    d.t4 = (uint32_t)t * 0x01010101u;
    d.keep_scale = (float)(256.0 / (double)(256 - t));
    d.c4 = (uint32_t)(256 - t) * 0x01010101u;
    d.c7 = d.c4 & 0x7F7F7F7Fu;
  }
  d.k0 = (uint32_t)seed;
  d.k1 = (uint32_t)(seed >> 32);
  return d;
}

// window: 0 for none, else >= 1 (a causal sliding window; one covering the
// whole sequence is the causal case and is run as such).  drop.t4 = 0: no
// dropout.
fa_status fwd_impl(const void* Q, const void* K, const void* V, void* O,
                   float* LSE, int B, int H, int N, int d, float scale,
                   int causal, int window, const fa::DropSpec& drop,
                   fa_dtype dt, void* stream) {
  fa_status st = check_shape(B, H, N, d, scale, (int)dt);
  if (st != FA_OK) return st;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
      !aligned16(LSE))
    return FA_ERR_INVALID_ARG;
  int dev;
  DeviceInfo info;
  if ((st = current_device(&dev, &info)) != FA_OK) return st;
  if (window >= N) window = 0;  // sees every earlier key: plain causal
  const fa::AttnShape s{B, H, N, d, scale, (causal || window > 0) ? 1 : 0,
                        window, drop};
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dt == FA_F32)
    return from_cuda(fa::launch_fwd_f32(
        s, static_cast<const float*>(Q), static_cast<const float*>(K),
        static_cast<const float*>(V), static_cast<float*>(O), LSE, cs));
  if (info.sm_major != 10 || info.sm_minor != 3) return FA_ERR_UNSUPPORTED;
  if ((st = get_encoder()) != FA_OK) return st;
  fa::TileMaps maps{};
  const int BH = B * H;
  if ((st = make_map(&maps.q, Q, BH, N, d)) != FA_OK) return st;
  if ((st = make_map(&maps.k, K, BH, N, d)) != FA_OK) return st;
  if ((st = make_map(&maps.v, V, BH, N, d)) != FA_OK) return st;
  if (d == 256)
    return from_cuda(fa::launch_fwd256_tc(s, maps, O, LSE, info.num_sms,
                                          fa::kWaitLimitNs, cs));
  return from_cuda(fa::launch_fwd_tc(s, maps, O, LSE, info.num_sms,
                                     fa::kWaitLimitNs, cs));
}

}  // namespace

FA_API fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O,
                        float* LSE, int B, int H, int N, int d, float scale,
                        int causal, fa_dtype dt, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, causal, 0, fa::DropSpec{},
                  dt, stream);
}

FA_API fa_status fa_fwd_window(const void* Q, const void* K, const void* V,
                               void* O, float* LSE, int B, int H, int N, int d,
                               float scale, int window, fa_dtype dt,
                               void* stream) {
  if (window < 1) return FA_ERR_INVALID_ARG;
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, 1, window, fa::DropSpec{},
                  dt, stream);
}

FA_API int fa_dropout_threshold(float dropout_p) { return threshold_of(dropout_p); }

FA_API fa_status fa_fwd_fp8(const void* Q, const void* K, const void* V,
                            void* O, float* LSE, int B, int H, int N, int d,
                            float scale, int causal, int window,
                            float q_descale, float k_descale, float v_descale,
                            void* stream) {
  fa_status st = check_shape(B, H, N, d, scale, (int)FA_BF16);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (window < 0 || !std::isfinite(q_descale) || !std::isfinite(k_descale) ||
      !std::isfinite(v_descale) || !(q_descale > 0.f) || !(k_descale > 0.f) ||
      !(v_descale > 0.f))
    return FA_ERR_INVALID_ARG;
  const float qk = scale * q_descale * k_descale;
  if (!std::isfinite(qk)) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
      !aligned16(LSE))
    return FA_ERR_INVALID_ARG;
  int dev;
  DeviceInfo info;
  if ((st = current_device(&dev, &info)) != FA_OK) return st;
  if (info.sm_major != 10 || info.sm_minor != 3) return FA_ERR_UNSUPPORTED;
  if (window >= N) window = 0;
  fa::AttnShape s{B, H, N, d, qk, (causal || window > 0) ? 1 : 0, window};
  s.fp8 = 1;
  s.v_descale = v_descale;
  if ((st = get_encoder()) != FA_OK) return st;
  fa::TileMaps maps{};
  const int BH = B * H;
  if ((st = make_map_u8(&maps.q, Q, BH, N, d)) != FA_OK) return st;
  if ((st = make_map_u8(&maps.k, K, BH, N, d)) != FA_OK) return st;
  if ((st = make_map_u8(&maps.v, V, BH, N, d)) != FA_OK) return st;
  return from_cuda(fa::launch_fwd_tc(s, maps, O, LSE, info.num_sms,
                                     fa::kWaitLimitNs,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

FA_API fa_status fa_fwd_dropout(const void* Q, const void* K, const void* V,
                                void* O, float* LSE, int B, int H, int N, int d,
                                float scale, int causal, int window,
                                float dropout_p, unsigned long long seed,
                                fa_dtype dt, void* stream) {
  const int t = threshold_of(dropout_p);
  if (window < 0 || t < 0) return FA_ERR_INVALID_ARG;
  return fwd_impl(Q, K, V, O, LSE, B, H, N, d, scale, causal, window,
                  drop_spec(t, seed), dt, stream);
}

FA_API fa_status fa_dropout_mask(unsigned char* keep, int B, int H, int N,
                                 float dropout_p, unsigned long long seed,
                                 void* stream) {
  const int t = threshold_of(dropout_p);
  if (!keep || t < 0 || B < 1 || H < 1 || N < 1 || N > 4 * 65535)
    return FA_ERR_INVALID_ARG;
  if ((long long)B * H >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  int dev;
  DeviceInfo info;
  fa_status st = current_device(&dev, &info);
  if (st != FA_OK) return st;
  fa::AttnShape s{B, H, N, 64, 1.f, 0, 0, drop_spec(t, seed)};
  return from_cuda(fa::launch_dropout_mask(s, keep,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

FA_API size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d, 1.0f, FA_BF16) != FA_OK) return 0;
  const size_t rows = (size_t)B * H * N;
  return align256(rows * sizeof(float)) + align256(rows * d * sizeof(float));
}

namespace {

fa_status bwd_impl(const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* LSE, void* dQ, void* dK,
                   void* dV, int B, int H, int N, int d, float scale,
                   int causal, int window, const fa::DropSpec& drop,
                   fa_dtype dt, void* workspace, size_t workspace_bytes,
                   void* stream) {
  fa_status st = check_shape(B, H, N, d, scale, (int)dt);
  if (st != FA_OK) return st;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
      !aligned16(dO) || !aligned16(LSE) || !aligned16(dQ) || !aligned16(dK) ||
      !aligned16(dV))
    return FA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < fa_bwd_workspace_size(B, H, N, d))
    return FA_ERR_INVALID_ARG;
  int dev;
  DeviceInfo info;
  if ((st = current_device(&dev, &info)) != FA_OK) return st;
  if (window >= N) window = 0;
  const fa::AttnShape s{B, H, N, d, scale, (causal || window > 0) ? 1 : 0,
                        window, drop};
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)B * H * N;
  float* Dvec = static_cast<float*>(workspace);
  float* dQacc = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          align256(rows * sizeof(float)));
  if (dt == FA_F32) {
    if ((st = from_cuda(fa::launch_bwd_pre(s, O, dO, 0, Dvec, nullptr, cs))) !=
        FA_OK)
      return st;
    return from_cuda(fa::launch_bwd_f32(
        s, static_cast<const float*>(Q), static_cast<const float*>(K),
        static_cast<const float*>(V), static_cast<const float*>(dO), LSE, Dvec,
        static_cast<float*>(dQ), static_cast<float*>(dK),
        static_cast<float*>(dV), cs));
  }
  if (info.sm_major != 10 || info.sm_minor != 3) return FA_ERR_UNSUPPORTED;
  if ((st = get_encoder()) != FA_OK) return st;
  fa::TileMaps maps{};
  const int BH = B * H;
  if (d == 256) {  // one half of d per work item, 64-query blocks
    if ((st = make_map(&maps.q, Q, BH, N, d, 64)) != FA_OK) return st;
    if ((st = make_map(&maps.k, K, BH, N, d)) != FA_OK) return st;
    if ((st = make_map(&maps.dO, dO, BH, N, d, 64)) != FA_OK) return st;
    if ((st = from_cuda(fa::launch_bwd_pre(s, O, dO, 1, Dvec, dQacc, cs))) != FA_OK)
      return st;
    if ((st = from_cuda(fa::launch_bwd256_tc(s, maps, LSE, Dvec, V, dQacc, dK, dV,
                                             info.num_sms, fa::kWaitLimitNs, cs))) !=
        FA_OK)
      return st;
    return from_cuda(fa::launch_dq_convert(s, dQacc, dQ, cs));
  }
  if ((st = make_map(&maps.q, Q, BH, N, d)) != FA_OK) return st;
  if ((st = make_map(&maps.k, K, BH, N, d)) != FA_OK) return st;
  if ((st = make_map(&maps.v, V, BH, N, d)) != FA_OK) return st;
  if ((st = make_map(&maps.dO, dO, BH, N, d)) != FA_OK) return st;
  if ((st = make_map_f32(&maps.dq_acc, dQacc, BH, N, d)) != FA_OK) return st;
  // dK and dV leave the backward kernel through TMA stores
  if ((st = make_map(&maps.dk, dK, BH, N, d)) != FA_OK) return st;
  if ((st = make_map(&maps.dv, dV, BH, N, d)) != FA_OK) return st;
  if ((st = from_cuda(fa::launch_bwd_pre(s, O, dO, 1, Dvec, dQacc, cs))) !=
      FA_OK)
    return st;
  const cudaError_t ke =
      (d == 64 && s.drop.t4 == 0)
          ? fa::launch_bwd64_tc(s, maps, LSE, Dvec, dK, dV, info.num_sms,
                                fa::kWaitLimitNs, cs)
          : fa::launch_bwd_tc(s, maps, LSE, Dvec, dQacc, dK, dV, info.num_sms,
                              fa::kWaitLimitNs, cs);
  if ((st = from_cuda(ke)) != FA_OK) return st;
  return from_cuda(fa::launch_dq_convert(s, dQacc, dQ, cs));
}

}  // namespace

FA_API fa_status fa_bwd(const void* Q, const void* K, const void* V,
                        const void* O, const void* dO, const float* LSE,
                        void* dQ, void* dK, void* dV, int B, int H, int N,
                        int d, float scale, int causal, fa_dtype dt,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal,
                  0, fa::DropSpec{}, dt, workspace, workspace_bytes, stream);
}

FA_API fa_status fa_bwd_window(const void* Q, const void* K, const void* V,
                               const void* O, const void* dO, const float* LSE,
                               void* dQ, void* dK, void* dV, int B, int H,
                               int N, int d, float scale, int window,
                               fa_dtype dt, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (window < 1) return FA_ERR_INVALID_ARG;
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, 1,
                  window, fa::DropSpec{}, dt, workspace, workspace_bytes, stream);
}

FA_API fa_status fa_bwd_dropout(const void* Q, const void* K, const void* V,
                                const void* O, const void* dO, const float* LSE,
                                void* dQ, void* dK, void* dV, int B, int H,
                                int N, int d, float scale, int causal,
                                int window, float dropout_p,
                                unsigned long long seed, fa_dtype dt,
                                void* workspace, size_t workspace_bytes,
                                void* stream) {
  const int t = threshold_of(dropout_p);
  if (window < 0 || t < 0) return FA_ERR_INVALID_ARG;
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, scale, causal,
                  window, drop_spec(t, seed), dt, workspace, workspace_bytes,
                  stream);
}

FA_API fa_status fa_last_device_status(void* stream) {
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const unsigned int words[6] = {fa::read_status_fwd_tc(cs),
                                 fa::read_status_fwd256_tc(cs),
                                 fa::read_status_bwd_tc(cs),
                                 fa::read_status_bwd64_tc(cs),
                                 fa::read_status_bwd256_tc(cs),
                                 fa::read_status_simt(cs)};
  fa_status out = FA_OK;
  for (unsigned int w : words) {
    if (w == 0xFFFFFFFFu) return FA_ERR_CUDA;
    if (w != 0 && out == FA_OK) out = static_cast<fa_status>(w & 0xFFu);
  }
  return out;
}

FA_API const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

FA_API fa_status fa_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 10000000u) return FA_ERR_INVALID_ARG;
  return from_cuda(fa::launch_selftest_timeout((uint64_t)limit_us * 1000ull,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

FA_API fa_status fa_fwd_schedule_census(int N, int causal, long long* out) {
  return fa_fwd_schedule_census_window(N, causal, 0, out);
}

FA_API fa_status fa_fwd_schedule_census_window(int N, int causal, int window,
                                               long long* out) {
  if (N < 1 || !out || window < 0) return FA_ERR_INVALID_ARG;
  fa::FwdSched sc;
  sc.init(1, N, causal ? 1 : 0, 1, window < N ? window : 0);
  long long computed = 0;
  for (int q = 0; q < sc.n_q_tiles; ++q) computed += sc.n_kv(q);
  out[0] = computed;
  out[1] = (long long)sc.n_q_tiles * sc.n_kv_total - computed;
  out[2] = sc.n_pairs;
  return FA_OK;
}

FA_API fa_status fa_fwd_schedule_cover(int BH, int N, int causal, int window, int d,
                                       int num_sms, int* counts, int* grid,
                                       int* items) {
  if (BH < 1 || N < 1 || window < 0 || num_sms < 1 || !counts) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const int win = window < N ? window : 0;
  // d = 64: single-block items for two workers per CTA; d = 128: pairs
  const bool groups = d == 64;
  const fa::FwdSched sc = groups ? fa::FwdSched::planned_groups(BH, N, causal ? 1 : 0, num_sms, win)
                                 : fa::FwdSched::planned(BH, N, causal ? 1 : 0, num_sms, win);
  const size_t n = (size_t)BH * sc.n_q_tiles;
  for (size_t i = 0; i < n; ++i) counts[i] = 0;
  const int nw = sc.n_waves();
  for (int v = 0; v < sc.grid; ++v)
    for (int w = 0; w < nw; ++w) {
      const int item = sc.item_of(v, w);
      if (item < 0) continue;
      int bh, q0;
      bool two = false;
      if (groups)
        sc.decode(item, bh, q0);
      else
        sc.decode_blocks(item, bh, q0, two);
      if (bh < 0 || bh >= BH || q0 < 0 || q0 + (two ? 1 : 0) >= sc.n_q_tiles)
        return FA_ERR_INVALID_ARG;  // an item outside the tensor
      ++counts[(size_t)bh * sc.n_q_tiles + q0];
      if (two) ++counts[(size_t)bh * sc.n_q_tiles + q0 + 1];
    }
  if (grid) *grid = groups ? sc.grid / 2 : sc.grid;
  if (items) *items = sc.total_items;
  return FA_OK;
}

FA_API int fa_version(void) { return 300; }
