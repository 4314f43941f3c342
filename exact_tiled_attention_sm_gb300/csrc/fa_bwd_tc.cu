// fa_bwd_tc.cu -- bf16 exact attention backward on sm_103a tensor cores.
//
// Recomputation instead of storage ("Flash Attention, From First Principles",
// "The backward pass -- resurrection"; "FlashAttention from scratch",
// follow-up on the backward pass): P is rebuilt tile by tile from Q, K and
// the forward's log-sum-exp, P = exp(scale*QK^T - LSE), and
//   dV += P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D = rowsum(dO * O),
//   dK += scale * dS^T Q,  dQ += scale * dS K.
//
// One persistent CTA per SM walks the items of BwdSched: a head and a block of
// 128 keys, whose K and V tiles stay resident in shared memory while the
// query blocks i stream past (K/V-outer order, so dK and dV accumulate in
// TMEM and are written once).  Per query block the tensor core computes the
// transposed tiles S^T = K Q_i^T and dP^T = V dO_i^T (rows = keys), the dS
// warpgroup turns them into P^T and scale*dS^T, and the tensor core then
// forms dV += P^T dO_i and dK += dS^T Q_i (P^T and dS^T read straight from
// TMEM) and dQ_i = dS K (dS read from shared memory); the dQ warpgroup adds
// dQ_i into the fp32 accumulator with vector atomics.
//
// Roles: warps 0-3 dS (one thread per key row), warps 4-7 dQ atomics and the
// dK/dV epilogue, warp 8 tensor-core issuer and TMEM owner, warp 9 loads
// (TMA for K, V, Q, dO; plain loads for LSE and D).
//
// TMEM: S^T [0,128) (P^T aliases its first 64 columns), dP^T [128,256) (dS^T
// aliases its first 64 columns, and dQ_i reuses the block once dK has read
// dS^T), dV [256, 256+d), dK [256+d, 256+2d).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_sched.cuh"
#include "fa_tiles.cuh"

namespace fa {
namespace bwdtc {

template <int D>
struct Cfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE_BYTES = CH * kChunkBytes;
  static constexpr int QST = 2;  // Q / dO ring stages
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + QST * TILE_BYTES;
  static constexpr int OFF_DS = OFF_DO + QST * TILE_BYTES;   // dS^T [128][128]
  static constexpr int OFF_STAT = OFF_DS + 2 * kChunkBytes;  // per stage
  static constexpr int STAT_BYTES = 2 * 128 * 4;             // lse2[128], D[128]
  static constexpr int OFF_BAR = OFF_STAT + QST * STAT_BYTES;
  static constexpr int B_KVFULL = 0, B_KVEMPTY = 1;
  static constexpr int B_QFULL = 2, B_QEMPTY = B_QFULL + QST;
  static constexpr int B_SDP = B_QEMPTY + QST;
  static constexpr int B_DSREADY = B_SDP + 1;
  static constexpr int B_DQFULL = B_DSREADY + 1;
  static constexpr int B_DQFREE = B_DQFULL + 1;
  static constexpr int B_DKDVDONE = B_DQFREE + 1;
  static constexpr int B_DKDVFREE = B_DKDVDONE + 1;
  static constexpr int B_MMADONE = B_DKDVFREE + 1;
  static constexpr int NBAR = B_MMADONE + 1;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_SS = idesc_bf16_f32(128, 128, 0, 0);
  static constexpr uint32_t IDESC_TS = idesc_bf16_f32(128, D, 0, 1);
  static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, D, 1, 1);
};

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;

struct Params {
  const float* LSE;
  const float* Dvec;
  float* dQacc;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  float scale;
  float scale_log2;
  uint64_t wait_limit_ns;
  BwdSched sched;
};

enum : uint32_t {
  SITE_L_KVEMPTY = 1, SITE_L_QEMPTY, SITE_M_KVFULL, SITE_M_QFULL, SITE_M_DQFREE,
  SITE_M_DSREADY, SITE_M_DKDVFREE, SITE_S_QFULL, SITE_S_SDP, SITE_Q_DQFULL,
  SITE_Q_DKDVDONE, SITE_DRAIN, SITE_ALIGN
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap mq,
               const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv,
               const __grid_constant__ CUtensorMap mdo, const Params p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + C::OFF_BAR + 8u * (uint32_t)i; };
  auto sQ = [&](int s) { return sb + C::OFF_Q + (uint32_t)s * C::TILE_BYTES; };
  auto sdO = [&](int s) { return sb + C::OFF_DO + (uint32_t)s * C::TILE_BYTES; };
  auto stat = [&](int s) {
    return reinterpret_cast<float*>(smem + C::OFF_STAT + s * C::STAT_BYTES);
  };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  volatile uint32_t* tmem_slot =
      reinterpret_cast<volatile uint32_t*>(smem + C::OFF_TMEM);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const BwdSched& sc = p.sched;
  const uint64_t lim = p.wait_limit_ns;
  const int N = sc.N;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KVFULL), 1);
    mbar_init(bar(C::B_KVEMPTY), 1);
    for (int s = 0; s < C::QST; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1 + 32);  // TMA arrive + 32 stat writers
      mbar_init(bar(C::B_QEMPTY + s), 1);
    }
    mbar_init(bar(C::B_SDP), 1);
    mbar_init(bar(C::B_DSREADY), 128);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQFREE), 128);
    mbar_init(bar(C::B_DKDVDONE), 1);
    mbar_init(bar(C::B_DKDVFREE), 128);
    mbar_init(bar(C::B_MMADONE), 1);
    *abort_flag = 0;
    if (sb & 1023u) record_timeout(abort_flag, SITE_ALIGN);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nw = sc.n_waves();

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      prefetch_tensormap(&mdo);
    }
    uint32_t qcnt = 0, it = 0;
    int kv_last = -1;
    uint32_t q_used = 0, q_par = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      if (it > 0 && !wait_warp(bar(C::B_KVEMPTY), (it - 1) & 1, abort_flag, lim,
                               SITE_L_KVEMPTY))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::TILE_BYTES);
        for (int c = 0; c < C::CH; ++c) {
          tma_load_3d(sb + C::OFF_K + c * kChunkBytes, &mk, bar(C::B_KVFULL),
                      c * 64, kb * 128, bh);
          tma_load_3d(sb + C::OFF_V + c * kChunkBytes, &mv, bar(C::B_KVFULL),
                      c * 64, kb * 128, bh);
        }
      }
      kv_last = (int)(it & 1);
      for (int i = sc.q_begin(kb); i < sc.n_blk; ++i) {
        const int s = qcnt % C::QST;
        const uint32_t ph = (qcnt / C::QST) & 1;
        if (!wait_warp(bar(C::B_QEMPTY + s), ph ^ 1, abort_flag, lim,
                       SITE_L_QEMPTY)) {
          ok = false;
          break;
        }
        // LSE (as log2) and D of the block's 128 queries; rows past N get
        // LSE = +inf so that their P is exactly 0
        float* st = stat(s);
        const size_t base = (size_t)bh * N;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qi = lane * 4 + e;
          const int q = i * 128 + qi;
          const bool valid = q < N;
          st[qi] = valid ? p.LSE[base + q] * 1.4426950408889634f : INFINITY;
          st[128 + qi] = valid ? p.Dvec[base + q] : 0.f;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::B_QFULL + s), 2 * C::TILE_BYTES);
          for (int c = 0; c < C::CH; ++c) {
            tma_load_3d(sQ(s) + c * kChunkBytes, &mq, bar(C::B_QFULL + s),
                        c * 64, i * 128, bh);
            tma_load_3d(sdO(s) + c * kChunkBytes, &mdo, bar(C::B_QFULL + s),
                        c * 64, i * 128, bh);
          }
        }
        mbar_arrive(bar(C::B_QFULL + s));
        q_used |= 1u << s;
        q_par = (q_par & ~(1u << s)) | (ph << s);
        ++qcnt;
      }
      ++it;
    }
    if (lane == 0) {  // every copy issued here lands before the CTA exits
      volatile int no_abort = 0;
      if (kv_last >= 0)
        wait_one(bar(C::B_KVFULL), (uint32_t)kv_last, &no_abort, lim, SITE_DRAIN);
      for (int s = 0; s < C::QST; ++s)
        if ((q_used >> s) & 1)
          wait_one(bar(C::B_QFULL + s), (q_par >> s) & 1, &no_abort, lim,
                   SITE_DRAIN);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- tensor core
    if (lane == 0) {
      uint32_t qcnt = 0, it = 0, g = 0;
      bool ok = true;
      const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V;
      const uint32_t sDS = sb + C::OFF_DS;
      for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
        const int item = sc.item_of(blockIdx.x, w);
        if (item < 0) continue;
        int bh, kb;
        sc.decode(item, bh, kb);
        if (!wait_one(bar(C::B_KVFULL), it & 1, abort_flag, lim, SITE_M_KVFULL))
          break;
        tc_fence_after();
        const int i0 = sc.q_begin(kb);
        for (int i = i0; i < sc.n_blk; ++i) {
          const int s = qcnt % C::QST;
          if (!wait_one(bar(C::B_QFULL + s), (qcnt / C::QST) & 1, abort_flag,
                        lim, SITE_M_QFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_rows_x_rows<D>(tmem + C::TM_S, sK, sQ(s), C::IDESC_SS);
          if (g > 0) {  // dQ of the previous block has been read out
            if (!wait_one(bar(C::B_DQFREE), (g - 1) & 1, abort_flag, lim,
                          SITE_M_DQFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          mma_rows_x_rows<D>(tmem + C::TM_DP, sV, sdO(s), C::IDESC_SS);
          umma_commit(bar(C::B_SDP));
          if (!wait_one(bar(C::B_DSREADY), g & 1, abort_flag, lim,
                        SITE_M_DSREADY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool first = (i == i0);
          if (first && it > 0) {  // previous item's dK/dV have been stored
            if (!wait_one(bar(C::B_DKDVFREE), (it - 1) & 1, abort_flag, lim,
                          SITE_M_DKDVFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          mma_tmem_x_rows(tmem + C::TM_DV, tmem + C::TM_S, sdO(s), C::IDESC_TS,
                          !first);
          mma_tmem_x_rows(tmem + C::TM_DK, tmem + C::TM_DP, sQ(s), C::IDESC_TS,
                          !first);
          umma_commit(bar(C::B_QEMPTY + s));
          ++qcnt;
          mma_colsT_x_rows(tmem + C::TM_DP, sDS, sK, C::IDESC_DQ);
          umma_commit(bar(C::B_DQFULL));
          ++g;
        }
        if (!ok) break;
        umma_commit(bar(C::B_KVEMPTY));
        umma_commit(bar(C::B_DKDVDONE));
        ++it;
      }
      umma_commit(bar(C::B_MMADONE));
      volatile int no_abort = 0;
      wait_one(bar(C::B_MMADONE), 0, &no_abort, lim, SITE_DRAIN);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------------- dS
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int r = warp * 32 + lane;  // key row within the block
    const float sl2 = p.scale_log2, scale = p.scale;
    uint32_t qcnt = 0, g = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      const int key = kb * 128 + r;
      const bool kvalid = key < N;
      for (int i = sc.q_begin(kb); i < sc.n_blk; ++i) {
        const int s = qcnt % C::QST;
        if (!wait_warp(bar(C::B_QFULL + s), (qcnt / C::QST) & 1, abort_flag,
                       lim, SITE_S_QFULL) ||
            !wait_warp(bar(C::B_SDP), g & 1, abort_flag, lim, SITE_S_SDP)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* lse2 = stat(s);
        const float* dvec = lse2 + 128;
        const int q0 = i * 128;
        const bool diag = sc.causal && i == kb;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t sr[32], dr[32];
          tmem_ld32(tmem + lane_off + C::TM_S + 32 * c, sr);
          tmem_ld32(tmem + lane_off + C::TM_DP + 32 * c, dr);
          tmem_ld_wait();
          reg_fence32(sr);
          reg_fence32(dr);
          uint32_t pp[16], dd[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float pv[2], dv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int qi = 32 * c + e + u;
              float pr = ex2_approx(__uint_as_float(sr[e + u]) * sl2 - lse2[qi]);
              if (!kvalid || (diag && q0 + qi < key)) pr = 0.f;
              pv[u] = pr;
              dv[u] = pr * (__uint_as_float(dr[e + u]) - dvec[qi]) * scale;
            }
            pp[e / 2] = pack_bf16x2(pv[0], pv[1]);
            dd[e / 2] = pack_bf16x2(dv[0], dv[1]);
          }
          tmem_st16(tmem + lane_off + C::TM_S + 16 * c, pp);
          tmem_st16(tmem + lane_off + C::TM_DP + 16 * c, dd);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v = make_uint4(dd[4 * k], dd[4 * k + 1], dd[4 * k + 2],
                                 dd[4 * k + 3]);
            *reinterpret_cast<uint4*>(smem + C::OFF_DS + swz_offset(r, 4 * c + k)) = v;
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::B_DSREADY));
        ++qcnt;
        ++g;
      }
    }
  } else {
    // ------------------------------------------------- dQ atomics, dK / dV
    const int wq = warp - 4;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int r = wq * 32 + lane;
    uint32_t g = 0, it = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      for (int i = sc.q_begin(kb); i < sc.n_blk; ++i) {
        if (!wait_warp(bar(C::B_DQFULL), g & 1, abort_flag, lim, SITE_Q_DQFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int q = i * 128 + r;
        float4* dst = reinterpret_cast<float4*>(
            p.dQacc + ((size_t)bh * N + (size_t)(q < N ? q : 0)) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + C::TM_DP + 32 * c, v);
          tmem_ld_wait();
          reg_fence32(v);
          if (q < N) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              atomicAdd(dst + 8 * c + k,
                        make_float4(__uint_as_float(v[4 * k]),
                                    __uint_as_float(v[4 * k + 1]),
                                    __uint_as_float(v[4 * k + 2]),
                                    __uint_as_float(v[4 * k + 3])));
          }
        }
        tc_fence_before();
        mbar_arrive(bar(C::B_DQFREE));
        ++g;
      }
      if (!ok) break;
      if (!wait_warp(bar(C::B_DKDVDONE), it & 1, abort_flag, lim,
                     SITE_Q_DKDVDONE))
        break;
      tc_fence_after();
      const int key = kb * 128 + r;
      const bool store = key < N;
      const size_t row = ((size_t)bh * N + (size_t)(store ? key : 0)) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* out = (which == 0 ? p.dV : p.dK) + row;
        const uint32_t col = which == 0 ? C::TM_DV : C::TM_DK;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + col + 32 * c, v);
          tmem_ld_wait();
          reg_fence32(v);
          uint4 o[4];
          uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            ow[k] = pack_bf16x2(__uint_as_float(v[2 * k]),
                                __uint_as_float(v[2 * k + 1]));
          if (store) {
            uint4* dstv = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
            for (int k = 0; k < 4; ++k) dstv[k] = o[k];
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_DKDVFREE));
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D>
cudaError_t launch(const AttnShape& s, const TileMaps& maps, const float* LSE,
                   const float* Dvec, float* dQacc, void* dK, void* dV,
                   int num_sms, uint64_t lim, cudaStream_t stream) {
  using C = Cfg<D>;
  static cudaError_t attr = cudaFuncSetAttribute(
      bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (attr != cudaSuccess) return attr;
  Params p;
  p.LSE = LSE;
  p.Dvec = Dvec;
  p.dQacc = dQacc;
  p.dK = reinterpret_cast<__nv_bfloat16*>(dK);
  p.dV = reinterpret_cast<__nv_bfloat16*>(dV);
  p.scale = s.scale;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.wait_limit_ns = lim;
  const int BH = s.B * s.H;
  const int n_blk = (s.N + 127) / 128;
  const int total = BH * n_blk;
  const int grid = total < num_sms ? total : num_sms;
  p.sched.init(BH, s.N, s.causal, grid);
  bwd_kernel<D><<<grid, kThreads, C::SMEM_BYTES, stream>>>(maps.q, maps.k, maps.v,
                                                             maps.dO, p);
  return cudaGetLastError();
}

}  // namespace bwdtc

cudaError_t launch_bwd_tc(const AttnShape& s, const TileMaps& maps,
                          const float* LSE, const float* Dvec, float* dQacc,
                          void* dK, void* dV, int num_sms,
                          uint64_t wait_limit_ns, cudaStream_t stream) {
  if (s.d == 64)
    return bwdtc::launch<64>(s, maps, LSE, Dvec, dQacc, dK, dV, num_sms,
                             wait_limit_ns, stream);
  return bwdtc::launch<128>(s, maps, LSE, Dvec, dQacc, dK, dV, num_sms,
                            wait_limit_ns, stream);
}

FA_DEFINE_STATUS_READER(read_status_bwd_tc)

}  // namespace fa
