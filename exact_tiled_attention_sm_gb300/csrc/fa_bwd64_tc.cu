// fa_bwd64_tc.cu -- bf16 exact attention backward for head dimension 64 on
// sm_103a tensor cores.
//
// The recomputation of the d <= 128 backward ("Flash Attention, From First
// Principles", "The backward pass -- resurrection"; "FlashAttention from
// scratch", follow-up on the backward pass), K/V-outer:
//   P = exp(scale*QK^T - LSE), dV += P^T dO, dP = dO V^T,
//   dS = P * (dP - D), dK += scale*dS^T Q, dQ += scale*dS K,
// with the tiles and products of fa_bwd_tc.cu (S^T and dP^T with keys as
// rows, P^T and dS^T feeding dV and dK from TMEM, dQ_i = dS K with dS read
// from shared memory).
//
// What differs at d = 64 is room: the tiles leave 128 TMEM columns and about
// 97 KiB of shared memory free.  So dQ_i goes into TMEM columns of its own
// (the next dP^T no longer waits for it to be read out) and is staged by a
// dedicated warpgroup in a two-slot fp32 ring of its own, from which a warp
// of its own adds it into the accumulator with TMA bulk reduce-adds.  The
// Q/dO stages are then free as soon as dV_i and dK_i have read them (not
// after a reduce), so S^T(i+1) is issued right after dV_i, and the dS
// warpgroups turn it into P^T(i+1) while the tensor core forms dK_i and dQ_i.
//
// Roles (four whole warpgroups, so that setmaxnreg can move registers
// between them): warps 0-7 the two dS warpgroups (64 query columns each; the
// dV and dK epilogue); warps 8-11 the dQ warpgroup (TMEM lane quarter =
// warp - 8, query rows); warp 12 tensor-core issuer and TMEM owner; warp 13
// loads (TMA for K, V, Q, dO; plain loads for LSE and D); warp 14 the dQ
// reduce-adds; warp 15 idle.
//
// TMEM: S^T [0,128), dP^T [128,256), dV [256,320), dK [320,384),
// dQ [384,448).  P^T overwrites columns [0,32) and [64,96) of S^T, dS^T the
// same columns of dP^T, each warpgroup inside the columns it has read.
// Dropout (the keep mask's regeneration) stays on fa_bwd_tc.cu's kernel.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_sched.cuh"
#include "fa_tiles.cuh"
#include "fa_trace.cuh"

namespace fa {
namespace bwd64 {

FA_TRACE_DEFINE(g_cta_trace, fa_cta_trace_bwd64)

// Executed by every warp of a warpgroup: lowers (dealloc) or raises (alloc)
// its per-thread register count, R a multiple of 8 in [24, 256].  A raise
// must not go below the warp's current count nor a lowering above it (the
// instruction is illegal otherwise); a raise waits until other warpgroups
// have released enough of the CTA's registers.
template <int R>
__device__ __forceinline__ void reg_dealloc() {
  static_assert(R >= 24 && R <= 256 && R % 8 == 0, "setmaxnreg count");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void reg_alloc() {
  static_assert(R >= 24 && R <= 256 && R % 8 == 0, "setmaxnreg count");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}

struct Params {
  const float* LSE;
  const float* Dvec;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  float scale;
  float scale_log2;
  uint64_t wait_limit_ns;
  BwdSched sched;
};

enum : uint32_t {
  SITE_L_KVEMPTY = 1, SITE_L_QEMPTY, SITE_R_STAGED, SITE_Q_SFREE, SITE_M_KVFULL, SITE_M_QFULL,
  SITE_M_DQFREE, SITE_M_DSREADY, SITE_M_DKDVFREE, SITE_S_QFULL, SITE_S_SFULL, SITE_Q_DQFULL,
  SITE_E_DKDVDONE, SITE_DRAIN, SITE_ALIGN, SITE_M_PREADY, SITE_S_DPFULL, SITE_M_DOFULL,
  SITE_E_STAGED, SITE_E_READ, SITE_S_EREAD
};

struct B64Cfg {
  static constexpr int D = 64;
  static constexpr int TILE_BYTES = kChunkBytes;        // [128][64] bf16
  static constexpr int QST = 2;
  static constexpr int DQ_SLOT = 2 * kChunkBytes;        // [128][64] fp32: two 32-column boxes
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + QST * TILE_BYTES;
  static constexpr int OFF_DS = OFF_DO + QST * TILE_BYTES;   // dS^T [128][128]
  static constexpr int OFF_DQS = OFF_DS + 2 * kChunkBytes;   // [2] dQ slots
  static constexpr int OFF_STAT = OFF_DQS + 2 * DQ_SLOT;
  static constexpr int STAT_BYTES = 2 * 128 * 4;
  static constexpr int OFF_BAR = OFF_STAT + QST * STAT_BYTES;
  static constexpr int B_KVFULL = 0, B_KVEMPTY = 1;
  static constexpr int B_QFULL = 2;                  // [QST] Q_i and the stats
  static constexpr int B_DOFULL = B_QFULL + QST;     // [QST] dO_i
  static constexpr int B_QEMPTY = B_DOFULL + QST;    // [QST] the stage's readers are done
  static constexpr int B_DQSTAGED = B_QEMPTY + QST;  // [2] a dQ slot filled
  static constexpr int B_DQSFREE = B_DQSTAGED + 2;   // [2] ... and read by its reduce-adds
  static constexpr int B_SFULL = B_DQSFREE + 2;
  static constexpr int B_DPFULL = B_SFULL + 1;
  static constexpr int B_PREADY = B_DPFULL + 1;
  static constexpr int B_DSREADY = B_PREADY + 1;
  static constexpr int B_DQFULL = B_DSREADY + 1;
  static constexpr int B_DQFREE = B_DQFULL + 1;
  static constexpr int B_DKDVDONE = B_DQFREE + 1;
  static constexpr int B_DKDVFREE = B_DKDVDONE + 1;
  static constexpr int B_MMADONE = B_DKDVFREE + 1;
  static constexpr int B_ESTAGED = B_MMADONE + 1;
  static constexpr int B_EREAD = B_ESTAGED + 1;
  static constexpr int NBAR = B_EREAD + 1;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 320, TM_DQ = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_SS = idesc_bf16_f32(128, 128, 0, 0);
  static constexpr uint32_t IDESC_TS = idesc_bf16_f32(128, D, 0, 1);
  static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, D, 1, 1);
};
static_assert(B64Cfg::SMEM_BYTES <= 227 * 1024, "shared memory");
static_assert(B64Cfg::OFF_DS % 1024 == 0 && B64Cfg::OFF_DQS % 1024 == 0, "swizzled tiles");

constexpr int kB64Threads = 512;
constexpr int kB64DqWarp0 = 8;
constexpr int kB64MmaWarp = 12;
constexpr int kB64LoadWarp = 13;
constexpr int kB64RedWarp = 14;
// launched with 128 registers a thread; the control warpgroup (issuer,
// loads, reduce-adds, one idle warp) gives 24 of them to the dS groups and
// the dQ group: 256 x 136 + 128 x 136 + 128 x 104 = 512 x 128
constexpr int kB64RegsDs = 136, kB64RegsDq = 136, kB64RegsCtl = 104;
static_assert(256 * kB64RegsDs + 128 * kB64RegsDq + 128 * kB64RegsCtl == kB64Threads * 128,
              "register split");
static_assert(kB64RegsDs >= 128 && kB64RegsDq >= 128 && kB64RegsCtl <= 128,
              "the dS and dQ groups are raised from the launch's 128, the control group lowered");

// p_half for one 32-query chunk c (0..3) of S^T: P^T into pr[0..31] and, as
// bf16, into TMEM at tm_s + pcol.
__device__ __forceinline__ void p_chunk(uint32_t tmem_row, uint32_t tm_s, const float* nlse2,
                                        int c, uint32_t pcol, int key, bool kvalid, bool diag,
                                        int window, bool edge, int q0, float sl2, float* pr) {
  uint32_t sr[32];
  tmem_ld32(tmem_row + tm_s + 32 * c, sr);
  tmem_ld_wait();
  reg_fence32(sr);
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  const ulonglong2* l4 = reinterpret_cast<const ulonglong2*>(nlse2 + 32 * c);
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const ulonglong2 lv = l4[e / 4];
    float* o = pr + e;
    f2_unpack(ffma2(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2x2, lv.x),
              o[0], o[1]);
    f2_unpack(ffma2(f2_pack(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), sl2x2,
                    lv.y),
              o[2], o[3]);
#pragma unroll
    for (int u = 0; u < 4; ++u) o[u] = ex2_approx(o[u]);
  }
  if (diag) {
#pragma unroll
    for (int x = 0; x < 32; ++x)
      if (q0 + 32 * c + x < key) pr[x] = 0.f;
  }
  if (edge) {
#pragma unroll
    for (int x = 0; x < 32; ++x)
      if (q0 + 32 * c + x - key >= window) pr[x] = 0.f;
  }
  if (__any_sync(0xffffffffu, !kvalid)) {
#pragma unroll
    for (int x = 0; x < 32; ++x) pr[x] = kvalid ? pr[x] : 0.f;
  }
  uint32_t pp[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) pp[k] = pack_bf16x2(pr[2 * k], pr[2 * k + 1]);
  tmem_st16(tmem_row + tm_s + pcol, pp);
}

// ds_half for one 32-query chunk c: scale*dS^T as bf16 into TMEM at
// tm_dp + pcol and into the swizzled dS^T tile at ds_tile (pieces 4c .. 4c+3
// of row r).
__device__ __forceinline__ void ds_chunk(uint32_t tmem_row, uint32_t tm_dp, uint8_t* ds_tile,
                                         const float* ndsc, int c, uint32_t pcol, int r,
                                         float scale, const float* pr) {
  uint32_t dr[32];
  tmem_ld32(tmem_row + tm_dp + 32 * c, dr);
  tmem_ld_wait();
  reg_fence32(dr);
  const uint64_t sc2 = f2_pack(scale, scale);
  const ulonglong2* d4 = reinterpret_cast<const ulonglong2*>(ndsc + 32 * c);
  uint32_t dd[16];
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const ulonglong2 dv = d4[e / 4];
    const float* pe = pr + e;
    float a0, a1, a2, a3;
    f2_unpack(fmul2(ffma2(f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), sc2,
                          dv.x),
                    f2_pack(pe[0], pe[1])),
              a0, a1);
    f2_unpack(fmul2(ffma2(f2_pack(__uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3])), sc2,
                          dv.y),
                    f2_pack(pe[2], pe[3])),
              a2, a3);
    dd[e / 2] = pack_bf16x2(a0, a1);
    dd[e / 2 + 1] = pack_bf16x2(a2, a3);
  }
  tmem_st16(tmem_row + tm_dp + pcol, dd);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(ds_tile + swz_offset(r, 4 * c + k)) =
        make_uint4(dd[4 * k], dd[4 * k + 1], dd[4 * k + 2], dd[4 * k + 3]);
}

__global__ void __launch_bounds__(kB64Threads, 1)
    bwd64_kernel(const __grid_constant__ CUtensorMap mq,
                 const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv,
                 const __grid_constant__ CUtensorMap mdo,
                 const __grid_constant__ CUtensorMap mdq,
                 const __grid_constant__ CUtensorMap mdk,
                 const __grid_constant__ CUtensorMap mdv, const Params p) {
  using C = B64Cfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + C::OFF_BAR + 8u * (uint32_t)i; };
  auto sQ = [&](int s) { return sb + C::OFF_Q + (uint32_t)s * C::TILE_BYTES; };
  auto sdO = [&](int s) { return sb + C::OFF_DO + (uint32_t)s * C::TILE_BYTES; };
  auto sDQ = [&](int k) { return sb + C::OFF_DQS + (uint32_t)k * C::DQ_SLOT; };
  auto stat = [&](int s) {
    return reinterpret_cast<float*>(smem + C::OFF_STAT + s * C::STAT_BYTES);
  };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_TMEM);
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
      mbar_init(bar(C::B_DOFULL + s), 1);
      mbar_init(bar(C::B_QEMPTY + s), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(C::B_DQSTAGED + k), 128);
      mbar_init(bar(C::B_DQSFREE + k), 1);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_PREADY), 256);
    mbar_init(bar(C::B_DSREADY), 256);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQFREE), 128);
    mbar_init(bar(C::B_DKDVDONE), 1);
    mbar_init(bar(C::B_DKDVFREE), 256);
    mbar_init(bar(C::B_MMADONE), 1);
    mbar_init(bar(C::B_ESTAGED), 256);
    mbar_init(bar(C::B_EREAD), 1);
    *abort_flag = 0;
    if (sb & 1023u) record_timeout(abort_flag, SITE_ALIGN);
    fence_barrier_init();
  }
  if (warp == kB64MmaWarp) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  FA_TRACE_MARK(g_cta_trace, 0);
  const uint32_t tmem = *tmem_slot;
  const int nw = sc.n_waves();

  if (warp > kB64RedWarp) {
    reg_dealloc<kB64RegsCtl>();  // the idle member of the control warpgroup
  } else if (warp == kB64RedWarp) {
    reg_dealloc<kB64RegsCtl>();
    // ---------------------------------------------------- dQ reduce-adds
    // Block k's dQ tile, staged in slot k % 2, is added into the fp32
    // accumulator (two 32-column boxes); once the copies have read the slot
    // it is handed back to the dQ warpgroup.
    if (lane == 0) prefetch_tensormap(&mdq);
    griddep_wait();  // the accumulator is zeroed by the pre-pass
    uint32_t k = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      const int iend = sc.q_end(kb);
      for (int i = sc.q_begin(kb); i <= iend; ++i) {
        const int slot = k & 1;
        if (!wait_warp(bar(C::B_DQSTAGED + slot), (k >> 1) & 1, abort_flag, lim,
                       SITE_R_STAGED)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          for (int c = 0; c < 2; ++c)
            tma_reduce_add_3d(&mdq, sDQ(slot) + c * kChunkBytes, 32 * c, i * 128, bh);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(bar(C::B_DQSFREE + slot));
        }
        __syncwarp();
        ++k;
      }
    }
    if (lane == 0) bulk_wait_group0();  // the adds complete before the CTA exits
    __syncwarp();
  } else if (warp == kB64LoadWarp) {
    reg_dealloc<kB64RegsCtl>();
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
    float lraw[4] = {0.f, 0.f, 0.f, 0.f}, draw[4] = {0.f, 0.f, 0.f, 0.f};
    auto fetch_stats = [&](int bh_, int i_) {
      const size_t base = (size_t)bh_ * N;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int q = min(i_ * 128 + lane * 4 + e, N - 1);
        lraw[e] = p.LSE[base + q];
        draw[e] = p.Dvec[base + q];
      }
    };
    griddep_wait();  // D comes from the pre-pass launched just before this grid
    for (int w = 0; w < nw; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh0, kb0;
      sc.decode(item, bh0, kb0);
      fetch_stats(bh0, sc.q_begin(kb0));
      break;
    }
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      int nbh = -1, ni = 0;
      for (int w2 = w + 1; w2 < nw; ++w2) {
        const int item2 = sc.item_of(blockIdx.x, w2);
        if (item2 < 0) continue;
        int kb2;
        sc.decode(item2, nbh, kb2);
        ni = sc.q_begin(kb2);
        break;
      }
      if (it > 0 && !wait_warp(bar(C::B_KVEMPTY), (it - 1) & 1, abort_flag, lim,
                               SITE_L_KVEMPTY))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::TILE_BYTES);
        tma_load_3d(sb + C::OFF_K, &mk, bar(C::B_KVFULL), 0, kb * 128, bh);
        tma_load_3d(sb + C::OFF_V, &mv, bar(C::B_KVFULL), 0, kb * 128, bh);
      }
      kv_last = (int)(it & 1);
      const int iend = sc.q_end(kb);
      for (int i = sc.q_begin(kb); i <= iend; ++i) {
        const int s = qcnt % C::QST;
        const uint32_t ph = (qcnt / C::QST) & 1;
        float lv[4], dv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool valid = i * 128 + lane * 4 + e < N;
          lv[e] = valid ? -lraw[e] * 1.4426950408889634f : -INFINITY;
          dv[e] = valid ? -draw[e] * p.scale : 0.f;
        }
        if (i + 1 <= iend)
          fetch_stats(bh, i + 1);
        else if (nbh >= 0)
          fetch_stats(nbh, ni);
        // the stage's previous block: its four products that read Q or dO
        // and its dS phase (the reader of the stats) are done
        if (qcnt >= (uint32_t)C::QST &&
            !wait_warp(bar(C::B_QEMPTY + s), ph ^ 1, abort_flag, lim, SITE_L_QEMPTY)) {
          ok = false;
          break;
        }
        float* st = stat(s);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          st[lane * 4 + e] = lv[e];
          st[128 + lane * 4 + e] = dv[e];
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::B_QFULL + s), C::TILE_BYTES);
          tma_load_3d(sQ(s), &mq, bar(C::B_QFULL + s), 0, i * 128, bh);
          mbar_arrive_expect_tx(bar(C::B_DOFULL + s), C::TILE_BYTES);
          tma_load_3d(sdO(s), &mdo, bar(C::B_DOFULL + s), 0, i * 128, bh);
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
        if ((q_used >> s) & 1) {
          wait_one(bar(C::B_QFULL + s), (q_par >> s) & 1, &no_abort, lim, SITE_DRAIN);
          wait_one(bar(C::B_DOFULL + s), (q_par >> s) & 1, &no_abort, lim, SITE_DRAIN);
        }
    }
    __syncwarp();
  } else if (warp == kB64MmaWarp) {
    reg_dealloc<kB64RegsCtl>();
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
        if (!wait_one(bar(C::B_KVFULL), it & 1, abort_flag, lim, SITE_M_KVFULL)) break;
        tc_fence_after();
        const int i0 = sc.q_begin(kb);
        // S^T = K Q^T of block qc (TMEM's S^T columns hold the previous
        // block's P^T until its dV product, issued earlier, has read it)
        auto issue_s = [&](uint32_t qc) -> bool {
          const int st = qc % C::QST;
          if (!wait_one(bar(C::B_QFULL + st), (qc / C::QST) & 1, abort_flag, lim,
                        SITE_M_QFULL))
            return false;
          tc_fence_after();
          mma_rows_x_rows<D>(tmem + C::TM_S, sK, sQ(st), C::IDESC_SS);
          umma_commit(bar(C::B_SFULL));
          return true;
        };
        if (!issue_s(qcnt)) break;
        const int iend = sc.q_end(kb);
        for (int i = i0; i <= iend; ++i) {
          const int s = qcnt % C::QST;
          if (!wait_one(bar(C::B_DOFULL + s), (qcnt / C::QST) & 1, abort_flag, lim,
                        SITE_M_DOFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_rows_x_rows<D>(tmem + C::TM_DP, sV, sdO(s), C::IDESC_SS);
          umma_commit(bar(C::B_DPFULL));
          if (!wait_one(bar(C::B_PREADY), g & 1, abort_flag, lim, SITE_M_PREADY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool first = (i == i0);
          if (first && it > 0) {  // the previous item's dK/dV have left TMEM
            if (!wait_one(bar(C::B_DKDVFREE), (it - 1) & 1, abort_flag, lim,
                          SITE_M_DKDVFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          mma_tmem2_x_rows(tmem + C::TM_DV, tmem + C::TM_S, tmem + C::TM_S + 64, sdO(s),
                           C::IDESC_TS, !first);
          // the next block's S^T, over P^T_i (read by the dV product above)
          if (i + 1 <= iend && !issue_s(qcnt + 1)) {
            ok = false;
            break;
          }
          if (!wait_one(bar(C::B_DSREADY), g & 1, abort_flag, lim, SITE_M_DSREADY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tmem2_x_rows(tmem + C::TM_DK, tmem + C::TM_DP, tmem + C::TM_DP + 64, sQ(s),
                           C::IDESC_TS, !first);
          umma_commit(bar(C::B_QEMPTY + s));  // Q_i, dO_i and the stats: no later reader
          if (g > 0) {  // the previous block's dQ has left its TMEM columns
            if (!wait_one(bar(C::B_DQFREE), (g - 1) & 1, abort_flag, lim, SITE_M_DQFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          mma_colsT_x_rows(tmem + C::TM_DQ, sDS, sK, C::IDESC_DQ);
          umma_commit(bar(C::B_DQFULL));
          ++qcnt;
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
  } else if (warp >= kB64DqWarp0) {
    reg_alloc<kB64RegsDq>();
    // ------------------------------------------------------------------ dQ
    // dQ_i (lanes = the block's queries, 64 columns = d) to registers, its
    // TMEM columns released, then staged as swizzled fp32 in slot g % 2 once
    // that slot's previous tile has been read by its reduce-adds.
    const int wq = warp - kB64DqWarp0;
    const uint32_t tmem_row = tmem + ((uint32_t)(wq * 32) << 16);
    const int r = wq * 32 + lane;
    uint32_t g = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      const int iend = sc.q_end(kb);
      for (int i = sc.q_begin(kb); i <= iend; ++i) {
        const int slot = g & 1;
        if (!wait_warp(bar(C::B_DQFULL), g & 1, abort_flag, lim, SITE_Q_DQFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[2][32];
        tmem_ld32(tmem_row + C::TM_DQ, v[0]);
        tmem_ld32(tmem_row + C::TM_DQ + 32, v[1]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_DQFREE));
        reg_fence32(v[0]);
        reg_fence32(v[1]);
        if (g >= 2 && !wait_warp(bar(C::B_DQSFREE + slot), ((g >> 1) & 1) ^ 1, abort_flag, lim,
                                 SITE_Q_SFREE)) {
          ok = false;
          break;
        }
        uint8_t* stg = smem + C::OFF_DQS + slot * C::DQ_SLOT + r * 128;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(stg + c * kChunkBytes + ((k ^ (r & 7)) << 4)) =
                make_uint4(v[c][4 * k], v[c][4 * k + 1], v[c][4 * k + 2], v[c][4 * k + 3]);
        fence_proxy_async_smem();
        mbar_arrive(bar(C::B_DQSTAGED + slot));
        ++g;
      }
    }
  } else {
    reg_alloc<kB64RegsDs>();
    // ------------------------------------------- dS (both warpgroups), dK, dV
    const int grp = warp >> 2;     // 0: query columns 0-63, 1: 64-127
    const int wq = warp & 3;       // TMEM lane quarter
    const uint32_t tmem_row = tmem + ((uint32_t)(wq * 32) << 16);
    const int r = wq * 32 + lane;  // key row
    const float sl2 = p.scale_log2;
    const float scale = p.scale;
    uint32_t qcnt = 0, g = 0, it = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      const int key = kb * 128 + r;
      const bool kvalid = key < N;
      const int iend = sc.q_end(kb);
      for (int i = sc.q_begin(kb); i <= iend; ++i) {
        const int s = qcnt % C::QST;
        if (!wait_warp(bar(C::B_QFULL + s), (qcnt / C::QST) & 1, abort_flag, lim,
                       SITE_S_QFULL) ||
            !wait_warp(bar(C::B_SFULL), g & 1, abort_flag, lim, SITE_S_SFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* lse2 = stat(s);
        const int q0 = i * 128;
        const bool diag = sc.causal && i == kb;
        const bool edge = sc.window_edge(i, kb);
        float pr[64];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          p_chunk(tmem_row, C::TM_S, lse2, 2 * grp + h, 64u * grp + 16u * h, key, kvalid, diag,
                  sc.window, edge, q0, sl2, pr + 32 * h);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_PREADY));
        if (!wait_warp(bar(C::B_DPFULL), g & 1, abort_flag, lim, SITE_S_DPFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the dS tile doubles as the previous item's dK staging
        if (i == sc.q_begin(kb) && it > 0 &&
            !wait_warp(bar(C::B_EREAD), 1, abort_flag, lim, SITE_S_EREAD)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
          ds_chunk(tmem_row, C::TM_DP, smem + C::OFF_DS, lse2 + 128, 2 * grp + h,
                   64u * grp + 16u * h, r, scale, pr + 32 * h);
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::B_DSREADY));
        ++qcnt;
        ++g;
      }
      if (!ok) break;
      if (!wait_warp(bar(C::B_DKDVDONE), it & 1, abort_flag, lim, SITE_E_DKDVDONE)) break;
      tc_fence_after();
      // dV, then dK, through the dS tile and TMA stores, as in bwd_kernel
      constexpr int NPG = D / 16;
      constexpr int NL = D / 64;
      uint32_t pv[4 * NPG], pk[4 * NPG];
      auto grab = [&](uint32_t tcol, uint32_t (&dst)[4 * NPG]) {
#pragma unroll
        for (int l = 0; l < NL; ++l) {
          uint32_t v[32];
          tmem_ld32(tmem_row + tcol + (D / 2) * grp + 32 * l, v);
          tmem_ld_wait();
          reg_fence32(v);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            dst[16 * l + k] = pack_bf16x2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
        }
      };
      grab(C::TM_DV, pv);
      grab(C::TM_DK, pk);
      tc_fence_before();
      mbar_arrive(bar(C::B_DKDVFREE));
      const bool leader = warp == 0 && lane == 0;
      auto put = [&](const uint32_t (&src)[4 * NPG], const CUtensorMap* map, uint32_t par) {
#pragma unroll
        for (int q = 0; q < NPG; ++q)
          *reinterpret_cast<uint4*>(smem + C::OFF_DS + swz_offset(r, NPG * grp + q)) =
              make_uint4(src[4 * q], src[4 * q + 1], src[4 * q + 2], src[4 * q + 3]);
        fence_proxy_async_smem();
        mbar_arrive(bar(C::B_ESTAGED));
        if (leader && wait_one(bar(C::B_ESTAGED), par, abort_flag, lim, SITE_E_STAGED)) {
          tma_store_3d(map, sb + C::OFF_DS, 0, kb * 128, bh);  // rows past N are cut
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(bar(C::B_EREAD));
        }
      };
      put(pv, &mdv, 0);
      if (!wait_warp(bar(C::B_EREAD), 0, abort_flag, lim, SITE_E_READ)) break;
      put(pk, &mdk, 1);
      ++it;
    }
    if (warp == 0 && lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  FA_TRACE_MARK(g_cta_trace, 1);
  if (warp == kB64MmaWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

cudaError_t launch(const AttnShape& s, const TileMaps& maps, const float* LSE,
                     const float* Dvec, void* dK, void* dV, int num_sms, uint64_t lim,
                     cudaStream_t stream) {
  using C = B64Cfg;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t attr = smem_limit_once(bwd64_kernel, C::SMEM_BYTES, attr_done);
  if (attr != cudaSuccess) return attr;
  // The register split adds up to the launch's 512 x 128 registers; a build
  // that launched with another count is refused rather than launched.
  cudaFuncAttributes fattr{};
  const cudaError_t fe = cudaFuncGetAttributes(&fattr, bwd64_kernel);
  if (fe != cudaSuccess) return fe;
  if (fattr.numRegs != 128) return cudaErrorInvalidConfiguration;
  Params p;
  p.LSE = LSE;
  p.Dvec = Dvec;
  p.dK = reinterpret_cast<__nv_bfloat16*>(dK);
  p.dV = reinterpret_cast<__nv_bfloat16*>(dV);
  p.scale = s.scale;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.wait_limit_ns = lim;
  const int BH = s.B * s.H;
  const int n_blk = (s.N + 127) / 128;
  const int total = BH * n_blk;
  const int grid = total < num_sms ? total : num_sms;
  p.sched.init(BH, s.N, s.causal, grid, s.window);
  return launch_after(bwd64_kernel, dim3(grid), dim3(kB64Threads), C::SMEM_BYTES, stream,
                      maps.q, maps.k, maps.v, maps.dO, maps.dq_acc, maps.dk, maps.dv, p);
}

}  // namespace bwd64

cudaError_t launch_bwd64_tc(const AttnShape& s, const TileMaps& maps, const float* LSE,
                            const float* Dvec, void* dK, void* dV, int num_sms,
                            uint64_t wait_limit_ns, cudaStream_t stream) {
  if (s.d != 64 || s.drop.t4 != 0) return cudaErrorInvalidValue;
  return bwd64::launch(s, maps, LSE, Dvec, dK, dV, num_sms, wait_limit_ns, stream);
}

FA_DEFINE_STATUS_READER(read_status_bwd64_tc)

}  // namespace fa
