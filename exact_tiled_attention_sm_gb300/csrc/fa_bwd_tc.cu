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
// transposed tiles S^T = K Q_i^T and dP^T = V dO_i^T (rows = keys); two
// warpgroups (64 query columns each) turn S^T into P^T while the tensor core
// still computes dP^T, then turn dP^T into scale*dS^T while it already forms
// dV += P^T dO_i; then dK += dS^T Q_i (P^T and dS^T read straight from TMEM,
// so these two products read only one operand from shared memory) and
// dQ_i = dS K (dS read from shared memory).  Shared-memory reads by anything
// other than the tensor core make progress mostly while it runs such
// TMEM-operand products.  dQ_i is copied out of TMEM by both warpgroups into the
// just-consumed Q_i / dO_i stage as swizzled fp32 (the tensor memory is
// released as soon as it has been read); the load warp, the stage's next
// user, adds it into the fp32 dQ accumulator in global memory with TMA bulk
// reduce-adds before reloading the stage, Q_i first.
//
// Roles: warps 0-3 dS for query columns 0-63, half of the dQ readout and the
// dV epilogue; warps 4-7 dS for columns 64-127, the other half of the dQ
// readout and the dK epilogue; warp 8 tensor-core issuer and TMEM owner;
// warp 9 loads (TMA for K, V, Q, dO; plain loads for LSE and D) and the dQ
// bulk reduce-adds.
//
// TMEM: S^T [0,128), dP^T [128,256), dV [256, 256+d), dK [256+d, 256+2d).
// P^T overwrites columns [0,32) (queries 0-63) and [64,96) (queries 64-127)
// of S^T, each half inside the columns its own warpgroup has already read;
// dS^T likewise inside dP^T; dQ_i then reuses the dP^T columns.
//
// With dropout (the DR variant) the forward's keep mask M (entries 0 or
// 256/(256 - t)) is regenerated from the same Philox counters: the tensor
// core gets P o M (zeroed entries; the factor is applied to dV once, in the
// epilogue), and dS = P * (M dP - D).  Each thread draws the keep bytes of
// its key row for the 64 queries of its half while it would otherwise wait
// for the next S^T: one Philox call per lane and 4 x 4 patch, a byte
// transpose inside the lane and a word transpose across the quad.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "fa_sched.cuh"
#include "fa_tiles.cuh"
#include "fa_trace.cuh"

namespace fa {
namespace bwdtc {

FA_TRACE_DEFINE(g_cta_trace, fa_cta_trace_bwd)

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
  static constexpr int STAT_BYTES = 2 * 128 * 4;  // -LSE*log2(e)[128], -D*scale[128]
  static constexpr int OFF_BAR = OFF_STAT + QST * STAT_BYTES;
  static constexpr int B_KVFULL = 0, B_KVEMPTY = 1;
  static constexpr int B_QFULL = 2;                 // Q_i and the stats
  static constexpr int B_DOFULL = B_QFULL + QST;    // dO_i
  static constexpr int B_STAGED = B_DOFULL + QST;
  static constexpr int B_SFULL = B_STAGED + QST;   // S^T in TMEM
  static constexpr int B_DPFULL = B_SFULL + 1;      // dP^T in TMEM
  static constexpr int B_PREADY = B_DPFULL + 1;     // P^T written
  static constexpr int B_DSREADY = B_PREADY + 1;    // dS^T written
  static constexpr int B_DQFULL = B_DSREADY + 1;
  static constexpr int B_DQFREE = B_DQFULL + 1;
  static constexpr int B_DKDVDONE = B_DQFREE + 1;
  static constexpr int B_DKDVFREE = B_DKDVDONE + 1;
  static constexpr int B_MMADONE = B_DKDVFREE + 1;
  static constexpr int B_ESTAGED = B_MMADONE + 1;   // dV or dK tile in the dS buffer
  static constexpr int B_EREAD = B_ESTAGED + 1;     // ... and read by its TMA store
  static constexpr int NBAR = B_EREAD + 1;
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
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  float scale;
  float scale_log2;
  uint64_t wait_limit_ns;
  DropSpec drop;  // used by the DR variant only
  BwdSched sched;
};

enum : uint32_t {
  SITE_L_KVEMPTY = 1, SITE_L_STAGED, SITE_M_KVFULL, SITE_M_QFULL, SITE_M_DQFREE,
  SITE_M_DSREADY, SITE_M_DKDVFREE, SITE_S_QFULL, SITE_S_SFULL, SITE_Q_DQFULL,
  SITE_E_DKDVDONE, SITE_DRAIN, SITE_ALIGN, SITE_M_PREADY, SITE_S_DPFULL,
  SITE_M_DOFULL, SITE_E_STAGED, SITE_E_READ, SITE_S_EREAD
};

// Keep words of key row `key` for the 64 queries q_base + (0..63): word c
// holds the keep flags (keep_flags: top bit of each byte) of queries
// q_base + 4c + (0..3).  Lane q of a quad (keys 4*(key/4) + 0..3) draws the query patches
// 4g + q, g = 0..3; each call's words are indexed by query, its bytes by key,
// so a byte transpose regroups them by key and a quad transpose hands each
// lane its own key's words.
__device__ __forceinline__ void key_row_keep_words(uint32_t (&kw)[16],
                                                   const DropSpec& d, int bh,
                                                   int key, int q_base, int lane) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const Philox4 o = philox4x32_10((uint32_t)key >> 2,
                                    ((uint32_t)q_base >> 2) + 4 * g + (uint32_t)(lane & 3),
                                    (uint32_t)bh, 0u, d.k0, d.k1);
    uint32_t a[4] = {o.x[0], o.x[1], o.x[2], o.x[3]};
    byte_transpose(a);
    quad_transpose(a, lane);
#pragma unroll
    for (int c = 0; c < 4; ++c) kw[4 * g + c] = keep_flags(a[c], d);
  }
}

// One warpgroup's half of the softmax-gradient step for query block i:
// chunks c0, c0+1 of 32 query columns; thread = key row r (TMEM lane).
// Phase P (needs only S^T): P^T = 2^(S*scale*log2(e) - LSE*log2(e)), kept in
// fp32 registers and written to TMEM as bf16 at `pcol` (columns relative to
// the S^T block, inside the columns this warpgroup has read).  `nlse2` holds
// -LSE*log2(e) per query (-inf past N, so those columns are exactly 0).
// DR: TMEM gets P with the dropped entries zeroed (kw: key_row_keep_words);
// pr keeps the undropped values.
template <bool DR>
__device__ __forceinline__ void p_half(uint32_t tmem_row, uint32_t tm_s,
                                       const float* nlse2, int c0, uint32_t pcol,
                                       int key, bool kvalid, bool diag,
                                       int window, bool edge, int q0,
                                       float sl2, float (&pr)[64],
                                       const uint32_t (&kw)[16]) {
  uint32_t sr[2][32];
  tmem_ld32(tmem_row + tm_s + 32 * c0, sr[0]);
  tmem_ld32(tmem_row + tm_s + 32 * (c0 + 1), sr[1]);
  tmem_ld_wait();
  reg_fence32(sr[0]);
  reg_fence32(sr[1]);
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  const ulonglong2* l4 = reinterpret_cast<const ulonglong2*>(nlse2 + 32 * c0);
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const ulonglong2 lv = l4[(32 * h + e) / 4];
      float* o = pr + 32 * h + e;
      f2_unpack(ffma2(f2_pack(__uint_as_float(sr[h][e]), __uint_as_float(sr[h][e + 1])),
                      sl2x2, lv.x),
                o[0], o[1]);
      f2_unpack(ffma2(f2_pack(__uint_as_float(sr[h][e + 2]), __uint_as_float(sr[h][e + 3])),
                      sl2x2, lv.y),
                o[2], o[3]);
#pragma unroll
      for (int u = 0; u < 4; ++u) o[u] = ex2_approx(o[u]);
    }
  // causal diagonal block: keys after the query are invisible; key rows past
  // N (ragged last block) are zeroed too (warp-uniform, rare branches)
  if (diag) {
#pragma unroll
    for (int x = 0; x < 64; ++x)
      if (q0 + 32 * c0 + x < key) pr[x] = 0.f;
  }
  // sliding window: a query more than window - 1 rows after the key is
  // past it (only tiles the window's left edge cuts)
  if (edge) {
#pragma unroll
    for (int x = 0; x < 64; ++x)
      if (q0 + 32 * c0 + x - key >= window) pr[x] = 0.f;
  }
  if (__any_sync(0xffffffffu, !kvalid)) {
#pragma unroll
    for (int x = 0; x < 64; ++x) pr[x] = kvalid ? pr[x] : 0.f;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pp[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      pp[k] = pack_bf16x2(pr[32 * h + 2 * k], pr[32 * h + 2 * k + 1]);
      if constexpr (DR) pp[k] &= pair_mask(kw[8 * h + (k >> 1)], k);
    }
    tmem_st16(tmem_row + tm_s + pcol + 16 * h, pp);
  }
}

// Phase dS (needs dP^T): scale*dS^T = P * (dP*scale - D*scale), written as
// bf16 to TMEM at `pcol` of the dP^T block (the dK product's A operand) and
// to the swizzled shared tile (row = key r; the dQ product's A operand).
// `ndsc` holds -D*scale per query.  DR: dP of dropped entries is zeroed and
// `scale` is scale * 256/(256 - t), which gives P * (M dP - D) * scale.
template <int D, bool DR>
__device__ __forceinline__ void ds_half(uint32_t tmem_row, uint8_t* smem,
                                        const float* ndsc, int c0, uint32_t pcol,
                                        int r, float scale,
                                        const float (&pr)[64],
                                        const uint32_t (&kw)[16]) {
  using C = Cfg<D>;
  uint32_t dr[2][32];
  tmem_ld32(tmem_row + C::TM_DP + 32 * c0, dr[0]);
  tmem_ld32(tmem_row + C::TM_DP + 32 * (c0 + 1), dr[1]);
  tmem_ld_wait();
  reg_fence32(dr[0]);
  reg_fence32(dr[1]);
  const uint64_t sc2 = f2_pack(scale, scale);
  const ulonglong2* d4 = reinterpret_cast<const ulonglong2*>(ndsc + 32 * c0);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = c0 + h;
    uint32_t dd[16];
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const ulonglong2 dv = d4[(32 * h + e) / 4];
      const float* pe = pr + 32 * h + e;
      uint32_t g0 = dr[h][e], g1 = dr[h][e + 1], g2 = dr[h][e + 2], g3 = dr[h][e + 3];
      if constexpr (DR) {
        const uint32_t w = kw[8 * h + e / 4];
        g0 &= elem_mask(w, 0);
        g1 &= elem_mask(w, 1);
        g2 &= elem_mask(w, 2);
        g3 &= elem_mask(w, 3);
      }
      float a0, a1, a2, a3;
      f2_unpack(fmul2(ffma2(f2_pack(__uint_as_float(g0), __uint_as_float(g1)), sc2, dv.x),
                      f2_pack(pe[0], pe[1])),
                a0, a1);
      f2_unpack(fmul2(ffma2(f2_pack(__uint_as_float(g2), __uint_as_float(g3)), sc2, dv.y),
                      f2_pack(pe[2], pe[3])),
                a2, a3);
      dd[e / 2] = pack_bf16x2(a0, a1);
      dd[e / 2 + 1] = pack_bf16x2(a2, a3);
    }
    tmem_st16(tmem_row + C::TM_DP + pcol + 16 * h, dd);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<uint4*>(smem + C::OFF_DS + swz_offset(r, 4 * c + k)) =
          make_uint4(dd[4 * k], dd[4 * k + 1], dd[4 * k + 2], dd[4 * k + 3]);
  }
}

// Reads one 128 x D fp32 accumulator (lanes = rows) and stores row r as bf16
// (times `mult` when MUL).
template <int D, bool MUL = false>
__device__ __forceinline__ void store_rows_bf16(uint32_t tmem_col,
                                                __nv_bfloat16* out, bool store,
                                                float mult = 1.f) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(tmem_col + 32 * c, v);
    tmem_ld_wait();
    reg_fence32(v);
    uint4 o[4];
    uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      float a = __uint_as_float(v[2 * k]), b = __uint_as_float(v[2 * k + 1]);
      if constexpr (MUL) {
        a *= mult;
        b *= mult;
      }
      ow[k] = pack_bf16x2(a, b);
    }
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[k] = o[k];
    }
  }
}

template <int D, bool DR>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap mq,
               const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv,
               const __grid_constant__ CUtensorMap mdo,
               const __grid_constant__ CUtensorMap mdq,
               const __grid_constant__ CUtensorMap mdk,
               const __grid_constant__ CUtensorMap mdv, const Params p) {
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
      mbar_init(bar(C::B_DOFULL + s), 1);
      mbar_init(bar(C::B_STAGED + s), 256);    // dQ tile staged in the stage
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_PREADY), 256);
    mbar_init(bar(C::B_DSREADY), 256);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQFREE), 256);
    mbar_init(bar(C::B_DKDVDONE), 1);
    mbar_init(bar(C::B_DKDVFREE), 256);
    mbar_init(bar(C::B_MMADONE), 1);
    mbar_init(bar(C::B_ESTAGED), 256);
    mbar_init(bar(C::B_EREAD), 1);
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
  FA_TRACE_MARK(g_cta_trace, 0);
  const uint32_t tmem = *tmem_slot;
  const int nw = sc.n_waves();
  // No early griddep_launch_dependents here: the dQ conversion launched
  // after this grid starts when it exits (signalling at the start measured
  // 1% slower at d = 128, where no conversion CTA fits beside this one).

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------- loads
    // A Q/dO stage is reused every QST query blocks.  Its previous block's
    // dQ tile sits in it as fp32 staging (written by the dQ warpgroup): this
    // warp adds that tile into the accumulator with bulk reduce-adds, waits
    // until they have read it, then loads the stage's next block.
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      prefetch_tensormap(&mdo);
      prefetch_tensormap(&mdq);
    }
    uint32_t qcnt = 0, it = 0;
    int kv_last = -1;
    uint32_t q_used = 0, q_par = 0;
    int pend_bh[C::QST], pend_q0[C::QST];  // staged dQ tile of each stage
    for (int s = 0; s < C::QST; ++s) pend_bh[s] = -1, pend_q0[s] = 0;
    // reduce-adds one half of the dQ tile staged in stage s: half 0 is the
    // part held in the Q buffer (columns [0, d/2)), half 1 the part in the dO
    // buffer.  Lane 0; returns once the bulk copies have read that buffer.
    auto reduce_half = [&](int s, int half) {
      if (lane == 0 && pend_bh[s] >= 0) {
#pragma unroll
        for (int c = 0; c < C::CH; ++c) {  // 32-column fp32 boxes
          const uint32_t src = (half ? sdO(s) : sQ(s)) + c * kChunkBytes;
          tma_reduce_add_3d(&mdq, src, 32 * (c + C::CH * half), pend_q0[s],
                            pend_bh[s]);
        }
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      __syncwarp();
    };
    // LSE and D of a block's 128 queries (4 per lane), loaded one block
    // ahead so that their latency is hidden behind a whole block of work:
    // raw values from clamped addresses, validity applied when they are
    // written to the stage
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
    // D and the zeroed dQ accumulator come from the pre-pass launched just
    // before this grid: this warp is their only reader (the statistics and
    // the bulk reduce-adds)
    griddep_wait();
    // the first block this CTA processes
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
      // the block after this item's last one: the next item's first block
      int nbh = -1, ni = 0;
      for (int w2 = w + 1; w2 < nw; ++w2) {
        const int item2 = sc.item_of(blockIdx.x, w2);
        if (item2 < 0) continue;
        int kb2;
        sc.decode(item2, nbh, kb2);
        ni = sc.q_begin(kb2);
        break;
      }
      // The stage this item's first block will use still holds the staged
      // dQ of an earlier block: add it out now, while the previous item's
      // last blocks are still being computed, instead of after the K/V swap.
      if (qcnt >= (uint32_t)C::QST) {
        const int s = qcnt % C::QST;
        if (!wait_warp(bar(C::B_STAGED + s), ((qcnt / C::QST) & 1) ^ 1, abort_flag,
                       lim, SITE_L_STAGED))
          break;
        reduce_half(s, 0);
        reduce_half(s, 1);
        pend_bh[s] = -1;
      }
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
      const int iend = sc.q_end(kb);
      for (int i = sc.q_begin(kb); i <= iend; ++i) {
        const int s = qcnt % C::QST;
        const uint32_t ph = (qcnt / C::QST) & 1;
        // -LSE*log2(e) and -D*scale of this block's queries (fetched during
        // the previous block); rows past N get -inf so that their P is
        // exactly 0.  Then the next block's values are requested.
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
        if (qcnt >= (uint32_t)C::QST) {
          if (!wait_warp(bar(C::B_STAGED + s), ph ^ 1, abort_flag, lim,
                         SITE_L_STAGED)) {
            ok = false;
            break;
          }
          reduce_half(s, 0);
        }
        float* st = stat(s);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          st[lane * 4 + e] = lv[e];
          st[128 + lane * 4 + e] = dv[e];
        }
        // Q_i first: S^T and the P phase need only Q_i and the stats
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::B_QFULL + s), C::TILE_BYTES);
          for (int c = 0; c < C::CH; ++c)
            tma_load_3d(sQ(s) + c * kChunkBytes, &mq, bar(C::B_QFULL + s),
                        c * 64, i * 128, bh);
        }
        mbar_arrive(bar(C::B_QFULL + s));
        if (qcnt >= (uint32_t)C::QST) reduce_half(s, 1);
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::B_DOFULL + s), C::TILE_BYTES);
          for (int c = 0; c < C::CH; ++c)
            tma_load_3d(sdO(s) + c * kChunkBytes, &mdo, bar(C::B_DOFULL + s),
                        c * 64, i * 128, bh);
        }
        pend_bh[s] = bh;
        pend_q0[s] = i * 128;
        q_used |= 1u << s;
        q_par = (q_par & ~(1u << s)) | (ph << s);
        ++qcnt;
      }
      ++it;
    }
    // the last QST blocks' dQ tiles (skipped after an abort)
    if (ok && !*abort_flag) {
      for (uint32_t k = qcnt > (uint32_t)C::QST ? qcnt - C::QST : 0; k < qcnt; ++k) {
        const int s = k % C::QST;
        if (!wait_warp(bar(C::B_STAGED + s), (k / C::QST) & 1, abort_flag, lim,
                       SITE_L_STAGED))
          break;
        reduce_half(s, 0);
        reduce_half(s, 1);
      }
    }
    if (lane == 0) {  // every copy issued here completes before the CTA exits
      bulk_wait_group0();
      volatile int no_abort = 0;
      if (kv_last >= 0)
        wait_one(bar(C::B_KVFULL), (uint32_t)kv_last, &no_abort, lim, SITE_DRAIN);
      for (int s = 0; s < C::QST; ++s)
        if ((q_used >> s) & 1) {
          wait_one(bar(C::B_QFULL + s), (q_par >> s) & 1, &no_abort, lim,
                   SITE_DRAIN);
          wait_one(bar(C::B_DOFULL + s), (q_par >> s) & 1, &no_abort, lim,
                   SITE_DRAIN);
        }
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
        // S^T = K Q_i^T of block qc into TMEM (the previous block's P^T has
        // been consumed by its dV product, issued earlier by this thread)
        auto issue_s = [&](uint32_t qc) -> bool {
          const int st = qc % C::QST;
          if (!wait_one(bar(C::B_QFULL + st), (qc / C::QST) & 1, abort_flag,
                        lim, SITE_M_QFULL))
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
          if (g > 0) {  // dQ of the previous block has left TMEM
            if (!wait_one(bar(C::B_DQFREE), (g - 1) & 1, abort_flag, lim,
                          SITE_M_DQFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!wait_one(bar(C::B_DOFULL + s), (qcnt / C::QST) & 1, abort_flag,
                        lim, SITE_M_DOFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_rows_x_rows<D>(tmem + C::TM_DP, sV, sdO(s), C::IDESC_SS);
          umma_commit(bar(C::B_DPFULL));
          if (!wait_one(bar(C::B_PREADY), g & 1, abort_flag, lim,
                        SITE_M_PREADY)) {
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
          mma_tmem2_x_rows(tmem + C::TM_DV, tmem + C::TM_S, tmem + C::TM_S + 64,
                           sdO(s), C::IDESC_TS, !first);
          if (!wait_one(bar(C::B_DSREADY), g & 1, abort_flag, lim,
                        SITE_M_DSREADY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tmem2_x_rows(tmem + C::TM_DK, tmem + C::TM_DP,
                           tmem + C::TM_DP + 64, sQ(s), C::IDESC_TS, !first);
          mma_colsT_x_rows(tmem + C::TM_DP, sDS, sK, C::IDESC_DQ);
          umma_commit(bar(C::B_DQFULL));
          // the next block's S^T: its Q/dO stage was refilled after the
          // stage's previous dQ tile had been reduced out, a full block ago
          if (i + 1 <= iend && !issue_s(qcnt + 1)) {
            ok = false;
            break;
          }
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
  } else {
    // ------------------------------------- dS (both warpgroups), dQ, dK, dV
    const int grp = warp >> 2;        // 0: query columns 0-63, 1: 64-127
    const int wq = warp & 3;          // TMEM lane quarter
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tmem_row = tmem + lane_off;
    const int r = wq * 32 + lane;     // key row (dS, dK, dV) / query row (dQ)
    const float sl2 = p.scale_log2;
    const float scale = DR ? p.scale * p.drop.keep_scale : p.scale;  // of dP
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
        uint32_t kw[16];
        if constexpr (DR) key_row_keep_words(kw, p.drop, bh, key, i * 128 + 64 * grp, lane);
        if (!wait_warp(bar(C::B_QFULL + s), (qcnt / C::QST) & 1, abort_flag,
                       lim, SITE_S_QFULL) ||
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
        p_half<DR>(tmem_row, C::TM_S, lse2, 2 * grp, 64u * grp, key, kvalid, diag,
                   sc.window, edge, q0, sl2, pr, kw);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_PREADY));
        if (!wait_warp(bar(C::B_DPFULL), g & 1, abort_flag, lim, SITE_S_DPFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the dS tile doubles as the previous item's dK staging: written
        // only once that tile's TMA store has read it
        if (!DR && i == sc.q_begin(kb) && it > 0 &&
            !wait_warp(bar(C::B_EREAD), 1, abort_flag, lim, SITE_S_EREAD)) {
          ok = false;
          break;
        }
        ds_half<D, DR>(tmem_row, smem, lse2 + 128, 2 * grp, 64u * grp, r, scale, pr, kw);
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::B_DSREADY));
        // dQ_i, both warpgroups, d/2 columns each: TMEM -> registers (the
        // columns are released at once for the next dP^T) -> swizzled fp32
        // staging in the consumed stage (group 0 in the Q buffer, group 1 in
        // the dO buffer), which the load warp bulk reduce-adds into the
        // accumulator before refilling the stage
        if (!wait_warp(bar(C::B_DQFULL), g & 1, abort_flag, lim, SITE_Q_DQFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          constexpr int NC = D / 64;  // 32-column chunks per group
          uint32_t v[NC][32];
#pragma unroll
          for (int c = 0; c < NC; ++c)
            tmem_ld32(tmem_row + C::TM_DP + 32 * (NC * grp + c), v[c]);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(bar(C::B_DQFREE));
          uint8_t* stg = smem + ((grp ? sdO(s) : sQ(s)) - sb) + r * 128;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            reg_fence32(v[c]);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<uint4*>(stg + c * kChunkBytes + ((k ^ (r & 7)) << 4)) =
                  make_uint4(v[c][4 * k], v[c][4 * k + 1], v[c][4 * k + 2], v[c][4 * k + 3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(C::B_STAGED + s));
        }
        ++qcnt;
        ++g;
      }
      if (!ok) break;
      if (!wait_warp(bar(C::B_DKDVDONE), it & 1, abort_flag, lim,
                     SITE_E_DKDVDONE))
        break;
      tc_fence_after();
      if constexpr (DR) {  // a row per thread (measured faster with dropout)
        const bool store = key < N;
        const size_t rowoff = ((size_t)bh * N + (size_t)(store ? key : 0)) * D;
        if (grp == 0)
          store_rows_bf16<D, true>(tmem_row + C::TM_DV, p.dV + rowoff, store,
                                   p.drop.keep_scale);
        else
          store_rows_bf16<D>(tmem_row + C::TM_DK, p.dK + rowoff, store);
        tc_fence_before();
        mbar_arrive(bar(C::B_DKDVFREE));
      } else {
        // dV, then dK, leave through the dS tile (free: the item's last dQ
        // product has completed) and TMA stores of whole 64-column boxes,
        // instead of a 2*D-byte row per thread.  Group g converts columns
        // [g*D/2, (g+1)*D/2) of both; TMEM is released once both are read.
        constexpr int NPG = D / 16;  // 16-byte pieces of a row per group
        constexpr int NL = D / 64;   // 32-column TMEM loads per group
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
              dst[16 * l + k] = pack_bf16x2(__uint_as_float(v[2 * k]),
                                            __uint_as_float(v[2 * k + 1]));
          }
        };
        grab(C::TM_DV, pv);
        grab(C::TM_DK, pk);
        tc_fence_before();
        mbar_arrive(bar(C::B_DKDVFREE));
        const bool leader = warp == 0 && lane == 0;
        // stage this thread's half row, then one thread stores the tile
        auto put = [&](const uint32_t (&src)[4 * NPG], const CUtensorMap* map,
                       uint32_t par) {
#pragma unroll
          for (int q = 0; q < NPG; ++q)
            *reinterpret_cast<uint4*>(smem + C::OFF_DS + swz_offset(r, NPG * grp + q)) =
                make_uint4(src[4 * q], src[4 * q + 1], src[4 * q + 2], src[4 * q + 3]);
          fence_proxy_async_smem();
          mbar_arrive(bar(C::B_ESTAGED));
          if (leader &&
              wait_one(bar(C::B_ESTAGED), par, abort_flag, lim, SITE_E_STAGED)) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c)  // rows past N are cut by the copy
              tma_store_3d(map, sb + C::OFF_DS + c * kChunkBytes, 64 * c, kb * 128, bh);
            bulk_commit_group();
            bulk_wait_group_read0();
            mbar_arrive(bar(C::B_EREAD));
          }
        };
        put(pv, &mdv, 0);
        if (!wait_warp(bar(C::B_EREAD), 0, abort_flag, lim, SITE_E_READ)) break;
        put(pk, &mdk, 1);
      }
      ++it;
    }
    // the last dK stores complete before the CTA exits
    if (!DR && warp == 0 && lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  FA_TRACE_MARK(g_cta_trace, 1);
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool DR>
cudaError_t launch(const AttnShape& s, const TileMaps& maps, const float* LSE,
                   const float* Dvec, void* dK, void* dV, int num_sms,
                   uint64_t lim, cudaStream_t stream) {
  using C = Cfg<D>;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t attr = smem_limit_once(bwd_kernel<D, DR>, C::SMEM_BYTES, attr_done);
  if (attr != cudaSuccess) return attr;
  Params p;
  p.LSE = LSE;
  p.Dvec = Dvec;
  p.dK = reinterpret_cast<__nv_bfloat16*>(dK);
  p.dV = reinterpret_cast<__nv_bfloat16*>(dV);
  p.scale = s.scale;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.wait_limit_ns = lim;
  p.drop = s.drop;
  const int BH = s.B * s.H;
  const int n_blk = (s.N + 127) / 128;
  const int total = BH * n_blk;
  const int grid = total < num_sms ? total : num_sms;
  p.sched.init(BH, s.N, s.causal, grid, s.window);
  // a dependent of the pre-pass launched just before (D, the zeroed dQ
  // accumulator): its set-up overlaps the pre-pass's last CTAs
  return launch_after(bwd_kernel<D, DR>, dim3(grid), dim3(kThreads), C::SMEM_BYTES, stream,
                      maps.q, maps.k, maps.v, maps.dO, maps.dq_acc, maps.dk, maps.dv, p);
}

}  // namespace bwdtc

cudaError_t launch_bwd_tc(const AttnShape& s, const TileMaps& maps,
                          const float* LSE, const float* Dvec, float* dQacc,
                          void* dK, void* dV, int num_sms,
                          uint64_t wait_limit_ns, cudaStream_t stream) {
  (void)dQacc;  // reached through maps.dq_acc
  const bool dr = s.drop.t4 != 0;
  const uint64_t lim = wait_limit_ns;
  if (s.d == 64)
    return dr ? bwdtc::launch<64, true>(s, maps, LSE, Dvec, dK, dV, num_sms, lim, stream)
              : bwdtc::launch<64, false>(s, maps, LSE, Dvec, dK, dV, num_sms, lim, stream);
  return dr ? bwdtc::launch<128, true>(s, maps, LSE, Dvec, dK, dV, num_sms, lim, stream)
            : bwdtc::launch<128, false>(s, maps, LSE, Dvec, dK, dV, num_sms, lim, stream);
}

FA_DEFINE_STATUS_READER(read_status_bwd_tc)

}  // namespace fa
