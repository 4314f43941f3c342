// fa_bwd256_tc.cu -- bf16 exact attention backward for head dimension 256 on
// sm_103a tensor cores.
//
// The same recomputation as the d <= 128 backward ("Flash Attention, From
// First Principles", "The backward pass -- resurrection"; "FlashAttention
// from scratch", follow-up on the backward pass):
//   P = exp(scale*QK^T - LSE), dV += P^T dO, dP = dO V^T,
//   dS = P * (dP - D), D = rowsum(dO * O), dK += scale*dS^T Q, dQ += scale*dS K,
// K/V-outer, so that dK and dV accumulate on chip and are written once.
//
// The d^2/M wall ("Flash Attention, From First Principles", "The rent
// arithmetic") in TMEM form: for 128 keys the two accumulators dV and dK
// alone take 2 x 256 of TMEM's 512 columns, leaving nothing for the score
// tiles.  So a work item (one head, one block of 128 keys) makes two passes
// over its query blocks, one per HALF of the head dimension, h: pass h
// accumulates dV[:, h] and dK[:, h] (128 columns each) and adds dQ[:, h];
// the score products S^T = K Q^T and dP^T = V dO^T contract over all 256
// columns and are computed in both passes (2 of the 5 products twice: 14 of
// the 10 counted N^2 d units).  K and V stay loaded across the two passes,
// and the next item's K and V rows are prefetched into L2 during the second
// pass.  Query blocks are
// 64 rows, so that K (64 KiB), a two-stage ring of Q_i and dO_i (4 x 32 KiB)
// and the dS tile fit in shared memory; V is the A operand of dP^T and lives
// in TMEM instead (it has no other reader).
//
// Per query block i, with P^T and dS^T rows = keys (TMEM lanes):
//   S^T  = K Q_i^T          SS, M = 128 keys, N = 64 queries, K = 256
//   dP^T = V dO_i^T         A = V from TMEM, B = dO_i
//   P^T  = 2^(S^T scale log2 e - LSE log2 e), written over S^T as bf16
//   dV_h += P^T dO_i[:, h]  A = P^T from TMEM, N = 128
//   dS^T = P^T * (dP^T scale - D scale), over dP^T (bf16) and into shared
//          memory as dS^T [key][query]
//   dK_h += dS^T Q_i[:, h]  A = dS^T from TMEM
//   dQ_h^T = K_h^T dS^T     SS, M = 128 (the half's d), N = 64 queries,
//                           K = 128 keys, over dP^T's columns
// and dQ_h^T goes from TMEM to registers (thread = one d, 32 queries) and is
// added to the fp32 dQ accumulator with coalesced red.global.add (a warp adds
// 32 consecutive floats of one query row per instruction).
//
// Roles: warps 0-3 query columns 0-31 of each block, the dV epilogue and
// V columns 0-127 into TMEM; warps 4-7 query columns 32-63, the dK epilogue
// and V columns 128-255; warps 8-11 (the dQ warpgroup) read dQ_h^T out of
// TMEM and add it to the accumulator, so that the dS warpgroups go from
// dS(i) straight on to P(i+1) while those adds run; warp 12 tensor-core
// issuer and TMEM owner; warp 13 TMA loads (K, Q_i, dO_i) and the per-query
// statistics (-LSE log2 e, -D scale) of each block.
//
// TMEM: S^T [0,64), dP^T [64,128), dV_h [128,256), dK_h [256,384),
// V [384,512) (bf16 pairs).  Warpgroup g writes its P^T into columns
// [32g, 32g+16) and its dS^T into [64+32g, 64+32g+16), inside the columns it
// has itself read, so the two groups never overwrite what the other still
// reads; the dV and dK products take their A operand from those two pieces.
//
// With dropout (the DR variant) the forward's keep mask is regenerated from
// the same Philox counters, as in the d <= 128 backward: P o M goes to the
// tensor core (dropped entries zeroed, the factor applied in dV's
// epilogue) and dS = P * (M dP - D).
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "fa_sched.cuh"
#include "fa_tiles.cuh"
#include "fa_trace.cuh"

namespace fa {
namespace bwd256 {

FA_TRACE_DEFINE(g_cta_trace, fa_cta_trace_bwd256)

constexpr int D = 256;
constexpr int BQ = 64;                      // queries per block
constexpr int HALF = 128;                   // columns of d per work item
constexpr int QCHUNK = 64 * 128;            // a 64-column chunk of 64 rows: 8 KiB
constexpr int QTILE = 4 * QCHUNK;           // Q_i or dO_i: [64][256] bf16, 32 KiB
constexpr int KTILE = 4 * kChunkBytes;      // K: [128][256] bf16, 64 KiB
constexpr int QST = 2;                      // Q / dO ring stages
constexpr int OFF_K = 0;
constexpr int OFF_Q = OFF_K + KTILE;
constexpr int OFF_DO = OFF_Q + QST * QTILE;
constexpr int OFF_DS = OFF_DO + QST * QTILE;  // dS^T [128 keys][64 queries] bf16
constexpr int OFF_STAT = OFF_DS + kChunkBytes;
constexpr int STAT_BYTES = 2 * BQ * 4;        // -LSE*log2(e)[64], -D*scale[64]
constexpr int OFF_BAR = OFF_STAT + QST * STAT_BYTES;
constexpr int B_KFULL = 0, B_KEMPTY = 1;
constexpr int B_QFULL = 2;                 // [QST] Q_i and the stats
constexpr int B_DOFULL = B_QFULL + QST;    // [QST] dO_i
constexpr int B_QEMPTY = B_DOFULL + QST;   // [QST] the stage's readers are done
constexpr int B_SFULL = B_QEMPTY + QST;
constexpr int B_DPFULL = B_SFULL + 1;
constexpr int B_PREADY = B_DPFULL + 1;
constexpr int B_DSREADY = B_PREADY + 1;
constexpr int B_DQFULL = B_DSREADY + 1;
constexpr int B_DQFREE = B_DQFULL + 1;
constexpr int B_VREADY = B_DQFREE + 1;
constexpr int B_DKDVDONE = B_VREADY + 1;
constexpr int B_DKDVFREE = B_DKDVDONE + 1;
constexpr int B_MMADONE = B_DKDVFREE + 1;
constexpr int NBAR = B_MMADONE + 1;
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM_BYTES = OFF_ABORT + 4;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
constexpr uint32_t TM_S = 0, TM_DP = 64, TM_DV = 128, TM_DK = 256, TM_V = 384;
constexpr uint32_t TMEM_COLS = 512;
// S^T and dP^T: M = 128 keys, N = 64 queries, both operands K-major
constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BQ, 0, 0);
// dV_h, dK_h: A from TMEM, B = Q_i or dO_i columns of half h read MN-major
constexpr uint32_t IDESC_KV = idesc_bf16_f32(128, HALF, 0, 1);
// dQ_h^T: A = K_h^T and B = dS^T, both MN-major
constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, BQ, 1, 1);

constexpr int kThreads = 448;
constexpr int kDqWarp0 = 8;   // warps 8-11: the dQ warpgroup
constexpr int kMmaWarp = 12;
constexpr int kLoadWarp = 13;

// Work items: (head, 128-key block kb), each walked twice (once per half of
// d).  Under the causal mask the query blocks of 64 rows visited by key
// block kb start at 2kb; with a sliding window of w keys they end at the
// block of the last query whose window still reaches the key block's last
// key.  Causal cost falls with kb, so items are listed kb-ascending inside
// head groups and taken in snake waves, as in the d <= 128 backward.
struct Sched {
  int BH, N, causal, window, grid;
  int n_kb, n_qb, group, total_items;

  __host__ __device__ void init(int bh, int n, int is_causal, int grid_size, int win) {
    BH = bh;
    N = n;
    window = win > 0 ? win : 0;
    causal = (is_causal || window > 0) ? 1 : 0;
    grid = grid_size;
    n_kb = (N + 127) / 128;
    n_qb = (N + BQ - 1) / BQ;
    int g = (causal ? kBwdGroupWaves : 1) * grid / n_kb;
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    group = g;
    total_items = BH * n_kb;
  }
  __host__ __device__ int n_waves() const { return (total_items + grid - 1) / grid; }
  __host__ __device__ int item_of(int cta, int w) const {
    const int pos = (w & 1) ? (grid - 1 - cta) : cta;
    const int i = w * grid + pos;
    return i < total_items ? i : -1;
  }
  __host__ __device__ void decode(int i, int& bh, int& kb) const {
    const int per_group = group * n_kb;
    const int full_groups = BH / group;
    const int full_items = full_groups * per_group;
    int g, r, gs;
    if (i < full_items) {
      g = i / per_group;
      r = i - g * per_group;
      gs = group;
    } else {
      g = full_groups;
      r = i - full_items;
      gs = BH - full_groups * group;
    }
    kb = r / gs;
    bh = g * group + r % gs;
  }
  __host__ __device__ int q_begin(int kb) const { return causal ? 2 * kb : 0; }
  __host__ __device__ int q_end(int kb) const {
    if (window == 0) return n_qb - 1;
    const int last_q = kb * 128 + 127 + window - 1;  // its window's newest row
    const int blk = last_q / BQ;
    return blk < n_qb - 1 ? blk : n_qb - 1;
  }
  // Does query block i share rows with key block kb (the causal diagonal)?
  __host__ __device__ bool diag(int i, int kb) const {
    return causal && i <= 2 * kb + 1;
  }
  // Does the window's left edge cut the tile (some query too far past some key)?
  __host__ __device__ bool window_edge(int i, int kb) const {
    return window > 0 && i * BQ + BQ - 1 - kb * 128 >= window;
  }
};

struct Params {
  const float* LSE;
  const float* Dvec;
  const __nv_bfloat16* V;
  float* dQacc;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  float scale;
  float scale_log2;
  uint64_t wait_limit_ns;
  DropSpec drop;  // DR variant only
  Sched sched;
};

enum : uint32_t {
  SITE_L_KEMPTY = 1, SITE_L_QEMPTY, SITE_M_KFULL, SITE_M_QFULL, SITE_M_DQFREE,
  SITE_M_DSREADY, SITE_M_DKDVFREE, SITE_S_QFULL, SITE_S_SFULL, SITE_Q_DQFULL,
  SITE_E_DKDVDONE, SITE_DRAIN, SITE_ALIGN, SITE_M_PREADY, SITE_S_DPFULL,
  SITE_M_DOFULL, SITE_M_VREADY
};

// K-major step kk (16 elements) of a tile whose 64-column chunks hold 64
// rows (8 KiB apart).
__host__ __device__ constexpr uint32_t kstep64(int kk) {
  return (uint32_t)(((kk >> 2) * QCHUNK + (kk & 3) * 32) >> 4);
}

// S^T (or dP^T) = A B^T over the 256 columns: A either K in shared memory
// (128-row chunks) or V in TMEM (bf16 pairs, 8 columns per step of 16), B a
// [64][256] tile (64-row chunks), 16 steps.
__device__ __forceinline__ void mma_scores_ss(uint32_t d_tmem, uint32_t sk, uint32_t sq) {
  const uint64_t da = kdesc(sk), db = kdesc(sq);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    umma_ss(d_tmem, da + kstep(kk), db + kstep64(kk), IDESC_S, kk > 0 ? 1u : 0u);
}
__device__ __forceinline__ void mma_scores_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t sq) {
  const uint64_t db = kdesc(sq);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    umma_ts(d_tmem, a_tmem + 8 * kk, db + kstep64(kk), IDESC_S, kk > 0 ? 1u : 0u);
}

// dV_h (or dK_h) (+)= A B: A (128 keys x 64 queries) in TMEM as the two
// warpgroups' pieces (queries 0-31 at a_tmem, 32-63 at a_tmem + 32; 8 columns
// per step of 16 queries), B = columns [128h, 128h + 128) of a [64][256] tile
// read MN-major (N runs = its chunks 2h and 2h + 1, 8 KiB apart).
__device__ __forceinline__ void mma_half_acc(uint32_t d_tmem, uint32_t a_tmem,
                                             uint32_t stile, int h, bool accumulate) {
  const uint64_t db = sdesc_sw128(stile + 2 * h * QCHUNK, QCHUNK, 1024);
#pragma unroll
  for (int kk = 0; kk < BQ / 16; ++kk)
    umma_ts(d_tmem, a_tmem + (kk >> 1) * 32 + (kk & 1) * 8, db + mstep(kk), IDESC_KV,
            (accumulate || kk > 0) ? 1u : 0u);
}

// Keep words of key row `key` for the 32 queries q_base + (0..31): word c
// holds the keep flags of queries q_base + 4c + (0..3) (the d <= 128
// backward's key_row_keep_words for half as many queries).
__device__ __forceinline__ void key_row_keep_words32(uint32_t (&kw)[8], const DropSpec& d,
                                                     int bh, int key, int q_base, int lane) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
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

template <bool DR>
__global__ void __launch_bounds__(kThreads, 1)
    bwd256_kernel(const __grid_constant__ CUtensorMap mq,
                  const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mdo, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + OFF_BAR + 8u * (uint32_t)i; };
  auto sQ = [&](int s) { return sb + OFF_Q + (uint32_t)s * QTILE; };
  auto sdO = [&](int s) { return sb + OFF_DO + (uint32_t)s * QTILE; };
  auto stat = [&](int s) {
    return reinterpret_cast<float*>(smem + OFF_STAT + s * STAT_BYTES);
  };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Sched& sc = p.sched;
  const uint64_t lim = p.wait_limit_ns;
  const int N = sc.N;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KFULL), 1);
    mbar_init(bar(B_KEMPTY), 1);
    for (int s = 0; s < QST; ++s) {
      mbar_init(bar(B_QFULL + s), 1 + 32);  // TMA arrive + 32 stat writers
      mbar_init(bar(B_DOFULL + s), 1);
      mbar_init(bar(B_QEMPTY + s), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_DPFULL), 1);
    mbar_init(bar(B_PREADY), 256);
    mbar_init(bar(B_DSREADY), 256);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQFREE), 128);
    mbar_init(bar(B_VREADY), 256);
    mbar_init(bar(B_DKDVDONE), 1);
    mbar_init(bar(B_DKDVFREE), 256);
    mbar_init(bar(B_MMADONE), 1);
    *abort_flag = 0;
    if (sb & 1023u) record_timeout(abort_flag, SITE_ALIGN);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  FA_TRACE_MARK(g_cta_trace, 0);
  const uint32_t tmem = *tmem_slot;
  const int nw = sc.n_waves();
  // The dQ conversion launched after this grid may start now: one of its
  // CTAs fits beside this one and waits (griddep_wait) for this grid to end.
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mdo);
    }
    uint32_t qcnt = 0, it = 0;
    int k_last = -1;
    uint32_t q_used = 0, q_par = 0;
    // LSE and D of a block's 64 queries (2 per lane), loaded one block ahead
    // from clamped addresses; validity applied when written to the stage
    float lraw[2] = {0.f, 0.f}, draw[2] = {0.f, 0.f};
    griddep_wait();  // D comes from the pre-pass launched just before
    auto fetch_stats = [&](int bh_, int i_) {
      const size_t base = (size_t)bh_ * N;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int q = min(i_ * BQ + lane * 2 + e, N - 1);
        lraw[e] = p.LSE[base + q];
        draw[e] = p.Dvec[base + q];
      }
    };
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
      int nbh = -1, nkb = 0, ni = 0;  // the next item and its first block
      for (int w2 = w + 1; w2 < nw; ++w2) {
        const int item2 = sc.item_of(blockIdx.x, w2);
        if (item2 < 0) continue;
        sc.decode(item2, nbh, nkb);
        ni = sc.q_begin(nkb);
        break;
      }
      if (it > 0 && !wait_warp(bar(B_KEMPTY), (it - 1) & 1, abort_flag, lim, SITE_L_KEMPTY))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_KFULL), KTILE);
        for (int c = 0; c < 4; ++c)
          tma_load_3d(sb + OFF_K + c * kChunkBytes, &mk, bar(B_KFULL), c * 64, kb * 128, bh);
      }
      k_last = (int)(it & 1);
      const int iend = sc.q_end(kb);
      for (int h = 0; h < 2 && ok; ++h)
      for (int i = sc.q_begin(kb); i <= iend; ++i) {
        if (h == 1 && i == sc.q_begin(kb) && nbh >= 0 && lane == 0) {
          // the next item's K tile into L2 while this item's second pass runs
          for (int c = 0; c < 4; ++c) tma_prefetch_l2_3d(&mk, c * 64, nkb * 128, nbh);
        }
        const int s = qcnt % QST;
        const uint32_t ph = (qcnt / QST) & 1;
        float lv[2], dv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool valid = i * BQ + lane * 2 + e < N;
          lv[e] = valid ? -lraw[e] * 1.4426950408889634f : -INFINITY;
          dv[e] = valid ? -draw[e] * p.scale : 0.f;
        }
        if (i + 1 <= iend)
          fetch_stats(bh, i + 1);
        else if (h == 0)
          fetch_stats(bh, sc.q_begin(kb));
        else if (nbh >= 0)
          fetch_stats(nbh, ni);
        // the stage's previous block: its S^T, dP^T, dV and dK products
        // (the readers of Q and dO) have completed
        if (qcnt >= (uint32_t)QST &&
            !wait_warp(bar(B_QEMPTY + s), ph ^ 1, abort_flag, lim, SITE_L_QEMPTY)) {
          ok = false;
          break;
        }
        float* st = stat(s);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          st[lane * 2 + e] = lv[e];
          st[BQ + lane * 2 + e] = dv[e];
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_QFULL + s), QTILE);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(sQ(s) + c * QCHUNK, &mq, bar(B_QFULL + s), c * 64, i * BQ, bh);
          mbar_arrive_expect_tx(bar(B_DOFULL + s), QTILE);
          for (int c = 0; c < 4; ++c)
            tma_load_3d(sdO(s) + c * QCHUNK, &mdo, bar(B_DOFULL + s), c * 64, i * BQ, bh);
        }
        mbar_arrive(bar(B_QFULL + s));
        q_used |= 1u << s;
        q_par = (q_par & ~(1u << s)) | (ph << s);
        ++qcnt;
      }
      ++it;
    }
    if (lane == 0) {  // every copy issued here lands before the CTA exits
      volatile int no_abort = 0;
      if (k_last >= 0) wait_one(bar(B_KFULL), (uint32_t)k_last, &no_abort, lim, SITE_DRAIN);
      for (int s = 0; s < QST; ++s)
        if ((q_used >> s) & 1) {
          wait_one(bar(B_QFULL + s), (q_par >> s) & 1, &no_abort, lim, SITE_DRAIN);
          wait_one(bar(B_DOFULL + s), (q_par >> s) & 1, &no_abort, lim, SITE_DRAIN);
        }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- tensor core
    if (lane == 0) {
      uint32_t qcnt = 0, it = 0, g = 0, hc = 0;
      bool ok = true;
      const uint32_t sK = sb + OFF_K, sDS = sb + OFF_DS;
      for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
        const int item = sc.item_of(blockIdx.x, w);
        if (item < 0) continue;
        int bh, kb;
        sc.decode(item, bh, kb);
        if (!wait_one(bar(B_KFULL), it & 1, abort_flag, lim, SITE_M_KFULL)) break;
        tc_fence_after();
        const int i0 = sc.q_begin(kb);
        // S^T of block qc into TMEM (the previous block's P^T has been read
        // by its dV product, issued earlier by this thread)
        auto issue_s = [&](uint32_t qc) -> bool {
          const int st = qc % QST;
          if (!wait_one(bar(B_QFULL + st), (qc / QST) & 1, abort_flag, lim, SITE_M_QFULL))
            return false;
          tc_fence_after();
          mma_scores_ss(tmem + TM_S, sK, sQ(st));
          umma_commit(bar(B_SFULL));
          return true;
        };
        if (!issue_s(qcnt)) break;
        // V of this item has been written into TMEM by the dS warpgroups
        // (after the previous item's products, which read the old V, had
        // completed)
        if (!wait_one(bar(B_VREADY), it & 1, abort_flag, lim, SITE_M_VREADY)) break;
        tc_fence_after();
        const int iend = sc.q_end(kb);
        for (int h = 0; h < 2 && ok; ++h) {
        for (int i = i0; i <= iend; ++i) {
          const int s = qcnt % QST;
          if (g > 0) {  // dQ^T of the previous block has left TMEM
            if (!wait_one(bar(B_DQFREE), (g - 1) & 1, abort_flag, lim, SITE_M_DQFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!wait_one(bar(B_DOFULL + s), (qcnt / QST) & 1, abort_flag, lim, SITE_M_DOFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_scores_ts(tmem + TM_DP, tmem + TM_V, sdO(s));
          umma_commit(bar(B_DPFULL));
          if (!wait_one(bar(B_PREADY), g & 1, abort_flag, lim, SITE_M_PREADY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool first = (i == i0);
          if (first && hc > 0) {  // the previous pass's dK, dV have been stored
            if (!wait_one(bar(B_DKDVFREE), (hc - 1) & 1, abort_flag, lim, SITE_M_DKDVFREE)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          mma_half_acc(tmem + TM_DV, tmem + TM_S, sdO(s), h, !first);
          if (!wait_one(bar(B_DSREADY), g & 1, abort_flag, lim, SITE_M_DSREADY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_half_acc(tmem + TM_DK, tmem + TM_DP, sQ(s), h, !first);
          umma_commit(bar(B_QEMPTY + s));  // Q_i and dO_i have no later reader
          mma_colsT_x_rows(tmem + TM_DP, sK + 2 * h * kChunkBytes, sDS, IDESC_DQ);
          umma_commit(bar(B_DQFULL));
          // the next block's S^T (the first block again after the first pass)
          if ((i + 1 <= iend || h == 0) && !issue_s(qcnt + 1)) {
            ok = false;
            break;
          }
          ++qcnt;
          ++g;
        }
        if (!ok) break;
        umma_commit(bar(B_DKDVDONE));
        ++hc;
        }
        if (!ok) break;
        umma_commit(bar(B_KEMPTY));
        ++it;
      }
      umma_commit(bar(B_MMADONE));
      volatile int no_abort = 0;
      wait_one(bar(B_MMADONE), 0, &no_abort, lim, SITE_DRAIN);
    }
    __syncwarp();
  } else if (warp >= kDqWarp0 && warp < kDqWarp0 + 4) {
    // ------------------------------------------------------------ dQ
    // dQ_h^T: TMEM lanes are d (128h + r), columns the block's 64 queries.
    // Each block's columns go to registers and are released at once (the
    // next dP^T is issued into them), then each of the 64 is added into the
    // accumulator row of its query by a warp-wide red (32 consecutive floats).
    const int wq = warp - kDqWarp0;  // TMEM lane quarter
    const uint32_t tmem_row = tmem + ((uint32_t)(wq * 32) << 16);
    const int r = wq * 32 + lane;
    griddep_wait();  // the accumulator is zeroed by the pre-pass
    uint32_t g = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      const int iend = sc.q_end(kb);
      for (int h = 0; h < 2 && ok; ++h)
        for (int i = sc.q_begin(kb); i <= iend; ++i) {
          if (!wait_warp(bar(B_DQFULL), g & 1, abort_flag, lim, SITE_Q_DQFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t v[2][32];
          tmem_ld32(tmem_row + TM_DP, v[0]);
          tmem_ld32(tmem_row + TM_DP + 32, v[1]);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(bar(B_DQFREE));
          reg_fence32(v[0]);
          reg_fence32(v[1]);
          const int q0 = i * BQ;
          float* dst = p.dQacc + ((size_t)bh * N + (size_t)q0) * D + HALF * h + r;
          const int nq = min(BQ, N - q0);
#pragma unroll
          for (int c = 0; c < BQ; ++c)
            if (c < nq) atomicAdd(dst + (size_t)c * D, __uint_as_float(v[c >> 5][c & 31]));
          ++g;
        }
    }
  } else {
    // ------------------------------------------- dS (both warpgroups), dK, dV
    const int grp = warp >> 2;     // query columns [32 grp, 32 grp + 32)
    const int wq = warp & 3;       // TMEM lane quarter
    const uint32_t tmem_row = tmem + ((uint32_t)(wq * 32) << 16);
    const int r = wq * 32 + lane;  // key row (P, dS, dK, dV) / d row (dQ^T)
    const float sl2 = p.scale_log2;
    const float scale = DR ? p.scale * p.drop.keep_scale : p.scale;  // of dP
    uint32_t qcnt = 0, g = 0, hc = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, kb;
      sc.decode(item, bh, kb);
      // the next item's V row of this thread (this group's 256 bytes) is
      // brought into L2 during the second pass
      const __nv_bfloat16* vnext = nullptr;
      for (int w2 = w + 1; w2 < nw; ++w2) {
        const int item2 = sc.item_of(blockIdx.x, w2);
        if (item2 < 0) continue;
        int nbh, nkb;
        sc.decode(item2, nbh, nkb);
        const int nkey = nkb * 128 + r;
        if (nkey < N) vnext = p.V + ((size_t)nbh * N + (size_t)nkey) * D + 128 * grp;
        break;
      }
      const int key = kb * 128 + r;
      const bool kvalid = key < N;
      // V row `key` into TMEM as bf16 pairs: this group's 128 columns of d
      // (64 TMEM columns); rows past N are zero
      {
        const uint4* vsrc = reinterpret_cast<const uint4*>(
            p.V + ((size_t)bh * N + (size_t)(kvalid ? key : 0)) * D + 128 * grp);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t vr[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 u = kvalid ? vsrc[8 * c + k] : make_uint4(0u, 0u, 0u, 0u);
            vr[4 * k] = u.x;
            vr[4 * k + 1] = u.y;
            vr[4 * k + 2] = u.z;
            vr[4 * k + 3] = u.w;
          }
          tmem_st32(tmem_row + TM_V + 64 * grp + 32 * c, vr);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_VREADY));
      }
      const int iend = sc.q_end(kb);
      for (int h = 0; h < 2 && ok; ++h) {
      if (h == 1 && vnext) {
        prefetch_l2(vnext);
        prefetch_l2(vnext + 64);
      }
      for (int i = sc.q_begin(kb); i <= iend; ++i) {
        const int s = qcnt % QST;
        const int q0 = i * BQ + 32 * grp;  // first query of this group's columns
        uint32_t kw[8];
        if constexpr (DR) key_row_keep_words32(kw, p.drop, bh, key, q0, lane);
        if (!wait_warp(bar(B_QFULL + s), (qcnt / QST) & 1, abort_flag, lim, SITE_S_QFULL) ||
            !wait_warp(bar(B_SFULL), g & 1, abort_flag, lim, SITE_S_SFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* st = stat(s);
        // ---- P^T = 2^(S scale log2 e - LSE log2 e) for 32 queries
        float pr[32];
        {
          uint32_t sr[32];
          tmem_ld32(tmem_row + TM_S + 32 * grp, sr);
          tmem_ld_wait();
          reg_fence32(sr);
          const uint64_t sl2x2 = f2_pack(sl2, sl2);
          const ulonglong2* l4 = reinterpret_cast<const ulonglong2*>(st + 32 * grp);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const ulonglong2 lv = l4[e / 4];
            f2_unpack(ffma2(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                            sl2x2, lv.x),
                      pr[e], pr[e + 1]);
            f2_unpack(ffma2(f2_pack(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])),
                            sl2x2, lv.y),
                      pr[e + 2], pr[e + 3]);
#pragma unroll
            for (int u = 0; u < 4; ++u) pr[e + u] = ex2_approx(pr[e + u]);
          }
          if (sc.diag(i, kb)) {  // keys after the query are invisible
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (q0 + x < key) pr[x] = 0.f;
          }
          if (sc.window_edge(i, kb)) {  // queries past the key's window
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (q0 + x - key >= sc.window) pr[x] = 0.f;
          }
          if (__any_sync(0xffffffffu, !kvalid)) {
#pragma unroll
            for (int x = 0; x < 32; ++x) pr[x] = kvalid ? pr[x] : 0.f;
          }
          uint32_t pp[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            pp[k] = pack_bf16x2(pr[2 * k], pr[2 * k + 1]);
            if constexpr (DR) pp[k] &= pair_mask(kw[k >> 1], k);
          }
          tmem_st16(tmem_row + TM_S + 32 * grp, pp);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PREADY));
        // ---- scale*dS^T = P * (dP*scale - D*scale), into TMEM and shared memory
        if (!wait_warp(bar(B_DPFULL), g & 1, abort_flag, lim, SITE_S_DPFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          uint32_t dr[32];
          tmem_ld32(tmem_row + TM_DP + 32 * grp, dr);
          tmem_ld_wait();
          reg_fence32(dr);
          const uint64_t sc2 = f2_pack(scale, scale);
          const ulonglong2* d4 = reinterpret_cast<const ulonglong2*>(st + BQ + 32 * grp);
          uint32_t dd[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const ulonglong2 dv = d4[e / 4];
            uint32_t g0 = dr[e], g1 = dr[e + 1], g2 = dr[e + 2], g3 = dr[e + 3];
            if constexpr (DR) {
              const uint32_t wk = kw[e / 4];
              g0 &= elem_mask(wk, 0);
              g1 &= elem_mask(wk, 1);
              g2 &= elem_mask(wk, 2);
              g3 &= elem_mask(wk, 3);
            }
            float a0, a1, a2, a3;
            f2_unpack(fmul2(ffma2(f2_pack(__uint_as_float(g0), __uint_as_float(g1)), sc2, dv.x),
                            f2_pack(pr[e], pr[e + 1])),
                      a0, a1);
            f2_unpack(fmul2(ffma2(f2_pack(__uint_as_float(g2), __uint_as_float(g3)), sc2, dv.y),
                            f2_pack(pr[e + 2], pr[e + 3])),
                      a2, a3);
            dd[e / 2] = pack_bf16x2(a0, a1);
            dd[e / 2 + 1] = pack_bf16x2(a2, a3);
          }
          tmem_st16(tmem_row + TM_DP + 32 * grp, dd);
          // dS^T row r, queries 32 grp .. + 31: 16-byte pieces 4 grp .. 4 grp + 3
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(smem + OFF_DS + r * 128 + (((4 * grp + k) ^ (r & 7)) << 4)) =
                make_uint4(dd[4 * k], dd[4 * k + 1], dd[4 * k + 2], dd[4 * k + 3]);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_DSREADY));
        ++qcnt;
        ++g;
      }
      if (!ok) break;
      if (!wait_warp(bar(B_DKDVDONE), hc & 1, abort_flag, lim, SITE_E_DKDVDONE)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool store = kvalid;
      const size_t rowoff = ((size_t)bh * N + (size_t)(store ? key : 0)) * D + HALF * h;
      // both groups hold all 128 key rows (lanes); group 0 stores dV_h,
      // group 1 dK_h, 128 columns each
#pragma unroll
      for (int c = 0; c < HALF / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem_row + (grp ? TM_DK : TM_DV) + 32 * c, v);
        tmem_ld_wait();
        reg_fence32(v);
        const float mult = (DR && grp == 0) ? p.drop.keep_scale : 1.f;
        uint4 o[4];
        uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          ow[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mult,
                              __uint_as_float(v[2 * k + 1]) * mult);
        if (store) {
          uint4* dstp = reinterpret_cast<uint4*>((grp ? p.dK : p.dV) + rowoff + 32 * c);
#pragma unroll
          for (int k = 0; k < 4; ++k) dstp[k] = o[k];
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_DKDVFREE));
      ++hc;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  FA_TRACE_MARK(g_cta_trace, 1);
  if (warp == kMmaWarp) tmem_dealloc(tmem, TMEM_COLS);
}

template <bool DR>
cudaError_t launch(const AttnShape& s, const TileMaps& maps, const float* LSE,
                   const float* Dvec, const void* V, float* dQacc, void* dK, void* dV,
                   int num_sms, uint64_t lim, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t attr = smem_limit_once(bwd256_kernel<DR>, SMEM_BYTES, attr_done);
  if (attr != cudaSuccess) return attr;
  Params p;
  p.LSE = LSE;
  p.Dvec = Dvec;
  p.V = reinterpret_cast<const __nv_bfloat16*>(V);
  p.dQacc = dQacc;
  p.dK = reinterpret_cast<__nv_bfloat16*>(dK);
  p.dV = reinterpret_cast<__nv_bfloat16*>(dV);
  p.scale = s.scale;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.wait_limit_ns = lim;
  p.drop = s.drop;
  const int BH = s.B * s.H;
  Sched probe;
  probe.init(BH, s.N, s.causal, num_sms, s.window);
  const int grid = probe.total_items < num_sms ? probe.total_items : num_sms;
  p.sched.init(BH, s.N, s.causal, grid, s.window);
  // a dependent of the pre-pass launched just before (D, the zeroed dQ
  // accumulator): its set-up overlaps the pre-pass's last CTAs
  return launch_after(bwd256_kernel<DR>, dim3(grid), dim3(kThreads), SMEM_BYTES, stream, maps.q,
                      maps.k, maps.dO, p);
}

}  // namespace bwd256

cudaError_t launch_bwd256_tc(const AttnShape& s, const TileMaps& maps,
                             const float* LSE, const float* Dvec, const void* V,
                             float* dQacc, void* dK, void* dV, int num_sms,
                             uint64_t wait_limit_ns, cudaStream_t stream) {
  return s.drop.t4 != 0
             ? bwd256::launch<true>(s, maps, LSE, Dvec, V, dQacc, dK, dV, num_sms,
                                    wait_limit_ns, stream)
             : bwd256::launch<false>(s, maps, LSE, Dvec, V, dQacc, dK, dV, num_sms,
                                     wait_limit_ns, stream);
}

FA_DEFINE_STATUS_READER(read_status_bwd256_tc)

}  // namespace fa
