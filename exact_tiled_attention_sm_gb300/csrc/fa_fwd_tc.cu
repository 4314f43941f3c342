// fa_fwd_tc.cu -- bf16 exact attention forward on sm_103a tensor cores.
//
// One persistent CTA per SM walks the work items of FwdSched (one head, two
// 128-row query blocks).  Roles, by warp:
//   warps 0-3  softmax group 0: owns query block 0 of the item (TMEM lanes
//              0-127, one thread per query row)
//   warps 4-7  softmax group 1: query block 1
//   warp  8    tensor-core issuer (one elected thread) and TMEM owner
//   warp  9    TMA producer (one elected thread)
// At d = 64 (SA, below) the two groups are independent pipelines, each with
// its own items (single query blocks), Q tile and K/V ring: warps 8 and 10
// issue the products of groups 0 and 1, warps 9 and 11 load their tiles.
//
// Data flow per key/value block j ("LLM Architecture Refresh [3]", section 4:
// queries outer, key/value blocks inner; "FlashAttention from scratch",
// Steps 1-3):
//   TMA    K_j, V_j  HBM -> shared memory (128-byte swizzled, 2-4 stage ring)
//   MMA    S_t = Q_t K_j^T             (tcgen05, fp32 accumulator in TMEM)
//   softmax t: S_t -> registers, scale by scale*log2(e), mask the diagonal /
//          ragged block, m = max(m, rowmax); the exponent reference r
//          follows m only when m has risen past it by more than 8 (log2),
//          alpha = 2^(r_old - r), P = 2^(S - r) < 2^8 (bf16, written back
//          over S_t in TMEM), l = alpha*l + rowsum(P), O_t *= alpha when a
//          row's reference moved (rare after its first block)
//   MMA    O_t += P_t V_j              (A operand straight from TMEM)
// and after the last block O = O_t / l, LSE = (m + log2 l) * ln 2 (the
// division deferred to the end, "FlashAttention from scratch", Step 3).
// The two query blocks ping-pong: while softmax group 0 works on S_0 the
// tensor core runs group 1's S_1 and P_1 V products, and vice versa.
//
// TMEM (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256),
// O_0 [256, 256+d), O_1 [256+d, 256+2d); P_t aliases the first 64 columns of
// S_t as packed bf16 pairs.
//
// At d = 64 (the SA layout) P_t has columns of its own, [384 + 64t, 448 +
// 64t), so S_t(j+1) no longer waits for P_t V_j: it is issued as soon as the
// softmax group has read S_t(j) out of TMEM (B_SFREE), and the group goes
// from block j straight to block j+1, holding P_t(j+1) in registers until
// P_t V_j has completed (B_PVDONE) and only then writing it (and rescaling
// O_t, when the reference moved).  Per key block a group then waits for one
// S product instead of for its P V and S products in turn.  Each group has
// its own issuing thread (with one thread for both, its barrier waits and
// commits between the bursts left the tensor pipe idle about half the time)
// and its own loads: group g is worker g * CTAs + cta of a schedule of
// single query blocks (FwdSched::planned_groups), with a 3-stage K/V ring
// of its own, so one group's item boundary and epilogue overlap the other
// group's blocks, and causal items are half as coarse.
//
// With dropout (the DR variant), each softmax thread also draws the keep
// bytes of its row: per 32-key quarter of a block, two Philox calls per lane
// give the quad's four rows x 32 keys, a quad transpose hands every lane its
// own row's words, and P is written to TMEM with the dropped entries zeroed.
// The row sum l stays that of the undropped row (so LSE is unchanged) and
// the factor 256/(256 - t) of kept entries is folded into the final 1/l.
//
// The E8 variant takes Q, K, V as 8-bit E4M3 with per-tensor factors: the
// same pipeline with 16 KiB tiles (d = 128 bytes per row), kind::f8f6f4 MMAs
// (K = 32), and P written to TMEM as E4M3 (32 columns per S_t) scaled by
// 2^8, so that the probabilities use the format's normal range; the 2^8 is
// taken out again with 1/l (l sums the same scaled values) and the LSE.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fa_internal.h"
#include "fa_philox.cuh"
#include "fa_sched.cuh"
#include "fa_tiles.cuh"
#include "fa_trace.cuh"

namespace fa {
namespace fwdtc {

FA_TRACE_DEFINE(g_cta_trace, fa_cta_trace_fwd)

template <int D, bool E8 = false>
struct Cfg {
  static constexpr int CH = E8 ? D / 128 : D / 64;  // 128-byte column chunks
  static constexpr int CHUNK_ELEMS = E8 ? 128 : 64;
  static constexpr int CHUNK_BYTES = 128 * 128;   // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = CH * CHUNK_BYTES;
  // SA (d = 64): S ahead of P V (P in its own TMEM columns), and the two
  // query-block groups as independent pipelines (own producer, issuer, Q
  // tile, K/V ring and stream of single-block items).
  static constexpr bool SA = (D == 64) && !E8;
  static constexpr int THREADS = SA ? 384 : 320;
  // SA: quarters of P held in registers before the wait for the previous
  // P V (the later quarters are written as they are computed)
  static constexpr int P_HELD = 2;
  static constexpr int NRING = SA ? 2 : 1;                 // K/V rings
  static constexpr int KST = SA ? 3 : ((CH == 1) ? 4 : 2);  // K stages per ring
  static constexpr int VST = KST;                          // V stages per ring
  static constexpr int OFF_Q = 0;  // Q tiles of query blocks (groups) 0, 1
  static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NRING * KST * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NRING * VST * TILE_BYTES;
  // barrier slots (the Q and ring barriers of group g at + g under SA)
  static constexpr int NQ = SA ? 2 : 1;  // Q tiles with barriers of their own
  static constexpr int B_QFULL = 0, B_QEMPTY = NQ;  // [NQ]
  static constexpr int B_KFULL = 2 * NQ, B_KEMPTY = B_KFULL + NRING * KST;
  static constexpr int B_VFULL = B_KEMPTY + NRING * KST;
  static constexpr int B_VEMPTY = B_VFULL + NRING * VST;
  static constexpr int B_SFULL = B_VEMPTY + NRING * VST;  // [2]
  static constexpr int B_PREADY = B_SFULL + 2;    // [2]
  static constexpr int B_ODONE = B_PREADY + 2;    // [2]
  static constexpr int B_SFREE = B_ODONE + 2;     // [2] (SA)
  static constexpr int B_PVDONE = B_SFREE + 2;    // [2] (SA)
  static constexpr int B_MMADONE = B_PVDONE + 2;  // [2]
  static constexpr int NBAR = B_MMADONE + 2;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEM + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 4;
  static constexpr uint32_t TM_S = 0;     // + 128 * t
  static constexpr uint32_t TM_O = 256;   // + D * t
  static constexpr uint32_t TM_P = SA ? 384 : 0;  // + 64 * t (SA; else P aliases S)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S =
      E8 ? idesc_e4m3_f32(128, 128, 0, 0) : idesc_bf16_f32(128, 128, 0, 0);
  static constexpr uint32_t IDESC_PV =
      E8 ? idesc_e4m3_f32(128, D, 0, 1) : idesc_bf16_f32(128, D, 0, 1);
  // S = Q K^T for one query block and one key block
  static __device__ __forceinline__ void mma_s(uint32_t d, uint32_t sq, uint32_t sk) {
    if constexpr (E8)
      mma_rows_x_rows_f8<D>(d, sq, sk, IDESC_S);
    else
      mma_rows_x_rows<D>(d, sq, sk, IDESC_S);
  }
  // O (+)= P V, P in TMEM
  static __device__ __forceinline__ void mma_pv(uint32_t d, uint32_t p, uint32_t sv,
                                                bool acc) {
    if constexpr (E8)
      mma_tmem_x_rows_f8(d, p, sv, IDESC_PV, acc);
    else
      mma_tmem_x_rows(d, p, sv, IDESC_PV, acc);
  }
};

constexpr int kMmaWarp = 8;    // issues the products (SA: group 0's); owns TMEM
constexpr int kTmaWarp = 9;    // loads (SA: group 0's)
constexpr int kMmaWarp1 = 10;  // (SA) issues group 1's products
constexpr int kTmaWarp1 = 11;  // (SA) loads group 1's tiles

struct Params {
  __nv_bfloat16* O;
  float* LSE;
  float scale_log2;  // scale * log2(e) (times the Q and K factors for E8)
  float v_descale;   // E8: the V factor
  uint64_t wait_limit_ns;
  DropSpec drop;     // used by the DR variant only
  FwdSched sched;
};

// Wait-site ids recorded with a timeout.
enum : uint32_t {
  SITE_P_QEMPTY = 1, SITE_P_KEMPTY, SITE_P_VEMPTY, SITE_M_QFULL, SITE_M_KFULL,
  SITE_M_VFULL, SITE_M_PREADY, SITE_S_SFULL, SITE_S_ODONE, SITE_DRAIN,
  SITE_ALIGN, SITE_M_SFREE, SITE_S_PVDONE
};

// W: the causal sliding-window variant, DR: dropout, E8: E4M3 inputs (each
// compiled separately, so that the plain kernels carry none of their
// bookkeeping).
template <int D, bool W, bool DR, bool E8>
__global__ void __launch_bounds__(Cfg<D, E8>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mq,
               const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const Params p) {
  using C = Cfg<D, E8>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  volatile uint32_t* tmem_slot =
      reinterpret_cast<volatile uint32_t*>(smem + C::OFF_TMEM);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const FwdSched& sc = p.sched;
  const uint64_t lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int g = 0; g < C::NQ; ++g) {
      mbar_init(bar(C::B_QFULL + g), 1);
      mbar_init(bar(C::B_QEMPTY + g), 1);
    }
    for (int s = 0; s < C::NRING * C::KST; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::NRING * C::VST; ++s) {
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_SFULL + t), 1);
      mbar_init(bar(C::B_PREADY + t), 128);
      mbar_init(bar(C::B_ODONE + t), 1);
      mbar_init(bar(C::B_SFREE + t), 128);
      mbar_init(bar(C::B_PVDONE + t), 1);
    }
    mbar_init(bar(C::B_MMADONE), 1);
    mbar_init(bar(C::B_MMADONE + 1), 1);
    // the swizzled tiles need 1024-byte alignment: refuse to run otherwise
    *abort_flag = (sb & 1023u) ? 1 : 0;
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

  auto sQ = [&](int t) { return sb + C::OFF_Q + (uint32_t)t * C::TILE_BYTES; };

  if (C::SA && (warp == kTmaWarp || warp == kTmaWarp1)) {
    // ------------------------------------------------------------ producer
    // (SA) Group g's loads: its Q tile, then its K/V blocks through its own
    // ring, for the single-block items of worker g*grid + cta.
    if (lane == 0) {
      const int g = warp == kTmaWarp ? 0 : 1;
      const int v = g * (int)gridDim.x + (int)blockIdx.x;
      if (g == 0) {
        prefetch_tensormap(&mq);
        prefetch_tensormap(&mk);
        prefetch_tensormap(&mv);
      }
      uint32_t kcnt = 0, vcnt = 0, qn = 0;
      uint32_t k_used = 0, k_par = 0, v_used = 0, v_par = 0;
      const uint32_t sq = sQ(g);
      const int kb = C::B_KFULL + g * C::KST, keb = C::B_KEMPTY + g * C::KST;
      const int vb = C::B_VFULL + g * C::VST, veb = C::B_VEMPTY + g * C::VST;
      const uint32_t sk0 = sb + C::OFF_K + (uint32_t)(g * C::KST) * C::TILE_BYTES;
      const uint32_t sv0 = sb + C::OFF_V + (uint32_t)(g * C::VST) * C::TILE_BYTES;
      const int nw = sc.n_waves();
      bool ok = true;
      for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
        const int item = sc.item_of(v, w);
        if (item < 0) continue;
        int bh, q;
        sc.decode(item, bh, q);
        const int jlo = W ? sc.kv_lo(q) : 0, jhi = sc.kv_hi(q);
        if (qn > 0 && !wait_one(bar(C::B_QEMPTY + g), (qn - 1) & 1, abort_flag, lim,
                                SITE_P_QEMPTY))
          break;
        mbar_arrive_expect_tx(bar(C::B_QFULL + g), C::TILE_BYTES);
        for (int c = 0; c < C::CH; ++c)
          tma_load_3d(sq + c * C::CHUNK_BYTES, &mq, bar(C::B_QFULL + g),
                      c * C::CHUNK_ELEMS, q * 128, bh);
        ++qn;
        for (int j = jlo; j <= jhi && ok; ++j) {
          {
            const int s = kcnt % C::KST;
            const uint32_t ph = (kcnt / C::KST) & 1;
            if (!wait_one(bar(keb + s), ph ^ 1, abort_flag, lim, SITE_P_KEMPTY)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(kb + s), C::TILE_BYTES);
            for (int c = 0; c < C::CH; ++c)
              tma_load_3d(sk0 + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &mk, bar(kb + s),
                          c * C::CHUNK_ELEMS, j * 128, bh);
            k_used |= 1u << s;
            k_par = (k_par & ~(1u << s)) | (ph << s);
            ++kcnt;
          }
          {
            const int s = vcnt % C::VST;
            const uint32_t ph = (vcnt / C::VST) & 1;
            if (!wait_one(bar(veb + s), ph ^ 1, abort_flag, lim, SITE_P_VEMPTY)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(vb + s), C::TILE_BYTES);
            for (int c = 0; c < C::CH; ++c)
              tma_load_3d(sv0 + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &mv, bar(vb + s),
                          c * C::CHUNK_ELEMS, j * 128, bh);
            v_used |= 1u << s;
            v_par = (v_par & ~(1u << s)) | (ph << s);
            ++vcnt;
          }
        }
      }
      // Drain: every copy this thread issued lands before the CTA exits.
      volatile int no_abort = 0;
      if (qn > 0)
        wait_one(bar(C::B_QFULL + g), (qn - 1) & 1, &no_abort, lim, SITE_DRAIN);
      for (int s = 0; s < C::KST; ++s)
        if ((k_used >> s) & 1)
          wait_one(bar(kb + s), (k_par >> s) & 1, &no_abort, lim, SITE_DRAIN);
      for (int s = 0; s < C::VST; ++s)
        if ((v_used >> s) & 1)
          wait_one(bar(vb + s), (v_par >> s) & 1, &no_abort, lim, SITE_DRAIN);
    }
    __syncwarp();
  } else if (!C::SA && warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      uint32_t kcnt = 0, vcnt = 0, it = 0;
      int last_q = -1;
      // per ring stage: bit s of *_used = a copy was issued into stage s,
      // bit s of *_par = the phase parity of the last such copy
      uint32_t k_used = 0, k_par = 0, v_used = 0, v_par = 0;
      const int nw = sc.n_waves();
      for (int w = 0; w < nw && !*abort_flag; ++w) {
        const int item = sc.item_of(blockIdx.x, w);
        if (item < 0) continue;
        int bh;
        int q0;
        bool valid1;  // the item holds query block q0 + 1 as well
        sc.decode_blocks(item, bh, q0, valid1);
        // key blocks of either query block: kv_lo(q0) .. kv_hi(last)
        const int jlo = W ? sc.kv_lo(q0) : 0;
        const int jhi = sc.kv_hi(valid1 ? q0 + 1 : q0);
        if (it > 0 &&
            !wait_one(bar(C::B_QEMPTY), (it - 1) & 1, abort_flag, lim,
                      SITE_P_QEMPTY))
          break;
        mbar_arrive_expect_tx(bar(C::B_QFULL),
                              (valid1 ? 2 : 1) * C::TILE_BYTES);
        for (int t = 0; t < (valid1 ? 2 : 1); ++t)
          for (int c = 0; c < C::CH; ++c)
            tma_load_3d(sQ(t) + c * C::CHUNK_BYTES, &mq, bar(C::B_QFULL),
                        c * C::CHUNK_ELEMS, (q0 + t) * 128, bh);
        last_q = it & 1;
        bool ok = true;
        for (int j = jlo; j <= jhi && ok; ++j) {
          {
            const int s = kcnt % C::KST;
            const uint32_t ph = (kcnt / C::KST) & 1;
            if (!wait_one(bar(C::B_KEMPTY + s), ph ^ 1, abort_flag, lim,
                          SITE_P_KEMPTY)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE_BYTES);
            const uint32_t dst = sb + C::OFF_K + s * C::TILE_BYTES;
            for (int c = 0; c < C::CH; ++c)
              tma_load_3d(dst + c * C::CHUNK_BYTES, &mk, bar(C::B_KFULL + s),
                          c * C::CHUNK_ELEMS, j * 128, bh);
            k_used |= 1u << s;
            k_par = (k_par & ~(1u << s)) | (ph << s);
            ++kcnt;
          }
          {
            const int s = vcnt % C::VST;
            const uint32_t ph = (vcnt / C::VST) & 1;
            if (!wait_one(bar(C::B_VEMPTY + s), ph ^ 1, abort_flag, lim,
                          SITE_P_VEMPTY)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE_BYTES);
            const uint32_t dst = sb + C::OFF_V + s * C::TILE_BYTES;
            for (int c = 0; c < C::CH; ++c)
              tma_load_3d(dst + c * C::CHUNK_BYTES, &mv, bar(C::B_VFULL + s),
                          c * C::CHUNK_ELEMS, j * 128, bh);
            v_used |= 1u << s;
            v_par = (v_par & ~(1u << s)) | (ph << s);
            ++vcnt;
          }
        }
        if (!ok) break;
        ++it;
      }
      // Drain: every copy this thread issued must have landed before the CTA
      // exits (normally all were consumed long ago and these return at once).
      volatile int no_abort = 0;
      if (last_q >= 0)
        wait_one(bar(C::B_QFULL), (uint32_t)last_q, &no_abort, lim, SITE_DRAIN);
      for (int s = 0; s < C::KST; ++s)
        if ((k_used >> s) & 1)
          wait_one(bar(C::B_KFULL + s), (k_par >> s) & 1, &no_abort, lim,
                   SITE_DRAIN);
      for (int s = 0; s < C::VST; ++s)
        if ((v_used >> s) & 1)
          wait_one(bar(C::B_VFULL + s), (v_par >> s) & 1, &no_abort, lim,
                   SITE_DRAIN);
    }
    __syncwarp();
  } else if (!C::SA && warp == kMmaWarp) {
    // ------------------------------------------------------------ tensor core
    // One issuing thread for both query blocks, in the order P_0 V_j,
    // S_0(j+1), P_1 V_j, S_1(j+1): each block's two products run as one burst
    // while the other block's softmax works.
    if (lane == 0) {
      uint32_t kcnt = 0, vcnt = 0, it = 0;
      uint32_t pcnt0 = 0, pcnt1 = 0;
      const int nw = sc.n_waves();
      for (int w = 0; w < nw && !*abort_flag; ++w) {
        const int item = sc.item_of(blockIdx.x, w);
        if (item < 0) continue;
        int bh;
        int q0;
        bool valid1;  // the item holds query block q0 + 1 as well
        sc.decode_blocks(item, bh, q0, valid1);
        // key-block range of each query block (tile 1's may start one block
        // later and ends one later under the causal mask; empty if absent)
        const int lo0 = W ? sc.kv_lo(q0) : 0, hi0 = sc.kv_hi(q0);
        const int lo1 = (W && valid1) ? sc.kv_lo(q0 + 1) : 0;
        const int hi1 = valid1 ? sc.kv_hi(q0 + 1) : -1;
        const int jlo = lo0, jhi = hi1 > hi0 ? hi1 : hi0;
        auto in_t = [&](int t, int j) {
          return t ? (j >= lo1 && j <= hi1) : (j >= lo0 && j <= hi0);
        };
        bool ok = wait_one(bar(C::B_QFULL), it & 1, abort_flag, lim, SITE_M_QFULL);
        if (!ok) break;
        tc_fence_after();
        {  // S_t for the first key block
          const int s = kcnt % C::KST;
          if (!wait_one(bar(C::B_KFULL + s), (kcnt / C::KST) & 1, abort_flag,
                        lim, SITE_M_KFULL))
            break;
          tc_fence_after();
          const uint32_t sk = sb + C::OFF_K + s * C::TILE_BYTES;
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (in_t(t, jlo)) {
              C::mma_s(tmem + C::TM_S + 128 * t, sQ(t), sk);
              umma_commit(bar(C::B_SFULL + t));
            }
          umma_commit(bar(C::B_KEMPTY + s));
          ++kcnt;
          // the Q tiles are read by S products only: with a single key block
          // they are free for the next item as soon as these complete
          if (jlo == jhi) umma_commit(bar(C::B_QEMPTY));
        }
        for (int j = jlo; j <= jhi && ok; ++j) {
          const int vs = vcnt % C::VST;
          if (!wait_one(bar(C::B_VFULL + vs), (vcnt / C::VST) & 1, abort_flag,
                        lim, SITE_M_VFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sv = sb + C::OFF_V + vs * C::TILE_BYTES;
          const int ks = kcnt % C::KST;
          const uint32_t sk = sb + C::OFF_K + ks * C::TILE_BYTES;
          bool k_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok) continue;
            if (in_t(t, j)) {
              uint32_t& pc = t ? pcnt1 : pcnt0;
              if (!wait_one(bar(C::B_PREADY + t), pc & 1, abort_flag, lim,
                            SITE_M_PREADY)) {
                ok = false;
                continue;
              }
              ++pc;
              tc_fence_after();
              C::mma_pv(tmem + C::TM_O + D * t, tmem + C::TM_S + 128 * t, sv,
                        j > (t ? lo1 : lo0));
              if (j == (t ? hi1 : hi0)) umma_commit(bar(C::B_ODONE + t));
            }
            if (in_t(t, j + 1)) {
              if (!k_ready) {
                if (!wait_one(bar(C::B_KFULL + ks), (kcnt / C::KST) & 1,
                              abort_flag, lim, SITE_M_KFULL)) {
                  ok = false;
                  continue;
                }
                tc_fence_after();
                k_ready = true;
              }
              C::mma_s(tmem + C::TM_S + 128 * t, sQ(t), sk);
              umma_commit(bar(C::B_SFULL + t));
            }
          }
          umma_commit(bar(C::B_VEMPTY + vs));
          ++vcnt;
          if (k_ready) {
            umma_commit(bar(C::B_KEMPTY + ks));
            ++kcnt;
          }
          // the item's last S products have been issued: the next item's Q
          // tiles may load while its last P V products and epilogue run
          if (ok && j + 1 == jhi) umma_commit(bar(C::B_QEMPTY));
        }
        if (!ok) break;
        ++it;
      }
      // every MMA issued by this thread completes before TMEM is released
      umma_commit(bar(C::B_MMADONE));
      volatile int no_abort = 0;
      wait_one(bar(C::B_MMADONE), 0, &no_abort, lim, SITE_DRAIN);
    }
    __syncwarp();
  } else if (C::SA && (warp == kMmaWarp || warp == kMmaWarp1)) {
    // ------------------------------------------------------------ tensor core
    // (SA) Group g's issuing thread: S_g(j+1) as soon as the softmax group
    // has read S_g(j) (S-free), then P_g V_j once P is written (P-ready), for
    // the single-block items of worker g*grid + cta, from the group's own
    // Q tile and K/V ring.
    if (lane == 0) {
      const int g = warp == kMmaWarp ? 0 : 1;
      const int v = g * (int)gridDim.x + (int)blockIdx.x;
      uint32_t kcnt = 0, vcnt = 0, it = 0;
      uint32_t pc = 0;  // P-ready phases consumed
      uint32_t si = 0;  // S products issued so far
      // S_g is overwritten only after the softmax group has read the
      // previous S_g out of TMEM
      auto s_free = [&]() -> bool {
        if (si > 0) {
          if (!wait_one(bar(C::B_SFREE + g), (si - 1) & 1, abort_flag, lim,
                        SITE_M_SFREE))
            return false;
          tc_fence_after();
        }
        ++si;
        return true;
      };
      const uint32_t tS = tmem + C::TM_S + 128 * g;
      const uint32_t tO = tmem + C::TM_O + D * g;
      const uint32_t tP = tmem + C::TM_P + 64 * g;
      const uint32_t sq = sQ(g);
      const int kb = C::B_KFULL + g * C::KST, keb = C::B_KEMPTY + g * C::KST;
      const int vb = C::B_VFULL + g * C::VST, veb = C::B_VEMPTY + g * C::VST;
      const uint32_t sk0 = sb + C::OFF_K + (uint32_t)(g * C::KST) * C::TILE_BYTES;
      const uint32_t sv0 = sb + C::OFF_V + (uint32_t)(g * C::VST) * C::TILE_BYTES;
      const int nw = sc.n_waves();
      for (int w = 0; w < nw && !*abort_flag; ++w) {
        const int item = sc.item_of(v, w);
        if (item < 0) continue;
        int bh, q;
        sc.decode(item, bh, q);
        const int lo = W ? sc.kv_lo(q) : 0, hi = sc.kv_hi(q);
        bool ok = wait_one(bar(C::B_QFULL + g), it & 1, abort_flag, lim, SITE_M_QFULL);
        if (!ok) break;
        tc_fence_after();
        {  // S for the first key block
          const int s = kcnt % C::KST;
          if (!wait_one(bar(kb + s), (kcnt / C::KST) & 1, abort_flag, lim,
                        SITE_M_KFULL))
            break;
          tc_fence_after();
          if (!s_free()) break;
          C::mma_s(tS, sq, sk0 + s * C::TILE_BYTES);
          umma_commit(bar(C::B_SFULL + g));
          umma_commit(bar(keb + s));
          ++kcnt;
          // the Q tile is read by S products only: free after the last one
          if (hi == lo) umma_commit(bar(C::B_QEMPTY + g));
        }
        for (int j = lo; j <= hi && ok; ++j) {
          const int vs = vcnt % C::VST;
          if (!wait_one(bar(vb + vs), (vcnt / C::VST) & 1, abort_flag, lim,
                        SITE_M_VFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (j + 1 <= hi) {  // S_g(j+1) first: P_g V_j reads P's own columns
            const int ks = kcnt % C::KST;
            if (!wait_one(bar(kb + ks), (kcnt / C::KST) & 1, abort_flag, lim,
                          SITE_M_KFULL) ||
                !s_free()) {
              ok = false;
              break;
            }
            tc_fence_after();
            C::mma_s(tS, sq, sk0 + ks * C::TILE_BYTES);
            umma_commit(bar(C::B_SFULL + g));
            umma_commit(bar(keb + ks));
            ++kcnt;
            if (j + 1 == hi) umma_commit(bar(C::B_QEMPTY + g));
          }
          // O_g += P_g V_j once the softmax group has written P_g
          if (!wait_one(bar(C::B_PREADY + g), pc & 1, abort_flag, lim,
                        SITE_M_PREADY)) {
            ok = false;
            break;
          }
          ++pc;
          tc_fence_after();
          C::mma_pv(tO, tP, sv0 + vs * C::TILE_BYTES, j > lo);
          umma_commit(bar(C::B_PVDONE + g));
          if (j == hi) umma_commit(bar(C::B_ODONE + g));
          umma_commit(bar(veb + vs));
          ++vcnt;
        }
        if (!ok) break;
        ++it;
      }
      // every MMA issued by this thread completes before TMEM is released
      umma_commit(bar(C::B_MMADONE + g));
      volatile int no_abort = 0;
      wait_one(bar(C::B_MMADONE + g), 0, &no_abort, lim, SITE_DRAIN);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;          // query block of the item
    const int wq = warp & 3;          // TMEM lane quarter
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S + 128 * t;
    const uint32_t tO = tmem + lane_off + C::TM_O + D * t;
    const uint32_t tP = C::SA ? tmem + lane_off + C::TM_P + 64 * t : tS;
    const float sl2 = p.scale_log2;
    uint32_t scnt = 0, ocnt = 0;
    const int nw = sc.n_waves();
    // (SA) the group's own worker; otherwise the CTA's pair items
    const int v = C::SA ? t * (int)gridDim.x + (int)blockIdx.x : (int)blockIdx.x;
    for (int w = 0; w < nw && !*abort_flag; ++w) {
      const int item = sc.item_of(v, w);
      if (item < 0) continue;
      int bh, q;
      if constexpr (C::SA) {
        sc.decode(item, bh, q);
      } else {
        int q0;
        bool two;
        sc.decode_blocks(item, bh, q0, two);
        if (t == 1 && !two) continue;
        q = q0 + t;
      }
      const int jlo = W ? sc.kv_lo(q) : 0, jhi = sc.kv_hi(q);
      const int row = q * 128 + wq * 32 + lane;
      float m = -INFINITY;     // running row maximum of the raw scores
      float mref = -INFINITY;  // exponent reference of l and O_t (log2 units)
      float l = 0.f;
      bool ok = true;
      for (int j = jlo; j <= jhi; ++j) {
        if (!wait_warp(bar(C::B_SFULL + t), scnt & 1, abort_flag, lim,
                       SITE_S_SFULL)) {
          ok = false;
          break;
        }
        ++scnt;
        tc_fence_after();
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(tS + 0, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_ld_wait();
        reg_fence32(r0);
        reg_fence32(r1);
        reg_fence32(r2);
        reg_fence32(r3);
        if constexpr (C::SA) {  // S_t may take the next block's product now
          tc_fence_before();
          mbar_arrive(bar(C::B_SFREE + t));
        }
        float x[128];  // raw scores q.k of this row
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(r0[i]);
          x[32 + i] = __uint_as_float(r1[i]);
          x[64 + i] = __uint_as_float(r2[i]);
          x[96 + i] = __uint_as_float(r3[i]);
        }
        if (sc.needs_mask(q, j) || (W && sc.window_edge(q, j))) {
          // visible keys: lo_k <= key < lim_k (the window's left edge, the
          // diagonal, the end of the sequence)
          const int k0 = j * 128;
          const int lim_k = sc.causal ? min(row + 1, sc.N) : sc.N;
          if constexpr (W) {
            const int lo_k = row - sc.window + 1;
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (k0 + i >= lim_k || k0 + i < lo_k) x[i] = -INFINITY;
          } else {
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (k0 + i >= lim_k) x[i] = -INFINITY;
          }
        }
        // Row maximum of the raw scores (scale > 0 commutes with max): eight
        // independent chains of three-input maxima, then a short tree.
        float mk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmax3(x[k], x[8 + k], x[16 + k]);
#pragma unroll
        for (int i = 24; i < 120; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) mk[k] = fmax3(mk[k], x[i + k], x[i + 8 + k]);
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], x[120 + k]);
        const float m_prev = m;
        m = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]),
                  fmax3(mk[6], mk[7], m));
        // Exponent reference in log2 units.  It moves to the new maximum only
        // when that exceeds it by more than kRefSlack, or when the row had no
        // visible key before this block: P = 2^(s - mref) stays below
        // 2^kRefSlack, which the fp32 sums and bf16 P hold without loss, and
        // O_t needs its rescale (TMEM round trips) only when the reference
        // moves, which after a row's first block is rare.  O / l and
        // LSE = mref + log2 l are the same whichever reference is used.  A row
        // with nothing visible yet keeps 0.  (E8: no slack, 2^8 P already
        // fills E4M3's range.)
        constexpr float kRefSlack = E8 ? 0.f : 8.f;
        const float cand = (m == -INFINITY) ? 0.f : m * sl2;
        const bool move = (m_prev == -INFINITY) || (cand > mref + kRefSlack);
        const float mref_new = move ? cand : mref;
        // alpha rescales what the row has accumulated so far.  A row that has
        // seen no key yet has nothing (l = 0, O_t = 0), so alpha = 0; under
        // the window this also covers a row whose first visible keys come in
        // a later block, where mref still holds the placeholder 0 and
        // 2^(0 - cand) would overflow for very negative scores (inf * 0).
        const float alpha =
            !move ? 1.f : ((W && m_prev == -INFINITY) ? 0.f : ex2_approx(mref - mref_new));
        mref = mref_new;
        // P = 2^(scale*log2(e)*s - mref): one packed fma per pair, row sum
        // in four packed accumulators
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        // (E8: 2^8 P, inside E4M3's normal range)
        const float nref = E8 ? 8.f - mref_new : -mref_new;
        const uint64_t nm2 = f2_pack(nref, nref);
        // O_t *= alpha is needed when a row of this warp moved its max (the
        // previous P V product into O_t completed before S_t of this block
        // did).  O's first 64 columns are requested (always, which keeps the
        // register allocation free of branches) before the last quarter of
        // the exponentials, so that their TMEM latency hides behind it.
        // (SA: the previous P V may still run; O and P_t are touched only
        // after it has completed, below.)
        const bool resc = j > jlo && __any_sync(0xffffffffu, alpha != 1.f);
        uint32_t oa[2][32];
        uint32_t pks[4][16];  // P of this row, 32 keys per quarter
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        bool pv_ok = true;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          if constexpr (C::SA) {
            if (h == C::P_HELD) {
              // P_t and O_t are free once the group's previous P V has
              // completed; the quarters held so far are written then
              const uint32_t b = scnt - 1;  // this block's index in the group
              if (b > 0) {
                pv_ok = wait_warp(bar(C::B_PVDONE + t), (b - 1) & 1, abort_flag,
                                  lim, SITE_S_PVDONE);
                if (!pv_ok) break;
                tc_fence_after();
              }
#pragma unroll
              for (int h2 = 0; h2 < C::P_HELD; ++h2) tmem_st16(tP + 16 * h2, pks[h2]);
            }
          }
          if (h == 3 && !C::SA) {
            tmem_ld32(tO + 0, oa[0]);
            tmem_ld32(tO + 32, oa[1]);
          }
          // keep bytes of this row for keys 32h + 4c + (0..3), c = 0..7: lane
          // q of the quad draws key patches q and 4 + q for the quad's four
          // rows (word = row mod 4), the transpose collects this row's words
          uint32_t kw[8];
          if constexpr (DR) {
            const uint32_t kp0 = (uint32_t)(j * 32 + 8 * h) + (uint32_t)(lane & 3);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const Philox4 o = philox4x32_10(kp0 + 4 * g, (uint32_t)row >> 2,
                                              (uint32_t)bh, 0u, p.drop.k0, p.drop.k1);
              uint32_t a[4] = {o.x[0], o.x[1], o.x[2], o.x[3]};
              quad_transpose(a, lane);
#pragma unroll
              for (int c = 0; c < 4; ++c) kw[4 * g + c] = keep_flags(a[c], p.drop);
            }
          }
          uint32_t(&pk)[16] = pks[h];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = 32 * h + 2 * i;
            float a, b;
            f2_unpack(ffma2(f2_pack(x[e], x[e + 1]), sl2x2, nm2), a, b);
            a = ex2_approx(a);
            b = ex2_approx(b);
            acc[i & 3] = fadd2(acc[i & 3], f2_pack(a, b));
            if constexpr (E8)
              pk[i] = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                               __NV_E4M3);
            else
              pk[i] = pack_bf16x2(a, b);
            if constexpr (DR) pk[i] &= pair_mask(kw[i >> 1], i);
          }
          if constexpr (E8) {  // four E4M3 values a column, key order
            uint32_t p8[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) p8[w] = __byte_perm(pk[2 * w], pk[2 * w + 1], 0x5410);
            tmem_st8(tS + 8 * h, p8);
          } else if constexpr (!C::SA) {
            tmem_st16(tS + 16 * h, pk);
          } else {
            if (h >= C::P_HELD) tmem_st16(tP + 16 * h, pk);
          }
        }
        if (!pv_ok) {
          ok = false;
          break;
        }
        float rs_lo, rs_hi;
        f2_unpack(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), rs_lo, rs_hi);
        l = l * alpha + (rs_lo + rs_hi);
        if constexpr (C::SA) {
          if (resc) {
            tmem_ld32(tO + 0, oa[0]);
            tmem_ld32(tO + 32, oa[1]);
            tmem_ld_wait();
            reg_fence32(oa[0]);
            reg_fence32(oa[1]);
          }
        } else {
          // the loaded registers stay untouched until the load has landed
          tmem_ld_wait();
          reg_fence32(oa[0]);
          reg_fence32(oa[1]);
        }
        if (resc) {
          const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a, b;
              f2_unpack(fmul2(f2_pack(__uint_as_float(oa[c][2 * i]),
                                      __uint_as_float(oa[c][2 * i + 1])),
                              al2),
                        a, b);
              oa[c][2 * i] = __float_as_uint(a);
              oa[c][2 * i + 1] = __float_as_uint(b);
            }
            tmem_st32(tO + 32 * c, oa[c]);
          }
#pragma unroll
          for (int c = 2; c < D / 32; ++c) {  // the remaining columns
            uint32_t ob[32];
            tmem_ld32(tO + 32 * c, ob);
            tmem_ld_wait();
            reg_fence32(ob);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a, b;
              f2_unpack(fmul2(f2_pack(__uint_as_float(ob[2 * i]),
                                      __uint_as_float(ob[2 * i + 1])),
                              al2),
                        a, b);
              ob[2 * i] = __float_as_uint(a);
              ob[2 * i + 1] = __float_as_uint(b);
            }
            tmem_st32(tO + 32 * c, ob);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::B_PREADY + t));
      }
      if (!ok) break;
      if (!wait_warp(bar(C::B_ODONE + t), ocnt & 1, abort_flag, lim,
                     SITE_S_ODONE))
        break;
      ++ocnt;
      tc_fence_after();
      // kept entries carry the factor 256/(256 - t)
      const float inv_l = (DR ? p.drop.keep_scale : E8 ? p.v_descale : 1.f) / l;
      const bool store = row < sc.N;
      __nv_bfloat16* orow = p.O + ((size_t)bh * sc.N + (size_t)(store ? row : 0)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c, o);
        tmem_ld_wait();
        reg_fence32(o);
        uint4 v[4];
        uint32_t* vw = reinterpret_cast<uint32_t*>(v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          vw[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l,
                              __uint_as_float(o[2 * i + 1]) * inv_l);
        if (store) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = v[i];
        }
      }
      if (store)
        p.LSE[(size_t)bh * sc.N + row] =
            (mref - (E8 ? 8.f : 0.f) + log2f(l)) * 0.69314718055994531f;
      // all TMEM reads of O_t are done before the next item's first P V
      // product (ordered by this group's next p_ready arrival)
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  FA_TRACE_MARK(g_cta_trace, 1);
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool W, bool DR, bool E8 = false>
cudaError_t launch(const AttnShape& s, const TileMaps& maps, void* O,
                   float* LSE, int num_sms, uint64_t lim, cudaStream_t stream) {
  using C = Cfg<D, E8>;
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t attr = smem_limit_once(fwd_kernel<D, W, DR, E8>, C::SMEM_BYTES, attr_done);
  if (attr != cudaSuccess) return attr;
  Params p;
  p.O = reinterpret_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.wait_limit_ns = lim;
  p.v_descale = s.v_descale;
  p.drop = s.drop;
  const int BH = s.B * s.H;
  p.sched = C::SA ? FwdSched::planned_groups(BH, s.N, s.causal, num_sms, s.window)
                  : FwdSched::planned(BH, s.N, s.causal, num_sms, s.window);
  const int grid = C::SA ? p.sched.grid / 2 : p.sched.grid;
  fwd_kernel<D, W, DR, E8><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(
      maps.q, maps.k, maps.v, p);
  return cudaGetLastError();
}

}  // namespace fwdtc

cudaError_t launch_fwd_tc(const AttnShape& s, const TileMaps& maps, void* O,
                          float* LSE, int num_sms, uint64_t wait_limit_ns,
                          cudaStream_t stream) {
  const int v = (s.window > 0 ? 1 : 0) + (s.drop.t4 != 0 ? 2 : 0);
  const uint64_t lim = wait_limit_ns;
  if (s.fp8)  // d = 128, no dropout (checked by the caller)
    return v & 1 ? fwdtc::launch<128, true, false, true>(s, maps, O, LSE, num_sms, lim, stream)
                 : fwdtc::launch<128, false, false, true>(s, maps, O, LSE, num_sms, lim, stream);
#define FA_FWD_CASE(DD)                                                        \
  switch (v) {                                                                 \
    case 0: return fwdtc::launch<DD, false, false>(s, maps, O, LSE, num_sms, lim, stream); \
    case 1: return fwdtc::launch<DD, true, false>(s, maps, O, LSE, num_sms, lim, stream);  \
    case 2: return fwdtc::launch<DD, false, true>(s, maps, O, LSE, num_sms, lim, stream);  \
    default: return fwdtc::launch<DD, true, true>(s, maps, O, LSE, num_sms, lim, stream);  \
  }
  if (s.d == 64) FA_FWD_CASE(64)
  FA_FWD_CASE(128)
#undef FA_FWD_CASE
}

FA_DEFINE_STATUS_READER(read_status_fwd_tc)

}  // namespace fa
