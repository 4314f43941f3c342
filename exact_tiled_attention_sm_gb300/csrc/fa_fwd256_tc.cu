// fa_fwd256_tc.cu -- bf16 exact attention forward for head dimension 256 on
// sm_103a tensor cores.
//
// At d = 256 one 128-row query block needs a 128-column S tile and a
// 256-column O accumulator in TMEM, so two blocks no longer fit in its 512
// columns (the d^2/M wall of "Flash Attention, From First Principles", "The
// rent arithmetic", in TMEM form).  A work item is therefore a single query
// block (FwdSched with one block per item), and the second half of TMEM holds
// a second S tile instead: S is double-buffered, so the tensor core computes
// S_{j+2} while the softmax works on S_{j+1}.
//
// Roles, by warp:
//   warps 0-3, 4-7  softmax warpgroups 0 and 1: both own all 128 rows of the
//                   block (warp w and w+4 share TMEM lanes 32(w%4)..), group
//                   g takes score columns [64g, 64g+64) and O columns
//                   [128g, 128g+128); the two halves of a row's maximum meet
//                   through shared memory once per key block, the two halves
//                   of its sum once per item
//   warp  8         tensor-core issuer and TMEM owner
//   warp  9         TMA producer
//
// Per key block j (queries outer, "LLM Architecture Refresh [3]", section 4):
//   MMA   S_j = Q K_j^T into S buffer j%2 (issued two blocks ahead)
//   softmax: max of both halves, the exponent reference (it follows the
//         max only when the max has risen past it by more than 8, log2),
//         alpha, P = 2^(S - reference) as bf16 over the block's first 64
//         columns, l, O *= alpha when a row's reference moved (after the
//         previous P V product has completed)
//   MMA   O += P_j V_j (P from TMEM, V MN-major, N = 256)
// and O = O / l, LSE = (m + log2 l) ln 2 once at the end.
//
// Shared memory: Q, K and V tiles of [128][256] bf16 (64 KiB each, four
// 128-byte-swizzled 64-column chunks); K and V are single-buffered, loaded as
// soon as the products reading the previous tile have completed.
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "fa_sched.cuh"
#include "fa_philox.cuh"
#include "fa_tiles.cuh"
#include "fa_trace.cuh"

namespace fa {
namespace fwd256 {

FA_TRACE_DEFINE(g_cta_trace, fa_cta_trace_fwd256)

constexpr int D = 256;
constexpr int CH = D / 64;
constexpr int TILE_BYTES = CH * kChunkBytes;  // 64 KiB
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;
constexpr int OFF_V = OFF_K + TILE_BYTES;
constexpr int OFF_XCH = OFF_V + TILE_BYTES;   // float [2 parity][2 group][128]
constexpr int OFF_XL = OFF_XCH + 2 * 2 * 128 * 4;  // float [2 group][128]
constexpr int OFF_BAR = OFF_XL + 2 * 128 * 4;
// barriers
constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = 3;
constexpr int B_VFULL = 4, B_VEMPTY = 5;
constexpr int B_SFULL = 6;    // [2] per S buffer
constexpr int B_PREADY = 8;   // [2] per S buffer (P lives there)
constexpr int B_PVDONE = 10;
constexpr int B_XCH = 11;     // [4 lane quarters][2 parity]: row-max halves
constexpr int B_XL = 19;      // [4 lane quarters]: row-sum halves
constexpr int B_MMADONE = 23;
constexpr int B_ODONE = 24;   // the item's last P V product has completed
constexpr int NBAR = 25;
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM_BYTES = OFF_ABORT + 4;
constexpr uint32_t TM_S = 0;    // + 128 * buffer
constexpr uint32_t TM_O = 256;  // 256 columns
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, 0, 1);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;

struct Params {
  __nv_bfloat16* O;
  float* LSE;
  float scale_log2;
  uint64_t wait_limit_ns;
  DropSpec drop;  // DR variant only
  FwdSched sched;
};

enum : uint32_t {
  SITE_P_QEMPTY = 1, SITE_P_KEMPTY, SITE_P_VEMPTY, SITE_M_QFULL, SITE_M_KFULL,
  SITE_M_VFULL, SITE_M_PREADY, SITE_S_SFULL, SITE_S_PVDONE, SITE_S_XCH,
  SITE_S_XL, SITE_DRAIN, SITE_ALIGN, SITE_S_ODONE
};

// W: causal sliding window; DR: dropout (keep bytes drawn per 32-key half as
// in the d <= 128 forward: two Philox calls per lane and a quad transpose).
template <bool W, bool DR>
__global__ void __launch_bounds__(kThreads, 1)
    fwd256_kernel(const __grid_constant__ CUtensorMap mq,
                  const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mv, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + OFF_BAR + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const FwdSched& sc = p.sched;
  const uint64_t lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_KFULL), 1);
    mbar_init(bar(B_KEMPTY), 1);
    mbar_init(bar(B_VFULL), 1);
    mbar_init(bar(B_VEMPTY), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_SFULL + b), 1);
      mbar_init(bar(B_PREADY + b), 256);
    }
    mbar_init(bar(B_PVDONE), 1);
    for (int i = 0; i < 8; ++i) mbar_init(bar(B_XCH + i), 2);
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_XL + i), 2);
    mbar_init(bar(B_MMADONE), 1);
    mbar_init(bar(B_ODONE), 1);
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

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    // Order of copies per item: Q, K_lo, then K_{j+1}, V_j for each j (the
    // order the tensor core consumes them in: S runs one block ahead of P V).
    if (lane == 0) {
      prefetch_tensormap(&mq);
      prefetch_tensormap(&mk);
      prefetch_tensormap(&mv);
      uint32_t kcnt = 0, vcnt = 0, qcnt = 0;
      bool ok = true;
      auto load_tile = [&](uint32_t dst, const CUtensorMap* m, int full, int row, int bh) {
        mbar_arrive_expect_tx(bar(full), TILE_BYTES);
        for (int c = 0; c < CH; ++c)
          tma_load_3d(dst + c * kChunkBytes, m, bar(full), c * 64, row, bh);
      };
      auto load_k = [&](int j, int bh) {
        if (!wait_one(bar(B_KEMPTY), (kcnt & 1) ^ 1, abort_flag, lim, SITE_P_KEMPTY))
          return false;
        load_tile(sb + OFF_K, &mk, B_KFULL, j * 128, bh);
        ++kcnt;
        return true;
      };
      for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
        const int item = sc.item_of(blockIdx.x, w);
        if (item < 0) continue;
        int bh, q;
        sc.decode(item, bh, q);
        const int jlo = W ? sc.kv_lo(q) : 0, jhi = sc.kv_hi(q);
        if (qcnt > 0 && !wait_one(bar(B_QEMPTY), (qcnt - 1) & 1, abort_flag, lim, SITE_P_QEMPTY))
          break;
        load_tile(sb + OFF_Q, &mq, B_QFULL, q * 128, bh);
        ++qcnt;
        if (!load_k(jlo, bh)) break;
        for (int j = jlo; j <= jhi; ++j) {
          if (j + 1 <= jhi && !load_k(j + 1, bh)) {
            ok = false;
            break;
          }
          if (!wait_one(bar(B_VEMPTY), (vcnt & 1) ^ 1, abort_flag, lim, SITE_P_VEMPTY)) {
            ok = false;
            break;
          }
          load_tile(sb + OFF_V, &mv, B_VFULL, j * 128, bh);
          ++vcnt;
        }
      }
      // every copy issued has landed before the CTA exits
      volatile int no_abort = 0;
      if (qcnt > 0) wait_one(bar(B_QFULL), (qcnt - 1) & 1, &no_abort, lim, SITE_DRAIN);
      if (kcnt > 0) wait_one(bar(B_KFULL), (kcnt - 1) & 1, &no_abort, lim, SITE_DRAIN);
      if (vcnt > 0) wait_one(bar(B_VFULL), (vcnt - 1) & 1, &no_abort, lim, SITE_DRAIN);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tensor core
    if (lane == 0) {
      uint32_t kcnt = 0, vcnt = 0, it = 0, gj = 0;  // gj: blocks done, all items
      bool ok = true;
      // S of global block index g into buffer g % 2 (needs K)
      auto issue_s = [&](uint32_t g) {
        if (!wait_one(bar(B_KFULL), kcnt & 1, abort_flag, lim, SITE_M_KFULL)) return false;
        tc_fence_after();
        mma_rows_x_rows<D>(tmem + TM_S + 128 * (g & 1), sb + OFF_Q, sb + OFF_K, IDESC_S);
        umma_commit(bar(B_SFULL + (g & 1)));
        umma_commit(bar(B_KEMPTY));
        ++kcnt;
        return true;
      };
      for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
        const int item = sc.item_of(blockIdx.x, w);
        if (item < 0) continue;
        int bh, q;
        sc.decode(item, bh, q);
        const int jlo = W ? sc.kv_lo(q) : 0, jhi = sc.kv_hi(q);
        if (!wait_one(bar(B_QFULL), it & 1, abort_flag, lim, SITE_M_QFULL)) break;
        tc_fence_after();
        if (!issue_s(gj)) break;
        if (jhi > jlo && !issue_s(gj + 1)) break;
        if (jhi <= jlo + 1) umma_commit(bar(B_QEMPTY));  // the item's last S
        for (int j = jlo; j <= jhi; ++j, ++gj) {
          if (!wait_one(bar(B_PREADY + (gj & 1)), (gj >> 1) & 1, abort_flag, lim,
                        SITE_M_PREADY) ||
              !wait_one(bar(B_VFULL), vcnt & 1, abort_flag, lim, SITE_M_VFULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tmem_x_rows(tmem + TM_O, tmem + TM_S + 128 * (gj & 1), sb + OFF_V,
                          IDESC_PV, j > jlo);
          umma_commit(bar(B_PVDONE));
          if (j == jhi) umma_commit(bar(B_ODONE));
          umma_commit(bar(B_VEMPTY));
          ++vcnt;
          // S two blocks ahead, into the buffer whose P was just consumed
          if (j + 2 <= jhi) {
            if (!issue_s(gj + 2)) {
              ok = false;
              break;
            }
            if (j + 2 == jhi) umma_commit(bar(B_QEMPTY));
          }
        }
        ++it;
      }
      umma_commit(bar(B_MMADONE));
      volatile int no_abort = 0;
      wait_one(bar(B_MMADONE), 0, &no_abort, lim, SITE_DRAIN);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int g = warp >> 2;   // column half
    const int wq = warp & 3;   // TMEM lane quarter
    const int rb = wq * 32 + lane;  // row within the block
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    float* xch = reinterpret_cast<float*>(smem + OFF_XCH);  // [par][g][128]
    float* xl = reinterpret_cast<float*>(smem + OFF_XL);    // [g][128]
    uint32_t gj = 0, it = 0;
    bool ok = true;
    for (int w = 0; w < nw && ok && !*abort_flag; ++w) {
      const int item = sc.item_of(blockIdx.x, w);
      if (item < 0) continue;
      int bh, q;
      sc.decode(item, bh, q);
      const int jlo = W ? sc.kv_lo(q) : 0, jhi = sc.kv_hi(q);
      const int row = q * 128 + rb;
      float m = -INFINITY, mref = -INFINITY, l = 0.f;
      for (int j = jlo; j <= jhi; ++j, ++gj) {
        const uint32_t buf = gj & 1;
        const uint32_t tS = tmem + lane_off + TM_S + 128 * buf;
        if (!wait_warp(bar(B_SFULL + buf), (gj >> 1) & 1, abort_flag, lim, SITE_S_SFULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(tS + 64 * g, r0);
        tmem_ld32(tS + 64 * g + 32, r1);
        tmem_ld_wait();
        reg_fence32(r0);
        reg_fence32(r1);
        float x[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(r0[i]);
          x[32 + i] = __uint_as_float(r1[i]);
        }
        if (sc.needs_mask(q, j) || (W && sc.window_edge(q, j))) {
          const int k0 = j * 128 + 64 * g;
          const int lim_k = sc.causal ? min(row + 1, sc.N) : sc.N;
          const int lo_k = W ? row - sc.window + 1 : 0;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (k0 + i >= lim_k || k0 + i < lo_k) x[i] = -INFINITY;
        }
        float mk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmax3(x[k], x[8 + k], x[16 + k]);
#pragma unroll
        for (int i = 24; i < 56; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) mk[k] = fmax3(mk[k], x[i + k], x[i + 8 + k]);
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], x[56 + k]);
        const float mp = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]),
                               fmaxf(mk[6], mk[7]));
        // the other half's maximum of this row (double-buffered by parity)
        // (arriving also orders both halves' reads of S before either half's
        // P overwrites columns of the other)
        xch[(buf * 2 + g) * 128 + rb] = mp;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_XCH + wq * 2 + buf));
        if (!wait_warp(bar(B_XCH + wq * 2 + buf), (gj >> 1) & 1, abort_flag, lim, SITE_S_XCH)) {
          ok = false;
          break;
        }
        __syncwarp();
        tc_fence_after();
        const float mo = xch[(buf * 2 + (g ^ 1)) * 128 + rb];
        // the exponent reference moves only when the maximum has risen by
        // more than 8 (log2 units) or the row had nothing visible before, so
        // that P < 2^8 and O is rarely rescaled; O / l and the LSE do not
        // depend on the reference
        const float m_prev = m;
        m = fmax3(m, mp, mo);
        const float cand = (m == -INFINITY) ? 0.f : m * sl2;
        const bool move = (m_prev == -INFINITY) || (cand > mref + 8.f);
        const float mref_new = move ? cand : mref;
        // a row that has seen no key yet has nothing to rescale: alpha = 0
        // (under the window its first visible keys may come in a later block,
        // where 2^(0 - cand) from the placeholder reference could overflow)
        const float alpha =
            !move ? 1.f : ((W && m_prev == -INFINITY) ? 0.f : ex2_approx(mref - mref_new));
        mref = mref_new;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t nm2 = f2_pack(-mref_new, -mref_new);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // keep flags of this row for keys 64g + 32h + 4c + (0..3)
          uint32_t kw[8];
          if constexpr (DR) {
            const uint32_t kp0 = (uint32_t)(j * 32 + 16 * g + 8 * h) + (uint32_t)(lane & 3);
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
              const Philox4 o = philox4x32_10(kp0 + 4 * gg, (uint32_t)row >> 2,
                                              (uint32_t)bh, 0u, p.drop.k0, p.drop.k1);
              uint32_t a[4] = {o.x[0], o.x[1], o.x[2], o.x[3]};
              quad_transpose(a, lane);
#pragma unroll
              for (int c = 0; c < 4; ++c) kw[4 * gg + c] = keep_flags(a[c], p.drop);
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = 32 * h + 2 * i;
            float a, b;
            f2_unpack(ffma2(f2_pack(x[e], x[e + 1]), sl2x2, nm2), a, b);
            a = ex2_approx(a);
            b = ex2_approx(b);
            acc[i & 3] = fadd2(acc[i & 3], f2_pack(a, b));
            pk[i] = pack_bf16x2(a, b);
            if constexpr (DR) pk[i] &= pair_mask(kw[i >> 1], i);
          }
          // P of keys 64g + 32h + (0..31): columns 32g + 16h .. + 15 (inside
          // the columns both halves have already read)
          tmem_st16(tS + 32 * g + 16 * h, pk);
        }
        float rs_lo, rs_hi;
        f2_unpack(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), rs_lo, rs_hi);
        l = l * alpha + (rs_lo + rs_hi);
        // O *= alpha on this half's 128 columns once the previous P V product
        // has completed.  Waiting on its phase by parity is exact here: the
        // one before it has completed (S_j was issued after it, or it belongs
        // to the previous item, whose completion the epilogue awaited), and
        // the next cannot start before this thread's p_ready arrival.
        if (j > jlo && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!wait_warp(bar(B_PVDONE), (gj - 1) & 1, abort_flag, lim, SITE_S_PVDONE)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t al2 = f2_pack(alpha, alpha);
          const uint32_t tO = tmem + lane_off + TM_O + 128 * g;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
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
        mbar_arrive(bar(B_PREADY + buf));
      }
      if (!ok) break;
      // epilogue: the item's last P V product (its own barrier: up to two P V
      // products may still be running here, which one parity cannot tell
      // apart), the two halves of l, O / l
      if (!wait_warp(bar(B_ODONE), it & 1, abort_flag, lim, SITE_S_ODONE)) break;
      tc_fence_after();
      xl[g * 128 + rb] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_XL + wq));
      if (!wait_warp(bar(B_XL + wq), it & 1, abort_flag, lim, SITE_S_XL)) break;
      __syncwarp();
      const float lt = l + xl[(g ^ 1) * 128 + rb];
      const float inv_l = (DR ? p.drop.keep_scale : 1.f) / lt;
      const bool store = row < sc.N;
      __nv_bfloat16* orow =
          p.O + ((size_t)bh * sc.N + (size_t)(store ? row : 0)) * D + 128 * g;
      const uint32_t tO = tmem + lane_off + TM_O + 128 * g;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
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
      if (store && g == 0)
        p.LSE[(size_t)bh * sc.N + row] = (mref + log2f(lt)) * 0.69314718055994531f;
      // O has been read before the next item's first P V product (ordered by
      // this thread's next p_ready arrival)
      tc_fence_before();
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  FA_TRACE_MARK(g_cta_trace, 1);
  if (warp == kMmaWarp) tmem_dealloc(tmem, TMEM_COLS);
}

template <bool W, bool DR>
cudaError_t launch(const AttnShape& s, const TileMaps& maps, void* O, float* LSE,
                   int num_sms, uint64_t lim, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  const cudaError_t attr = smem_limit_once(fwd256_kernel<W, DR>, SMEM_BYTES, attr_done);
  if (attr != cudaSuccess) return attr;
  Params p;
  p.O = reinterpret_cast<__nv_bfloat16*>(O);
  p.LSE = LSE;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.wait_limit_ns = lim;
  p.drop = s.drop;
  const int BH = s.B * s.H;
  FwdSched probe;
  probe.init(BH, s.N, s.causal, num_sms, s.window, 1);
  const int grid = probe.total_items < num_sms ? probe.total_items : num_sms;
  p.sched.init(BH, s.N, s.causal, grid, s.window, 1);
  fwd256_kernel<W, DR><<<grid, kThreads, SMEM_BYTES, stream>>>(maps.q, maps.k, maps.v, p);
  return cudaGetLastError();
}

}  // namespace fwd256

cudaError_t launch_fwd256_tc(const AttnShape& s, const TileMaps& maps, void* O,
                             float* LSE, int num_sms, uint64_t wait_limit_ns,
                             cudaStream_t stream) {
  const uint64_t lim = wait_limit_ns;
  const bool w = s.window > 0;
  if (s.drop.t4 != 0)
    return w ? fwd256::launch<true, true>(s, maps, O, LSE, num_sms, lim, stream)
             : fwd256::launch<false, true>(s, maps, O, LSE, num_sms, lim, stream);
  return w ? fwd256::launch<true, false>(s, maps, O, LSE, num_sms, lim, stream)
           : fwd256::launch<false, false>(s, maps, O, LSE, num_sms, lim, stream);
}

FA_DEFINE_STATUS_READER(read_status_fwd256_tc)

}  // namespace fa
