/*
 * fa.h -- C ABI of the exact tiled attention library (libfa.so) for one
 * sm_103a GPU.
 *
 * What it computes.  For every batch b and head h, with Q, K, V the N x d
 * slices of that head:
 *
 *     O = softmax(scale * Q K^T) V,        LSE_r = m_r + ln(l_r),
 *
 * tile by tile with an online softmax: a running row max m and a running row
 * sum l rescale the partial output when a later key/value block raises the
 * max (the forward keeps its exponent reference until the max has risen past
 * it by a factor 2^8, which leaves O / l and LSE unchanged and makes the
 * rescale rare), and the division by l happens once at the end ("Flash Attention,
 * From First Principles", sections "Online softmax -- the game" through "The
 * scaffold"; "LLM Architecture Refresh [3]", section 4).  The N x N score
 * matrix never reaches device memory.  With causal != 0, key k is visible to
 * query r only when k <= r (queries and keys share one length N); key blocks
 * that lie entirely in the future are skipped and only diagonal blocks are
 * masked ("LLM Architecture Refresh [3]", section 7).  The backward pass
 * recomputes the probabilities from Q, K and the saved LSE,
 * P = exp(scale*QK^T - LSE), and forms dV = P^T dO, dP = dO V^T,
 * D = rowsum(dO * O), dS = P * (dP - D), dQ = scale * dS K,
 * dK = scale * dS^T Q ("FlashAttention from scratch", follow-up "How do you
 * implement the backward pass of flash attention?").
 *
 * Conventions shared by every entry point.
 *   - Tensors are caller-owned device memory, contiguous, in [B][H][N][d]
 *     order (batch, heads, sequence, head dimension), base pointers 16-byte
 *     aligned.  O, dQ, dK, dV have the input dtype; LSE is fp32 [B][H][N],
 *     natural log.
 *   - dt = FA_BF16: bf16 inputs, fp32 accumulation on the tensor cores.
 *     dt = FA_F32: fp32 inputs and arithmetic throughout (CUDA cores).
 *   - d must be 64, 128 or 256; N >= 1; B, H >= 1; B*H*N*d must fit in
 *     2^31 elements per tensor; scale must be finite.
 *   - d = 256 (the d^2/M wall of "Flash Attention, From First Principles",
 *     "The rent arithmetic": one query block's S and O fill the tensor
 *     memory): the bf16 forward runs on the tensor cores with one 128-row
 *     query block per work item; the bf16 backward runs on the CUDA cores in
 *     fp32 arithmetic (its tensor-core layout would need 768 TMEM columns);
 *     fp32 inputs run on the CUDA cores as for every d.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  The returned status covers argument checks and the
 *     launch only; device-side failures (a bounded wait that ran out) are
 *     reported by fa_last_device_status().
 *   - Argument errors return before anything is launched.  The library
 *     allocates no device memory in fa_fwd / fa_bwd.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned, bad scale  */
  FA_ERR_UNSUPPORTED = 2, /* d not in {64,128,256}, unknown dtype, no sm_103a */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed              */
  FA_ERR_TIMEOUT = 4      /* a device-side bounded wait ran out             */
} fa_status;

typedef enum { FA_BF16 = 0, FA_F32 = 1 } fa_dtype;

/* Forward pass.  Reads Q, K, V; writes O and LSE.  Steps: schedule (causal
 * tile skip), TMA tile loads, S = scale*Q K^T, diagonal/ragged masking,
 * online softmax with deferred division, O += P V, epilogue.
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA. */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O,
                 float* LSE, int B, int H, int N, int d, float scale,
                 int causal, fa_dtype dt, void* stream);

/* Bytes of device workspace fa_bwd needs: an fp32 dQ accumulator
 * [B][H][N][d] and D = rowsum(dO * O) [B][H][N], each 256-byte aligned.
 * Returns 0 for sizes fa_bwd would reject. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/* Backward pass.  Reads Q, K, V, O, dO and the forward's LSE; writes dQ, dK,
 * dV.  `workspace` is caller-owned device memory of at least
 * fa_bwd_workspace_size() bytes (256-byte aligned); its contents on entry do
 * not matter and on return are unspecified.  Steps: D and zeroed dQ
 * accumulator; per key block, recompute S and P from LSE, dV += P^T dO,
 * dP = dO V^T, dS = P*(dP - D), dK += scale*dS^T Q, dQacc += scale*dS K
 * (fp32 bulk reduce-adds); dQ = dQacc converted to the input dtype.
 * In bf16 the call is three launches on `stream` (D and the zeroed
 * accumulator; the backward kernel; the conversion).  The second and third
 * are programmatic dependent launches: each may start while the one before
 * it ends and waits on the device for that one's results.  Work queued on
 * `stream` before the call, or after it, is ordered against the whole call
 * as usual, stream capture included.
 * Errors: as fa_fwd, plus FA_ERR_INVALID_ARG for a short workspace. */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O,
                 const void* dO, const float* LSE, void* dQ, void* dK,
                 void* dV, int B, int H, int N, int d, float scale,
                 int causal, fa_dtype dt, void* workspace,
                 size_t workspace_bytes, void* stream);

/* Causal sliding window ("LLM Architecture Refresh [3]", section 5, the
 * sliding-window contrast: each query attends only to the last `window`
 * keys, itself included), forward and backward.  Key k is visible to query r
 * iff r - window + 1 <= k <= r.  The arguments and conventions are those of
 * fa_fwd / fa_bwd with `causal` replaced by `window`; a window of N or more
 * is the causal computation.  Key blocks entirely older than a query block's
 * window are skipped like future ones, and only blocks a mask edge cuts are
 * masked element by element.
 * Errors: as fa_fwd / fa_bwd, plus FA_ERR_INVALID_ARG for window < 1. */
fa_status fa_fwd_window(const void* Q, const void* K, const void* V, void* O,
                        float* LSE, int B, int H, int N, int d, float scale,
                        int window, fa_dtype dt, void* stream);
fa_status fa_bwd_window(const void* Q, const void* K, const void* V,
                        const void* O, const void* dO, const float* LSE,
                        void* dQ, void* dK, void* dV, int B, int H, int N,
                        int d, float scale, int window, fa_dtype dt,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Attention dropout ("Flash Attention, From First Principles", "Honesty
 * time -- the confession list", item 4: the extra lines of the paper's
 * algorithm 2), forward and backward.  After the softmax each probability
 * p_rk is multiplied by M_rk = keep_rk * 256 / (256 - t), keep_rk in {0, 1},
 * so O = (P o M) V; LSE is that of the undropped row.  The backward uses
 * dV = (P o M)^T dO, dS = P o (M o dP - D) with D = rowsum(dO * O).
 *   - t = round(256 * dropout_p), ties to even (fa_dropout_threshold); each
 *     entry is dropped with probability t/256.  dropout_p must be finite and
 *     round to t <= 255; t = 0 is the computation without dropout.
 *   - keep_rk comes from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 *     random numbers: as easy as 1, 2, 3", SC'11) with key (seed & 0xFFFFFFFF,
 *     seed >> 32) and counter (k/4, r/4, b*H + h, 0): byte (k mod 4) of output
 *     word (r mod 4) is (r, k)'s, and keep_rk = (byte >= t).  The mask is a
 *     pure function of (seed, head, r, k): no state is kept between calls,
 *     and fa_bwd_dropout with the forward's seed regenerates the forward's
 *     mask exactly.
 *   - causal and window select the mask as in fa_fwd / fa_fwd_window: window
 *     = 0 means none (causal decides), window >= 1 a causal sliding window.
 * The other arguments and conventions are those of fa_fwd / fa_bwd.
 * Errors: as fa_fwd / fa_bwd, plus FA_ERR_INVALID_ARG for window < 0 or a
 * dropout_p outside the range above. */
fa_status fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O,
                         float* LSE, int B, int H, int N, int d, float scale,
                         int causal, int window, float dropout_p,
                         unsigned long long seed, fa_dtype dt, void* stream);
fa_status fa_bwd_dropout(const void* Q, const void* K, const void* V,
                         const void* O, const void* dO, const float* LSE,
                         void* dQ, void* dK, void* dV, int B, int H, int N,
                         int d, float scale, int causal, int window,
                         float dropout_p, unsigned long long seed, fa_dtype dt,
                         void* workspace, size_t workspace_bytes, void* stream);

/* The byte threshold t of a dropout probability (see fa_fwd_dropout), or -1
 * when fa_fwd_dropout would reject it.  Pure host arithmetic. */
int fa_dropout_threshold(float dropout_p);

/* Writes the keep mask of fa_fwd_dropout to `keep`: caller-owned device
 * memory of B*H*N*N bytes in [B][H][r][k] order, 1 where (r, k) is kept and
 * 0 where it is dropped (for every pair, whatever the causal or window
 * mask).  For inspection and testing; the attention entry points never
 * store the mask.  Asynchronous on `stream`.
 * Errors: FA_ERR_INVALID_ARG for a null pointer, B, H or N < 1, N > 262140,
 * or a dropout_p fa_dropout_threshold rejects; FA_ERR_CUDA. */
fa_status fa_dropout_mask(unsigned char* keep, int B, int H, int N,
                          float dropout_p, unsigned long long seed,
                          void* stream);

/* Forward pass with 8-bit inputs (the low-precision arithmetic the pages
 * credit to FlashAttention-3: "LLM Architecture Refresh [3]", section 8;
 * "FlashAttention from scratch", "Trade-offs and edge cases").
 * Q, K, V are OCP FP8 E4M3 bytes (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; no infinities), [B][H][N][d], standing for q_descale * Q,
 * k_descale * K and v_descale * V.  Computes the attention of those values:
 * S = scale * q_descale * k_descale * (Q K^T) with exact 8-bit products and
 * fp32 accumulation, P = exp(S - rowmax) rounded to E4M3 (times 2^8) for the
 * P V product, O = v_descale * (P V) / rowsum(P) written as bf16, and LSE
 * (fp32, natural log) as in fa_fwd.  causal and window as in
 * fa_fwd_dropout.  The rounding of P to E4M3 (3 mantissa bits) bounds the
 * error of O by about 2^-4 * sum_k p_k |v_k| per element.
 * Errors: FA_ERR_UNSUPPORTED for d != 128 or a device other than sm_103;
 * FA_ERR_INVALID_ARG for non-positive or non-finite factors, window < 0, and
 * the shape and alignment errors of fa_fwd. */
fa_status fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O,
                     float* LSE, int B, int H, int N, int d, float scale,
                     int causal, int window, float q_descale, float k_descale,
                     float v_descale, void* stream);

/* Size of the device scratch array that fa_bwd_noalloc uses in place of a
 * caller workspace: 64 MiB of static device memory, reserved on a GPU when
 * the code holding it is loaded there (with CUDA's default lazy loading: at
 * the first fa_bwd_noalloc call on that GPU) and held until the process
 * exits. */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64u << 20)

/* The backward pass for callers that cannot allocate device memory.  Some
 * callers only ever receive input and output buffers and have no way to
 * obtain more: a plugin whose host framework owns every device allocation
 * and hands out no allocator, a latency-critical loop where the implicit
 * synchronisation of cudaMalloc is not acceptable, or a deployment with a
 * device-memory budget fixed up front.  This entry point takes the
 * same arguments as fa_bwd minus the workspace and uses a
 * FA_BWD_NOALLOC_SCRATCH_BYTES array owned by the library instead; it calls
 * no cudaMalloc, cudaFree or other allocating routine.  (The pages have no
 * counterpart of this entry point: it is plumbing of this library.)
 *   - Sizes whose fa_bwd_workspace_size() exceeds the scratch are rejected
 *     with FA_ERR_INVALID_ARG before anything is launched (for d = 128 that
 *     is B*H*N above about 130,000 rows: 32 heads of 2048 fit, 32 of 4096 do
 *     not).  Other argument errors are those of fa_bwd.
 *   - The first call on a device is its set-up: it looks up the array's
 *     device address there (cudaGetSymbolAddress, with that device current)
 *     and keeps it.  That lookup loads the library's device code on that
 *     device if it is not loaded yet, which reserves the array: the one
 *     moment this entry point takes device memory, and it can synchronise.
 *     Make that first call before any stream capture and outside
 *     latency-critical loops (a warm-up call on each device does it).
 *   - The kept address belongs to the device's current context: after
 *     cudaDeviceReset on a device it is no longer valid, and this entry
 *     point must not be called there again in the same process.
 *   - All calls in the process share the one array and it keeps the last
 *     call's contents; the backward clears what must start at zero itself.
 *     Calls that overlap on the GPU (different streams, or several host
 *     threads) race on the array: serialise them. */
fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V,
                         const void* O, const void* dO, const float* LSE,
                         void* dQ, void* dK, void* dV, int B, int H, int N,
                         int d, float scale, int causal, fa_dtype dt,
                         void* stream);

/* Synchronises `stream`, then returns and clears the device-side status of
 * this library's kernels on the current device: FA_OK, or FA_ERR_TIMEOUT if
 * a bounded wait ran out since the last call (the kernel that gave up
 * skipped its remaining work, so its outputs are incomplete).  FA_ERR_CUDA
 * if the synchronisation itself failed. */
fa_status fa_last_device_status(void* stream);

/* Short English name of a status code (static storage). */
const char* fa_status_string(fa_status s);

/* Failure-detection self test: launches one CTA whose single wait is on a
 * barrier that nothing ever completes, with the given time limit in
 * microseconds (1..10,000,000).  The wait gives up, records FA_ERR_TIMEOUT
 * and the kernel exits normally; fa_last_device_status() then reports it.
 * Touches no user memory. */
fa_status fa_selftest_wait_timeout(unsigned int limit_us, void* stream);

/* Host-side view of the forward scheduler for one head: how many 128x128
 * (query block, key block) tiles the forward kernel computes and skips, and
 * how many work items (pairs of 128-row query blocks) it schedules.  Pure
 * host arithmetic, no GPU needed.  out = {computed, skipped, items}. */
fa_status fa_fwd_schedule_census(int N, int causal, long long* out);

/* As fa_fwd_schedule_census, with a causal sliding window of `window` keys
 * when window > 0 (window = 0: the mask selected by `causal`). */
fa_status fa_fwd_schedule_census_window(int N, int causal, int window,
                                        long long* out);

/* Host-side walk of the forward kernel's work list for BH heads of N rows
 * on a GPU with num_sms SMs, as a launch of fa_fwd at head dimension d would
 * plan it (d = 64: single query blocks for the two query-block groups of
 * each CTA; d = 128: pairs of query blocks).  counts[bh * ceil(N/128) + q]
 * is set to the number of work items that hold query block q of head bh
 * (every entry should be 1); *grid and *items, each when not NULL, to the
 * number of CTAs launched and of items in the list.  counts must hold
 * BH * ceil(N/128) ints.  window > 0 selects a causal sliding window, as in
 * fa_fwd_window.  Pure host arithmetic, no GPU needed.  Returns
 * FA_ERR_INVALID_ARG for BH, N or num_sms below 1, window < 0, a null
 * counts, or an item that would fall outside the tensor, and
 * FA_ERR_UNSUPPORTED for d other than 64 and 128.  No counterpart on the
 * pages: it exposes the scheduler so that its cover can be tested. */
fa_status fa_fwd_schedule_cover(int BH, int N, int causal, int window, int d,
                                int num_sms, int* counts, int* grid, int* items);

/* Library version, major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
