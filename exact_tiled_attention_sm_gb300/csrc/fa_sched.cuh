// fa_sched.cuh -- the forward kernel's causal tile scheduler (host + device).
//
// A work item is one head (b, h) and one pair of consecutive 128-row query
// blocks (rows [256*pair, 256*pair + 256)), or one query block for kernels
// that hold a single block (blocks_per_item = 1; "pair" is then the block).  For query block q, the key
// blocks visited are j = kv_lo(q) .. kv_hi(q): all of them without a mask;
// up to the diagonal (kv_hi = q) under the causal mask, where a key block
// whose first key lies after the query block's last row is never loaded or
// multiplied ("LLM Architecture Refresh [3]", section 7); and with a sliding
// window of w keys (query r sees keys r-w+1 .. r, section 5's contrast) also
// from the block holding the first row's oldest visible key, so blocks that
// are entirely too old are skipped the same way.  Only the blocks a mask
// edge cuts (the diagonal, the window's left edge, a ragged last block) are
// masked element by element.
//
// Balance.  Causal items cost in proportion to (pair + 1), so within a group
// of heads items are listed heaviest first, and a persistent grid takes the
// list in waves of `grid` items with the CTA order reversed on every other
// wave ("snake"), pairing heavy with light items.  Without a mask every item
// costs the same and only the last, partial wave is uneven: when its pairs
// fill at most half a wave, each is split into its two query blocks, which
// the CTAs then take one each (a single-block item runs one softmax group
// and finishes sooner).  Locality.  The list is
// grouped by heads, `group` heads (about kGroupWaves waves of items) at a
// time, so the K/V blocks that the running CTAs stream are shared through L2
// instead of re-read from HBM.
#pragma once

namespace fa {

// Under the causal mask a head group holds about this many waves of items:
// enough for the snake order to pair heavy with light items within the
// group, few enough heads that the group's K/V (forward) or Q/dO (backward)
// mostly stay in L2.  Eight waves balance the per-CTA work to within 2-3% on
// the measured shapes (N = 2048 ... 32768), where four left the last,
// partial group's heaviest items in one wave (a 21% loss at N = 16384).
// Without the mask every item costs the same and one wave per group keeps the
// most reuse.
constexpr int kGroupWaves = 8;
// The backward's items hold more per head in L2 (Q, dO and the fp32 dQ
// accumulator): eight waves of heads measured 6% slower than four, which
// balance its N = 2048 training shape equally well.
constexpr int kBwdGroupWaves = 4;

struct FwdSched {
  int BH, N, causal, window, grid;
  int n_q_tiles, n_pairs, n_kv_total, group, total_items;
  int split_from;  // items from here on are single query blocks of split pairs

  // window > 0: causal sliding window of `window` keys (implies causal).
  // n_pairs counts the items of one head (pairs, or blocks when
  // blocks_per_item = 1).
  __host__ __device__ void init(int bh, int n, int is_causal, int grid_size,
                                int win = 0, int blocks_per_item = 2) {
    BH = bh;
    N = n;
    window = win > 0 ? win : 0;
    causal = (is_causal || window > 0) ? 1 : 0;
    grid = grid_size;
    n_q_tiles = (N + 127) / 128;
    n_kv_total = n_q_tiles;
    n_pairs = (n_q_tiles + blocks_per_item - 1) / blocks_per_item;
    int g = (causal ? kGroupWaves : 1) * grid / n_pairs;
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    group = g;
    total_items = BH * n_pairs;
    split_from = total_items;
    const int tail = total_items % grid;
    if (blocks_per_item == 2 && !causal && (n_q_tiles & 1) == 0 && tail > 0 &&
        2 * tail <= grid) {
      split_from = total_items - tail;
      total_items += tail;
    }
  }

  // The forward launch's schedule: a grid of num_sms CTAs, or one CTA per
  // item when the items do not fill it (two-block items).
  static FwdSched planned(int bh, int n, int is_causal, int num_sms, int win = 0) {
    FwdSched probe;
    probe.init(bh, n, is_causal, num_sms, win);
    FwdSched sc;
    sc.init(bh, n, is_causal,
            probe.total_items < num_sms ? probe.total_items : num_sms, win);
    return sc;
  }

  // The d = 64 forward's schedule: single-block items for two workers per
  // CTA (its two query-block groups, worker g * CTAs + cta), so `grid`
  // counts workers and the launch takes grid / 2 CTAs of at most num_sms.
  static FwdSched planned_groups(int bh, int n, int is_causal, int num_sms, int win = 0) {
    FwdSched probe;
    probe.init(bh, n, is_causal, 2 * num_sms, win, 1);
    int ctas = (probe.total_items + 1) / 2;
    if (ctas > num_sms) ctas = num_sms;
    FwdSched sc;
    sc.init(bh, n, is_causal, 2 * ctas, win, 1);
    return sc;
  }

  // Number of waves a CTA walks through.
  __host__ __device__ int n_waves() const {
    return (total_items + grid - 1) / grid;
  }

  // Item taken by CTA `cta` in wave `w`, or -1 if that slot is past the end.
  __host__ __device__ int item_of(int cta, int w) const {
    int pos = (w & 1) ? (grid - 1 - cta) : cta;
    int i = w * grid + pos;
    return i < total_items ? i : -1;
  }

  // Item index -> (flat head bh, query-block pair).
  __host__ __device__ void decode(int i, int& bh, int& pair) const {
    const int per_group = group * n_pairs;
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
    pair = n_pairs - 1 - r / gs;  // heaviest pairs first within a group
    bh = g * group + r % gs;
  }

  // Item index -> (flat head bh, first query block q0, whether the item also
  // holds block q0 + 1), for items of up to two blocks.
  __host__ __device__ __forceinline__ void decode_blocks(int i, int& bh, int& q0,
                                                        bool& two) const {
    int pair;
    const bool single = i >= split_from;
    const int u = i - split_from;
    decode(single ? split_from + (u >> 1) : i, bh, pair);
    q0 = 2 * pair + (single ? (u & 1) : 0);
    two = !single && (2 * pair + 1 < n_q_tiles);
  }

  // First and last key block visited by query block q (q < n_q_tiles).
  __host__ __device__ int kv_lo(int q) const {
    if (window == 0) return 0;
    const int first_key = q * 128 - window + 1;  // oldest key row q*128 sees
    return first_key <= 0 ? 0 : first_key / 128;
  }
  __host__ __device__ int kv_hi(int q) const {
    const int n = !causal ? n_kv_total
                          : (q + 1 < n_kv_total ? q + 1 : n_kv_total);
    return n - 1;
  }
  // Number of key blocks visited by query block q.
  __host__ __device__ int n_kv(int q) const { return kv_hi(q) - kv_lo(q) + 1; }

  // Does key block j of query block q need an element mask for the causal
  // diagonal or the ragged end?  (window_edge: for the window's left edge.)
  __host__ __device__ bool needs_mask(int q, int j) const {
    return (causal && j == q) || (j == n_kv_total - 1 && (N & 127) != 0);
  }
  __host__ __device__ bool window_edge(int q, int j) const {
    return window > 0 && j * 128 < q * 128 + 128 - window;
  }
};

// The backward kernel's scheduler: a work item is one head and one 128-key
// block kb; the CTA keeps K_kb and V_kb resident and walks the query blocks
// i = q_begin(kb) .. q_end(kb) (i >= kb under the causal mask: query blocks
// that lie entirely before the key block see none of it; with a sliding
// window also i <= the block of the last query whose window still reaches
// the key block's last key).  Causal cost is
// proportional to n_blk - kb, so items are listed kb-ascending (heaviest
// first) inside head groups, and taken in snake waves as in FwdSched.
struct BwdSched {
  int BH, N, causal, window, grid;
  int n_blk, group, total_items;

  // window > 0: causal sliding window of `window` keys (implies causal).
  __host__ __device__ void init(int bh, int n, int is_causal, int grid_size,
                                int win = 0) {
    BH = bh;
    N = n;
    window = win > 0 ? win : 0;
    causal = (is_causal || window > 0) ? 1 : 0;
    grid = grid_size;
    n_blk = (N + 127) / 128;
    int g = (causal ? kBwdGroupWaves : 1) * grid / n_blk;
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    group = g;
    total_items = BH * n_blk;
  }

  __host__ __device__ int n_waves() const {
    return (total_items + grid - 1) / grid;
  }

  __host__ __device__ int item_of(int cta, int w) const {
    int pos = (w & 1) ? (grid - 1 - cta) : cta;
    int i = w * grid + pos;
    return i < total_items ? i : -1;
  }

  __host__ __device__ void decode(int i, int& bh, int& kb) const {
    const int per_group = group * n_blk;
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

  __host__ __device__ int q_begin(int kb) const { return causal ? kb : 0; }
  // Last query block that sees any key of block kb (inclusive).
  __host__ __device__ int q_end(int kb) const {
    if (window == 0) return n_blk - 1;
    const int last_q = kb * 128 + 127 + window - 1;  // its window's newest row
    const int blk = last_q / 128;
    return blk < n_blk - 1 ? blk : n_blk - 1;
  }
  // Does query block i see some key of block kb only partly (the window's
  // left edge cuts the tile)?
  __host__ __device__ bool window_edge(int i, int kb) const {
    return window > 0 && (i - kb) * 128 + 127 >= window;
  }
};

}  // namespace fa
