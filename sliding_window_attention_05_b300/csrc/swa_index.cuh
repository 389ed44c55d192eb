// swa_index.cuh -- index arithmetic of SWA(w, s) shared by the host launcher
// and the device kernels: ring-cache slots, the prefill tiling plan, the
// per-query-block tile list (band-aware schedule) and the in-tile mask.
//
// Key set of query t (explainer of arXiv 2608.28444, section "核心方法 / 1."):
//   K(t) = { j : j <= t and (j >= t - w + 1 or j < s) }.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define SWA_HD __host__ __device__ __forceinline__
#else
#define SWA_HD inline
#endif

namespace swa {

SWA_HD int imin(int a, int b) { return a < b ? a : b; }
SWA_HD int imax(int a, int b) { return a > b ? a : b; }
SWA_HD int cdiv(int a, int b) { return (a + b - 1) / b; }
SWA_HD int round_up(int a, int b) { return cdiv(a, b) * b; }

// Ring-cache slot of position p (wiblog.cn long-context SWA article, section
// "与 KV Cache 的配合：轮转替换策略": the oldest window entry is overwritten and
// the slot is found modulo the window). The first s positions keep slots
// 0..s-1 for good; later positions cycle through slots s..s+w-1.
SWA_HD long long ring_slot(long long p, int w, int s) {
  return p < s ? p : s + (p - s) % w;
}

// Number of valid cache slots once position p has been appended.
SWA_HD int ring_valid(long long p, int w, int s) {
  long long n = p + 1;
  long long cap = (long long)s + w;
  return (int)(n < cap ? n : cap);
}

// Membership of key j in K(t), intersected with the tile's owned key range
// [own_lo, own_hi) so that no pair is counted by two tiles.
SWA_HD bool admit(int t, int j, int w, int s, int own_lo, int own_hi) {
  return j >= own_lo && j < own_hi && j <= t && (j >= t - w + 1 || j < s);
}

// ---------------------------------------------------------------- prefill plan
//
// A CTA work item is one query block: Tq consecutive query positions of one
// (batch, KV head), packed with all G = Hq/Hkv query heads of that KV head into
// the M = 128 rows of one tensor-core tile (row r <-> position t0 + r / G,
// head kvh * G + r % G). Packing the group shrinks the key span a block needs
// from (w + 127) to (w + Tq - 1) keys.
//
// A block visits a short list of key tiles (at most kMaxTileKeys keys each,
// the MMA's N): its band tiles, which cover the window part of every row, and
// the sink keys. The sinks ride in the first band tile (a second TMA box in
// the same shared-memory slot) when that tile has room, otherwise they form
// tiles of their own. Every tile not listed is skipped: no load, no MMA, no
// exponential.
constexpr int kMaxTileKeys = 192;

struct PrefillPlan {
  int G;          // query heads per KV head
  int Tq;         // query positions per block
  int bpi;        // query blocks per work item (1, or 2: a pair sharing its key tiles)
  int kmax;       // widest key tile (MMA N)
  int rows;       // Tq * G <= 128 (rows past this stay zero)
  int n_band;     // keys per band tile (multiple of 16, <= kMaxTileKeys)
  int s_box;      // keys per sink box (multiple of 16, <= 128), 0 if s == 0
  int n_sink;     // sink boxes, ceil(s / 128); 0 if s == 0
  int merge;      // 1: the (single) sink box rides in the first band tile
  int sink_last;  // 1: otherwise the (single) sink box may ride in a block's
                  // last band tile (when its owned keys fit in n_band - s_box
                  // columns), ahead of a band box loaded s_box rows shorter
  int slot_keys;  // keys one K/V ring slot holds: the widest tile
  int steady_tiles;  // tiles a block far from the sequence start visits
  int nqb;        // query blocks per (batch, KV head)
  float inv_band; // 1 / n_band (device-side division by n_band)
};

// ceil(x / p.n_band) for x >= 0. Below 2^22 the device path multiplies by
// the float reciprocal and corrects the quotient by one step either way.
SWA_HD int cdiv_band(const PrefillPlan &p, int x) {
#if defined(__CUDA_ARCH__)
  const int y = x + p.n_band - 1;
  if (y >= (1 << 22)) return y / p.n_band;
  int q = (int)((float)y * p.inv_band);
  if (q * p.n_band > y) --q;
  if ((q + 1) * p.n_band <= y) ++q;
  return q;
#else
  return cdiv(x, p.n_band);
#endif
}

// kmax: widest key tile; bpi: query blocks per work item. A pair item
// (bpi = 2) covers blocks qb and qb + 1, whose key ranges differ only by Tq
// keys at either end, so one list of key tiles serves both. allow_sink_last:
// the kernel can load a shortened band box (sink_last below).
SWA_HD PrefillPlan make_plan(int L, int Hq, int Hkv, int w, int s, int kmax = kMaxTileKeys,
                             int bpi = 1, int allow_sink_last = 0) {
  PrefillPlan p;
  p.G = Hq / Hkv;
  p.Tq = 128 / p.G;
  p.bpi = bpi;
  p.kmax = kmax;
  p.rows = p.Tq * p.G;
  p.nqb = cdiv(L, p.Tq);
  // Band tiles: spread the steady-state span (w + bpi * Tq - 1 keys) evenly
  // over the fewest tiles of at most kmax keys, rounded up to the MMA's N
  // granularity of 16.
  long long span = (long long)imin(w, L) + (long long)bpi * p.Tq - 1;
  if (span > L) span = L;
  // Tile widths are kept to multiples of 32 keys so that the two softmax
  // warps sharing a row (bpi = 1) take equal halves of every tile (and run
  // the same code).
  const int nt = (int)((span + kmax - 1) / kmax);
  p.n_band = imin(kmax, round_up(cdiv((int)span, nt), 32));
  if (s > 0) {
    p.n_sink = cdiv(s, 128);
    p.s_box = imin(128, round_up(cdiv(s, p.n_sink), 16));
  } else {
    p.n_sink = 0;
    p.s_box = 0;
  }
  p.merge = (p.n_sink == 1 && round_up(p.s_box + p.n_band, 32) <= kmax) ? 1 : 0;
  if (p.merge) p.n_band = round_up(p.s_box + p.n_band, 32) - p.s_box;
  p.inv_band = 1.0f / (float)p.n_band;
  // The sink box rides in the last band tile when that tile owns at most
  // n_band - s_box keys in the steady state (the span's remainder): one tile
  // fewer per block than a tile of sinks alone.
  const int nb_steady = cdiv((int)span, p.n_band);
  const int own_last_steady = (int)span - (nb_steady - 1) * p.n_band;
  p.sink_last = (allow_sink_last && bpi == 1 && !p.merge && p.n_sink == 1 &&
                 p.s_box < p.n_band && own_last_steady <= p.n_band - p.s_box)
                    ? 1
                    : 0;
  p.steady_tiles = (p.merge || p.sink_last ? 0 : p.n_sink) + nb_steady;
  p.slot_keys = p.merge ? p.s_box + p.n_band : imax(p.n_band, p.s_box);
  return p;
}

// The tiles one work item visits (for a pair, both blocks' keys): tiles of sink boxes first (when the sinks
// ride in neither the first nor the last band tile), then band tiles that cover [lo, t_last].
struct BlockTiles {
  int t0;          // first query position of the block
  int t_last;      // last valid query position (< L)
  int lo;          // first key of the band part
  int n_sink;      // tiles made of sink boxes only
  int sink_first;  // 1: the first band tile also carries the sink box
  int sink_last;   // 1: the last band tile also carries the sink box
  int n_tiles;     // all tiles
};

// kMaySinkLast = false compiles the sink_last case out (kernels whose plan
// never sets it).
template <bool kMaySinkLast = true>
SWA_HD BlockTiles block_tiles(const PrefillPlan &p, int qb, int L, int w, int s) {
  BlockTiles b;
  b.t0 = qb * p.Tq;
  b.t_last = imin(b.t0 + p.bpi * p.Tq, L) - 1;
  int lo = imax(0, b.t0 - w + 1);  // leftmost window key of any row in the block
  b.n_sink = 0;
  b.sink_first = 0;
  b.sink_last = 0;
  if (s > 0 && lo >= s) {          // sinks lie left of every row's window
    if (p.merge) {
      b.sink_first = 1;
    } else if (kMaySinkLast && p.sink_last &&
               b.t_last - lo + 1 - (cdiv_band(p, b.t_last - lo + 1) - 1) * p.n_band <=
                   p.n_band - p.s_box) {
      b.sink_last = 1;             // the last band tile owns few enough keys
    } else {
      b.n_sink = p.n_sink;
    }
  } else if (s > 0) {
    lo = 0;                        // window reaches the sinks: one merged range
  }
  b.lo = lo;
  b.n_tiles = b.n_sink + cdiv_band(p, b.t_last - lo + 1);
  return b;
}

// The work items of one persistent CTA: item = first, first + stride, ...
// Each item is a query block qb of one (batch, KV head) pair bh, with
// item = (nqb - 1 - qb) * BH + bh, so the longest blocks of a causal prompt
// come first. Advancing costs no division.
struct ItemWalker {
  int item, stride, n_items, BH, nqb;
  int q, rem;    // item / BH, item % BH
  int sq, sr;    // stride / BH, stride % BH
  SWA_HD ItemWalker(int first, int stride_, int n_items_, int BH_, int nqb_)
      : item(first), stride(stride_), n_items(n_items_), BH(BH_), nqb(nqb_) {
    q = first / BH;
    rem = first % BH;
    sq = stride / BH;
    sr = stride % BH;
  }
  SWA_HD bool valid() const { return item < n_items; }
  SWA_HD int qb() const { return nqb - 1 - q; }
  SWA_HD int bh() const { return rem; }
  SWA_HD void next() {
    item += stride;
    q += sq;
    rem += sr;
    if (rem >= BH) {
      rem -= BH;
      ++q;
    }
  }
};

// One key tile. Its ncols columns are, in order: n_sink_cols columns holding
// the sink box keys sink_key0, sink_key0 + 1, ... (loaded with the sink tensor
// map), then the band columns holding keys k0, k0 + 1, ... of which the tile
// owns [own_lo, own_hi) (no key is owned by two tiles of a block).
struct Tile {
  int n_sink_cols;
  int sink_key0;
  int k0;
  int own_lo;
  int own_hi;
  int ncols;     // MMA N (multiple of 16, <= kMaxTileKeys)
  bool full;     // every (row, key) pair of the tile is admitted for the
                 // item's first block: no mask needed
};

// Whether every (row, key) pair of tile t is admitted for the query rows of
// the block t0q .. t0q + Tq - 1: all columns are owned band keys and, for every
// row q, inside [q - w + 1, q] (the in-band interior tiles, which need no mask).
// For a pair item, each of its two blocks asks this for itself.
SWA_HD bool tile_full_for(const Tile &t, int t0q, int Tq, int w) {
  const bool owned_all = t.n_sink_cols == 0 && (t.own_hi - t.own_lo) == t.ncols;
  const bool causal_ok = t.k0 + t.ncols - 1 <= t0q;
  const bool window_ok = t.k0 >= t0q + Tq - 1 - w + 1;
  return owned_all && causal_ok && window_ok;
}

template <bool kMaySinkLast = true>
SWA_HD Tile tile_at(const PrefillPlan &p, const BlockTiles &b, int i, int w, int s) {
  Tile t;
  if (i < b.n_sink) {            // a tile of one sink box
    t.n_sink_cols = p.s_box;
    t.sink_key0 = i * p.s_box;
    t.k0 = 0;
    t.own_lo = t.own_hi = 0;     // no band keys
    t.ncols = p.s_box;
    t.full = false;
    return t;
  }
  const int bi = i - b.n_sink;
  // the sink box rides in the first band tile (merge) or the last (sink_last);
  // either way its columns come first, the band keys after them
  t.n_sink_cols =
      ((b.sink_first && bi == 0) || (kMaySinkLast && b.sink_last && i == b.n_tiles - 1))
          ? p.s_box
          : 0;
  t.sink_key0 = 0;
  t.k0 = b.lo + bi * p.n_band;
  t.own_lo = t.k0;
  t.own_hi = imin(t.k0 + p.n_band, b.t_last + 1);
  // the loaded band box is n_band keys; columns past the owned keys are masked
  t.ncols = imin(t.n_sink_cols + p.n_band, round_up(t.n_sink_cols + t.own_hi - t.own_lo, 32));
  t.full = tile_full_for(t, b.t0, p.Tq, w);
  return t;
}

// The key held by column c of a tile.
SWA_HD int tile_key(const Tile &t, int c) {
  return c < t.n_sink_cols ? t.sink_key0 + c : t.k0 + (c - t.n_sink_cols);
}

// Whether query t admits column c of a tile (the tile's share of K(t)).
SWA_HD bool tile_admit(const Tile &t, int c, int q, int w, int s) {
  if (t.full) return true;
  const int j = tile_key(t, c);
  if (c < t.n_sink_cols) return j < s && j <= q;
  return admit(q, j, w, s, t.own_lo, t.own_hi);
}

// The admitted columns of a tile for query t form at most two ranges of
// column indices, [a_lo, a_hi) (band keys inside the window) and [b_lo, b_hi)
// (sink keys); either may be empty.
struct ColRanges {
  int a_lo, a_hi, b_lo, b_hi;
};

SWA_HD ColRanges tile_ranges(const Tile &t, int q, int w, int s) {
  ColRanges r;
  const int off = t.n_sink_cols - t.k0;  // column of band key j is j + off
  r.a_lo = imax(t.own_lo, q - w + 1) + off;
  r.a_hi = imin(t.own_hi, q + 1) + off;
  if (t.n_sink_cols > 0) {
    r.b_lo = 0;
    r.b_hi = imax(0, imin(imin(s, q + 1) - t.sink_key0, t.n_sink_cols));
  } else {
    // band keys below s are sinks too (the window reaches the sinks)
    r.b_lo = t.own_lo + off;
    r.b_hi = imin(imin(t.own_hi, s), q + 1) + off;
  }
  return r;
}

}  // namespace swa
