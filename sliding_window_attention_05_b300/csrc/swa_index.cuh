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
struct PrefillPlan {
  int G;          // query heads per KV head
  int Tq;         // query positions per block
  int rows;       // Tq * G <= 128 (rows past this stay zero)
  int n_band;     // keys per band tile (multiple of 16, <= 128)
  int s_box;      // keys per sink tile (multiple of 16, <= 128), 0 if s == 0
  int n_sink;     // sink tiles per block, 0 if s == 0
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

SWA_HD PrefillPlan make_plan(int L, int Hq, int Hkv, int w, int s) {
  PrefillPlan p;
  p.G = Hq / Hkv;
  p.Tq = 128 / p.G;
  p.rows = p.Tq * p.G;
  p.nqb = cdiv(L, p.Tq);
  // Band tiles: spread the steady-state span (w + Tq - 1 keys) evenly over the
  // fewest tiles of at most 128 keys, rounded up to the MMA's N granularity.
  long long span = (long long)imin(w, L) + p.Tq - 1;
  if (span > L) span = L;
  int nt = (int)((span + 127) / 128);
  p.n_band = imin(128, round_up(cdiv((int)span, nt), 16));
  p.inv_band = 1.0f / (float)p.n_band;
  if (s > 0) {
    p.n_sink = cdiv(s, 128);
    p.s_box = imin(128, round_up(cdiv(s, p.n_sink), 16));
  } else {
    p.n_sink = 0;
    p.s_box = 0;
  }
  return p;
}

// The tiles one query block visits: optional sink tiles first (so the running
// maximum is seen early), then band tiles that cover [lo, t_last]. Every tile
// not listed is skipped: no load, no MMA, no exponential.
struct BlockTiles {
  int t0;        // first query position of the block
  int t_last;    // last valid query position (< L)
  int lo;        // first key of the band part
  int n_sink;    // separate sink tiles (0 when the window reaches the sinks)
  int n_tiles;   // sink tiles + band tiles
};

SWA_HD BlockTiles block_tiles(const PrefillPlan &p, int qb, int L, int w, int s) {
  BlockTiles b;
  b.t0 = qb * p.Tq;
  b.t_last = imin(b.t0 + p.Tq, L) - 1;
  int lo = imax(0, b.t0 - w + 1);  // leftmost window key of any row in the block
  if (s > 0 && lo >= s) {
    b.n_sink = p.n_sink;           // sinks lie left of every row's window
  } else {
    b.n_sink = 0;
    if (s > 0) lo = 0;             // window reaches the sinks: one merged range
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

struct Tile {
  int k0;        // first key row loaded
  int own_lo;    // keys this tile is responsible for: [own_lo, own_hi)
  int own_hi;
  int ncols;     // MMA N: keys multiplied (multiple of 16, <= box rows)
  bool sink;     // loaded with the sink tensor map (box of s_box rows)
  bool full;     // every (row, key) pair of the tile is admitted: no mask needed
};

SWA_HD Tile tile_at(const PrefillPlan &p, const BlockTiles &b, int i, int w, int s) {
  Tile t;
  if (i < b.n_sink) {
    t.sink = true;
    t.own_lo = i * p.s_box;
    t.own_hi = imin(s, t.own_lo + p.s_box);
    t.k0 = t.own_lo;
    t.ncols = p.s_box;
  } else {
    t.sink = false;
    t.k0 = b.lo + (i - b.n_sink) * p.n_band;
    t.own_lo = t.k0;
    t.own_hi = imin(t.k0 + p.n_band, b.t_last + 1);
    t.ncols = imin(p.n_band, round_up(t.own_hi - t.own_lo, 16));
  }
  // Mask-free when all ncols keys are owned and, for every row t of the block
  // (t0 .. t0+Tq-1), inside [t - w + 1, t]: the in-band interior tiles.
  int t_hi = b.t0 + p.Tq - 1;
  bool owned_all = (t.own_hi - t.own_lo) == t.ncols;
  bool causal_ok = t.k0 + t.ncols - 1 <= b.t0;
  bool window_ok = t.k0 >= t_hi - w + 1;
  t.full = owned_all && causal_ok && window_ok && !t.sink;
  return t;
}

}  // namespace swa
