// prefill.cuh -- SWA(w, s) prefill on sm_103a: TMA + tcgen05 (TMEM) flash
// attention that visits only the key tiles inside each query block's window
// plus the sink tile.
//
// Method: explainer of arXiv 2608.28444, section "核心方法 / 1. 训练免费的
// SWA(w, s)" (x_t equation; swa_mask definition). Tile skipping: "Hybrid Sliding
// Window Attention" page, section "三、3. FlashAttention-2 / FlashAttention-3".
//
// Work item: one query block = Tq positions x G query heads of one
// (batch, KV head), packed as the M = 128 rows of the tile (row r <-> position
// t0 + r / G, head kvh * G + r % G). A persistent CTA walks its items
// (item = cta, cta + grid, ...); per item it visits the block's tile list
// (swa_index.cuh): sink tile(s) first, then the band tiles.
//
// Warp roles (384 threads, one CTA per SM):
//   warp 0      TMA producer: Q (double buffered) and a ring of K/V tiles, in the
//               MMA's consumption order
//   warp 1      TMEM owner and MMA issuer (one thread), in the order
//                 S_g = Q K_g^T      -> TMEM buffer g % 2      (fp32)
//                 O  += P_{g-1} V_{g-1}                        (fp32)
//               P_{g-1} is read from TMEM (it overwrites S_{g-1} in place), so
//               the tensor core computes S_g while the softmax warps still
//               work on tile g-1, and the softmax never waits for a P buffer.
//   warp 2      output store (TMA tensor store; plain stores for a block that
//               starts before row 0 of out)
//   warps 4-11  softmax + epilogue in two warpgroups; warps 4 + q and 8 + q own
//               TMEM lanes 32q .. 32q + 31 (tile rows) and split each tile's
//               columns: in-tile mask (edge chunks only), online softmax with
//               lazy rescaling, P (bf16) to TMEM, O rescale in TMEM when the
//               running max grows by more than 2^8, and at block end O / l -> bf16.
//
// Shared memory: Q 2 x (D/64) x 16 KB and a ring of K/V slots sized to the
// plan's largest tile. Every operand is stored as 64-column chunks of 128-byte
// rows with the 128-byte swizzle, which is what TMA writes and what the MMA
// descriptors describe.
//
// Tensor memory (512 columns): S/P buffer 0 at 0, S/P buffer 1 at 192, O at 384.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm100_ptx.cuh"
#include "swa_index.cuh"

namespace swa {

constexpr int kTileRows = 128;                // M of every MMA
constexpr int kChunkBytes = kTileRows * 128;  // one 64-column chunk of a 128-row tile
constexpr int kTmemCols = 512;
constexpr int kTmemS0 = 0;                    // S/P buffers at columns 0 and 192
constexpr int kTmemSStride = kMaxTileKeys;
constexpr int kTmemO = 2 * kMaxTileKeys;      // O at columns 384 .. 384 + d
constexpr int kPrefillThreads = 384;
constexpr int kSoftmaxWarp0 = 4;                // warps 4-11: two softmax warpgroups
constexpr int kMaxStages = 8;
constexpr float kRescaleThreshold = 8.0f;     // log2 units: rescale O when max grows > 2^8

// The order in which the three roles visit a block's tiles. The sink-last
// kernel visits them last to first: its last tile holds the sink box and the
// most recent keys, whose scores usually set a row's running maximum, so the
// older band tiles visited after it seldom raise that maximum past the
// lazy-rescale threshold. (Visited last, the sinks raised it in most warps,
// each of which then rescaled O right before the block's last P V.) The
// online softmax does not depend on the order.
template <bool kSinkLast>
__device__ __forceinline__ Tile tile_visit(const PrefillPlan &p, const BlockTiles &b, int i, int w,
                                           int s) {
  return tile_at<kSinkLast>(p, b, kSinkLast ? b.n_tiles - 1 - i : i, w, s);
}

struct PrefillArgs {
  __nv_bfloat16 *out;
  float *lse;         // [B, Hq, L] log-sum-exp of each row's scores (natural log), or null
  int B, L, Hq, Hkv, w, s;
  int qb_first;       // query blocks below it are not computed (pair kernel;
                      // the single-block kernel drops them through n_items)
  int q_off;          // K/V rows before row 0 of q and out: query row t of the
                      // key/value layout is row t - q_off of q and out, which
                      // hold L - q_off rows (0 for a whole prompt)
  float scale_log2;   // scale * log2(e)
  PrefillPlan plan;
  int n_items;
  int stages;         // K/V ring slots
  int kv_chunk;       // bytes of one 64-column chunk of a K/V slot
  int sep_stage;      // 1: the output is staged in a buffer of its own, so a Q
                      // buffer is free as soon as its block's last S is done;
                      // 0: the output is staged in the block's Q buffer
};

// Shared memory of one CTA.
template <int D>
struct PrefillSmem {
  static constexpr int kQBytes = (D / 64) * kChunkBytes;  // one Q tile
  static constexpr int kBarBytes = 256;
  // row-max exchange [parity][half][row], then row-sum exchange [half][row]
  static constexpr int kXchgBytes = (2 * 2 * 128 + 2 * 128) * 4;
  // keys held by one K/V slot: the widest tile of the plan
  static int chunk_bytes(const PrefillPlan &p) { return p.slot_keys * 128; }
  static int slot_bytes(const PrefillPlan &p) { return (D / 64) * chunk_bytes(p); }
  static size_t fixed_bytes(bool sep_stage) {
    return 1024 /* alignment slack */ + (sep_stage ? 3 : 2) * (size_t)kQBytes + kBarBytes +
           kXchgBytes;
  }
  static size_t bytes(const PrefillPlan &p, int stages, bool sep_stage) {
    return fixed_bytes(sep_stage) + (size_t)stages * slot_bytes(p);
  }
  static int stages(const PrefillPlan &p, int max_smem, bool sep_stage) {
    long long st = ((long long)max_smem - (long long)fixed_bytes(sep_stage)) / slot_bytes(p);
    return (int)(st > kMaxStages ? kMaxStages : st);
  }
  // A separate output buffer is used when the K/V ring still keeps enough
  // stages: two (the K and V of the one tile) when a block visits a single
  // tile, four otherwise.
  static bool use_sep_stage(const PrefillPlan &p, int max_smem) {
    return stages(p, max_smem, true) >= (p.steady_tiles == 1 ? 2 : 4);
  }
};

// Bit e set iff tile column c0 + e (0 <= e < 16) lies in [lo, hi).
__device__ __forceinline__ uint32_t range_bits16(int c0, int lo, int hi) {
  const int l = imin(imax(lo - c0, 0), 16);
  const int h = imin(imax(hi - c0, 0), 16);
  return ((1u << h) - 1u) & ~((1u << l) - 1u);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Online-softmax step for this thread's share of one S tile row. Two warps
// (one per softmax warpgroup) own the same 32 TMEM lanes and split the tile's
// 16-key chunks: this warp takes NC chunks starting at chunk c_first. Their
// partial row maxima are exchanged through shared memory, so both apply the
// same running max. The chunk count is a template parameter so the code is
// straight-line for each width: no chunk is skipped by predication.
//   s_row         TMEM address of the row's S values (column 0 of the tile);
//                 P (bf16, two per column) is written back over them
//   mask          0: every (row, key) pair of the tile is admitted; otherwise
//                 the row admits the tile columns [a_lo, a_hi) and
//                 [b_lo, b_hi) (either range may be empty)
//   my_max/partner_max  exchange slots of this row; bar_id: named barrier
//                 shared with the partner warp (64 threads)
//   m_used        running max (log2 units), identical in both warps
//   l_part        running sum over this warp's columns
//   factor        set to the O rescale factor (1: no rescale needed)
template <int NC>
__device__ __forceinline__ void softmax_part(uint32_t s_row, int c_first, int mask, int a_lo,
                                             int a_hi, int b_lo, int b_hi, float cl2,
                                             float *my_max, const float *partner_max,
                                             int bar_id, float &m_used, float &l_part,
                                             float &factor) {
  constexpr int kN = NC * 16 > 0 ? NC * 16 : 1;
  float x[kN];
#pragma unroll
  for (int c = 0; c < NC; ++c)
    tmem_ld16(s_row + (c_first + c) * 16, *reinterpret_cast<float(*)[16]>(&x[c * 16]));
  if (NC > 0) tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < NC; ++c) reg_fence16(*reinterpret_cast<float(*)[16]>(&x[c * 16]));
  if (mask != 0) {
    // A chunk is masked only when some row of the warp does not admit all of
    // its 16 keys (the decision is warp-uniform).
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int c0 = (c_first + c) * 16;
      const uint32_t bits = range_bits16(c0, a_lo, a_hi) | range_bits16(c0, b_lo, b_hi);
      if (__any_sync(0xffffffffu, bits != 0xFFFFu)) {
#pragma unroll
        for (int e = 0; e < 16; ++e) x[c * 16 + e] = (bits >> e) & 1u ? x[c * 16 + e] : -INFINITY;
      }
    }
  }
  // partial row max of the raw scores: eight independent chains, three-input
  // max (two keys per instruction)
  float m_part;
  if constexpr (NC == 0) {
    m_part = -INFINITY;
  } else {
    constexpr int kN = NC * 16;
    float mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = x[k];
    int e = 8;
#pragma unroll
    for (; e + 16 <= kN; e += 16)
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], x[e + k], x[e + 8 + k]);
#pragma unroll
    for (; e < kN; e += 8)
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], x[e + k]);
    m_part = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
  }
  *my_max = m_part;
  named_bar_sync(bar_id, 64);
  const float m_tile = fmaxf(m_part, *partner_max) * cl2;  // scale > 0: max commutes with it
  const float m_new = fmaxf(m_used, m_tile);
  factor = 1.f;
  if (m_used == -INFINITY) {
    m_used = m_new;  // nothing accumulated yet for this row
  } else if (m_new > m_used + kRescaleThreshold) {
    factor = fast_exp2(m_used - m_new);
    m_used = m_new;
    l_part *= factor;
  }
  const float msub = (m_used == -INFINITY) ? 0.f : m_used;
  // four chains of paired sums
  float sum[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) sum[k] = 0.f;
  // P = 2^(x * scale * log2 e - m) as bf16: 16 keys -> 8 packed columns; the
  // scale-and-shift runs two keys per instruction (fma.rn.f32x2)
#pragma unroll
  for (int c = 0; c < NC; ++c) {
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      float y0, y1;
      fma2_bc(y0, y1, x[c * 16 + e], x[c * 16 + e + 1], cl2, -msub);
      x[c * 16 + e] = fast_exp2(y0);
      x[c * 16 + e + 1] = fast_exp2(y1);
      const int k = (e >> 1) & 3;
      add2(sum[2 * k], sum[2 * k + 1], x[c * 16 + e], x[c * 16 + e + 1]);
    }
    const float *p = &x[c * 16];
    tmem_st8(s_row + (c_first + c) * 8, pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
             pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]), pack_bf16x2(p[8], p[9]),
             pack_bf16x2(p[10], p[11]), pack_bf16x2(p[12], p[13]), pack_bf16x2(p[14], p[15]));
  }
  add2(sum[0], sum[1], sum[2], sum[3]);
  add2(sum[4], sum[5], sum[6], sum[7]);
  add2(sum[0], sum[1], sum[4], sum[5]);
  l_part += sum[0] + sum[1];
}

// O (+)= P V for one tile of nk (1 .. kMaxTileKeys / 16) 16-key steps. The
// MMAs are guarded instead of branched over: the tensor core overlaps
// consecutive MMAs of a thread only when no branch separates their issue.
__device__ __forceinline__ void pv_group(int nk, uint32_t accumulate, uint32_t o_tmem,
                                         uint32_t p_tmem, uint64_t vd, uint32_t idesc) {
  umma_ts_if(o_tmem, p_tmem, vd, idesc, accumulate, 1u);
#pragma unroll
  for (int kk = 1; kk < kMaxTileKeys / 16; ++kk)
    umma_ts_if(o_tmem, p_tmem + kk * 8, vd + kk * 128, idesc, 1u, kk < nk ? 1u : 0u);
}

// kSinkLast: the plan may carry the sink box in a block's last band tile
// (plan.sink_last); the other instantiation compiles that case out.
template <int D, bool kSinkLast>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    swa_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_ks,
                       const __grid_constant__ CUtensorMap tm_vs,
                       const __grid_constant__ CUtensorMap tm_kb,
                       const __grid_constant__ CUtensorMap tm_vb,
                       const __grid_constant__ CUtensorMap tm_o, const PrefillArgs a) {
  constexpr int kQBytes = PrefillSmem<D>::kQBytes;
  constexpr int kChunks = D / 64;
  constexpr int kSteps = D / 16;  // K steps of the S = Q K^T product

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int stages = a.stages;
  const int kv_chunk = a.kv_chunk;
  const int slot_bytes = kChunks * kv_chunk;
  uint8_t *sQ = smem;                               // 2 x kQBytes
  uint8_t *sStage = a.sep_stage ? sQ + 2 * kQBytes : nullptr;  // kQBytes (optional)
  uint8_t *sKV = sQ + (a.sep_stage ? 3 : 2) * kQBytes;        // stages x slot_bytes
  uint64_t *bars = reinterpret_cast<uint64_t *>(sKV + (size_t)stages * slot_bytes);
  uint64_t *q_full = bars + 0;      // [2]
  uint64_t *q_empty = bars + 2;     // [2]
  uint64_t *s_full = bars + 4;      // [2]
  uint64_t *p_full = bars + 6;      // [1]
  uint64_t *pv_done = bars + 7;     // [1]
  uint64_t *o_full = bars + 8;      // [1]
  uint64_t *mma_done = bars + 9;    // [1]
  uint64_t *kv_full = bars + 10;    // [stages <= 8]
  uint64_t *kv_empty = bars + 18;   // [stages <= 8]
  uint64_t *epi_staged = bars + 26; // [1] output tile staged in shared memory
  uint64_t *stage_free = bars + 29; // [1] separate staging buffer read by TMA
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 27);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 28);
  float *xchg = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) +
                                          PrefillSmem<D>::kBarBytes);  // [2][2][128] + [2][128]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const PrefillPlan &plan = a.plan;

  if (threadIdx.x == 0) {
    mbar_init(&q_full[0], 1);
    mbar_init(&q_full[1], 1);
    mbar_init(&q_empty[0], 1);
    mbar_init(&q_empty[1], 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 8);
    mbar_init(pv_done, 1);
    mbar_init(o_full, 1);
    mbar_init(mma_done, 1);
    mbar_init(epi_staged, 8);
    mbar_init(stage_free, 1);
    for (int i = 0; i < stages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (plan.rows < kTileRows) {
    // Rows past Tq * G are never written by TMA: keep them zero in both Q
    // buffers so their (unused) scores stay finite.
    for (int i = threadIdx.x; i < 2 * kQBytes / 16; i += blockDim.x)
      reinterpret_cast<uint4 *>(sQ)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above touched only this CTA's own resources; global memory is
  // read and written only after the kernels this one depends on are done.
  grid_launch_dependents();
  grid_dependency_wait();

  const int BH = a.B * a.Hkv;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (plan.n_sink) {
        tma_prefetch_desc(&tm_ks);
        tma_prefetch_desc(&tm_vs);
      }
      if (kSinkLast) {
        tma_prefetch_desc(&tm_kb);
        tma_prefetch_desc(&tm_vb);
      }
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t u = 0;        // K/V loads issued (two per tile)
      int slot = 0;          // ring slot of load u
      uint32_t phase = 0;    // (u / stages) & 1
      int q_issued = 0;      // Q loads issued (one per item)
      int it = 0;
      bool ok = true;
      // The ring is filled in the order the MMA warp consumes it: K of tile g,
      // then V of tile g - 1 (S_g is issued before P V_{g-1}, across blocks
      // too), and the last V at the end. K_g then reuses the slot of a V that
      // was consumed two tiles earlier, so its load is in flight long before
      // S_g needs it. Q of a block follows the K of its first tile; every load
      // before it is consumed by an MMA that does not need that Q.
      Tile prev{};
      int prev_b = 0, prev_kvh = 0;
      bool have_prev = false, done = false;
      ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, plan.nqb);
      int i = 0, b = 0, kvh = 0;
      BlockTiles bt{};
      if (wk.valid()) {
        b = wk.bh() / a.Hkv;
        kvh = wk.bh() % a.Hkv;
        bt = block_tiles<kSinkLast>(plan, wk.qb(), a.L, a.w, a.s);
      } else {
        done = true;
      }
      while (ok && (!done || have_prev)) {
        Tile tl{};
        if (!done) tl = tile_visit<kSinkLast>(plan, bt, i, a.w, a.s);
        for (int half = 0; half < 2; ++half) {  // 0: K of this tile, 1: V of the previous one
          if (half == 0 && done) continue;
          if (half == 1 && !have_prev) continue;
          const Tile &t = half == 0 ? tl : prev;
          const int tb = half == 0 ? b : prev_b, th = half == 0 ? kvh : prev_kvh;
          // slot rows [0, n_sink_cols): the sink box; then the band box, which
          // is s_box rows shorter in a last band tile that carries the sinks
          // (with sink_last the only band tiles with sink columns)
          const bool band = t.ncols > t.n_sink_cols;
          const bool short_band = kSinkLast && band && t.n_sink_cols > 0;
          const int band_rows = short_band ? plan.n_band - plan.s_box : plan.n_band;
          const uint32_t tile_bytes =
              (uint32_t)(kChunks * 128 * (t.n_sink_cols + (band ? band_rows : 0)));
          if (!mbar_wait(&kv_empty[slot], phase ^ 1, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&kv_full[slot], tile_bytes);
          uint8_t *dst = sKV + slot * slot_bytes;
          for (int c = 0; c < kChunks; ++c) {
            if (t.n_sink_cols)
              tma_load_4d(dst + c * kv_chunk, half == 0 ? &tm_ks : &tm_vs, &kv_full[slot],
                          c * 64, th, t.sink_key0, tb, pol_kv);
            if (band)
              tma_load_4d(dst + c * kv_chunk + t.n_sink_cols * 128,
                          short_band ? (half == 0 ? &tm_kb : &tm_vb)
                                     : (half == 0 ? &tm_k : &tm_v),
                          &kv_full[slot], c * 64, th, t.k0, tb, pol_kv);
          }
          ++u;
          if (++slot == stages) { slot = 0; phase ^= 1; }
          if (half == 0 && i == 0) {
            const int qbuf = it & 1;
            if (!mbar_wait(&q_empty[qbuf], ((it >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(&q_full[qbuf], (uint32_t)(kChunks * 64 * plan.rows * 2));
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(sQ + qbuf * kQBytes + c * kChunkBytes, &tm_q, &q_full[qbuf], c * 64,
                          kvh * plan.G, bt.t0 - a.q_off, b, pol_q);
            ++q_issued;
          }
        }
        if (!ok) break;
        have_prev = !done;
        if (done) break;
        prev = tl;
        prev_b = b;
        prev_kvh = kvh;
        if (++i == bt.n_tiles) {
          i = 0;
          ++it;
          wk.next();
          if (wk.valid()) {
            b = wk.bh() / a.Hkv;
            kvh = wk.bh() % a.Hkv;
            bt = block_tiles<kSinkLast>(plan, wk.qb(), a.L, a.w, a.s);
          } else {
            done = true;
          }
        }
      }
      if (!ok) {
        // Let the loads that may still be in flight land before the CTA can
        // exit: a slot (or Q buffer) is only refilled after its previous load
        // was consumed, so only the last `stages` K/V loads and the last two Q
        // loads can be outstanding.
        const uint32_t first = u > (uint32_t)stages ? u - stages : 0;
        for (uint32_t v = first; v < u; ++v)
          mbar_wait(&kv_full[v % stages], (v / stages) & 1, abort_flag, 200000000ull, false);
        for (int j = q_issued > 2 ? q_issued - 2 : 0; j < q_issued; ++j)
          mbar_wait(&q_full[j & 1], (j >> 1) & 1, abort_flag, 200000000ull, false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the control flow, so descriptors and counters stay
    // warp-uniform; lane 0 issues each tile's MMAs as one straight-line group
    // (the tensor core overlaps consecutive MMAs of a thread only when no
    // branch separates them) followed by its commits. The descriptors are
    // built once and advanced by adding 16-byte address units, and ring
    // slots/phases are tracked with counters (no division).
    const bool leader = lane == 0;
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      const bool r = mbar_wait(bar, parity, abort_flag);
      return __all_sync(0xffffffffu, r);
    };
    const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
    const uint64_t qd0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t kd0 = sdesc_sw128(smem_u32(sKV), 16, 1024);
    const uint64_t vd0 = sdesc_sw128(smem_u32(sKV), (uint32_t)kv_chunk, 1024);
    const uint32_t slot_step = (uint32_t)slot_bytes >> 4;
    const uint32_t kvc16 = (uint32_t)kv_chunk >> 4;
    // ring slot / phase of the next load consumed: the ring holds K_g, V_{g-1},
    // K_{g+1}, V_g, ... in the order of the MMAs below
    uint32_t cs = 0, cph = 0;
    auto consume = [&]() {
      if (++cs == (uint32_t)stages) { cs = 0; cph ^= 1; }
    };
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    // the tile whose S has been issued but whose P V is still pending
    bool pend = false;
    uint32_t pend_g = 0;
    int pend_ncols = 0;
    bool pend_first = false, pend_last = false;

    auto issue_pv = [&]() -> bool {
      if (!warp_wait(p_full, pend_g & 1)) return false;
      if (!warp_wait(&kv_full[cs], cph)) return false;
      tc_fence_after();
      // A = P (TMEM, 8 columns per 16 keys), B = V (MN-major: d contiguous)
      const uint32_t p_tmem = tmem_base + kTmemS0 + (pend_g & 1) * kTmemSStride;
      const uint64_t vd = vd0 + cs * slot_step;
      const uint32_t o_tmem = tmem_base + kTmemO;
      if (leader) {
        pv_group(pend_ncols >> 4, pend_first ? 0u : 1u, o_tmem, p_tmem, vd, idesc_pv);
        umma_commit(&kv_empty[cs]);
        umma_commit(pv_done);
        if (pend_last) umma_commit(o_full);
      }
      __syncwarp();
      consume();
      return true;
    };

    for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, plan.nqb); ok && wk.valid();
         wk.next(), ++it) {
      const BlockTiles bt = block_tiles<kSinkLast>(plan, wk.qb(), a.L, a.w, a.s);
      const int qbuf = it & 1;
      const uint64_t qd = qd0 + (uint32_t)qbuf * (uint32_t)(kQBytes >> 4);
      if (!warp_wait(&q_full[qbuf], (it >> 1) & 1)) { ok = false; break; }
      for (int i = 0; i < bt.n_tiles; ++i, ++g) {
        const Tile tl = tile_visit<kSinkLast>(plan, bt, i, a.w, a.s);
        if (!warp_wait(&kv_full[cs], cph)) { ok = false; break; }
        tc_fence_after();
        // S_g is issued before P V_{g-1} (which needs the softmax of tile g - 1),
        // also across blocks, so the tensor core computes S_g while the
        // softmax warps still work on tile g - 1. S_g overwrites buffer g % 2,
        // whose P_{g-2} feeds P V_{g-2}: that MMA was issued before this one
        // and tcgen05 MMAs of one thread execute in issue order.
        const uint32_t idesc_s = idesc_bf16_f32(128, tl.ncols, false);
        const uint32_t s_tmem = tmem_base + kTmemS0 + (g & 1) * kTmemSStride;
        const uint64_t kd = kd0 + cs * slot_step;
        if (leader) {
          umma_ss<0>(s_tmem, qd, kd, idesc_s);
#pragma unroll
          for (int kk = 1; kk < kSteps; ++kk) {
            const uint32_t qoff = (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2;
            const uint32_t koff = (kk >> 2) * kvc16 + (kk & 3) * 2;
            umma_ss<1>(s_tmem, qd + qoff, kd + koff, idesc_s);
          }
          umma_commit(&kv_empty[cs]);
          umma_commit(&s_full[g & 1]);
          if (a.sep_stage && i == bt.n_tiles - 1) umma_commit(&q_empty[qbuf]);
        }
        __syncwarp();
        consume();
        if (pend && !issue_pv()) { ok = false; break; }
        pend = true;
        pend_g = g;
        pend_ncols = tl.ncols;
        pend_first = (i == 0);
        pend_last = (i == bt.n_tiles - 1);
      }
    }
    if (ok && pend) issue_pv();
    // drain: every MMA issued by lane 0 completes before TMEM is freed
    if (leader) {
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, abort_flag, 200000000ull, false);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ output store
    // The softmax warps stage each finished block, bf16, in the Q buffer it
    // was computed from (same swizzled layout as the Q tile). Lane 0 stores it
    // with TMA and then frees the buffer for the next Q load. A block that
    // starts before row 0 of out (q_off > 0: its first rows are K/V rows that
    // have no query) is copied by the whole warp with plain stores instead,
    // row by row from row 0 of out on, since a TMA store may not start at a
    // negative coordinate.
    if (lane == 0) tma_prefetch_desc(&tm_o);
    const int out_rows = a.L - a.q_off;
    int it = 0;
    for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, plan.nqb); wk.valid();
         wk.next(), ++it) {
      const int qb = wk.qb();
      const int b = wk.bh() / a.Hkv, kvh = wk.bh() % a.Hkv;
      const int qbuf = it & 1;
      int staged = 1;
      if (lane == 0) staged = mbar_wait(epi_staged, it & 1, abort_flag) ? 1 : 0;
      staged = __shfl_sync(0xffffffffu, staged, 0);
      __syncwarp();
      if (!staged) break;
      const uint8_t *src = a.sep_stage ? sStage : sQ + qbuf * kQBytes;
      const int row0 = qb * plan.Tq - a.q_off;  // out row of the block's first position
      if (row0 >= 0) {
        if (lane == 0) {
          for (int c = 0; c < kChunks; ++c)
            tma_store_4d(&tm_o, src + c * kChunkBytes, c * 64, kvh * plan.G, row0, b);
          tma_store_commit();
          tma_store_wait_read();
        }
      } else {
        for (int i = lane; i < plan.rows * (D / 8); i += 32) {
          const int r = i / (D / 8), u = i % (D / 8);  // tile row, 16-byte unit
          const int orow = row0 + r / plan.G;
          if (orow < 0 || orow >= out_rows) continue;
          const int ch = u / 8, unit = u % 8;
          const uint4 val = *reinterpret_cast<const uint4 *>(src + ch * kChunkBytes + r * 128 +
                                                             ((unit ^ (r & 7)) << 4));
          *reinterpret_cast<uint4 *>(
              a.out + (((size_t)b * out_rows + orow) * a.Hq + kvh * plan.G + r % plan.G) * D +
              ch * 64 + unit * 8) = val;
        }
        // the buffer is next written by TMA (a Q load) or by the softmax warps
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(a.sep_stage ? stage_free : &q_empty[qbuf]);
    }
    if (lane == 0) tma_store_wait_all();
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------ softmax + epilogue
    // Warps 4-7 and 8-11 form two warpgroups. Warp 4 + q and warp 8 + q both
    // own TMEM lanes 32q .. 32q + 31 (tile rows) and split each tile's
    // columns: the first warpgroup takes the first ceil(nch / 2) chunks.
    const int sub = (warp - kSoftmaxWarp0) & 3;   // TMEM lane quarter
    const int half = (warp - kSoftmaxWarp0) >> 2; // column half
    const int r = sub * 32 + lane;                // tile row owned by this thread
    const int bar_id = 1 + sub;                   // named barrier of the warp pair
    const uint32_t lane_addr = tmem_base + ((uint32_t)(sub * 32) << 16);
    const float cl2 = a.scale_log2;
    // every lane polls; the outcome is made warp-uniform so a timeout on one
    // lane cannot leave the warp diverged before a .sync.aligned instruction
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      const bool r = mbar_wait(bar, parity, abort_flag);
      return __all_sync(0xffffffffu, r);
    };
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    const int row_pos = r / plan.G;      // position of this row within a block
    for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, plan.nqb); ok && wk.valid();
         wk.next(), ++it) {
      const BlockTiles bt = block_tiles<kSinkLast>(plan, wk.qb(), a.L, a.w, a.s);
      const int t = bt.t0 + row_pos;     // query position of this row
      float m_used = -INFINITY;          // running max (scaled, log2 units)
      float l_part = 0.f;                // sum over this warp's columns
      for (int i = 0; i < bt.n_tiles; ++i, ++g) {
        const Tile tl = tile_visit<kSinkLast>(plan, bt, i, a.w, a.s);
        if (!warp_wait(&s_full[g & 1], (g >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t s_row = lane_addr + kTmemS0 + (g & 1) * kTmemSStride;
        int mask = 0;
        ColRanges cr{0, 0, 0, 0};
        if (!tl.full) {
          mask = 1;
          cr = tile_ranges(tl, t, a.w, a.s);
        }
        const int nch = tl.ncols >> 4;
        const int n0 = (nch + 1) >> 1;   // chunks of the first warpgroup
        const int c_first = half ? n0 : 0;
        const int my_n = half ? nch - n0 : n0;
        float *xc = xchg + (g & 1) * 256;
        float *my_max = xc + half * 128 + r;
        const float *partner_max = xc + (half ^ 1) * 128 + r;
        float factor;
#define SWA_SOFTMAX_PART(N)                                                                  \
  softmax_part<N>(s_row, c_first, mask, cr.a_lo, cr.a_hi, cr.b_lo, cr.b_hi, cl2, my_max,      \
                  partner_max, bar_id, m_used, l_part, factor)
        switch (my_n) {
          case 0: SWA_SOFTMAX_PART(0); break;
          case 1: SWA_SOFTMAX_PART(1); break;
          case 2: SWA_SOFTMAX_PART(2); break;
          case 3: SWA_SOFTMAX_PART(3); break;
          case 4: SWA_SOFTMAX_PART(4); break;
          case 5: SWA_SOFTMAX_PART(5); break;
          default: SWA_SOFTMAX_PART(6); break;
        }
#undef SWA_SOFTMAX_PART
        tmem_wait_st();
        // P V of the previous tile must be complete before O is rescaled (and
        // it is waited for on every tile so the barrier's phases stay in step).
        if (g > 0 && !warp_wait(pv_done, (g - 1) & 1)) { ok = false; break; }
        if (__any_sync(0xffffffffu, factor != 1.f)) {
          // each warp of the pair rescales its half of O's columns
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[16];
            const uint32_t oa = lane_addr + kTmemO + half * (D / 2) + c * 16;
            tmem_ld16(oa, o);
            tmem_wait_ld();
            reg_fence16(o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= factor;
            tmem_st16(oa, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);  // one arrival per softmax warp
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      // O / l -> bf16 into the Q buffer of this block (free: every MMA that
      // read it completed before O did), in the swizzled layout of the output
      // tensor map; the store warp writes it out with TMA. Each warp of the
      // pair converts half of the columns.
      // (own slots: the partner reads them before it passes the next tile's
      // barrier, and this warp writes them again only after that)
      float *xl = xchg + 512;
      xl[half * 128 + r] = l_part;
      named_bar_sync(bar_id, 64);
      const float l_sum = l_part + xl[(half ^ 1) * 128 + r];
      if (a.lse != nullptr && half == 0 && r < plan.rows && t < a.L) {
        // m_used is in log2 units of the scaled scores
        const int hq = (wk.bh() % a.Hkv) * plan.G + r % plan.G;
        a.lse[((size_t)(wk.bh() / a.Hkv) * a.Hq + hq) * a.L + t] =
            (m_used + log2f(l_sum)) * 0.6931471805599453f;
      }
      if (!warp_wait(o_full, it & 1)) { ok = false; break; }
      // a separate staging buffer is free once the previous block's store read it
      if (a.sep_stage && !warp_wait(stage_free, (it & 1) ^ 1)) { ok = false; break; }
      tc_fence_after();
      const float inv_l = 1.0f / l_sum;
      const uint32_t stage_row =
          smem_u32(a.sep_stage ? sStage : sQ + (it & 1) * kQBytes) + r * 128;
      float o[D / 2];
#pragma unroll
      for (int j = 0; j < D / 32; ++j)
        tmem_ld16(lane_addr + kTmemO + half * (D / 2) + j * 16,
                  *reinterpret_cast<float(*)[16]>(&o[j * 16]));
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < D / 32; ++j) reg_fence16(*reinterpret_cast<float(*)[16]>(&o[j * 16]));
      if (r < plan.rows) {
#pragma unroll
        for (int u = 0; u < D / 16; ++u) {  // 16-byte unit: 8 columns
          const int col = half * (D / 2) + u * 8;
          const int ch = col / 64, unit = (col % 64) / 8;
          const float *v = &o[u * 8];
          st_shared_v4(stage_row + ch * kChunkBytes + ((unit ^ (r & 7)) << 4),
                       pack_bf16x2(v[0] * inv_l, v[1] * inv_l),
                       pack_bf16x2(v[2] * inv_l, v[3] * inv_l),
                       pack_bf16x2(v[4] * inv_l, v[5] * inv_l),
                       pack_bf16x2(v[6] * inv_l, v[7] * inv_l));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_staged);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace swa
