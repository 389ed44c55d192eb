// prefill_pair.cuh -- SWA(w, s) prefill on sm_103a, two query blocks per work
// item: TMA + tcgen05 (TMEM) flash attention whose two 128-row query tiles
// share every key/value tile.
//
// Method: explainer of arXiv 2608.28444, section "核心方法 / 1. 训练免费的
// SWA(w, s)" (x_t equation; swa_mask definition). Tile skipping: "Hybrid Sliding
// Window Attention" page, section "三、3. FlashAttention-2 / FlashAttention-3".
//
// Work item: the query blocks qb (tile A) and qb + 1 (tile B) of one
// (batch, KV head), each packed as in prefill.cuh (Tq positions x G heads =
// 128 rows). Their key ranges differ only by Tq keys at either end, so the
// item visits one list of key tiles covering both (swa_index.cuh with
// bpi = 2) and every K/V tile loaded feeds four MMAs instead of two.
//
// Warp roles (384 threads, one CTA per SM):
//   warp 0      TMA producer: Q_A and Q_B (one buffer each), then a ring of
//               K/V tiles in the order K_0, V_0, K_1, V_1, ...
//   warp 1      TMEM owner and MMA issuer (one thread), per item
//                 S_A0 S_B0 | PV_A0 S_A1 | PV_B0 S_B1 | PV_A1 S_A2 | ...
//               S_X(j) lands in tile X's S columns; P_X(j) overwrites it in
//               place and feeds O_X += P_X(j) V_j; S_X(j + 1) is issued after
//               that MMA (tcgen05 MMAs of one thread run in issue order).
//               While warpgroup A computes the softmax of tile j, the tensor
//               core runs P_B(j-1) V_{j-1} and S_B(j), and the other way round.
//   warp 2      output store: TMA store of each finished tile (plain stores
//               for a tile that starts before row 0 of out)
//   warps 4-7   softmax + epilogue of tile A, warps 8-11 of tile B: one thread
//               per tile row (TMEM lane), whole rows (no partner exchange).
//
// Shared memory: Q_A, Q_B and an output staging tile, (D/64) x 16 KB each, and
// a ring of K/V slots of the plan's widest tile. Tensor memory (512 columns):
// S_A at 0, S_B at 128, O_A at 256, O_B at 256 + D.
//
// Registers: the launch gives every thread 168 (384 x 168 = 64,512); the
// first warpgroup (producer, MMA, store) then gives back down to 80 and the two
// softmax warpgroups take 208 each, which holds a whole 128-column S row:
// 128 x 80 + 256 x 208 = 64,512. Code after a register re-split calls no
// out-of-line function (the bounded waits here are the inlined variant).
//
// Measured on B300 this kernel is 25-40% slower than the single-block kernel
// (prefill.cuh) at windows 64 to 2048: the lone MMA thread shares its SM
// partition with two softmax warps, and the N = 128 S MMAs read 8 KB of
// shared memory each, so the tensor pipe stays about 25% busy. The library
// runs it only when it is selected (swa_prefill_select).
#pragma once

#include "prefill.cuh"

namespace swa {

constexpr int kPairThreads = 384;
constexpr int kPairRegsLaunch = 168;  // 65536 / 384, rounded down to a multiple of 8
constexpr int kPairRegsLow = 80;      // warps 0-3
constexpr int kPairRegsHigh = 208;    // warps 4-11
static_assert(128 * kPairRegsLow + 256 * kPairRegsHigh <= kPairThreads * kPairRegsLaunch,
              "register shares exceed the launch allocation");

template <int D>
struct PairSmem {
  static constexpr int kTileKeys = 128;                   // widest key tile (MMA N)
  static constexpr int kQBytes = (D / 64) * kChunkBytes;  // one 128-row tile of D columns
  static constexpr int kBarBytes = 512;   // 32 mbarriers / words (see the kernel)
  static int chunk_bytes(const PrefillPlan &p) { return p.slot_keys * 128; }
  static int slot_bytes(const PrefillPlan &p) { return (D / 64) * chunk_bytes(p); }
  static size_t fixed_bytes() {
    return 1024 /* alignment slack */ + 3 * (size_t)kQBytes + kBarBytes;
  }
  static size_t bytes(const PrefillPlan &p, int stages) {
    return fixed_bytes() + (size_t)stages * slot_bytes(p);
  }
  static int stages(const PrefillPlan &p, int max_smem) {
    long long st = ((long long)max_smem - (long long)fixed_bytes()) / slot_bytes(p);
    return (int)(st > kMaxStages ? kMaxStages : st);
  }
};

// Online-softmax step over one whole S tile row of NC 16-key chunks (the
// thread owns the row: no exchange with another warp).
//   s_row   TMEM address of the row's S values; P (bf16, two per column) is
//           written back over them
//   mask    0: every column is admitted; otherwise the row admits the tile
//           columns [a_lo, a_hi) and [b_lo, b_hi) (either may be empty)
//   m_used  running max (log2 units of the scaled scores); l_sum running sum
//   factor  set to the O rescale factor (1: no rescale needed)
template <int NC>
__device__ __forceinline__ void softmax_row(uint32_t s_row, int mask, int a_lo, int a_hi,
                                            int b_lo, int b_hi, float cl2, float &m_used,
                                            float &l_sum, float &factor) {
  float x[NC * 16];
#pragma unroll
  for (int c = 0; c < NC; ++c)
    tmem_ld16(s_row + c * 16, *reinterpret_cast<float(*)[16]>(&x[c * 16]));
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < NC; ++c) reg_fence16(*reinterpret_cast<float(*)[16]>(&x[c * 16]));
  if (mask != 0) {
    // A 16-key chunk is masked only when some row of the warp does not admit
    // all of its keys (the decision is warp-uniform).
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int c0 = c * 16;
      const uint32_t bits = range_bits16(c0, a_lo, a_hi) | range_bits16(c0, b_lo, b_hi);
      if (__any_sync(0xffffffffu, bits != 0xFFFFu)) {
#pragma unroll
        for (int e = 0; e < 16; ++e) x[c * 16 + e] = (bits >> e) & 1u ? x[c * 16 + e] : -INFINITY;
      }
    }
  }
  constexpr int kChains = 8;
  float mx[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) mx[k] = x[k];
#pragma unroll
  for (int e = kChains; e < NC * 16; ++e) mx[e % kChains] = fmaxf(mx[e % kChains], x[e]);
#pragma unroll
  for (int k = 1; k < kChains; ++k) mx[0] = fmaxf(mx[0], mx[k]);
  const float m_tile = mx[0] * cl2;  // scale > 0: max commutes with it
  const float m_new = fmaxf(m_used, m_tile);
  factor = 1.f;
  if (m_used == -INFINITY) {
    m_used = m_new;  // nothing accumulated yet for this row
  } else if (m_new > m_used + kRescaleThreshold) {
    factor = fast_exp2(m_used - m_new);
    m_used = m_new;
    l_sum *= factor;
  }
  const float msub = (m_used == -INFINITY) ? 0.f : m_used;
  float sum[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) sum[k] = 0.f;
  // P = 2^(x * scale * log2 e - m) as bf16: 16 keys -> 8 packed columns
#pragma unroll
  for (int c = 0; c < NC; ++c) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      x[c * 16 + e] = fast_exp2(fmaf(x[c * 16 + e], cl2, -msub));
      sum[e % kChains] += x[c * 16 + e];
    }
    const float *p = &x[c * 16];
    tmem_st8(s_row + c * 8, pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
             pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]), pack_bf16x2(p[8], p[9]),
             pack_bf16x2(p[10], p[11]), pack_bf16x2(p[12], p[13]), pack_bf16x2(p[14], p[15]));
  }
#pragma unroll
  for (int k = 1; k < kChains; ++k) sum[0] += sum[k];
  l_sum += sum[0];
}

// O (+)= P V for one tile of nk (1 .. kSteps) 16-key steps, guarded rather
// than branched so the group issues back to back.
template <int kSteps>
__device__ __forceinline__ void pv_steps(int nk, uint32_t accumulate, uint32_t o_tmem,
                                         uint32_t p_tmem, uint64_t vd, uint32_t idesc) {
  umma_ts_if(o_tmem, p_tmem, vd, idesc, accumulate, 1u);
#pragma unroll
  for (int kk = 1; kk < kSteps; ++kk)
    umma_ts_if(o_tmem, p_tmem + kk * 8, vd + kk * 128, idesc, 1u, kk < nk ? 1u : 0u);
}

template <int D>
__global__ void __launch_bounds__(kPairThreads, 1)
    swa_prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_ks,
                            const __grid_constant__ CUtensorMap tm_vs,
                            const __grid_constant__ CUtensorMap tm_o, const PrefillArgs a) {
  using Smem = PairSmem<D>;
  constexpr int kQBytes = Smem::kQBytes;
  constexpr int kN = Smem::kTileKeys;
  constexpr int kChunks = D / 64;
  constexpr int kSteps = D / 16;      // K steps of S = Q K^T
  constexpr int kPvSteps = kN / 16;   // K steps of O += P V for the widest tile
  constexpr int kTmemO0 = 2 * kN;     // O_A; O_B at kTmemO0 + D

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int stages = a.stages;
  const int kv_chunk = a.kv_chunk;
  const int slot_bytes = kChunks * kv_chunk;
  uint8_t *sQ = smem;                      // Q_A, Q_B
  uint8_t *sStage = sQ + 2 * kQBytes;      // output staging tile
  uint8_t *sKV = sStage + kQBytes;         // stages x slot_bytes
  uint64_t *bars = reinterpret_cast<uint64_t *>(sKV + (size_t)stages * slot_bytes);
  uint64_t *q_full = bars + 0;       // [2] (A, B)
  uint64_t *q_empty = bars + 2;      // [2]
  uint64_t *s_full = bars + 4;       // [2]
  uint64_t *p_full = bars + 6;       // [2], 4 arrivals (the tile's softmax warps)
  uint64_t *o_full = bars + 8;       // [2]
  uint64_t *mma_done = bars + 10;    // [1]
  uint64_t *epi_staged = bars + 11;  // [1], 4 arrivals
  // [2]: stage_free[h] completes when the store of the other tile's last
  // staging has read the buffer, so warpgroup h waits for every one of its
  // phases in turn (a waiter that skipped phases could mistake an old phase
  // for the one it wants)
  uint64_t *stage_free = bars + 12;
  uint64_t *kv_full = bars + 14;     // [stages <= 8]
  uint64_t *kv_empty = bars + 22;    // [stages <= 8]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 30);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 31);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const PrefillPlan &plan = a.plan;

  if (threadIdx.x == 0) {
    for (int h = 0; h < 2; ++h) {
      mbar_init(&q_full[h], 1);
      mbar_init(&q_empty[h], 1);
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], 4);
      mbar_init(&o_full[h], 1);
    }
    mbar_init(mma_done, 1);
    mbar_init(epi_staged, 4);
    mbar_init(&stage_free[0], 1);
    mbar_init(&stage_free[1], 1);
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
  // pair index p (items run from the last pair down) -> first block of the pair
  const int npairs = cdiv(plan.nqb - a.qb_first, 2);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<kPairRegsLow>();
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (plan.n_sink) {
        tma_prefetch_desc(&tm_ks);
        tma_prefetch_desc(&tm_vs);
      }
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t u = 0;        // K/V loads issued
      int slot = 0;          // ring slot of load u
      uint32_t phase = 0;    // (u / stages) & 1
      int it = 0;
      int q_issued[2] = {0, 0};  // Q loads issued into each buffer
      bool ok = true;
      for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, npairs); ok && wk.valid();
           wk.next(), ++it) {
        const int b = wk.bh() / a.Hkv, kvh = wk.bh() % a.Hkv;
        const int qb = a.qb_first + 2 * wk.qb();
        const BlockTiles bt = block_tiles<false>(plan, qb, a.L, a.w, a.s);
        for (int i = 0; ok && i < bt.n_tiles; ++i) {
          const Tile t = tile_at<false>(plan, bt, i, a.w, a.s);
          const bool band = t.ncols > t.n_sink_cols;
          const uint32_t tile_bytes =
              (uint32_t)(kChunks * 128 * (t.n_sink_cols + (band ? plan.n_band : 0)));
          for (int kv = 0; kv < 2; ++kv) {  // K of tile i, then its V
            if (!mbar_wait_inl(&kv_empty[slot], phase ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(&kv_full[slot], tile_bytes);
            uint8_t *dst = sKV + slot * slot_bytes;
            for (int c = 0; c < kChunks; ++c) {
              if (t.n_sink_cols)
                tma_load_4d(dst + c * kv_chunk, kv == 0 ? &tm_ks : &tm_vs, &kv_full[slot],
                            c * 64, kvh, t.sink_key0, b, pol_kv);
              if (band)
                tma_load_4d(dst + c * kv_chunk + t.n_sink_cols * 128, kv == 0 ? &tm_k : &tm_v,
                            &kv_full[slot], c * 64, kvh, t.k0, b, pol_kv);
            }
            ++u;
            if (++slot == stages) { slot = 0; phase ^= 1; }
            if (i == 0 && kv == 0) {
              // the item's queries follow its first K tile
              for (int h = 0; h < 2; ++h) {
                if (!mbar_wait_inl(&q_empty[h], (it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(&q_full[h], (uint32_t)(kChunks * 64 * plan.rows * 2));
                for (int c = 0; c < kChunks; ++c)
                  tma_load_4d(sQ + h * kQBytes + c * kChunkBytes, &tm_q, &q_full[h], c * 64,
                              kvh * plan.G, (qb + h) * plan.Tq - a.q_off, b, pol_q);
                ++q_issued[h];
              }
              if (!ok) break;
            }
          }
        }
      }
      if (!ok) {
        // Let the loads that may still be in flight land before the CTA can
        // exit: a slot is only refilled after its previous load was consumed,
        // so only the last `stages` K/V loads can be outstanding, and each Q
        // buffer holds at most one load.
        const uint32_t first = u > (uint32_t)stages ? u - stages : 0;
        for (uint32_t v = first; v < u; ++v)
          mbar_wait_inl(&kv_full[v % stages], (v / stages) & 1, abort_flag, 200000000ull, false);
        for (int h = 0; h < 2; ++h)
          if (q_issued[h] > 0)
            mbar_wait_inl(&q_full[h], (q_issued[h] - 1) & 1, abort_flag, 200000000ull, false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 alone runs this loop (waits, MMAs and commits): no warp-wide
    // vote or reconvergence sits between the MMA groups.
    setmaxnreg_dec<kPairRegsLow>();
    if (lane == 0) {
      const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      const uint64_t qd0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t kd0 = sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t vd0 = sdesc_sw128(smem_u32(sKV), (uint32_t)kv_chunk, 1024);
      const uint32_t slot_step = (uint32_t)slot_bytes >> 4;
      const uint32_t kvc16 = (uint32_t)kv_chunk >> 4;
      // ring position of the next K/V load consumed in order (K_0 V_0 K_1 ...)
      uint32_t ks = 0, kph = 0;   // slot and phase of the item's next K
      uint32_t gt = 0;            // tiles issued for each query tile (the same for A and B)
      int it = 0;
      bool ok = true;
      auto advance = [&](uint32_t &slot, uint32_t &ph, uint32_t by) {
        slot += by;
        while (slot >= (uint32_t)stages) { slot -= (uint32_t)stages; ph ^= 1u; }
      };
      // S_h = Q_h K^T for a tile of ncols keys whose K sits in ring slot kslot
      auto issue_s = [&](int h, uint32_t kslot, int ncols) {
        const uint32_t idesc_s = idesc_bf16_f32(128, ncols, false);
        const uint32_t s_tmem = tmem_base + h * kN;
        const uint64_t qd = qd0 + (uint32_t)h * (uint32_t)(kQBytes >> 4);
        const uint64_t kd = kd0 + kslot * slot_step;
        umma_ss<0>(s_tmem, qd, kd, idesc_s);
#pragma unroll
        for (int kk = 1; kk < kSteps; ++kk) {
          const uint32_t qoff = (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2;
          const uint32_t koff = (kk >> 2) * kvc16 + (kk & 3) * 2;
          umma_ss<1>(s_tmem, qd + qoff, kd + koff, idesc_s);
        }
      };
      for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, npairs); ok && wk.valid();
           wk.next(), ++it) {
        const int qb = a.qb_first + 2 * wk.qb();
        const BlockTiles bt = block_tiles<false>(plan, qb, a.L, a.w, a.s);
        const int n = bt.n_tiles;
        if (!mbar_wait_inl(&q_full[0], it & 1, abort_flag) ||
            !mbar_wait_inl(&q_full[1], it & 1, abort_flag)) {
          ok = false;
          break;
        }
        // S of the first tile for both query tiles
        int cur_ncols = tile_at<false>(plan, bt, 0, a.w, a.s).ncols;
        if (!mbar_wait_inl(&kv_full[ks], kph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        issue_s(0, ks, cur_ncols);
        umma_commit(&s_full[0]);
        if (n == 1) umma_commit(&q_empty[0]);
        issue_s(1, ks, cur_ncols);
        umma_commit(&s_full[1]);
        umma_commit(&kv_empty[ks]);
        if (n == 1) umma_commit(&q_empty[1]);
        for (int j = 0; j < n; ++j, ++gt) {
          uint32_t vs = ks, vph = kph;   // V_j follows K_j
          advance(vs, vph, 1);
          uint32_t ks1 = vs, kph1 = vph; // K_{j+1} follows V_j
          advance(ks1, kph1, 1);
          const bool more = j + 1 < n;
          const int nxt_ncols = more ? tile_at<false>(plan, bt, j + 1, a.w, a.s).ncols : 0;
          if (!mbar_wait_inl(&kv_full[vs], vph, abort_flag)) { ok = false; break; }
          // A = P (TMEM, 8 columns per 16 keys), B = V (MN-major: d contiguous)
          const uint64_t vd = vd0 + vs * slot_step;
          for (int h = 0; h < 2; ++h) {
            if (!mbar_wait_inl(&p_full[h], gt & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            pv_steps<kPvSteps>(cur_ncols >> 4, j > 0 ? 1u : 0u, tmem_base + kTmemO0 + h * D,
                               tmem_base + h * kN, vd, idesc_pv);
            if (h == 1) umma_commit(&kv_empty[vs]);
            if (!more) {
              umma_commit(&o_full[h]);
              continue;
            }
            if (h == 0 && !mbar_wait_inl(&kv_full[ks1], kph1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_s(h, ks1, nxt_ncols);
            umma_commit(&s_full[h]);
            if (h == 1) umma_commit(&kv_empty[ks1]);
            if (j + 2 == n) umma_commit(&q_empty[h]);
          }
          if (!ok) break;
          cur_ncols = nxt_ncols;
          ks = ks1;   // after the last tile: the next item's first K
          kph = kph1;
        }
      }
      // drain: every MMA issued here completes before TMEM is freed
      umma_commit(mma_done);
      mbar_wait_inl(mma_done, 0, abort_flag, 200000000ull, false);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ output store
    setmaxnreg_dec<kPairRegsLow>();
    // Tiles are staged in turn (A, B, A, B, ...) in one buffer. Lane 0 stores
    // each with TMA; a tile that starts before row 0 of out (q_off > 0) is
    // copied by the whole warp with plain stores, row by row from row 0 on,
    // since a TMA store may not start at a negative coordinate.
    if (lane == 0) tma_prefetch_desc(&tm_o);
    const int out_rows = a.L - a.q_off;
    uint32_t use = 0;
    bool ok = true;
    for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, npairs); ok && wk.valid();
         wk.next()) {
      const int b = wk.bh() / a.Hkv, kvh = wk.bh() % a.Hkv;
      for (int h = 0; h < 2; ++h, ++use) {
        const int qb = a.qb_first + 2 * wk.qb() + h;
        int staged = 1;
        if (lane == 0) staged = mbar_wait_inl(epi_staged, use & 1, abort_flag) ? 1 : 0;
        staged = __shfl_sync(0xffffffffu, staged, 0);
        __syncwarp();
        if (!staged) { ok = false; break; }
        const int row0 = qb * plan.Tq - a.q_off;  // out row of the tile's first position
        if (row0 >= out_rows) {
          // every row lies past the end of out (the second block of the last pair)
        } else if (row0 >= 0) {
          if (lane == 0) {
            for (int c = 0; c < kChunks; ++c)
              tma_store_4d(&tm_o, sStage + c * kChunkBytes, c * 64, kvh * plan.G, row0, b);
            tma_store_commit();
            tma_store_wait_read();
          }
        } else {
          for (int i = lane; i < plan.rows * (D / 8); i += 32) {
            const int r = i / (D / 8), u8 = i % (D / 8);  // tile row, 16-byte unit
            const int orow = row0 + r / plan.G;
            if (orow < 0 || orow >= out_rows) continue;
            const int ch = u8 / 8, unit = u8 % 8;
            const uint4 val = *reinterpret_cast<const uint4 *>(sStage + ch * kChunkBytes + r * 128 +
                                                               ((unit ^ (r & 7)) << 4));
            *reinterpret_cast<uint4 *>(
                a.out + (((size_t)b * out_rows + orow) * a.Hq + kvh * plan.G + r % plan.G) * D +
                ch * 64 + unit * 8) = val;
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) mbar_arrive(&stage_free[h ^ 1]);  // the other tile stages next
      }
    }
    if (lane == 0) tma_store_wait_all();
  } else if (warp == 3) {
    setmaxnreg_dec<kPairRegsLow>();  // idle; the whole warpgroup re-splits
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    setmaxnreg_inc<kPairRegsHigh>();
    const int h = (warp - kSoftmaxWarp0) >> 2;    // query tile: 0 = A, 1 = B
    const int sub = warp & 3;                     // TMEM lane quarter
    const int r = sub * 32 + lane;                // tile row owned by this thread
    const uint32_t lane_addr = tmem_base + ((uint32_t)(sub * 32) << 16);
    const uint32_t s_row = lane_addr + h * kN;
    const uint32_t o_row = lane_addr + kTmemO0 + h * D;
    const float cl2 = a.scale_log2;
    // every lane polls; the outcome is made warp-uniform so a timeout on one
    // lane cannot leave the warp diverged before a .sync.aligned instruction
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      const bool rr = mbar_wait_inl(bar, parity, abort_flag);
      return __all_sync(0xffffffffu, rr);
    };
    uint32_t gt = 0;
    int it = 0;
    bool ok = true;
    const int row_pos = r / plan.G;      // position of this row within a block
    for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, npairs); ok && wk.valid();
         wk.next(), ++it) {
      const int qb0 = a.qb_first + 2 * wk.qb();
      const BlockTiles bt = block_tiles<false>(plan, qb0, a.L, a.w, a.s);
      const int t0q = (qb0 + h) * plan.Tq;  // first position of this query tile
      const int t = t0q + row_pos;          // query position of this row
      float m_used = -INFINITY;             // running max (scaled, log2 units)
      float l_sum = 0.f;
      for (int i = 0; i < bt.n_tiles; ++i, ++gt) {
        const Tile tl = tile_at<false>(plan, bt, i, a.w, a.s);
        if (!warp_wait(&s_full[h], gt & 1)) { ok = false; break; }
        tc_fence_after();
        int mask = 0;
        ColRanges cr{0, 0, 0, 0};
        if (!tile_full_for(tl, t0q, plan.Tq, a.w)) {
          mask = 1;
          cr = tile_ranges(tl, t, a.w, a.s);
        }
        float factor;
#define SWA_SOFTMAX_ROW(N) \
  softmax_row<N>(s_row, mask, cr.a_lo, cr.a_hi, cr.b_lo, cr.b_hi, cl2, m_used, l_sum, factor)
        static_assert(kN == 128, "softmax dispatch covers 1..8 chunks");
        switch (tl.ncols >> 4) {
          case 1: SWA_SOFTMAX_ROW(1); break;
          case 2: SWA_SOFTMAX_ROW(2); break;
          case 3: SWA_SOFTMAX_ROW(3); break;
          case 4: SWA_SOFTMAX_ROW(4); break;
          case 5: SWA_SOFTMAX_ROW(5); break;
          case 6: SWA_SOFTMAX_ROW(6); break;
          case 7: SWA_SOFTMAX_ROW(7); break;
          default: SWA_SOFTMAX_ROW(8); break;
        }
#undef SWA_SOFTMAX_ROW
        tmem_wait_st();
        // O_h has no MMA in flight here: S_h of this tile was issued after
        // P V of the previous one, and MMAs of one thread complete in order.
        if (__any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            float o[16];
            tmem_ld16(o_row + c * 16, o);
            tmem_wait_ld();
            reg_fence16(o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= factor;
            tmem_st16(o_row + c * 16, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[h]);  // one arrival per softmax warp
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      // O / l -> bf16 into the staging tile (tiles take turns: A, B, A, ...;
      // the store of the previous one must have read the buffer), in the
      // swizzled layout of the output tensor map.
      if (a.lse != nullptr && r < plan.rows && t < a.L) {
        // m_used is in log2 units of the scaled scores
        const int hq = (wk.bh() % a.Hkv) * plan.G + r % plan.G;
        a.lse[((size_t)(wk.bh() / a.Hkv) * a.Hq + hq) * a.L + t] =
            (m_used + log2f(l_sum)) * 0.6931471805599453f;
      }
      if (!warp_wait(&o_full[h], it & 1)) { ok = false; break; }
      // completion c of stage_free[h] (1-based): tile A of item it needs the
      // store of tile B of item it - 1 (c = it), tile B of item it needs the
      // store of tile A of item it (c = it + 1)
      const int c = h == 0 ? it : it + 1;
      if (c > 0 && !warp_wait(&stage_free[h], (uint32_t)(c - 1) & 1u)) { ok = false; break; }
      tc_fence_after();
      const float inv_l = 1.0f / l_sum;
      const uint32_t stage_row = smem_u32(sStage) + r * 128;
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        float o[16];
        tmem_ld16(o_row + j * 16, o);
        tmem_wait_ld();
        reg_fence16(o);
        if (r < plan.rows) {
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {  // 16-byte unit: 8 columns
            const int col = j * 16 + q2 * 8;
            const int ch = col / 64, unit = (col % 64) / 8;
            const float *v = &o[q2 * 8];
            st_shared_v4(stage_row + ch * kChunkBytes + ((unit ^ (r & 7)) << 4),
                         pack_bf16x2(v[0] * inv_l, v[1] * inv_l),
                         pack_bf16x2(v[2] * inv_l, v[3] * inv_l),
                         pack_bf16x2(v[4] * inv_l, v[5] * inv_l),
                         pack_bf16x2(v[6] * inv_l, v[7] * inv_l));
          }
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
