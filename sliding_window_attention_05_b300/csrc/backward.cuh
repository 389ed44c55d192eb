// backward.cuh -- gradients of the SWA(w, s) prefill on sm_103a: dQ, dK, dV
// for an upstream gradient dO, with tcgen05 MMAs (TMEM accumulators) and the
// same band-aware tile schedule as the forward pass.
//
// The pages give no backward formulas; they mention SWA-aware fine-tuning
// ("如何将Sliding Window Attention Adaptation应用到你的LLM项目中", section
// "微调：提升SWAA适应性"). What is computed is the chain rule applied to the
// forward definition (explainer of arXiv 2608.28444, section "核心方法 / 1.":
// the x_t equation with the swa_mask key set). For every row (b, hq, t) and
// key j in K(t), with P the softmax weights of the forward pass:
//   dP_tj = dO_t . v_j,   D_t = sum_j P_tj dP_tj = dO_t . O_t,
//   dS_tj = P_tj (dP_tj - D_t),
//   dQ_t  = scale sum_j dS_tj k_j,
//   dK_j  = scale sum_t dS_tj q_t,   dV_j = sum_t P_tj dO_t,
// where k_j, v_j belong to KV head hq / (Hq / Hkv): dK and dV sum over the
// query heads of a group. P is recomputed from the scores and the forward's
// row log-sum-exp: P_tj = 2^(scale log2(e) q_t . k_j - lse_t log2(e)).
//
// Kernels (launched in this order by swa_prefill_backward):
//   swa_bwd_pre_kernel   D_t = dO_t . O_t (fp32) for every row; clears the
//                        fp32 accumulators of the sink keys
//   swa_bwd_dq_kernel    one query block per work item, as the forward: for
//                        every key tile of the block, S = Q K^T and
//                        dP = dO V^T (TMEM), then the softmax warps form dS
//                        (bf16, over S in TMEM), then dQ += dS K (TMEM)
//   swa_bwd_dkv_kernel   one key tile (128 keys of one KV head) per CTA, over
//                        the query blocks whose rows attend to it:
//                        S^T = K Q^T and dP^T = V dO^T (TMEM), the softmax
//                        warps form P^T and dS^T (bf16, in TMEM), then
//                        dV += P^T dO and dK += dS^T Q (TMEM). Band tiles hold
//                        keys j >= s, attended by rows t in [j, j + w - 1]; the
//                        sink keys (j < s), attended by every later row, are
//                        split over CTAs by chunks of query blocks whose
//                        partial sums are added into fp32 accumulators
//   swa_bwd_sink_out_kernel  the sink keys' accumulators -> bf16 dK, dV rows
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "prefill.cuh"
#include "sm100_ptx.cuh"
#include "swa_index.cuh"

namespace swa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBwdSinkChunk = 16;   // query blocks per sink work item

struct BwdArgs {
  const __nv_bfloat16 *out, *dout;  // [B, L, Hq, d]
  const float *lse;                 // [B, Hq, L] natural log
  float *D;                         // [B, Hq, L] dO . O
  float *sink_dk, *sink_dv;         // [B, Hkv, s_eff, d] fp32 accumulators
  __nv_bfloat16 *dq, *dk, *dv;      // [B, L, Hq, d], [B, L, Hkv, d] x 2
  int B, L, Hq, Hkv, w, s, s_eff;   // s_eff = min(s, L)
  float scale, scale_log2;
  PrefillPlan plan;                 // the forward's tiling (dQ kernel)
  int n_items;                      // work items of the launch
  int stages;
  int kv_chunk;
  int n_band_tiles;                 // band key tiles per (b, KV head)
  int n_sink_items;                 // sink work items per (b, KV head)
};

// ---------------------------------------------------------------- D = dO . O

// D[b, hq, t] = sum_c dO[b, t, hq, c] O[b, t, hq, c] in fp32, for every row.
// Rows are numbered r = (b * Hq + hq) * L + t, the index of D, so the writes
// are contiguous. D / 8 threads take one row, 16 bytes each (32 / (D / 8) rows
// per warp pass), and every warp keeps four passes of loads in flight (a
// grid-stride loop). The first threads also clear the sink keys' accumulators.
template <int D>
__global__ void swa_bwd_pre_kernel(const BwdArgs a, long long n_rows, long long n_sink) {
  grid_launch_dependents();
  grid_dependency_wait();
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long i = gtid; i < n_sink; i += nthreads) {
    a.sink_dk[i] = 0.f;
    a.sink_dv[i] = 0.f;
  }
  constexpr int kTpr = D / 8;        // threads per row
  constexpr int kRpw = 32 / kTpr;    // rows per warp pass
  constexpr int kPasses = 4;         // passes in flight
  const int lane = threadIdx.x % 32;
  const int sub = lane / kTpr, c = lane % kTpr;
  const long long warp = gtid / 32, nwarps = nthreads / 32;
  for (long long base = warp * (kRpw * kPasses); base < n_rows;
       base += nwarps * (kRpw * kPasses)) {
    uint4 ov[kPasses], gv[kPasses];
#pragma unroll
    for (int u = 0; u < kPasses; ++u) {
      const long long r = base + u * kRpw + sub;
      ov[u] = gv[u] = make_uint4(0, 0, 0, 0);
      if (r < n_rows) {
        const long long t = r % a.L, bh = r / a.L;            // bh = b * Hq + hq
        const long long hq = bh % a.Hq, b = bh / a.Hq;
        const long long off = ((b * a.L + t) * a.Hq + hq) * D + c * 8;
        ov[u] = *reinterpret_cast<const uint4 *>(a.out + off);
        gv[u] = *reinterpret_cast<const uint4 *>(a.dout + off);
      }
    }
#pragma unroll
    for (int u = 0; u < kPasses; ++u) {
      const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&ov[u]);
      const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&gv[u]);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(o2[e]), gf = __bfloat1622float2(g2[e]);
        acc = fmaf(of.x, gf.x, fmaf(of.y, gf.y, acc));
      }
#pragma unroll
      for (int off = kTpr / 2; off >= 1; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long long r = base + u * kRpw + sub;
      if (c == 0 && r < n_rows) a.D[r] = acc;
    }
  }
}

// The sink keys' fp32 accumulators -> bf16 rows 0 .. s_eff - 1 of dk and dv
// (dK takes the scale here).
__global__ void swa_bwd_sink_out_kernel(const BwdArgs a, int d) {
  grid_launch_dependents();
  grid_dependency_wait();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long n = (long long)a.B * a.Hkv * a.s_eff * d;
  if (i >= n) return;
  const int c = (int)(i % d);
  const int j = (int)((i / d) % a.s_eff);
  const int kvh = (int)((i / ((long long)d * a.s_eff)) % a.Hkv);
  const long long b = i / ((long long)d * a.s_eff * a.Hkv);
  const size_t dst = (((size_t)b * a.L + j) * a.Hkv + kvh) * d + c;
  a.dk[dst] = __float2bfloat16_rn(a.sink_dk[i] * a.scale);
  a.dv[dst] = __float2bfloat16_rn(a.sink_dv[i]);
}

// ---------------------------------------------------------------- dQ

// Shared memory of the dQ kernel: Q and dO tiles of the current block, then
// a ring of K/V slots (the forward's tiles, up to kMaxTileKeys keys).
template <int D>
struct BwdDqSmem {
  static constexpr int kTile = (D / 64) * kChunkBytes;  // one 128-row tile
  static int slot_bytes(const PrefillPlan &p) { return (D / 64) * p.slot_keys * 128; }
  static size_t fixed_bytes() { return 1024 + 2 * (size_t)kTile + 256; }
  static size_t bytes(const PrefillPlan &p, int stages) {
    return fixed_bytes() + (size_t)stages * slot_bytes(p);
  }
  static int stages(const PrefillPlan &p, int max_smem) {
    long long st = ((long long)max_smem - (long long)fixed_bytes()) / slot_bytes(p);
    return (int)(st > kMaxStages ? kMaxStages : st);
  }
};

// Warp roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 4-11
// the row work: warps 4 + q and 8 + q own TMEM lanes 32q .. 32q + 31 (tile
// rows) and split each tile's 16-key chunks (dS is elementwise given lse and
// D, so the two need no exchange) and the dQ columns of the epilogue.
// Tensor memory: S at column 0, dP at 192, dQ at 384.
// Per tile g the MMA warp issues S_g = Q K_g^T and dP_g = dO V_g^T, the row
// warps turn them into dS_g (bf16, written over S_g), then the MMA warp issues
// dQ += dS_g K_g (A = dS from TMEM, B = K_g with d contiguous); the next tile's
// S and dP follow it in issue order, so they never overwrite dS before it is
// read. The ring holds K_g then V_g; V_g's slot is released after dP_g, K_g's
// after the dQ product.
template <int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    swa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_ks,
                      const __grid_constant__ CUtensorMap tm_vs, const BwdArgs a) {
  constexpr int kTile = BwdDqSmem<D>::kTile;
  constexpr int kChunks = D / 64;
  constexpr int kSteps = D / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int stages = a.stages;
  const int kv_chunk = a.kv_chunk;
  const int slot_bytes = kChunks * kv_chunk;
  uint8_t *sQ = smem;
  uint8_t *sDO = sQ + kTile;
  uint8_t *sKV = sDO + kTile;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sKV + (size_t)stages * slot_bytes);
  uint64_t *q_full = bars + 0;     // Q and dO of the item landed
  uint64_t *q_empty = bars + 1;    // every MMA reading Q / dO of the item done
  uint64_t *s_full = bars + 2;     // S and dP of the tile computed
  uint64_t *ds_full = bars + 3;    // dS written (8 warps)
  uint64_t *dq_full = bars + 4;    // the item's last dQ product done
  uint64_t *dq_free = bars + 5;    // dQ read out (8 warps)
  uint64_t *mma_done = bars + 6;
  uint64_t *kv_full = bars + 8;    // [stages <= 8]
  uint64_t *kv_empty = bars + 16;  // [stages <= 8]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 24);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 25);
  // [4] per TMEM lane quarter: both warps of the pair have read the tile's S
  // (each warp's dS goes over S columns that may hold the partner's chunks)
  uint64_t *pair_read = bars + 26;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const PrefillPlan &plan = a.plan;
  const int BH = a.B * a.Hkv;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 8);
    for (int q = 0; q < 4; ++q) mbar_init(&pair_read[q], 2);
    mbar_init(mma_done, 1);
    for (int i = 0; i < stages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (plan.rows < kTileRows) {
    for (int i = threadIdx.x; i < 2 * kTile / 16; i += blockDim.x)
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
  grid_launch_dependents();
  grid_dependency_wait();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t u = 0;
      int slot = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, plan.nqb); ok && wk.valid();
           wk.next(), ++it) {
        const int b = wk.bh() / a.Hkv, kvh = wk.bh() % a.Hkv;
        const BlockTiles bt = block_tiles<false>(plan, wk.qb(), a.L, a.w, a.s);
        // Q and dO of the block, once the previous block's MMAs are done
        if (!mbar_wait(q_empty, (it & 1) ^ 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(q_full, (uint32_t)(2 * kChunks * 64 * plan.rows * 2));
        for (int c = 0; c < kChunks; ++c) {
          tma_load_4d(sQ + c * kChunkBytes, &tm_q, q_full, c * 64, kvh * plan.G, bt.t0, b, pol_q);
          tma_load_4d(sDO + c * kChunkBytes, &tm_do, q_full, c * 64, kvh * plan.G, bt.t0, b, pol_q);
        }
        for (int i = 0; i < bt.n_tiles && ok; ++i) {
          const Tile t = tile_at<false>(plan, bt, i, a.w, a.s);
          const bool band = t.ncols > t.n_sink_cols;
          const uint32_t bytes =
              (uint32_t)(kChunks * 128 * (t.n_sink_cols + (band ? plan.n_band : 0)));
          for (int half = 0; half < 2; ++half) {  // K, then V
            if (!mbar_wait(&kv_empty[slot], phase ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(&kv_full[slot], bytes);
            uint8_t *dst = sKV + slot * slot_bytes;
            for (int c = 0; c < kChunks; ++c) {
              if (t.n_sink_cols)
                tma_load_4d(dst + c * kv_chunk, half ? &tm_vs : &tm_ks, &kv_full[slot], c * 64,
                            kvh, t.sink_key0, b, pol_kv);
              if (band)
                tma_load_4d(dst + c * kv_chunk + t.n_sink_cols * 128, half ? &tm_v : &tm_k,
                            &kv_full[slot], c * 64, kvh, t.k0, b, pol_kv);
            }
            ++u;
            if (++slot == stages) { slot = 0; phase ^= 1; }
          }
        }
      }
      if (!ok) {
        const uint32_t first = u > (uint32_t)stages ? u - stages : 0;
        for (uint32_t v = first; v < u; ++v)
          mbar_wait(&kv_full[v % stages], (v / stages) & 1, abort_flag, 200000000ull, false);
        mbar_wait(q_full, (it & 1), abort_flag, 200000000ull, false);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const bool leader = lane == 0;
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    const uint32_t idesc_dq = idesc_bf16_f32(128, D, true);
    const uint64_t qd = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dod = sdesc_sw128(smem_u32(sDO), 16, 1024);
    const uint64_t kd0 = sdesc_sw128(smem_u32(sKV), 16, 1024);
    const uint64_t kmn0 = sdesc_sw128(smem_u32(sKV), (uint32_t)kv_chunk, 1024);
    const uint32_t slot_step = (uint32_t)slot_bytes >> 4;
    const uint32_t kvc16 = (uint32_t)kv_chunk >> 4;
    const uint32_t s_tmem = tmem_base + 0, dp_tmem = tmem_base + kMaxTileKeys,
                   dq_tmem = tmem_base + 2 * kMaxTileKeys;
    uint32_t cs = 0, cph = 0;
    auto consume = [&]() {
      if (++cs == (uint32_t)stages) { cs = 0; cph ^= 1; }
    };
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, plan.nqb); ok && wk.valid();
         wk.next(), ++it) {
      const BlockTiles bt = block_tiles<false>(plan, wk.qb(), a.L, a.w, a.s);
      if (!warp_wait(q_full, it & 1)) { ok = false; break; }
      for (int i = 0; i < bt.n_tiles; ++i, ++g) {
        const Tile tl = tile_at<false>(plan, bt, i, a.w, a.s);
        const uint32_t ks = cs;
        if (!warp_wait(&kv_full[ks], cph)) { ok = false; break; }
        consume();
        const uint32_t vs = cs;
        if (!warp_wait(&kv_full[vs], cph)) { ok = false; break; }
        consume();
        tc_fence_after();
        const uint32_t idesc_s = idesc_bf16_f32(128, tl.ncols, false);
        if (leader) {
          const uint64_t kd = kd0 + ks * slot_step, vd = kd0 + vs * slot_step;
#pragma unroll
          for (int kk = 0; kk < kSteps; ++kk) {
            const uint32_t qoff = (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2;
            const uint32_t koff = (kk >> 2) * kvc16 + (kk & 3) * 2;
            umma_bf16_ss(s_tmem, qd + qoff, kd + koff, idesc_s, kk > 0 ? 1u : 0u);
            umma_bf16_ss(dp_tmem, dod + qoff, vd + koff, idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(&kv_empty[vs]);
          umma_commit(s_full);
          if (i == bt.n_tiles - 1) umma_commit(q_empty);
        }
        __syncwarp();
        // dQ += dS K once the row warps have formed dS; the first product of
        // an item overwrites dQ, after the previous item's epilogue read it
        if (!warp_wait(ds_full, g & 1)) { ok = false; break; }
        if (i == 0 && !warp_wait(dq_free, (it & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
          pv_group(tl.ncols >> 4, i == 0 ? 0u : 1u, dq_tmem, s_tmem, kmn0 + ks * slot_step,
                   idesc_dq);
          umma_commit(&kv_empty[ks]);
          if (i == bt.n_tiles - 1) umma_commit(dq_full);
        }
        __syncwarp();
      }
    }
    if (leader) {
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, abort_flag, 200000000ull, false);
    }
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0) {
    // ---------------------------------------------------------- row warps
    const int sub = (warp - kSoftmaxWarp0) & 3;   // TMEM lane quarter
    const int half = (warp - kSoftmaxWarp0) >> 2; // chunk half
    const int r = sub * 32 + lane;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(sub * 32) << 16);
    const uint32_t s_row = lane_addr, dp_row = lane_addr + kMaxTileKeys,
                   dq_row = lane_addr + 2 * kMaxTileKeys;
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    uint32_t g = 0;
    int it = 0;
    bool ok = true;
    for (ItemWalker wk(blockIdx.x, gridDim.x, a.n_items, BH, plan.nqb); ok && wk.valid();
         wk.next(), ++it) {
      const int b = wk.bh() / a.Hkv, kvh = wk.bh() % a.Hkv;
      const BlockTiles bt = block_tiles<false>(plan, wk.qb(), a.L, a.w, a.s);
      const int t = bt.t0 + r / plan.G;
      const int hq = kvh * plan.G + r % plan.G;
      const bool valid = r < plan.rows && t < a.L;
      const size_t ri = ((size_t)b * a.Hq + hq) * a.L + t;
      // P = 2^(x scale log2 e - lse log2 e); an invalid row gets P = 0
      const float lse2 = valid ? a.lse[ri] * kLog2e : INFINITY;
      const float Dr = valid ? a.D[ri] : 0.f;
      for (int i = 0; i < bt.n_tiles; ++i, ++g) {
        const Tile tl = tile_at<false>(plan, bt, i, a.w, a.s);
        if (!warp_wait(s_full, g & 1)) { ok = false; break; }
        tc_fence_after();
        ColRanges cr{0, tl.ncols, 0, 0};
        if (!tl.full) cr = tile_ranges(tl, t, a.w, a.s);
        // this warp's chunks: the first half of the tile's 16-key chunks for
        // warps 4-7, the rest for warps 8-11. dS of chunk c (bf16, 8 columns)
        // goes over S columns 8c .. 8c + 7, which may hold a chunk the partner
        // has not read yet: dS is kept in registers until both have read S.
        constexpr int kMaxMine = (kMaxTileKeys / 16 + 1) / 2;
        const int nch = tl.ncols >> 4, n0 = (nch + 1) >> 1;
        const int c_lo = half ? n0 : 0, my_n = half ? nch - n0 : n0;
        uint32_t pk[kMaxMine][8];
#pragma unroll
        for (int k = 0; k < kMaxMine; ++k) {
          if (k < my_n) {
            const int c = c_lo + k;
            float x[16], y[16];
            tmem_ld16(s_row + c * 16, x);
            tmem_ld16(dp_row + c * 16, y);
            tmem_wait_ld();
            reg_fence16(x);
            reg_fence16(y);
            const uint32_t bits = range_bits16(c * 16, cr.a_lo, cr.a_hi) |
                                  range_bits16(c * 16, cr.b_lo, cr.b_hi);
            float ds[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float p =
                  ((bits >> e) & 1u) ? fast_exp2(fmaf(x[e], a.scale_log2, -lse2)) : 0.f;
              ds[e] = p * (y[e] - Dr);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[k][e] = pack_bf16x2(ds[2 * e], ds[2 * e + 1]);
          }
        }
        // both warps of the pair have read S (bounded wait, one arrival per warp)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pair_read[sub]);
        if (!warp_wait(&pair_read[sub], g & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kMaxMine; ++k)
          if (k < my_n)
            tmem_st8(s_row + (c_lo + k) * 8, pk[k][0], pk[k][1], pk[k][2], pk[k][3], pk[k][4],
                     pk[k][5], pk[k][6], pk[k][7]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full);
      }
      if (!ok) break;
      // epilogue: dQ = scale * (dS K) -> bf16, one row per thread
      if (!warp_wait(dq_full, it & 1)) { ok = false; break; }
      tc_fence_after();
      __nv_bfloat16 *dst = a.dq + (((size_t)b * a.L + t) * a.Hq + hq) * D;
      // each warp of the pair converts half of the D columns
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        const int c = half * (D / 32) + cc;
        float o[16];
        tmem_ld16(dq_row + c * 16, o);
        tmem_wait_ld();
        reg_fence16(o);
        if (valid) {
          uint4 u0, u1;
          u0.x = pack_bf16x2(o[0] * a.scale, o[1] * a.scale);
          u0.y = pack_bf16x2(o[2] * a.scale, o[3] * a.scale);
          u0.z = pack_bf16x2(o[4] * a.scale, o[5] * a.scale);
          u0.w = pack_bf16x2(o[6] * a.scale, o[7] * a.scale);
          u1.x = pack_bf16x2(o[8] * a.scale, o[9] * a.scale);
          u1.y = pack_bf16x2(o[10] * a.scale, o[11] * a.scale);
          u1.z = pack_bf16x2(o[12] * a.scale, o[13] * a.scale);
          u1.w = pack_bf16x2(o[14] * a.scale, o[15] * a.scale);
          reinterpret_cast<uint4 *>(dst + c * 16)[0] = u0;
          reinterpret_cast<uint4 *>(dst + c * 16)[1] = u1;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------- dK, dV

// Shared memory of the dK/dV kernel: the CTA's K and V tiles (128 keys), then
// a ring of (Q block, dO block) slot pairs, plus the per-column row data of
// each ring stage (lse, D, position).
template <int D>
struct BwdDkvSmem {
  static constexpr int kTile = (D / 64) * kChunkBytes;
  static constexpr int kStages = 2;
  static constexpr size_t kRowData = 128 * 12;  // lse2, D, t per column
  static size_t bytes() {
    return 1024 + 2 * (size_t)kTile + (size_t)kStages * 2 * kTile + kStages * kRowData + 256;
  }
};

// Work item of a dK/dV CTA: a band tile (keys [k0, k0 + 128) with k0 = s +
// 128 i, attended by rows [k0, k0 + 127 + w - 1]) or a sink item (keys
// [128 m, 128 m + 128) of the s_eff sinks, a chunk of kBwdSinkChunk query
// blocks from the start).
struct DkvItem {
  int b, kvh, k0, nkeys, qb_lo, qb_hi;  // query blocks qb_lo .. qb_hi (inclusive)
  bool sink;
};

__device__ __forceinline__ DkvItem dkv_item(const BwdArgs &a, int idx) {
  DkvItem it;
  const int per_bh = a.n_band_tiles + a.n_sink_items;
  const int bh = idx / per_bh, j = idx % per_bh;
  it.b = bh / a.Hkv;
  it.kvh = bh % a.Hkv;
  const int Tq = a.plan.Tq;
  if (j < a.n_band_tiles) {
    it.sink = false;
    it.k0 = a.s + 128 * j;
    it.nkeys = imin(128, a.L - it.k0);
    const long long last = imin((long long)a.L - 1, (long long)it.k0 + it.nkeys - 1 + a.w - 1);
    it.qb_lo = it.k0 / Tq;
    it.qb_hi = (int)(last / Tq);
  } else {
    it.sink = true;
    const int n_chunks = cdiv(a.plan.nqb, kBwdSinkChunk);
    const int m = (j - a.n_band_tiles) / n_chunks, c = (j - a.n_band_tiles) % n_chunks;
    it.k0 = 128 * m;
    it.nkeys = imin(128, a.s_eff - it.k0);
    it.qb_lo = imax(c * kBwdSinkChunk, it.k0 / Tq);
    it.qb_hi = imin(a.plan.nqb - 1, c * kBwdSinkChunk + kBwdSinkChunk - 1);
  }
  return it;
}

// Warp roles as the dQ kernel; tensor memory: S^T at 0, dP^T at 128, dV at
// 256, dK at 384 (keys in lanes). Per query block: S^T = K Q^T and
// dP^T = V dO^T, then the key warps form P^T and dS^T (bf16, over S^T and dP^T),
// then dV += P^T dO and dK += dS^T Q (B operands with d contiguous); the next
// block's products follow in issue order.
template <int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    swa_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_kt,
                       const __grid_constant__ CUtensorMap tm_vt, const BwdArgs a) {
  using Smem = BwdDkvSmem<D>;
  constexpr int kTile = Smem::kTile;
  constexpr int kChunks = D / 64;
  constexpr int kSteps = D / 16;
  constexpr int kStages = Smem::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sK = smem;
  uint8_t *sV = sK + kTile;
  uint8_t *sRing = sV + kTile;                    // [stage][Q, dO] x kTile
  float *sRow = reinterpret_cast<float *>(sRing + (size_t)kStages * 2 * kTile);  // [stage][3][128]
  uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sRow) +
                                                kStages * Smem::kRowData);
  uint64_t *kv_full = bars + 0;    // the CTA's K and V tiles landed
  uint64_t *st_full = bars + 1;    // S^T and dP^T computed
  uint64_t *pt_full = bars + 2;    // P^T and dS^T written (4 warps)
  uint64_t *acc_full = bars + 3;   // the last dV / dK products done
  uint64_t *mma_done = bars + 4;
  uint64_t *row_full = bars + 5;   // [kStages] the stage's row data written (4 warps)
  uint64_t *ring_full = bars + 8;  // [kStages]
  uint64_t *ring_empty = bars + 10;  // [kStages]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 12);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 13);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const PrefillPlan &plan = a.plan;
  const DkvItem item = dkv_item(a, blockIdx.x);
  const int n_steps = item.qb_hi - item.qb_lo + 1;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(st_full, 1);
    mbar_init(pt_full, 4);
    mbar_init(acc_full, 1);
    mbar_init(mma_done, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&row_full[i], 4);
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (plan.rows < kTileRows) {
    for (int i = threadIdx.x; i < kStages * 2 * kTile / 16; i += blockDim.x)
      reinterpret_cast<uint4 *>(sRing)[i] = make_uint4(0, 0, 0, 0);
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
  grid_launch_dependents();
  grid_dependency_wait();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      mbar_arrive_expect_tx(kv_full, (uint32_t)(2 * kChunks * 128 * 128));
      for (int c = 0; c < kChunks; ++c) {
        tma_load_4d(sK + c * kChunkBytes, &tm_kt, kv_full, c * 64, item.kvh, item.k0, item.b, pol);
        tma_load_4d(sV + c * kChunkBytes, &tm_vt, kv_full, c * 64, item.kvh, item.k0, item.b, pol);
      }
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n_steps; ++i) {
        const int st = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (!mbar_wait(&ring_empty[st], ph ^ 1, abort_flag)) { ok = false; break; }
        const int qb = item.qb_lo + i;
        uint8_t *dq_ = sRing + (size_t)st * 2 * kTile;
        mbar_arrive_expect_tx(&ring_full[st], (uint32_t)(2 * kChunks * 64 * plan.rows * 2));
        for (int c = 0; c < kChunks; ++c) {
          tma_load_4d(dq_ + c * kChunkBytes, &tm_q, &ring_full[st], c * 64, item.kvh * plan.G,
                      qb * plan.Tq, item.b, pol);
          tma_load_4d(dq_ + kTile + c * kChunkBytes, &tm_do, &ring_full[st], c * 64,
                      item.kvh * plan.G, qb * plan.Tq, item.b, pol);
        }
        ++issued;
      }
      // the CTA's own K/V tiles land before it can exit (bounded, not abortable)
      mbar_wait(kv_full, 0, abort_flag, 200000000ull, false);
      if (!ok) {
        for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
          mbar_wait(&ring_full[i % kStages], (i / kStages) & 1, abort_flag, 200000000ull, false);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const bool leader = lane == 0;
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    const uint32_t idesc_st = idesc_bf16_f32(128, 128, false);
    const uint32_t idesc_acc = idesc_bf16_f32(128, D, true);
    const uint64_t kd = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t vd = sdesc_sw128(smem_u32(sV), 16, 1024);
    const uint32_t st_tmem = tmem_base, dpt_tmem = tmem_base + 128,
                   dv_tmem = tmem_base + 256, dk_tmem = tmem_base + 384;
    bool ok = warp_wait(kv_full, 0);
    for (int i = 0; ok && i < n_steps; ++i) {
      const int st = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      if (!warp_wait(&ring_full[st], ph)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ring_addr = smem_u32(sRing + (size_t)st * 2 * kTile);
      const uint64_t qd = sdesc_sw128(ring_addr, 16, 1024);
      const uint64_t dod = sdesc_sw128(ring_addr + kTile, 16, 1024);
      if (leader) {
        // S^T = K Q^T, dP^T = V dO^T (M = 128 keys, N = 128 rows)
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
          const uint32_t off = (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2;
          umma_bf16_ss(st_tmem, kd + off, qd + off, idesc_st, kk > 0 ? 1u : 0u);
          umma_bf16_ss(dpt_tmem, vd + off, dod + off, idesc_st, kk > 0 ? 1u : 0u);
        }
        umma_commit(st_full);
      }
      __syncwarp();
      if (!warp_wait(pt_full, i & 1)) { ok = false; break; }
      tc_fence_after();
      if (leader) {
        // dV += P^T dO, dK += dS^T Q (K = 128 rows; B with d contiguous)
        const uint64_t qmn = sdesc_sw128(ring_addr, kChunkBytes, 1024);
        const uint64_t domn = sdesc_sw128(ring_addr + kTile, kChunkBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          umma_bf16_ts(dv_tmem, st_tmem + kk * 8, domn + kk * 128, idesc_acc,
                       (i > 0 || kk > 0) ? 1u : 0u);
          umma_bf16_ts(dk_tmem, dpt_tmem + kk * 8, qmn + kk * 128, idesc_acc,
                       (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&ring_empty[st]);
        if (i == n_steps - 1) umma_commit(acc_full);
      }
      __syncwarp();
    }
    if (leader) {
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, abort_flag, 200000000ull, false);
    }
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4) {
    // ---------------------------------------------------------- key warps
    const int sub = warp - kSoftmaxWarp0;
    const int r = sub * 32 + lane;           // key lane (and row-data column)
    const uint32_t lane_addr = tmem_base + ((uint32_t)(sub * 32) << 16);
    const int j = item.k0 + r;               // this lane's key
    const bool key_ok = r < item.nkeys;
    auto warp_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    bool ok = true;
    for (int i = 0; i < n_steps; ++i) {
      const int st = i % kStages;
      const int qb = item.qb_lo + i;
      // row data of the block's 128 rows (column c = r): lse (log2 units), D, t
      float *rd = sRow + st * 3 * 128;
      {
        const int t = qb * plan.Tq + r / plan.G;
        const int hq = item.kvh * plan.G + r % plan.G;
        const bool valid = r < plan.rows && t < a.L;
        const size_t ri = ((size_t)item.b * a.Hq + hq) * a.L + t;
        rd[r] = valid ? a.lse[ri] * kLog2e : INFINITY;
        rd[128 + r] = valid ? a.D[ri] : 0.f;
        reinterpret_cast<int *>(rd)[256 + r] = valid ? t : -1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&row_full[st]);
      if (!warp_wait(&row_full[st], (uint32_t)(i / kStages) & 1u)) { ok = false; break; }
      if (!warp_wait(st_full, i & 1)) { ok = false; break; }
      tc_fence_after();
      const int *tcol = reinterpret_cast<const int *>(rd) + 256;
      for (int c = 0; c < 8; ++c) {
        float x[16], y[16];
        tmem_ld16(lane_addr + c * 16, x);
        tmem_ld16(lane_addr + 128 + c * 16, y);
        tmem_wait_ld();
        reg_fence16(x);
        reg_fence16(y);
        float p[16], ds[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = c * 16 + e;
          const int t = tcol[col];
          // key j is in K(t): j <= t and (t - j < w, or j a sink)
          const bool adm = key_ok && t >= j && (item.sink || t - j < a.w);
          p[e] = adm ? fast_exp2(fmaf(x[e], a.scale_log2, -rd[col])) : 0.f;
          ds[e] = p[e] * (y[e] - rd[128 + col]);
        }
        tmem_st8(lane_addr + c * 8, pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                 pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]), pack_bf16x2(p[8], p[9]),
                 pack_bf16x2(p[10], p[11]), pack_bf16x2(p[12], p[13]),
                 pack_bf16x2(p[14], p[15]));
        tmem_st8(lane_addr + 128 + c * 8, pack_bf16x2(ds[0], ds[1]), pack_bf16x2(ds[2], ds[3]),
                 pack_bf16x2(ds[4], ds[5]), pack_bf16x2(ds[6], ds[7]),
                 pack_bf16x2(ds[8], ds[9]), pack_bf16x2(ds[10], ds[11]),
                 pack_bf16x2(ds[12], ds[13]), pack_bf16x2(ds[14], ds[15]));
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pt_full);
    }
    if (ok && n_steps > 0 && warp_wait(acc_full, 0)) {
      // epilogue: dV and dK rows of this lane's key
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        float dvv[16], dkk[16];
        tmem_ld16(lane_addr + 256 + c * 16, dvv);
        tmem_ld16(lane_addr + 384 + c * 16, dkk);
        tmem_wait_ld();
        reg_fence16(dvv);
        reg_fence16(dkk);
        if (!key_ok) continue;
        if (item.sink) {
          const size_t base = ((((size_t)item.b * a.Hkv + item.kvh) * a.s_eff) + j) * D + c * 16;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            atomicAdd(a.sink_dv + base + e, dvv[e]);
            atomicAdd(a.sink_dk + base + e, dkk[e]);
          }
        } else {
          const size_t base = (((size_t)item.b * a.L + j) * a.Hkv + item.kvh) * D + c * 16;
          uint4 v0, v1, k0_, k1_;
          v0.x = pack_bf16x2(dvv[0], dvv[1]); v0.y = pack_bf16x2(dvv[2], dvv[3]);
          v0.z = pack_bf16x2(dvv[4], dvv[5]); v0.w = pack_bf16x2(dvv[6], dvv[7]);
          v1.x = pack_bf16x2(dvv[8], dvv[9]); v1.y = pack_bf16x2(dvv[10], dvv[11]);
          v1.z = pack_bf16x2(dvv[12], dvv[13]); v1.w = pack_bf16x2(dvv[14], dvv[15]);
          const float sc = a.scale;
          k0_.x = pack_bf16x2(dkk[0] * sc, dkk[1] * sc); k0_.y = pack_bf16x2(dkk[2] * sc, dkk[3] * sc);
          k0_.z = pack_bf16x2(dkk[4] * sc, dkk[5] * sc); k0_.w = pack_bf16x2(dkk[6] * sc, dkk[7] * sc);
          k1_.x = pack_bf16x2(dkk[8] * sc, dkk[9] * sc); k1_.y = pack_bf16x2(dkk[10] * sc, dkk[11] * sc);
          k1_.z = pack_bf16x2(dkk[12] * sc, dkk[13] * sc); k1_.w = pack_bf16x2(dkk[14] * sc, dkk[15] * sc);
          reinterpret_cast<uint4 *>(a.dv + base)[0] = v0;
          reinterpret_cast<uint4 *>(a.dv + base)[1] = v1;
          reinterpret_cast<uint4 *>(a.dk + base)[0] = k0_;
          reinterpret_cast<uint4 *>(a.dk + base)[1] = k1_;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace swa
