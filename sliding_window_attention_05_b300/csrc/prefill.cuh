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
// Warp roles (256 threads, one CTA per SM):
//   warp 0      TMA producer: Q (double buffered) and a ring of K/V tiles
//   warp 1      TMEM owner and MMA issuer (one thread):
//                 S_g = Q K_g^T  -> TMEM buffer g % 2   (tcgen05, fp32)
//                 O  += P_g V_g  -> TMEM                 (tcgen05, fp32)
//               S_{g+1} is issued before O += P_g V_g so the tensor core
//               works on the next tile while the softmax warps finish this one
//   warps 4-7   softmax + epilogue, one thread per tile row (TMEM lane):
//               in-tile mask, online softmax with lazy rescaling, P (bf16) to
//               shared memory, O rescale in TMEM when the running max grows by
//               more than 2^8, and at block end O / l -> bf16 -> global.
//
// Shared memory (d = 128): Q 2 x 32 KB, K/V ring 4 x 32 KB, P 32 KB. Every
// operand is stored as 64-column chunks of 128-byte rows with the 128-byte
// swizzle, which is what TMA writes and what the MMA descriptors describe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sm100_ptx.cuh"
#include "swa_index.cuh"

namespace swa {

constexpr int kTileRows = 128;             // M of every MMA
constexpr int kChunkBytes = kTileRows * 128;  // one 64-column chunk of a 128-row tile
constexpr int kPBytes = 2 * kChunkBytes;   // P tile: 128 rows x up to 128 keys, bf16
constexpr int kTmemCols = 512;
constexpr int kTmemS0 = 0;                 // S buffers at columns 0 and 128
constexpr int kTmemO = 256;                // O at columns 256 .. 256 + d
constexpr int kPrefillThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when max grows > 2^8

struct PrefillArgs {
  __nv_bfloat16 *out;
  int B, L, Hq, Hkv, w, s;
  float scale_log2;   // scale * log2(e)
  PrefillPlan plan;
  int n_items;
  int stages;         // K/V ring slots
};

template <int D>
struct PrefillSmem {
  static constexpr int kQBytes = (D / 64) * kChunkBytes;  // one Q (or K or V) tile
  static size_t bytes(int stages) {
    return 1024 /* alignment slack */ + 2 * (size_t)kQBytes + (size_t)stages * kQBytes + kPBytes +
           256 /* barriers and the TMEM address */;
  }
};

template <int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    swa_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_ks,
                       const __grid_constant__ CUtensorMap tm_vs, const PrefillArgs a) {
  constexpr int kQBytes = PrefillSmem<D>::kQBytes;
  constexpr int kChunks = D / 64;
  constexpr int kSteps = D / 16;  // K steps of the S = Q K^T product

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int stages = a.stages;
  uint8_t *sQ = smem;                               // 2 x kQBytes
  uint8_t *sKV = sQ + 2 * kQBytes;                  // stages x kQBytes
  uint8_t *sP = sKV + (size_t)stages * kQBytes;     // kPBytes
  uint64_t *bars = reinterpret_cast<uint64_t *>(sP + kPBytes);
  uint64_t *q_full = bars + 0;      // [2]
  uint64_t *q_empty = bars + 2;     // [2]
  uint64_t *s_full = bars + 4;      // [2]
  uint64_t *p_full = bars + 6;      // [1]
  uint64_t *pv_done = bars + 7;     // [1]
  uint64_t *o_full = bars + 8;      // [1]
  uint64_t *mma_done = bars + 9;    // [1]
  uint64_t *kv_full = bars + 10;    // [stages <= 8]
  uint64_t *kv_empty = bars + 18;   // [stages <= 8]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 26);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 27);

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
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(o_full, 1);
    mbar_init(mma_done, 1);
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
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t g = 0;  // global tile counter of this CTA
      int it = 0;
      int last_q_parity[2] = {-1, -1};
      int last_kv_parity[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
      bool ok = true;
      for (int item = blockIdx.x; ok && item < a.n_items; item += gridDim.x, ++it) {
        const int qb = plan.nqb - 1 - item / BH;
        const int bh = item % BH;
        const int b = bh / a.Hkv, kvh = bh % a.Hkv;
        const BlockTiles bt = block_tiles(plan, qb, a.L, a.w, a.s);
        const int qbuf = it & 1;
        if (!mbar_wait(&q_empty[qbuf], ((it >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&q_full[qbuf], (uint32_t)(kChunks * 64 * plan.rows * 2));
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(sQ + qbuf * kQBytes + c * kChunkBytes, &tm_q, &q_full[qbuf], c * 64,
                      kvh * plan.G, bt.t0, b, pol_q);
        last_q_parity[qbuf] = (it >> 1) & 1;
        for (int i = 0; i < bt.n_tiles; ++i, ++g) {
          const Tile tl = tile_at(plan, bt, i, a.w, a.s);
          const int box = tl.sink ? plan.s_box : plan.n_band;
          const uint32_t tile_bytes = (uint32_t)(kChunks * 64 * box * 2);
          for (int half = 0; half < 2; ++half) {  // 0: K, 1: V
            const uint32_t u = 2 * g + half;
            const int slot = (int)(u % stages);
            const uint32_t use = u / stages;
            if (!mbar_wait(&kv_empty[slot], (use & 1) ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(&kv_full[slot], tile_bytes);
            const CUtensorMap *tm =
                half == 0 ? (tl.sink ? &tm_ks : &tm_k) : (tl.sink ? &tm_vs : &tm_v);
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(sKV + slot * kQBytes + c * kChunkBytes, tm, &kv_full[slot], c * 64, kvh,
                          tl.k0, b, pol_kv);
            last_kv_parity[slot] = use & 1;
          }
          if (!ok) break;
        }
      }
      if (!ok) {
        // Let the loads already in flight land before the CTA can exit.
        for (int i = 0; i < 2; ++i)
          if (last_q_parity[i] >= 0) mbar_wait(&q_full[i], last_q_parity[i], abort_flag, 200000000ull, false);
        for (int i = 0; i < stages; ++i)
          if (last_kv_parity[i] >= 0) mbar_wait(&kv_full[i], last_kv_parity[i], abort_flag, 200000000ull, false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_base = smem_u32(sQ), kv_base = smem_u32(sKV), p_base = smem_u32(sP);
      const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      // the tile whose S has been issued but whose P V is still pending
      bool pend = false;
      uint32_t pend_g = 0;
      int pend_ncols = 0;
      bool pend_first = false, pend_last = false;

      auto issue_pv = [&](uint32_t gg, int ncols, bool first, bool last) -> bool {
        if (!mbar_wait(p_full, gg & 1, abort_flag)) return false;
        const uint32_t u = 2 * gg + 1;
        const int slot = (int)(u % stages);
        if (!mbar_wait(&kv_full[slot], (u / stages) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t v_base = kv_base + slot * kQBytes;
        for (int kk = 0; kk < ncols / 16; ++kk) {
          // A = P (K-major, 64-key chunks), B = V (MN-major: d contiguous)
          const uint64_t adesc = sdesc_sw128(p_base + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(v_base + kk * 2048, kChunkBytes, 1024);
          umma_bf16_ss(tmem_base + kTmemO, adesc, bdesc, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
        umma_commit(&kv_empty[slot]);
        umma_commit(pv_done);
        if (last) umma_commit(o_full);
        return true;
      };

      for (int item = blockIdx.x; ok && item < a.n_items; item += gridDim.x, ++it) {
        const int qb = plan.nqb - 1 - item / BH;
        const BlockTiles bt = block_tiles(plan, qb, a.L, a.w, a.s);
        const int qbuf = it & 1;
        if (!mbar_wait(&q_full[qbuf], (it >> 1) & 1, abort_flag)) { ok = false; break; }
        for (int i = 0; i < bt.n_tiles; ++i, ++g) {
          const Tile tl = tile_at(plan, bt, i, a.w, a.s);
          const uint32_t u = 2 * g;
          const int slot = (int)(u % stages);
          if (!mbar_wait(&kv_full[slot], (u / stages) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t idesc_s = idesc_bf16_f32(128, tl.ncols, false);
          const uint32_t qa = q_base + qbuf * kQBytes, kb = kv_base + slot * kQBytes;
#pragma unroll
          for (int kk = 0; kk < kSteps; ++kk) {
            const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
            umma_bf16_ss(tmem_base + kTmemS0 + (g & 1) * 128, sdesc_sw128(qa + off, 16, 1024),
                         sdesc_sw128(kb + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(&kv_empty[slot]);
          umma_commit(&s_full[g & 1]);
          if (i == bt.n_tiles - 1) umma_commit(&q_empty[qbuf]);
          if (pend && !issue_pv(pend_g, pend_ncols, pend_first, pend_last)) { ok = false; break; }
          pend = true;
          pend_g = g;
          pend_ncols = tl.ncols;
          pend_first = (i == 0);
          pend_last = (i == bt.n_tiles - 1);
        }
      }
      if (ok && pend) issue_pv(pend_g, pend_ncols, pend_first, pend_last);
      // drain: every MMA issued by this thread completes before TMEM is freed
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, abort_flag, 200000000ull, false);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------ softmax + epilogue
    const int sub = warp - kSoftmaxWarp0;  // TMEM lane quarter
    const int r = sub * 32 + lane;         // tile row owned by this thread
    const uint32_t lane_addr = tmem_base + ((uint32_t)(sub * 32) << 16);
    const uint32_t p_row = smem_u32(sP) + r * 128;
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
    for (int item = blockIdx.x; ok && item < a.n_items; item += gridDim.x, ++it) {
      const int qb = plan.nqb - 1 - item / BH;
      const int bh = item % BH;
      const int b = bh / a.Hkv, kvh = bh % a.Hkv;
      const BlockTiles bt = block_tiles(plan, qb, a.L, a.w, a.s);
      const int t = bt.t0 + r / plan.G;  // query position of this row
      float m_used = -INFINITY;          // running max (scaled, log2 units)
      float l_sum = 0.f;
      for (int i = 0; i < bt.n_tiles; ++i, ++g) {
        const Tile tl = tile_at(plan, bt, i, a.w, a.s);
        if (!warp_wait(&s_full[g & 1], (g >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        float x[128];
        const uint32_t s_addr = lane_addr + kTmemS0 + (g & 1) * 128;
        const int nch = tl.ncols >> 4;  // 16-column chunks (ncols is a multiple of 16)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (c < nch) tmem_ld16(s_addr + c * 16, *reinterpret_cast<float(*)[16]>(&x[c * 16]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (c < nch) reg_fence16(*reinterpret_cast<float(*)[16]>(&x[c * 16]));
        if (!tl.full) {
          // The admitted columns of this row form at most two ranges: the
          // window part [max(own_lo, t-w+1), min(own_hi, t+1)) and the sink
          // part [own_lo, min(own_hi, s, t+1)).
          const int a_lo = imax(tl.own_lo, t - a.w + 1) - tl.k0;
          const int a_hi = imin(tl.own_hi, t + 1) - tl.k0;
          const int b_lo = tl.own_lo - tl.k0;
          const int b_hi = imin(imin(tl.own_hi, a.s), t + 1) - tl.k0;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if (c < nch) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int col = c * 16 + e;
                const bool in = (col >= a_lo && col < a_hi) || (col >= b_lo && col < b_hi);
                x[col] = in ? x[col] : -INFINITY;
              }
            }
        }
        // row max of the raw scores, eight independent chains
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (c < nch) {
#pragma unroll
            for (int e = 0; e < 16; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], x[c * 16 + e]);
          }
#pragma unroll
        for (int k = 1; k < 8; ++k) mx8[0] = fmaxf(mx8[0], mx8[k]);
        const float m_tile = mx8[0] * cl2;  // scale > 0, so the max commutes with it
        const float m_new = fmaxf(m_used, m_tile);
        float factor = 1.f;
        bool rescale = false;
        if (m_used == -INFINITY) {
          m_used = m_new;  // nothing accumulated yet for this row
        } else if (m_new > m_used + kRescaleThreshold) {
          factor = fast_exp2(m_used - m_new);
          m_used = m_new;
          l_sum *= factor;
          rescale = true;
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        float sum8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sum8[k] = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (c < nch) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              x[c * 16 + e] = fast_exp2(fmaf(x[c * 16 + e], cl2, -msub));
              sum8[e & 7] += x[c * 16 + e];
            }
          }
        float rs = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
                   ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        l_sum += rs;
        // P buffer is free once the previous tile's P V has completed; that
        // also makes O current for the rescale below.
        if (g > 0 && !warp_wait(pv_done, (g - 1) & 1)) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (c < nch) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int u = 2 * c + h;  // 16-byte unit: keys 8u .. 8u+7
              const uint32_t addr = p_row + (u >> 3) * kChunkBytes + (((u & 7) ^ (r & 7)) << 4);
              st_shared_v4(addr, pack_bf16x2(x[u * 8 + 0], x[u * 8 + 1]),
                           pack_bf16x2(x[u * 8 + 2], x[u * 8 + 3]),
                           pack_bf16x2(x[u * 8 + 4], x[u * 8 + 5]),
                           pack_bf16x2(x[u * 8 + 6], x[u * 8 + 7]));
            }
          }
        fence_proxy_async_smem();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            float o[16];
            tmem_ld16(lane_addr + kTmemO + c * 16, o);
            tmem_wait_ld();
            reg_fence16(o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= factor;
            tmem_st16(lane_addr + kTmemO + c * 16, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);  // one arrival per softmax warp
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!warp_wait(o_full, it & 1)) { ok = false; break; }
      tc_fence_after();
      const float inv_l = 1.0f / l_sum;
      const bool store = (r < plan.rows) && (t < a.L);
      __nv_bfloat16 *orow =
          a.out + (((size_t)b * a.L + t) * a.Hq + (size_t)kvh * plan.G + (r % plan.G)) * D;
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        float o[16];
        tmem_ld16(lane_addr + kTmemO + c * 16, o);
        tmem_wait_ld();
        reg_fence16(o);
        if (store) {
          uint4 v0, v1;
          v0.x = pack_bf16x2(o[0] * inv_l, o[1] * inv_l);
          v0.y = pack_bf16x2(o[2] * inv_l, o[3] * inv_l);
          v0.z = pack_bf16x2(o[4] * inv_l, o[5] * inv_l);
          v0.w = pack_bf16x2(o[6] * inv_l, o[7] * inv_l);
          v1.x = pack_bf16x2(o[8] * inv_l, o[9] * inv_l);
          v1.y = pack_bf16x2(o[10] * inv_l, o[11] * inv_l);
          v1.z = pack_bf16x2(o[12] * inv_l, o[13] * inv_l);
          v1.w = pack_bf16x2(o[14] * inv_l, o[15] * inv_l);
          reinterpret_cast<uint4 *>(orow + c * 16)[0] = v0;
          reinterpret_cast<uint4 *>(orow + c * 16)[1] = v1;
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace swa
