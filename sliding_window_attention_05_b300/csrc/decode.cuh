// decode.cuh -- rolling KV cache append and SWA(w, s) decode on sm_103a.
//
// Cache layout: K and V each [B, Hkv, s + w, d] bf16. Slots 0..s-1 hold the
// sink positions 0..s-1 for good; slots s..s+w-1 form the circular window
// (wiblog.cn long-context SWA article, section "与 KV Cache 的配合：轮转替换策略":
// the oldest entry is evicted, the slot is found modulo the window). After
// position p has been appended, slots 0 .. min(p+1, s+w)-1 hold exactly the key
// set K(p) of the x_t equation with sinks, so decode needs no mask.
//
// Decode is bandwidth-bound (about 4 flop per byte of cache read): it runs on
// the CUDA cores. One CTA (4 warps) serves one (sequence, KV head, head group,
// split): the G query heads sharing the KV head are packed so every K/V row is
// read from memory once for all of them. Each key row (d bf16) is spread over
// d/8 lanes that each load 16 bytes, so a warp-wide load covers 256 or 512
// contiguous bytes; dot products are reduced with xor-shuffles.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sm100_ptx.cuh"
#include "swa_index.cuh"

namespace swa {

// ---------------------------------------------------------------- append

// One thread moves 16 bytes of K and 16 bytes of V of one (b, token, kvh).
__global__ void swa_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                  uint4 *__restrict__ kcache, uint4 *__restrict__ vcache,
                                  const int *__restrict__ pos_start, int T, int Hkv, int d, int w,
                                  int s) {
  const int b = blockIdx.y;
  const int vec_per_row = d / 8;
  const long long n = (long long)T * Hkv * vec_per_row;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n) return;
  const int c = (int)(idx % vec_per_row);
  const int kvh = (int)((idx / vec_per_row) % Hkv);
  const int i = (int)(idx / ((long long)vec_per_row * Hkv));
  const int p0 = pos_start[b];
  if (p0 < 0) {
    if (idx == 0) record_error(kErrNegativePosition);
    return;
  }
  const long long p = (long long)p0 + i;
  const long long p_last = (long long)p0 + T - 1;
  // A token that a later token of this call overwrites again is skipped.
  const bool survives = p < s || p >= p_last - w + 1;
  if (!survives) return;
  const long long slot = ring_slot(p, w, s);
  const long long src = (((long long)b * T + i) * Hkv + kvh) * vec_per_row + c;
  const long long dst = (((long long)b * Hkv + kvh) * (s + w) + slot) * vec_per_row + c;
  kcache[dst] = k_new[src];
  vcache[dst] = v_new[src];
}

// ---------------------------------------------------------------- decode

constexpr int kDecodeWarps = 4;

__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

struct DecodeArgs {
  const __nv_bfloat16 *q;
  const __nv_bfloat16 *kc;
  const __nv_bfloat16 *vc;
  const int *pos;
  __nv_bfloat16 *out;
  float *part_o;     // [B, Hq, splits, D] when splits > 1
  float2 *part_ml;   // [B, Hq, splits] (running max in log2 units, sum)
  int Hq, Hkv, w, s, splits;
  float scale_log2;
};

// HG query heads per CTA (a divisor of G); D = head dimension.
// Key chunks of KPW * U keys are processed per warp iteration, double-buffered.
template <int D, int HG>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    swa_decode_kernel(const DecodeArgs a) {
  constexpr int LPK = D / 8;          // lanes per key row (16 bytes each)
  constexpr int KPW = 32 / LPK;       // keys per warp-wide load
  constexpr int U = HG >= 4 ? 2 : 4;  // loads per lane per chunk
  constexpr int CH = KPW * U;         // keys per chunk

  const int split = blockIdx.x;
  const int G = a.Hq / a.Hkv;
  const int hgroups = G / HG;
  const int kvh = blockIdx.y / hgroups;
  const int hg = blockIdx.y % hgroups;
  const int b = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kg = lane / LPK;          // which key of a warp-wide load
  const int dl = lane % LPK;          // which 8-element slice of d

  const int pos = a.pos[b];
  if (pos < 0) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) record_error(kErrNegativePosition);
    return;
  }
  const int n = ring_valid(pos, a.w, a.s);
  const int per_split = cdiv(n, a.splits);
  const int k_begin = imin(n, split * per_split);
  const int k_end = imin(n, k_begin + per_split);

  // queries of the HG heads, this lane's slice, pre-scaled to log2 units
  float qf[HG][8];
  const int hq0 = kvh * G + hg * HG;
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(a.q + ((size_t)b * a.Hq + hq0 + h) * D + dl * 8);
    bf16x8_to_f32(raw, qf[h]);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[h][e] *= a.scale_log2;
  }

  const size_t row_base = ((size_t)b * a.Hkv + kvh) * (size_t)(a.s + a.w);
  const uint4 *kc = reinterpret_cast<const uint4 *>(a.kc + row_base * D) + dl;
  const uint4 *vc = reinterpret_cast<const uint4 *>(a.vc + row_base * D) + dl;

  float m[HG], l[HG], o[HG][8];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
  }

  // chunks of this split are dealt round-robin to the warps; two register
  // buffers alternate (static indices) so the next chunk's loads are in flight
  // while the current one is reduced
  const int n_chunks = cdiv(k_end - k_begin, CH);
  uint4 ka[U], va[U], kb[U], vb[U];
  auto load_chunk = [&](int ci, uint4 (&kr)[U], uint4 (&vr)[U]) {
    const int base = k_begin + ci * CH;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = base + u * KPW + kg;
      if (key < k_end) {
        kr[u] = ld_stream_v4(kc + (size_t)key * LPK);
        vr[u] = ld_stream_v4(vc + (size_t)key * LPK);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  auto consume = [&](int ci, const uint4 (&kr)[U], const uint4 (&vr)[U]) {
    const int base = k_begin + ci * CH;
    float sc[HG][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[8];
      bf16x8_to_f32(kr[u], kf);
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(qf[h][e], kf[e], acc);
        sc[h][u] = acc;
      }
    }
    // sum the partial dots over the LPK lanes of each key
#pragma unroll
    for (int off = LPK / 2; off >= 1; off /= 2)
#pragma unroll
      for (int h = 0; h < HG; ++h)
#pragma unroll
        for (int u = 0; u < U; ++u) sc[h][u] += __shfl_xor_sync(0xffffffffu, sc[h][u], off);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool valid = base + u * KPW + kg < k_end;
#pragma unroll
      for (int h = 0; h < HG; ++h)
        if (!valid) sc[h][u] = -INFINITY;
    }
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      float cm = sc[h][0];
#pragma unroll
      for (int u = 1; u < U; ++u) cm = fmaxf(cm, sc[h][u]);
#pragma unroll
      for (int off = LPK; off < 32; off *= 2) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
      const float m_new = fmaxf(m[h], cm);  // finite: every chunk holds a valid key
      const float f = fast_exp2(m[h] - m_new);
      m[h] = m_new;
      l[h] *= f;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[h][e] *= f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float p = fast_exp2(sc[h][u] - m_new);
        l[h] += p;
        float vf[8];
        bf16x8_to_f32(vr[u], vf);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] = fmaf(p, vf[e], o[h][e]);
      }
    }
  };

  constexpr int W = kDecodeWarps;
  if (warp < n_chunks) load_chunk(warp, ka, va);
  for (int ci = warp; ci < n_chunks; ci += 2 * W) {
    if (ci + W < n_chunks) load_chunk(ci + W, kb, vb);
    consume(ci, ka, va);
    if (ci + W >= n_chunks) break;
    if (ci + 2 * W < n_chunks) load_chunk(ci + 2 * W, ka, va);
    consume(ci + W, kb, vb);
  }

  // combine the KPW key groups of the warp (same d slice, different keys)
#pragma unroll
  for (int h = 0; h < HG; ++h) {
#pragma unroll
    for (int off = LPK; off < 32; off *= 2) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], off);
    }
  }

  // combine the warps through shared memory
  __shared__ float sm_m[kDecodeWarps][HG], sm_l[kDecodeWarps][HG];
  __shared__ float sm_o[kDecodeWarps][HG][D];
  if (lane < LPK) {
#pragma unroll
    for (int h = 0; h < HG; ++h) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sm_o[warp][h][dl * 8 + e] = o[h][e];
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      sm_m[warp][h] = m[h];
      sm_l[warp][h] = l[h];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < HG * D; idx += blockDim.x) {
    const int h = idx / D, e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int wi = 0; wi < kDecodeWarps; ++wi) M = fmaxf(M, sm_m[wi][h]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int wi = 0; wi < kDecodeWarps; ++wi) {
        const float f = fast_exp2(sm_m[wi][h] - M);  // 0 for warps without keys
        num += f * sm_o[wi][h][e];
        den += f * sm_l[wi][h];
      }
    }
    const int hq = hq0 + h;
    if (a.splits == 1) {
      a.out[((size_t)b * a.Hq + hq) * D + e] = __float2bfloat16_rn(num / den);
    } else {
      const size_t pi = ((size_t)b * a.Hq + hq) * a.splits + split;
      a.part_o[pi * D + e] = num;
      if (e == 0) a.part_ml[pi] = make_float2(M, den);
    }
  }
}

// Merge the per-split partial results: one CTA per (b, hq), one thread per d.
template <int D>
__global__ void __launch_bounds__(D) swa_decode_combine_kernel(const float *__restrict__ part_o,
                                                               const float2 *__restrict__ part_ml,
                                                               __nv_bfloat16 *__restrict__ out,
                                                               int splits) {
  const size_t bh = blockIdx.x;
  const int e = threadIdx.x;
  float M = -INFINITY;
  for (int i = 0; i < splits; ++i) M = fmaxf(M, part_ml[bh * splits + i].x);
  float num = 0.f, den = 0.f;
  for (int i = 0; i < splits; ++i) {
    const float2 ml = part_ml[bh * splits + i];
    if (ml.y > 0.f) {
      const float f = fast_exp2(ml.x - M);
      num += f * part_o[(bh * splits + i) * D + e];
      den += f * ml.y;
    }
  }
  out[bh * D + e] = __float2bfloat16_rn(num / den);
}

// ---------------------------------------------------------------- key-mask export

// One CTA per query row: replays the prefill tile schedule and in-tile mask of
// that row's query block and records every admitted (row, key) pair.
__global__ void swa_keymask_kernel(PrefillPlan plan, int L, int w, int s, int row0, int nrows,
                                   uint32_t *bits, int *counts) {
  const int r = blockIdx.x;
  if (r >= nrows) return;
  const int t = row0 + r;
  const int words = cdiv(L, 32);
  uint32_t *row_bits = bits + (size_t)r * words;
  for (int i = threadIdx.x; i < words; i += blockDim.x) row_bits[i] = 0u;
  __shared__ int cnt;
  if (threadIdx.x == 0) cnt = 0;
  __syncthreads();
  const int qb = t / plan.Tq;
  const BlockTiles bt = block_tiles(plan, qb, L, w, s);
  int local = 0;
  for (int i = 0; i < bt.n_tiles; ++i) {
    const Tile tl = tile_at(plan, bt, i, w, s);
    // the same column ranges the prefill softmax keeps unmasked
    const ColRanges cr = tile_ranges(tl, t, w, s);
    for (int c = threadIdx.x; c < tl.ncols; c += blockDim.x) {
      const int j = tile_key(tl, c);
      const bool ok = tl.full || (c >= cr.a_lo && c < cr.a_hi) || (c >= cr.b_lo && c < cr.b_hi);
      if (ok && j >= 0 && j < L) {
        atomicOr(&row_bits[j / 32], 1u << (j % 32));
        ++local;
      }
    }
  }
  atomicAdd(&cnt, local);
  __syncthreads();
  if (threadIdx.x == 0) counts[r] = cnt;
}

}  // namespace swa
