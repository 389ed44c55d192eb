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
// split): the query heads sharing the KV head are packed, so every K/V row is
// read from memory once for all of them. Each warp stages its own run of the
// CTA's slots (at most kDecodeMaxKeys per CTA) with bulk asynchronous copies
// issued at the start, so all of the CTA's bytes are in flight at once, and
// computes on its rows as soon as they land.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sm100_ptx.cuh"
#include "swa_index.cuh"

namespace swa {

// ---------------------------------------------------------------- append

// Only the tokens that survive the call are visited: token i (position
// p0 + i) survives iff p0 + i < s (a sink) or i >= T - w (among the last w).
// Survivor k of sequence b is token k if k < h, else token max(h, T - w) + k - h,
// where h = clamp(s - p0, 0, T); there are at most min(T, s + w) of them.
// One thread moves 16 bytes of K and 16 bytes of V of one (b, survivor, kvh).
__global__ void swa_append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                  uint4 *__restrict__ kcache, uint4 *__restrict__ vcache,
                                  const int *__restrict__ pos_start, int T, int Hkv, int d, int w,
                                  int s, int max_survivors) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.y;
  const int vec_per_row = d / 8;
  const long long n = (long long)max_survivors * Hkv * vec_per_row;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n) return;
  const int c = (int)(idx % vec_per_row);
  const int kvh = (int)((idx / vec_per_row) % Hkv);
  const int k = (int)(idx / ((long long)vec_per_row * Hkv));
  const int p0 = pos_start[b];
  if (p0 < 0) {
    if (idx == 0) record_error(kErrNegativePosition);
    return;
  }
  const int h = imin(imax(s - p0, 0), T);       // survivors at the front (sinks)
  const int tail0 = imax(h, T - w);             // first survivor of the tail
  const int i = k < h ? k : tail0 + (k - h);    // token index
  if (i >= T) return;
  const long long p = (long long)p0 + i;
  const long long slot = ring_slot(p, w, s);
  const long long src = (((long long)b * T + i) * Hkv + kvh) * vec_per_row + c;
  const long long dst = (((long long)b * Hkv + kvh) * (s + w) + slot) * vec_per_row + c;
  kcache[dst] = k_new[src];
  vcache[dst] = v_new[src];
}

// Paged form of the append: the same survivors, written to row p % page_size
// of the physical page table[b][p / page_size] of the pools
// [n_pages, Hkv, page_size, d]. An unmapped (or out-of-range) page is skipped
// and flagged.
__global__ void swa_paged_append_kernel(const uint4 *__restrict__ k_new,
                                        const uint4 *__restrict__ v_new, uint4 *__restrict__ kpool,
                                        uint4 *__restrict__ vpool, const int *__restrict__ table,
                                        const int *__restrict__ pos_start, int T, int Hkv, int d,
                                        int w, int s, int max_survivors, int page_size,
                                        int max_pages, int n_pages) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.y;
  const int vec_per_row = d / 8;
  const long long n = (long long)max_survivors * Hkv * vec_per_row;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n) return;
  const int c = (int)(idx % vec_per_row);
  const int kvh = (int)((idx / vec_per_row) % Hkv);
  const int k = (int)(idx / ((long long)vec_per_row * Hkv));
  const int p0 = pos_start[b];
  if (p0 < 0) {
    if (idx == 0) record_error(kErrNegativePosition);
    return;
  }
  const int h = imin(imax(s - p0, 0), T);
  const int tail0 = imax(h, T - w);
  const int i = k < h ? k : tail0 + (k - h);
  if (i >= T) return;
  const long long p = (long long)p0 + i;
  const long long lp = p / page_size;
  const int page = lp < max_pages ? table[(long long)b * max_pages + lp] : -1;
  if (page < 0 || page >= n_pages) {
    record_error(kErrMissingPage);
    return;
  }
  const long long src = (((long long)b * T + i) * Hkv + kvh) * vec_per_row + c;
  const long long dst =
      (((long long)page * Hkv + kvh) * page_size + p % page_size) * vec_per_row + c;
  kpool[dst] = k_new[src];
  vpool[dst] = v_new[src];
}

// ---------------------------------------------------------------- decode

constexpr int kDecodeThreads = 128;
constexpr int kDecodeMaxKeys = 256;   // slots one CTA stages (128 KB of K+V at d = 128)
constexpr int kDecodeMaxHeads = 4;    // query heads one CTA packs
constexpr uint64_t kDecodeWaitNs = 2000000000ull;   // bounded wait for the staged data
constexpr uint64_t kDecodeDrainNs = 200000000ull;   // bounded drain on the failure path

// Bulk asynchronous copy global -> shared of `bytes` (a multiple of 16, both
// addresses 16-byte aligned), completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

struct DecodeArgs {
  const __nv_bfloat16 *q;
  const __nv_bfloat16 *kc;
  const __nv_bfloat16 *vc;
  const __nv_bfloat16 *k_new;  // [B, Hkv, D] token appended at pos[b] first (or null)
  const __nv_bfloat16 *v_new;
  __nv_bfloat16 *kc_w;         // the caches, writable (used with k_new)
  __nv_bfloat16 *vc_w;
  const int *pos;
  __nv_bfloat16 *out;
  float *part_o;     // [B, Hq, splits, D] when splits > 1
  float2 *part_ml;   // [B, Hq, splits] (running max in log2 units, sum)
  int Hq, Hkv, w, s, splits;
  int max_keys;      // slots one CTA stages at most (sizes its shared memory)
  float scale_log2;
  // paged layout (kc/vc are then the page pools [n_pages, Hkv, page_size, D])
  const int *page_table;  // [B, max_pages]
  int page_size, max_pages, n_pages;
  // bounded waits: the limit of each wait for staged data; stall != 0 (test
  // aid) issues no copy at all, so every wait runs out and the kernel must
  // leave through its failure path
  uint64_t wait_ns;
  int stall;
};

constexpr int kDecodeChunk = kDecodeMaxKeys;  // keys per chunk: one chunk per CTA
constexpr int kDecodeMaxChunks = kDecodeMaxKeys / kDecodeChunk;

// Dynamic shared memory of one decode CTA.
template <int D, int HG>
struct DecodeSmem {
  static size_t bytes(int max_keys) {
    return 128 /* alignment */ + 256 /* barriers */ + 2 * (size_t)max_keys * D * 2 +
           2 * (size_t)(max_keys < kDecodeChunk ? max_keys : kDecodeChunk) * HG * 4 /* P */ +
           3 * HG * 4 + 16 +
           (size_t)kDecodeThreads * HG * 8;
  }
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<uint64_t *>(&a)), "l"(*reinterpret_cast<uint64_t *>(&b)),
        "l"(*reinterpret_cast<uint64_t *>(&c)));
  return *reinterpret_cast<float2 *>(&r);
}

// two bf16 (low half first) -> two floats
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// HG query heads per CTA (a divisor of G, at most 4); D = head dimension.
//
// The CTA's slots are consumed in chunks of kDecodeChunk keys (the K and V of
// every chunk requested at once, one bulk copy each with its own barrier) with
// an online softmax across chunks; with kDecodeChunk = kDecodeMaxKeys a CTA
// has a single chunk, K first and V second, so the scores start while V is
// still arriving.
//
// kPaged: the cache is paged. The CTA's keys are then the positions of K(pos)
// in order (the sinks, then pos - w + 1 .. pos), and each run of them inside
// one page is one bulk copy; key order does not change the result.
//
// Failure path: a wait that runs out (bounded by a.wait_ns) records
// kErrWaitTimeout; the CTA then skips the rest of the arithmetic, waits
// (bounded, not abortable) for the copies it issued, and exits without writing
// anything. A stalled test launch (a.stall) issues no copy, so its waits run
// out.
template <int D, int HG, bool kPaged>
__global__ void __launch_bounds__(kDecodeThreads) swa_decode_kernel(const DecodeArgs a) {
  constexpr int LPK = 8;            // lanes per key row in the score phase
  constexpr int EPL = D / LPK;      // elements of a row per lane (16 or 8)
  constexpr int kPairs = D / 2;     // column pairs of a row
  constexpr int kParts = kDecodeThreads / kPairs;  // key parts in the P V phase
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *dsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 127) &
                                             ~uintptr_t(127));
  uint64_t *bar_k = reinterpret_cast<uint64_t *>(dsm);                  // [kDecodeMaxChunks]
  uint64_t *bar_v = bar_k + kDecodeMaxChunks;                           // [kDecodeMaxChunks]
  __nv_bfloat16 *sK = reinterpret_cast<__nv_bfloat16 *>(dsm + 256);     // [max_keys][D]
  __nv_bfloat16 *sV = sK + (size_t)a.max_keys * D;                       // [max_keys][D]
  const int pchunk = imin(kDecodeChunk, a.max_keys);                  // keys of a P buffer
  float *sP = reinterpret_cast<float *>(sV + (size_t)a.max_keys * D);  // [2][pchunk][HG]
  float *sM = sP + 2 * pchunk * HG;                                    // [HG] running max
  float *sL = sM + HG;                                                 // [HG] running sum
  float *sF = sL + HG;                                                 // [HG] rescale factor
  float2 *sO = reinterpret_cast<float2 *>(                             // [kParts][HG][kPairs]
      (reinterpret_cast<uintptr_t>(sF + HG) + 15) & ~uintptr_t(15));
  __shared__ int abort_word;
  __shared__ int missing_page;

  const int split = blockIdx.x;
  const int G = a.Hq / a.Hkv;
  const int hgroups = G / HG;
  const int kvh = blockIdx.y / hgroups;
  const int hg = blockIdx.y % hgroups;
  const int b = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int hq0 = kvh * G + hg * HG;

  grid_launch_dependents();
  grid_dependency_wait();
  const int pos = a.pos[b];
  if (pos < 0) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) record_error(kErrNegativePosition);
    return;
  }
  const int n = ring_valid(pos, a.w, a.s);
  const int per_split = cdiv(n, a.splits);
  const int k_begin = imin(n, split * per_split);
  const int nk = imin(n, k_begin + per_split) - k_begin;  // <= max_keys
  const int n_chunks = cdiv(nk, kDecodeChunk);
  // With k_new: the token at position pos goes to ring slot(pos). Every CTA
  // that stages that slot patches its shared-memory copy; the first head
  // group's CTA also writes it to the cache.
  int append_row = -1;
  if (a.k_new != nullptr) {
    const int slot = (int)ring_slot(pos, a.w, a.s);
    if (slot >= k_begin && slot < k_begin + nk) {
      append_row = slot - k_begin;
      if (hg == 0 && threadIdx.x < D / 4) {
        const size_t src = ((size_t)b * a.Hkv + kvh) * D;
        const size_t dst = (((size_t)b * a.Hkv + kvh) * (size_t)(a.s + a.w) + slot) * D;
        const int u = threadIdx.x % (D / 8);
        if (threadIdx.x < D / 8)
          reinterpret_cast<uint4 *>(a.kc_w + dst)[u] = reinterpret_cast<const uint4 *>(a.k_new + src)[u];
        else
          reinterpret_cast<uint4 *>(a.vc_w + dst)[u] = reinterpret_cast<const uint4 *>(a.v_new + src)[u];
      }
    }
  }

  const size_t row_base = ((size_t)b * a.Hkv + kvh) * (size_t)(a.s + a.w) + k_begin;
  if (threadIdx.x == 0) {
    abort_word = 0;
    missing_page = 0;
    for (int c = 0; c < n_chunks; ++c) {
      mbar_init(&bar_k[c], 1);
      mbar_init(&bar_v[c], 1);
    }
    fence_mbar_init();
  }
  if constexpr (kPaged) {
    // keys k_begin .. k_begin + nk - 1 of the list [sinks | window] (one chunk:
    // nk <= kDecodeMaxKeys); every page is checked before any copy is issued
    if (threadIdx.x == 0 && nk > 0 && !a.stall) {
      const int ns = imin(a.s, pos + 1);              // sink positions held
      const long long lo = imax(a.s, pos - a.w + 1);  // first window position
      const int *tbl = a.page_table + (size_t)b * a.max_pages;
      for (int pass = 0; pass < 2 && !missing_page; ++pass) {
        if (pass == 1) {
          mbar_arrive_expect_tx(&bar_k[0], (uint32_t)nk * D * 2);
          mbar_arrive_expect_tx(&bar_v[0], (uint32_t)nk * D * 2);
        }
        for (int i = k_begin; i < k_begin + nk;) {
          const long long p = i < ns ? i : lo + (i - ns);
          const int seg_end = i < ns ? imin(k_begin + nk, ns) : k_begin + nk;
          const long long lp = p / a.page_size;
          const int row = (int)(p % a.page_size);
          const int len = imin(seg_end - i, a.page_size - row);
          const int page = lp < a.max_pages ? tbl[lp] : -1;
          if (page < 0 || page >= a.n_pages) {
            missing_page = 1;
            record_error(kErrMissingPage);
            break;
          }
          if (pass == 1) {
            const size_t src = (((size_t)page * a.Hkv + kvh) * a.page_size + row) * D;
            const uint32_t bytes = (uint32_t)len * D * 2;
            bulk_load(sK + (size_t)(i - k_begin) * D, a.kc + src, bytes, &bar_k[0]);
            bulk_load(sV + (size_t)(i - k_begin) * D, a.vc + src, bytes, &bar_v[0]);
          }
          i += len;
        }
      }
    }
  } else if (threadIdx.x == 0 && !a.stall) {
    // every chunk's K first, then every chunk's V: the scores need K first
    for (int c = 0; c < n_chunks; ++c) {
      const int kc = imin(kDecodeChunk, nk - c * kDecodeChunk);
      const uint32_t bytes = (uint32_t)kc * D * 2;
      mbar_arrive_expect_tx(&bar_k[c], bytes);
      bulk_load(sK + (size_t)c * kDecodeChunk * D, a.kc + (row_base + c * kDecodeChunk) * D,
                bytes, &bar_k[c]);
    }
    for (int c = 0; c < n_chunks; ++c) {
      const int kc = imin(kDecodeChunk, nk - c * kDecodeChunk);
      const uint32_t bytes = (uint32_t)kc * D * 2;
      mbar_arrive_expect_tx(&bar_v[c], bytes);
      bulk_load(sV + (size_t)c * kDecodeChunk * D, a.vc + (row_base + c * kDecodeChunk) * D,
                bytes, &bar_v[c]);
    }
  }
  if (threadIdx.x < HG) {
    sM[threadIdx.x] = -INFINITY;
    sL[threadIdx.x] = 0.f;
  }
  // queries of the HG heads, this lane's slice as pairs, pre-scaled to log2 units
  const int kg = lane / LPK;   // which of the 4 keys of a warp step
  const int dl = lane % LPK;   // which slice of d
  float2 q2[HG][EPL / 2];
#pragma unroll
  for (int h = 0; h < HG; ++h) {
#pragma unroll
    for (int v = 0; v < EPL / 8; ++v) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(a.q + ((size_t)b * a.Hq + hq0 + h) * D +
                                                         dl * EPL + v * 8);
      const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = bf16x2_to_f2(wd[e]);
        q2[h][v * 4 + e] = make_float2(f.x * a.scale_log2, f.y * a.scale_log2);
      }
    }
  }
  const int cp = threadIdx.x % kPairs, part = threadIdx.x / kPairs;  // P V phase mapping
  float2 o2[HG];
#pragma unroll
  for (int h = 0; h < HG; ++h) o2[h] = make_float2(0.f, 0.f);
  __syncthreads();  // barriers initialised
  if (kPaged && missing_page) return;  // nothing was copied
  // chunks whose copies thread 0 has seen land, and whether a wait ran out
  int landed = 0;
  bool failed = false;

  for (int c = 0; c < n_chunks; ++c) {
    const int j_base = c * kDecodeChunk;
    const int kc = imin(kDecodeChunk, nk - j_base);
    float *sPc = sP + (c & 1) * pchunk * HG;  // [pchunk][HG]
    // one thread polls the barrier; the others sleep in __syncthreads (which
    // also tells every thread whether the wait ran out)
    failed = __syncthreads_or(threadIdx.x == 0 && !mbar_wait(&bar_k[c], 0, &abort_word, a.wait_ns));
    if (failed) break;
    if (append_row >= j_base && append_row < j_base + kc) {
      // the appended token's slot: its staged row still holds the old entry
      if (threadIdx.x < D / 8)
        reinterpret_cast<uint4 *>(sK + (size_t)append_row * D)[threadIdx.x] =
            reinterpret_cast<const uint4 *>(a.k_new + ((size_t)b * a.Hkv + kvh) * D)[threadIdx.x];
      __syncthreads();
    }
    // ---- scores of the chunk: each warp step covers 4 keys, 8 lanes per key
    for (int j0 = warp * 4; j0 < kc; j0 += 4 * (kDecodeThreads / 32)) {
      const int j = j0 + kg;
      float2 acc2[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) acc2[h] = make_float2(0.f, 0.f);
      if (j < kc) {
#pragma unroll
        for (int v = 0; v < EPL / 8; ++v) {
          const uint4 raw =
              *reinterpret_cast<const uint4 *>(sK + (size_t)(j_base + j) * D + dl * EPL + v * 8);
          const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kf = bf16x2_to_f2(wd[e]);
#pragma unroll
            for (int h = 0; h < HG; ++h) acc2[h] = ffma2(q2[h][v * 4 + e], kf, acc2[h]);
          }
        }
      }
      float acc[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) acc[h] = acc2[h].x + acc2[h].y;
#pragma unroll
      for (int off = LPK / 2; off >= 1; off /= 2)
#pragma unroll
        for (int h = 0; h < HG; ++h) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], off);
      if (dl == 0 && j < kc) {
#pragma unroll
        for (int h = 0; h < HG; ++h) sPc[j * HG + h] = acc[h];
      }
    }
    __syncthreads();
    // ---- online softmax update of each head (warp h)
    if (warp < HG) {
      float mc = -INFINITY;
      for (int j = lane; j < kc; j += 32) mc = fmaxf(mc, sPc[j * HG + warp]);
#pragma unroll
      for (int off = 16; off >= 1; off /= 2) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
      const float m_old = sM[warp];
      const float m_new = fmaxf(m_old, mc);
      float ls = 0.f;
      for (int j = lane; j < kc; j += 32) {
        const float p = fast_exp2(sPc[j * HG + warp] - m_new);
        sPc[j * HG + warp] = p;
        ls += p;
      }
#pragma unroll
      for (int off = 16; off >= 1; off /= 2) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      if (lane == 0) {
        const float f = m_old == -INFINITY ? 0.f : fast_exp2(m_old - m_new);
        sF[warp] = f;
        sM[warp] = m_new;
        sL[warp] = sL[warp] * f + ls;
      }
    }
    failed = __syncthreads_or(threadIdx.x == 0 && !mbar_wait(&bar_v[c], 0, &abort_word, a.wait_ns));
    if (failed) break;
    landed = c + 1;
    if (append_row >= j_base && append_row < j_base + kc) {
      if (threadIdx.x < D / 8)
        reinterpret_cast<uint4 *>(sV + (size_t)append_row * D)[threadIdx.x] =
            reinterpret_cast<const uint4 *>(a.v_new + ((size_t)b * a.Hkv + kvh) * D)[threadIdx.x];
      __syncthreads();
    }
    // ---- O = O * f + P V over the chunk: thread = (column pair, key part);
    // one V pair feeds all HG heads (consecutive threads: consecutive pairs)
    {
      float f[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) f[h] = sF[h];
#pragma unroll
      for (int h = 0; h < HG; ++h) o2[h] = make_float2(o2[h].x * f[h], o2[h].y * f[h]);
      const int per_part = cdiv(kc, kParts);
      const int j_lo = imin(kc, part * per_part), j_hi = imin(kc, j_lo + per_part);
      const uint32_t *vcol = reinterpret_cast<const uint32_t *>(sV + (size_t)j_base * D) + cp;
      for (int j = j_lo; j < j_hi; ++j) {
        const float2 vf = bf16x2_to_f2(vcol[(size_t)j * kPairs]);
        float pr[HG];
        if constexpr (HG == 4) {
          const float4 p4 = *reinterpret_cast<const float4 *>(sPc + j * 4);
          pr[0] = p4.x; pr[1] = p4.y; pr[2] = p4.z; pr[3] = p4.w;
        } else {
#pragma unroll
          for (int h = 0; h < HG; ++h) pr[h] = sPc[j * HG + h];
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) o2[h] = ffma2(make_float2(pr[h], pr[h]), vf, o2[h]);
      }
    }
    // the next chunk writes the other P buffer; the one after that reuses
    // this one only after the next chunk's barrier
  }
  if (failed || a.stall) {
    // failure path: every copy issued lands before the CTA exits (bounded, not
    // abortable), and nothing is written
    if (threadIdx.x == 0 && !a.stall) {
      for (int c = landed; c < n_chunks; ++c) {
        mbar_wait(&bar_k[c], 0, &abort_word, kDecodeDrainNs, false);
        mbar_wait(&bar_v[c], 0, &abort_word, kDecodeDrainNs, false);
      }
    }
    return;
  }
#pragma unroll
  for (int h = 0; h < HG; ++h) sO[(part * HG + h) * kPairs + cp] = o2[h];
  __syncthreads();
  for (int item = threadIdx.x; item < HG * kPairs; item += kDecodeThreads) {
    const int h = item / kPairs, cq = item % kPairs;
    float2 o = sO[h * kPairs + cq];
#pragma unroll
    for (int pp = 1; pp < kParts; ++pp) {
      const float2 x = sO[(pp * HG + h) * kPairs + cq];
      o.x += x.x;
      o.y += x.y;
    }
    const int hq = hq0 + h;
    if (a.splits == 1) {
      const float inv = 1.0f / sL[h];
      reinterpret_cast<uint32_t *>(a.out + ((size_t)b * a.Hq + hq) * D)[cq] =
          pack_bf16x2(o.x * inv, o.y * inv);
    } else {
      const size_t pi = ((size_t)b * a.Hq + hq) * a.splits + split;
      reinterpret_cast<float2 *>(a.part_o + pi * D)[cq] = o;
      if (cq == 0) a.part_ml[pi] = nk > 0 ? make_float2(sM[h], sL[h]) : make_float2(-INFINITY, 0.f);
    }
  }
}

// Merge the per-split partial results of one (b, hq) per CTA, as the
// log-sum-exp combine of split-KV decoding does:
//   out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i,   M = max_i m_i,
// over the splits i holding keys (l_i > 0). The splits' weights are computed
// once per chunk of kCombineChunk splits into shared memory; the partial rows
// are then summed by kCombineThreads / (D / 4) thread groups, each reading one
// whole row as float4 columns, so many independent loads are in flight.
constexpr int kCombineThreads = 256;
constexpr int kCombineChunk = 1024;

__device__ __forceinline__ float block_reduce_256(float v, float *s_red, bool is_max) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
#pragma unroll
  for (int off = 16; off >= 1; off /= 2) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float r = s_red[0];
#pragma unroll
  for (int i = 1; i < kCombineThreads / 32; ++i) r = is_max ? fmaxf(r, s_red[i]) : r + s_red[i];
  __syncthreads();  // s_red may be written again
  return r;
}

template <int D>
__global__ void __launch_bounds__(kCombineThreads) swa_decode_combine_kernel(
    const float *__restrict__ part_o, const float2 *__restrict__ part_ml,
    __nv_bfloat16 *__restrict__ out, int splits) {
  constexpr int kCols = D / 4;                      // float4 columns of a row
  constexpr int kGroups = kCombineThreads / kCols;  // rows summed side by side
  __shared__ float s_f[kCombineChunk];
  __shared__ float s_red[kCombineThreads / 32];
  __shared__ float4 s_part[kGroups][kCols];
  grid_launch_dependents();
  grid_dependency_wait();
  const size_t bh = blockIdx.x;
  const float2 *ml = part_ml + bh * splits;
  const float4 *po = reinterpret_cast<const float4 *>(part_o + bh * splits * D);
  const int tid = threadIdx.x;
  float M = -INFINITY;
  for (int i = tid; i < splits; i += kCombineThreads) M = fmaxf(M, ml[i].x);
  M = block_reduce_256(M, s_red, true);
  const int c4 = tid % kCols, grp = tid / kCols;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int c0 = 0; c0 < splits; c0 += kCombineChunk) {
    const int n = imin(kCombineChunk, splits - c0);
    for (int i = tid; i < n; i += kCombineThreads) {
      const float2 x = ml[c0 + i];
      const float f = x.y > 0.f ? fast_exp2(x.x - M) : 0.f;
      s_f[i] = f;
      den = fmaf(f, x.y, den);
    }
    __syncthreads();
#pragma unroll 4
    for (int i = grp; i < n; i += kGroups) {
      const float f = s_f[i];
      // a split without keys is not read (its partial row carries no weight)
      const float4 x = f != 0.f ? po[(size_t)(c0 + i) * kCols + c4] : make_float4(0.f, 0.f, 0.f, 0.f);
      acc.x = fmaf(f, x.x, acc.x);
      acc.y = fmaf(f, x.y, acc.y);
      acc.z = fmaf(f, x.z, acc.z);
      acc.w = fmaf(f, x.w, acc.w);
    }
    __syncthreads();  // s_f is rewritten by the next chunk
  }
  den = block_reduce_256(den, s_red, false);
  s_part[grp][c4] = acc;
  __syncthreads();
  if (tid < kCols) {
    float4 o = s_part[0][tid];
#pragma unroll
    for (int g = 1; g < kGroups; ++g) {
      const float4 x = s_part[g][tid];
      o.x += x.x;
      o.y += x.y;
      o.z += x.z;
      o.w += x.w;
    }
    reinterpret_cast<uint2 *>(out + bh * D)[tid] =
        make_uint2(pack_bf16x2(o.x / den, o.y / den), pack_bf16x2(o.z / den, o.w / den));
  }
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
  // a pair item starts at the even block (a whole prompt: no blocks skipped)
  const BlockTiles bt = block_tiles(plan, plan.bpi == 2 ? (qb & ~1) : qb, L, w, s);
  int local = 0;
  for (int i = 0; i < bt.n_tiles; ++i) {
    const Tile tl = tile_at(plan, bt, i, w, s);
    // the same column ranges the prefill softmax keeps unmasked
    const bool full = tile_full_for(tl, qb * plan.Tq, plan.Tq, w);
    const ColRanges cr = tile_ranges(tl, t, w, s);
    for (int c = threadIdx.x; c < tl.ncols; c += blockDim.x) {
      const int j = tile_key(tl, c);
      const bool ok = full || (c >= cr.a_lo && c < cr.a_hi) || (c >= cr.b_lo && c < cr.b_hi);
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
