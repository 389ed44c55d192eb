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
constexpr int kDecodeWarps = kDecodeThreads / 32;
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

// Dynamic shared memory of one decode CTA:
//   barriers   K and V barrier of each warp
//   sK, sV     [max_keys][D] bf16 staged rows
//   sS         [max_keys][HG] fp32 scores (unscaled)
//   sP         [max_keys][HG] float2 (p, p): the weight twice, so that the
//              value product takes a ready operand pair
//   sO         [warps][HG][D] fp32 partial outputs
//   sQ         [HG][D] fp32 query rows
//   sML        [warps][HG] float2 (max, sum)
// (every region starts on a 16-byte boundary)
template <int D, int HG>
struct DecodeSmem {
  static constexpr size_t kBar = 128;
  __host__ __device__ static constexpr size_t up16(size_t x) { return (x + 15) & ~size_t(15); }
  __host__ __device__ static size_t k_off() { return kBar; }
  __host__ __device__ static size_t v_off(int mk) { return k_off() + up16((size_t)mk * D * 2); }
  __host__ __device__ static size_t s_off(int mk) { return v_off(mk) + up16((size_t)mk * D * 2); }
  __host__ __device__ static size_t p_off(int mk) { return s_off(mk) + up16((size_t)mk * HG * 4); }
  __host__ __device__ static size_t o_off(int mk) { return p_off(mk) + up16((size_t)mk * HG * 8); }
  __host__ __device__ static size_t q_off(int mk) { return o_off(mk) + up16((size_t)kDecodeWarps * HG * D * 4); }
  __host__ __device__ static size_t ml_off(int mk) { return q_off(mk) + up16((size_t)HG * D * 4); }
  __host__ __device__ static size_t bytes(int mk) { return 128 /* alignment */ + ml_off(mk) + kDecodeWarps * HG * 8; }
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

// Issue the bulk copies of one warp's keys [j_lo, j_hi) (keys numbered from
// the CTA's first key k_begin; paged: the positions of K(pos) in order, the
// sinks then pos - w + 1 .. pos, one copy per run inside a page). Returns
// false, with nothing issued, when a page is unmapped or out of range.
template <int D, bool kPaged>
__device__ __forceinline__ bool decode_issue(const DecodeArgs &a, int b, int kvh, int pos,
                                             int k_begin, int j_lo, int j_hi,
                                             __nv_bfloat16 *sK, __nv_bfloat16 *sV,
                                             uint64_t *bar_k, uint64_t *bar_v) {
  const uint32_t bytes = (uint32_t)(j_hi - j_lo) * D * 2;
  if constexpr (kPaged) {
    const int ns = imin(a.s, pos + 1);              // sink positions held
    const long long lo = imax(a.s, pos - a.w + 1);  // first window position
    const int *tbl = a.page_table + (size_t)b * a.max_pages;
    for (int pass = 0; pass < 2; ++pass) {          // check every page, then copy
      if (pass == 1) {
        mbar_arrive_expect_tx(bar_k, bytes);
        mbar_arrive_expect_tx(bar_v, bytes);
      }
      for (int i = k_begin + j_lo; i < k_begin + j_hi;) {
        const long long p = i < ns ? i : lo + (i - ns);
        const int seg_end = i < ns ? imin(k_begin + j_hi, ns) : k_begin + j_hi;
        const long long lp = p / a.page_size;
        const int row = (int)(p % a.page_size);
        const int len = imin(seg_end - i, a.page_size - row);
        const int page = lp < a.max_pages ? tbl[lp] : -1;
        if (page < 0 || page >= a.n_pages) return false;
        if (pass == 1) {
          const size_t src = (((size_t)page * a.Hkv + kvh) * a.page_size + row) * D;
          const size_t dst = (size_t)(i - k_begin) * D;
          bulk_load(sK + dst, a.kc + src, (uint32_t)len * D * 2, bar_k);
          bulk_load(sV + dst, a.vc + src, (uint32_t)len * D * 2, bar_v);
        }
        i += len;
      }
    }
  } else {
    const size_t row0 = ((size_t)b * a.Hkv + kvh) * (size_t)(a.s + a.w) + k_begin + j_lo;
    mbar_arrive_expect_tx(bar_k, bytes);
    bulk_load(sK + (size_t)j_lo * D, a.kc + row0 * D, bytes, bar_k);
    mbar_arrive_expect_tx(bar_v, bytes);
    bulk_load(sV + (size_t)j_lo * D, a.vc + row0 * D, bytes, bar_v);
  }
  return true;
}

// HG query heads per CTA (a divisor of G, at most 4); D = head dimension.
//
// One CTA (4 warps) serves one (sequence, KV head, head group, split). Its
// keys are cut into four contiguous runs, one per warp (in whole groups of 4
// keys). Each warp stages its own run of K and of V with one bulk copy each
// (its own barriers), so it starts as soon as its rows land, and computes, with
// no block-wide barrier, its scores (8 lanes per key, 16 elements of d each,
// all HG heads at once: every K element is read and converted once for the
// group), the softmax of its keys and its share of P V (each lane 4 columns of
// d for all HG heads). The four partial results (max, sum, O) are merged at the
// end, or, when the cache is split over CTAs, written as one partial per split
// for the combine kernel.
//
// Failure path: a wait that runs out records kErrWaitTimeout and sets the
// CTA's abort word; a paged CTA that meets an unmapped page records
// kErrMissingPage. Then every warp skips its arithmetic, the CTA waits
// (bounded, not abortable) for the copies it issued, and exits without
// writing any output.
//
// kPaged: the cache is paged (see decode_issue); key order does not change
// the result.
template <int D, int HG, bool kPaged>
__global__ void __launch_bounds__(kDecodeThreads, 4) swa_decode_kernel(const DecodeArgs a) {
  constexpr int LPK = 8;            // lanes per key row in the score phase
  constexpr int EPL = D / LPK;      // elements of a row per lane (16 or 8)
  constexpr int CPL = D / 32;       // output columns per lane in the value phase (4 or 2)
  using Smem = DecodeSmem<D, HG>;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t *dsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 127) &
                                             ~uintptr_t(127));
  const int mk = a.max_keys;
  uint64_t *bar_k = reinterpret_cast<uint64_t *>(dsm);           // [warps]
  uint64_t *bar_v = bar_k + kDecodeWarps;                        // [warps]
  volatile int *abort_word = reinterpret_cast<volatile int *>(bar_v + kDecodeWarps);
  volatile int *page_fault = abort_word + 1;
  __nv_bfloat16 *sK = reinterpret_cast<__nv_bfloat16 *>(dsm + Smem::k_off());
  __nv_bfloat16 *sV = reinterpret_cast<__nv_bfloat16 *>(dsm + Smem::v_off(mk));
  float *sS = reinterpret_cast<float *>(dsm + Smem::s_off(mk));
  float2 *sP = reinterpret_cast<float2 *>(dsm + Smem::p_off(mk));
  float *sO = reinterpret_cast<float *>(dsm + Smem::o_off(mk));
  float *sQ = reinterpret_cast<float *>(dsm + Smem::q_off(mk));
  float2 *sML = reinterpret_cast<float2 *>(dsm + Smem::ml_off(mk));

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
  // this warp's run of keys: whole groups of 4, spread evenly over the warps
  const int ngroups = cdiv(nk, 4);
  const int j_lo = imin(nk, (warp * ngroups / kDecodeWarps) * 4);
  const int j_hi = imin(nk, ((warp + 1) * ngroups / kDecodeWarps) * 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecodeWarps; ++i) {
      mbar_init(&bar_k[i], 1);
      mbar_init(&bar_v[i], 1);
    }
    *abort_word = 0;
    *page_fault = 0;
    fence_mbar_init();
  }
  // the query rows of the HG heads (contiguous in q): kQWpt bf16 pairs per
  // thread are loaded now and converted once the copies are under way
  constexpr int kQWords = HG * D / 2;                                     // 32 .. 256
  constexpr int kQWpt = kQWords > kDecodeThreads ? kQWords / kDecodeThreads : 1;  // 1 or 2
  constexpr int kQThreads = kQWords / kQWpt;
  uint32_t qraw[2] = {0u, 0u};
  if (threadIdx.x < kQThreads) {
    const __nv_bfloat16 *qsrc = a.q + ((size_t)b * a.Hq + hq0) * D + threadIdx.x * kQWpt * 2;
    if constexpr (kQWpt == 2) {
      const uint2 u = *reinterpret_cast<const uint2 *>(qsrc);
      qraw[0] = u.x;
      qraw[1] = u.y;
    } else {
      qraw[0] = *reinterpret_cast<const uint32_t *>(qsrc);
    }
  }
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
  __syncthreads();  // barriers initialised

  // ---- stage: lane 0 of each warp copies the warp's run of K and of V
  int issued = 0;
  if (lane == 0 && j_hi > j_lo && !a.stall) {
    if (decode_issue<D, kPaged>(a, b, kvh, pos, k_begin, j_lo, j_hi, sK, sV, &bar_k[warp],
                                &bar_v[warp])) {
      issued = 1;
    } else {
      *page_fault = 1;
      record_error(kErrMissingPage);
    }
  }
  issued = __shfl_sync(0xffffffffu, issued, 0);
  // query rows -> fp32 in shared memory
  if (threadIdx.x < kQThreads) {
    float *qd = sQ + threadIdx.x * kQWpt * 2;
    if constexpr (kQWpt == 2) {
      const float2 f0 = bf16x2_to_f2(qraw[0]), f1 = bf16x2_to_f2(qraw[1]);
      *reinterpret_cast<float4 *>(qd) = make_float4(f0.x, f0.y, f1.x, f1.y);
    } else {
      *reinterpret_cast<float2 *>(qd) = bf16x2_to_f2(qraw[0]);
    }
  }
  __syncthreads();

  const bool mine = j_hi > j_lo && (issued || a.stall);  // this warp has rows coming
  float m_w = -INFINITY, l_w = 0.f;                      // head lane % HG, over my keys
  bool wrote_o = false;
  bool ok = mine;
  if (ok) {
    // every lane polls; the outcome is made warp-uniform
    ok = __all_sync(0xffffffffu, mbar_wait(&bar_k[warp], 0, abort_word, a.wait_ns));
  }
  if (ok) {
    const int kg = lane / LPK;   // which of the 4 keys of a warp step
    const int dl = lane % LPK;   // which slice of d
    if (append_row >= j_lo && append_row < j_hi && lane < D / 8) {
      // the appended token's slot: its staged row still holds the old entry
      reinterpret_cast<uint4 *>(sK + (size_t)append_row * D)[lane] =
          reinterpret_cast<const uint4 *>(a.k_new + ((size_t)b * a.Hkv + kvh) * D)[lane];
    }
    // this lane's slice of the HG query rows
    float2 q2[HG][EPL / 2];
#pragma unroll
    for (int h = 0; h < HG; ++h)
#pragma unroll
      for (int v = 0; v < EPL / 4; ++v) {
        const float4 f = *reinterpret_cast<const float4 *>(sQ + h * D + dl * EPL + v * 4);
        q2[h][2 * v] = make_float2(f.x, f.y);
        q2[h][2 * v + 1] = make_float2(f.z, f.w);
      }
    __syncwarp();
    // ---- scores: a warp step covers 4 keys, 8 lanes per key
    constexpr int kSpan = LPK / HG;  // lanes that end up holding one head's total
    for (int j0 = j_lo; j0 < j_hi; j0 += 4) {
      const int j = j0 + kg;
      float2 acc2[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) acc2[h] = make_float2(0.f, 0.f);
      if (j < j_hi) {
#pragma unroll
        for (int v = 0; v < EPL / 8; ++v) {
          const uint4 raw =
              *reinterpret_cast<const uint4 *>(sK + (size_t)j * D + dl * EPL + v * 8);
          const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kf = bf16x2_to_f2(wd[e]);
#pragma unroll
            for (int h = 0; h < HG; ++h) acc2[h] = ffma2(q2[h][v * 4 + e], kf, acc2[h]);
          }
        }
      }
      // reduce over the 8 lanes of the key, scattering the heads: lane dl ends
      // with the total of head dl / kSpan
      float tot;
      if constexpr (HG == 4) {
        const float a0 = acc2[0].x + acc2[0].y, a1 = acc2[1].x + acc2[1].y;
        const float a2 = acc2[2].x + acc2[2].y, a3 = acc2[3].x + acc2[3].y;
        const bool b2 = (dl & 4) != 0, b1 = (dl & 2) != 0;
        float k0 = b2 ? a2 : a0, k1 = b2 ? a3 : a1;
        const float s0 = b2 ? a0 : a2, s1 = b2 ? a1 : a3;
        k0 += __shfl_xor_sync(0xffffffffu, s0, 4);
        k1 += __shfl_xor_sync(0xffffffffu, s1, 4);
        tot = b1 ? k1 : k0;
        tot += __shfl_xor_sync(0xffffffffu, b1 ? k0 : k1, 2);
        tot += __shfl_xor_sync(0xffffffffu, tot, 1);
      } else if constexpr (HG == 2) {
        const float a0 = acc2[0].x + acc2[0].y, a1 = acc2[1].x + acc2[1].y;
        const bool b2 = (dl & 4) != 0;
        tot = b2 ? a1 : a0;
        tot += __shfl_xor_sync(0xffffffffu, b2 ? a0 : a1, 4);
        tot += __shfl_xor_sync(0xffffffffu, tot, 2);
        tot += __shfl_xor_sync(0xffffffffu, tot, 1);
      } else {
        tot = acc2[0].x + acc2[0].y;
        tot += __shfl_xor_sync(0xffffffffu, tot, 4);
        tot += __shfl_xor_sync(0xffffffffu, tot, 2);
        tot += __shfl_xor_sync(0xffffffffu, tot, 1);
      }
      if (j < j_hi && (dl % kSpan) == 0) sS[j * HG + dl / kSpan] = tot;
    }
    __syncwarp();
    // ---- softmax over my keys: lane = r * HG + h
    {
      constexpr int R = 32 / HG;
      const int h = lane % HG, r = lane / HG;
      float mx = -INFINITY;
      for (int j = j_lo + r; j < j_hi; j += R) mx = fmaxf(mx, sS[j * HG + h]);
#pragma unroll
      for (int off = HG; off < 32; off *= 2) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      m_w = mx * a.scale_log2;           // scale > 0: the max commutes with it
      float ls = 0.f;
      for (int j = j_lo + r; j < j_hi; j += R) {
        const float p = fast_exp2(fmaf(sS[j * HG + h], a.scale_log2, -m_w));
        sP[j * HG + h] = make_float2(p, p);
        ls += p;
      }
#pragma unroll
      for (int off = HG; off < 32; off *= 2) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      l_w = ls;
    }
    ok = __all_sync(0xffffffffu, mbar_wait(&bar_v[warp], 0, abort_word, a.wait_ns));
    if (ok) {
      if (append_row >= j_lo && append_row < j_hi && lane < D / 8) {
        reinterpret_cast<uint4 *>(sV + (size_t)append_row * D)[lane] =
            reinterpret_cast<const uint4 *>(a.v_new + ((size_t)b * a.Hkv + kvh) * D)[lane];
      }
      __syncwarp();
      // ---- O += P V over my keys: lane = CPL consecutive columns, all heads
      float2 o2[HG][CPL / 2];
#pragma unroll
      for (int h = 0; h < HG; ++h)
#pragma unroll
        for (int c = 0; c < CPL / 2; ++c) o2[h][c] = make_float2(0.f, 0.f);
      const __nv_bfloat16 *vcol = sV + lane * CPL;
#pragma unroll 2
      for (int j = j_lo; j < j_hi; ++j) {
        float2 vf[CPL / 2];
        if constexpr (CPL == 4) {
          const uint2 u = *reinterpret_cast<const uint2 *>(vcol + (size_t)j * D);
          vf[0] = bf16x2_to_f2(u.x);
          vf[1] = bf16x2_to_f2(u.y);
        } else {
          vf[0] = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(vcol + (size_t)j * D));
        }
        float2 pr[HG];
        if constexpr (HG >= 2) {
#pragma unroll
          for (int h = 0; h < HG; h += 2) {
            const float4 p4 = *reinterpret_cast<const float4 *>(sP + j * HG + h);
            pr[h] = make_float2(p4.x, p4.y);
            pr[h + 1] = make_float2(p4.z, p4.w);
          }
        } else {
          pr[0] = sP[j];
        }
#pragma unroll
        for (int h = 0; h < HG; ++h)
#pragma unroll
          for (int c = 0; c < CPL / 2; ++c) o2[h][c] = ffma2(pr[h], vf[c], o2[h][c]);
      }
      // the warp's partial O -> shared memory
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        float *dst = sO + ((size_t)warp * HG + h) * D + lane * CPL;
        if constexpr (CPL == 4)
          *reinterpret_cast<float4 *>(dst) =
              make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
        else
          *reinterpret_cast<float2 *>(dst) = o2[h][0];
      }
      wrote_o = true;
    }
  }
  if (!ok) {
    m_w = -INFINITY;
    l_w = 0.f;
  }
  if (!wrote_o) {
    // no keys, or a failed wait: an empty partial
#pragma unroll
    for (int h = 0; h < HG; ++h) {
      float *dst = sO + ((size_t)warp * HG + h) * D + lane * CPL;
      if constexpr (CPL == 4)
        *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
      else
        *reinterpret_cast<float2 *>(dst) = make_float2(0.f, 0.f);
    }
  }
  // ---- the warp's (max, sum) -> shared memory
  if (lane < HG) sML[warp * HG + lane] = make_float2(m_w, l_w);
  __syncthreads();
  if (*abort_word || *page_fault || a.stall) {
    // failure path: let this warp's copies land before the CTA exits; write nothing
    if (lane == 0 && issued) {
      mbar_wait(&bar_k[warp], 0, abort_word, kDecodeDrainNs, false);
      mbar_wait(&bar_v[warp], 0, abort_word, kDecodeDrainNs, false);
    }
    return;
  }
  // ---- merge the warps' partials: thread = (head, column pair)
  for (int item = threadIdx.x; item < HG * (D / 2); item += kDecodeThreads) {
    const int h = item / (D / 2), cp = item % (D / 2);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, sML[w * HG + h].x);
    float2 o = make_float2(0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        const float2 ml = sML[w * HG + h];
        const float f = fast_exp2(ml.x - M);   // 0 for a warp without keys
        const float2 x = reinterpret_cast<const float2 *>(sO + ((size_t)w * HG + h) * D)[cp];
        o.x = fmaf(f, x.x, o.x);
        o.y = fmaf(f, x.y, o.y);
        den = fmaf(f, ml.y, den);
      }
    }
    const int hq = hq0 + h;
    if (a.splits == 1) {
      const float inv = 1.0f / den;
      reinterpret_cast<uint32_t *>(a.out + ((size_t)b * a.Hq + hq) * D)[cp] =
          pack_bf16x2(o.x * inv, o.y * inv);
    } else {
      const size_t pi = ((size_t)b * a.Hq + hq) * a.splits + split;
      reinterpret_cast<float2 *>(a.part_o + pi * D)[cp] = o;
      if (cp == 0) a.part_ml[pi] = make_float2(M, den);
    }
  }
}

// Merge the per-split partial results: one CTA per (b, hq), one thread per d.
template <int D>
__global__ void __launch_bounds__(D) swa_decode_combine_kernel(const float *__restrict__ part_o,
                                                               const float2 *__restrict__ part_ml,
                                                               __nv_bfloat16 *__restrict__ out,
                                                               int splits) {
  grid_launch_dependents();
  grid_dependency_wait();
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
