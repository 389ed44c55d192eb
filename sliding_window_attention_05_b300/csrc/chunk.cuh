// chunk.cuh -- chunked prefill into a rolling KV cache on sm_103a.
//
// A long prompt can be prefilled in chunks (wiblog.cn long-context SWA
// article, section "长 Prompt 的分块处理与工程实现": Mistral processes the
// prompt in window-sized pieces and fills the rolling cache as it goes). The
// T queries of a chunk at positions pos0 .. pos0 + T - 1 need, from before
// pos0, only the sinks (j < s) and the positions pos0 - w + 1 .. pos0 - 1;
// the ring cache holds exactly those once every position < pos0 has been
// appended (and, while pos0 <= s + w - 1, every position < pos0).
//
// The chunk runs through the prefill kernel on a contiguous staging copy of
// the keys and values whose row index differs from the position by a
// constant over the window part, so the kernel's band, causal and sink rules
// carry over unchanged:
//   pos0 <= s + w - 1: rows 0 .. pos0 - 1 are positions 0 .. pos0 - 1;
//   otherwise:         rows 0 .. s - 1 are the sinks, rows s .. s + w - 2 are
//                      positions pos0 - w + 1 .. pos0 - 1;
// then the T chunk rows. The queries stay in the caller's q: the kernel reads
// staged row n_pre + i from row i of q and writes it to row i of out. Query
// blocks made only of prefix rows are not computed; the prefix rows of the
// first computed block read zero queries (the TMA fill value below row 0 of
// q: finite scores) and their outputs are not stored.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sm100_ptx.cuh"
#include "swa_index.cuh"

namespace swa {

// Rows of the staged prefix for a chunk starting at pos0.
SWA_HD long long chunk_prefix_rows(long long pos0, int w, int s) {
  const long long keep = (long long)s + w - 1;
  return pos0 < keep ? pos0 : keep;
}

// Position held by prefix row r (r < chunk_prefix_rows(pos0, w, s)).
SWA_HD long long chunk_prefix_pos(long long r, long long pos0, int w, int s) {
  if (pos0 <= (long long)s + w - 1 || r < s) return r;
  return pos0 - w + 1 + (r - s);
}

// Where the staging reads the kept cache rows from: a ring cache
// [B, Hkv, s + w, d] (table == nullptr) or the pages of a paged pool
// [n_pages, Hkv, page_size, d] through a page table [B, max_pages].
struct ChunkSource {
  const uint4 *kcache, *vcache;
  const int *table;
  int page_size, max_pages, n_pages;
};

// Stage the key/value rows [prefix | chunk] into kx, vx [B, Lx, Hkv, d] with
// Lx = n_pre + T. The queries and outputs are not staged: the prefill kernel
// reads q and writes out at row (staged row - n_pre). One thread moves 16
// bytes of one (b, row, K or V head). Thread 0 of sequence 0 also writes pos0
// into pos_out[B] for the append that follows. A prefix row whose page is
// unmapped is staged as zeros and flagged in the device error word.
__global__ void swa_chunk_stage_kernel(const uint4 *__restrict__ k_new,
                                       const uint4 *__restrict__ v_new, const ChunkSource src,
                                       uint4 *__restrict__ kx, uint4 *__restrict__ vx,
                                       int *__restrict__ pos_out, int B, int T, int Hkv, int d,
                                       int w, int s, long long pos0, int n_pre) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.y;
  const int vpr = d / 8;                    // 16-byte units per row of one head
  const int heads = 2 * Hkv;                // K heads, then V heads
  const long long Lx = (long long)n_pre + T;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0 && idx < B) pos_out[idx] = (int)pos0;
  if (idx >= Lx * heads * vpr) return;
  const int c = (int)(idx % vpr);
  const int h = (int)((idx / vpr) % heads);
  const long long r = idx / ((long long)vpr * heads);
  const bool is_v = h >= Hkv;
  const int kvh = is_v ? h - Hkv : h;
  const long long dst = (((long long)b * Lx + r) * Hkv + kvh) * vpr + c;
  uint4 val = make_uint4(0, 0, 0, 0);
  if (r < n_pre) {
    const long long p = chunk_prefix_pos(r, pos0, w, s);
    long long at;
    if (src.table == nullptr) {
      at = (((long long)b * Hkv + kvh) * (s + w) + ring_slot(p, w, s)) * vpr + c;
    } else {
      const long long lp = p / src.page_size;
      const int page = lp < src.max_pages ? src.table[(long long)b * src.max_pages + lp] : -1;
      if (page < 0 || page >= src.n_pages) {
        record_error(kErrMissingPage);
        at = -1;
      } else {
        at = (((long long)page * Hkv + kvh) * src.page_size + p % src.page_size) * vpr + c;
      }
    }
    if (at >= 0) val = is_v ? src.vcache[at] : src.kcache[at];
  } else {
    const long long at = (((long long)b * T + (r - n_pre)) * Hkv + kvh) * vpr + c;
    val = is_v ? v_new[at] : k_new[at];
  }
  (is_v ? vx : kx)[dst] = val;
}

}  // namespace swa
