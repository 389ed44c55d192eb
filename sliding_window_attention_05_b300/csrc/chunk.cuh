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
// The chunk runs through the prefill kernel on a contiguous staging copy
// whose row index differs from the position by a constant over the window
// part, so the kernel's band, causal and sink rules carry over unchanged:
//   pos0 <= s + w - 1: rows 0 .. pos0 - 1 are positions 0 .. pos0 - 1;
//   otherwise:         rows 0 .. s - 1 are the sinks, rows s .. s + w - 2 are
//                      positions pos0 - w + 1 .. pos0 - 1;
// then the T chunk rows. Query blocks made only of prefix rows are not
// computed; the prefix rows of the first computed block get zero queries
// (finite scores) and their outputs are not used.
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

// Stage [prefix | chunk] rows: qx [B, Lx, Hq, d], kx/vx [B, Lx, Hkv, d] with
// Lx = n_pre + T; query rows below q_row0 (blocks the prefill skips) are not
// written. One thread moves 16 bytes of one (b, row, head) of the Hq + 2 Hkv
// heads. Thread 0 also writes pos0 into pos_out[B] for the append
// that follows.
__global__ void swa_chunk_stage_kernel(const uint4 *__restrict__ q, const uint4 *__restrict__ k_new,
                                       const uint4 *__restrict__ v_new,
                                       const uint4 *__restrict__ kcache,
                                       const uint4 *__restrict__ vcache, uint4 *__restrict__ qx,
                                       uint4 *__restrict__ kx, uint4 *__restrict__ vx,
                                       int *__restrict__ pos_out, int B, int T, int Hq, int Hkv,
                                       int d, int w, int s, long long pos0, int n_pre,
                                       int q_row0) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.y;
  const int vpr = d / 8;                    // 16-byte units per row of one head
  const int heads = Hq + 2 * Hkv;
  const long long Lx = (long long)n_pre + T;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0 && idx < B) pos_out[idx] = (int)pos0;
  if (idx >= Lx * heads * vpr) return;
  const int c = (int)(idx % vpr);
  const int h = (int)((idx / vpr) % heads);
  const long long r = idx / ((long long)vpr * heads);
  if (h < Hq) {  // query rows (those below q_row0 are never read)
    if (r < q_row0) return;
    const long long dst = (((long long)b * Lx + r) * Hq + h) * vpr + c;
    if (r < n_pre)
      qx[dst] = make_uint4(0, 0, 0, 0);
    else
      qx[dst] = q[(((long long)b * T + (r - n_pre)) * Hq + h) * vpr + c];
    return;
  }
  const bool is_v = h >= Hq + Hkv;
  const int kvh = h - Hq - (is_v ? Hkv : 0);
  const long long dst = (((long long)b * Lx + r) * Hkv + kvh) * vpr + c;
  uint4 val;
  if (r < n_pre) {
    const long long slot = ring_slot(chunk_prefix_pos(r, pos0, w, s), w, s);
    const long long src = (((long long)b * Hkv + kvh) * (s + w) + slot) * vpr + c;
    val = is_v ? vcache[src] : kcache[src];
  } else {
    const long long src = (((long long)b * T + (r - n_pre)) * Hkv + kvh) * vpr + c;
    val = is_v ? v_new[src] : k_new[src];
  }
  (is_v ? vx : kx)[dst] = val;
}

// out[b, i] = ox[b, n_pre + i] for the T chunk rows (16 bytes per thread).
__global__ void swa_chunk_out_kernel(const uint4 *__restrict__ ox, uint4 *__restrict__ out, int T,
                                     int Hq, int d, int n_pre) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.y;
  const long long row_units = (long long)Hq * (d / 8);
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)T * row_units) return;
  const long long Lx = (long long)n_pre + T;
  out[(long long)b * T * row_units + idx] = ox[((long long)b * Lx + n_pre) * row_units + idx];
}

}  // namespace swa
