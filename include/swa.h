/*
 * swa.h -- C ABI of libswa.so: causal sliding-window attention with attention
 * sinks, SWA(w, s), on NVIDIA B300 (sm_103a).
 *
 * The operation (explainer page of arXiv 2608.28444, "滑动窗口注意力（SWA）配
 * sinks 比 post-training 线性注意力更划算", section "核心方法 / 1. 训练免费的
 * SWA(w, s)": the x_t equation and the swa_mask definition):
 *
 *   query t (0-indexed) attends to the key set
 *       K(t) = { j : j <= t  and  (j >= t - w + 1  or  j < s) },
 *   i.e. the last w tokens (t itself included) plus the first s tokens
 *   ("sinks"), and returns  sum_{j in K(t)} softmax_j(scale * q_t . k_j) v_j.
 *
 * Query head hq reads key/value head hq / (Hq / Hkv) (grouped-query attention;
 * wiblog.cn long-context SWA article, section "SWA 的核心机制", Mistral 7B with
 * 8 KV heads). Decode runs over a rolling KV cache of s pinned sink slots plus w
 * window slots (same article, section "与 KV Cache 的配合：轮转替换策略").
 *
 * Conventions for every call:
 *  - Tensors are dense, row-major, bf16 (2 bytes per element) unless stated;
 *    the last dimension (d) is contiguous. All tensor pointers are DEVICE
 *    pointers owned by the caller; the library keeps no pointer after a call
 *    returns and allocates no device memory.
 *  - Device pointers must be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (NULL = legacy default stream) and
 *    never synchronises. Argument errors are detected on the host before any
 *    launch; nothing is launched in that case.
 *  - Inputs must be finite. scale must be finite and > 0.
 *  - Return value: SWA_OK, or an SWA_ERR_* code; swa_last_error() gives a
 *    text description of the last failure on the calling thread.
 *  - Supported head dimensions: d in {64, 128}. Group size Hq / Hkv in 1..128.
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SWA_API __attribute__((visibility("default")))
#else
#define SWA_API
#endif

/* Identical to cudaStream_t. */
typedef struct CUstream_st *swa_stream_t;

enum swa_status {
    SWA_OK = 0,
    SWA_ERR_INVALID_ARG = 1, /* null pointer, bad size, w < 1, Hq % Hkv != 0 ... */
    SWA_ERR_UNSUPPORTED = 2, /* valid but not implemented here (e.g. d = 96)   */
    SWA_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed         */
    SWA_ERR_DEVICE = 4       /* no usable sm_103a device                       */
};

/* Prefill: out = SWA(w, s) attention of every query of a prompt.
 *   q   [B, L, Hq,  d]  bf16        k, v [B, L, Hkv, d]  bf16
 *   out [B, L, Hq,  d]  bf16 (written; must not alias q, k or v)
 * Requires B, L >= 1, w >= 1, s >= 0, Hq % Hkv == 0. w >= L gives full causal
 * attention; s > 0 adds the sinks. Accumulation is fp32, probabilities are
 * rounded to bf16 before the value product, the output is rounded to bf16
 * (round to nearest even). Only key tiles that intersect a query block's
 * window, plus the sink tile, are loaded or multiplied (explainer of
 * "Hybrid Sliding Window Attention", section "三、3. FlashAttention-2 /
 * FlashAttention-3": tiles outside the window are skipped). */
SWA_API int swa_prefill(const void *q, const void *k, const void *v, void *out,
                int B, int L, int Hq, int Hkv, int d, int w, int s,
                float scale, swa_stream_t stream);

/* Prefill that also writes each row's log-sum-exp of its scaled scores,
 *   lse[b, hq, t] = log(sum_{j in K(t)} exp(scale * q_t . k_j))   (natural log),
 * as fp32 [B, Hq, L] (4-byte aligned): what swa_prefill_backward needs to
 * recompute the softmax weights. Otherwise identical to swa_prefill. */
SWA_API int swa_prefill_lse(const void *q, const void *k, const void *v, void *out, float *lse,
                            int B, int L, int Hq, int Hkv, int d, int w, int s, float scale,
                            swa_stream_t stream);

/* Backward of the prefill: the gradients of the outputs with respect to q, k
 * and v for an upstream gradient dout. The pages give no backward formulas;
 * they mention SWA-aware fine-tuning (the SWAA page, "如何将Sliding Window
 * Attention Adaptation应用到你的LLM项目中", section "微调：提升SWAA适应性"). This
 * is the chain rule applied to the forward definition above: for every row
 * (b, hq, t) and key j in K(t), with P the forward's softmax weights,
 *   dP_tj = dout_t . v_j,  D_t = dout_t . out_t,  dS_tj = P_tj (dP_tj - D_t),
 *   dq_t = scale sum_j dS_tj k_j,  dk_j = scale sum_t dS_tj q_t,
 *   dv_j = sum_t P_tj dout_t,
 * with dk and dv summed over the query heads of each KV head group.
 *   q, out, dout [B, L, Hq, d] bf16; k, v [B, L, Hkv, d] bf16 (the forward's
 *   inputs and output); lse fp32 [B, Hq, L] from swa_prefill_lse on the same
 *   inputs; dq [B, L, Hq, d], dk, dv [B, L, Hkv, d] bf16 (written in full).
 *   workspace: caller-owned device memory of at least
 *   swa_prefill_backward_workspace_size(...) bytes, 16-byte aligned.
 * Only the key tiles inside each query block's window (plus the sinks) are
 * visited, as in the forward pass. Products run on the tensor cores with fp32
 * accumulation; P and dS are rounded to bf16 before their products; the
 * gradients are rounded to bf16. */
SWA_API size_t swa_prefill_backward_workspace_size(int B, int L, int Hq, int Hkv, int d, int s);
SWA_API int swa_prefill_backward(const void *q, const void *k, const void *v, const void *out,
                                 const void *dout, const float *lse, void *dq, void *dk, void *dv,
                                 int B, int L, int Hq, int Hkv, int d, int w, int s, float scale,
                                 void *workspace, size_t workspace_bytes, swa_stream_t stream);

/* Ring-cache append: store T consecutive new tokens of every sequence (the
 * rolling cache of the wiblog.cn long-context SWA article, section
 * "与 KV Cache 的配合：轮转替换策略", with the s sinks of the SWA(w, s) explainer,
 * section "工程落地与实践" item 3: 64 + 4 = 68 slots at w = 64, s = 4).
 *   k_new, v_new [B, T, Hkv, d] bf16     kcache, vcache [B, Hkv, s + w, d] bf16
 *   pos_start    DEVICE int32[B]: position of token 0 of this call, per sequence
 * Token i of sequence b has position p = pos_start[b] + i and goes to slot
 *   slot(p) = p                   if p < s      (sink slots, kept forever)
 *           = s + (p - s) mod w   otherwise     (window slots, oldest evicted)
 * Tokens that a later token of the same call evicts again are not written.
 * Positions must be appended in order across calls (each call continues where
 * the previous one ended); positions < 0 are skipped and flagged in the
 * device error word. */
SWA_API int swa_cache_append(const void *k_new, const void *v_new, void *kcache, void *vcache,
                     const int *pos_start, int B, int T, int Hkv, int d, int w, int s,
                     swa_stream_t stream);

/* Chunked prefill into a ring cache: the T prompt tokens at positions
 * pos0 .. pos0 + T - 1 of every sequence (one pos0 for the whole batch) attend
 * over the keys the cache still holds plus the chunk's own keys, and are then
 * appended to the cache. Row i of out equals row pos0 + i of swa_prefill over
 * the whole prompt (wiblog.cn long-context SWA article, section
 * "长 Prompt 的分块处理与工程实现": a long prompt is prefilled in pieces while
 * the rolling cache fills).
 *   q [B, T, Hq, d]; k_new, v_new [B, T, Hkv, d]; out [B, T, Hq, d] (written)
 *   kcache, vcache [B, Hkv, s + w, d]: every position < pos0 must already have
 *   been appended (swa_cache_append, swa_append_decode or earlier chunks). The
 *   rows a chunk needs from before pos0 are the sinks and the last w - 1
 *   positions, which the ring keeps.
 *   workspace: caller-owned device memory of at least
 *   swa_prefill_chunk_workspace_size(...) bytes, 16-byte aligned; its size grows
 *   with (min(pos0, s + w - 1) + T) rows of k and v.
 * The work: a staging kernel lays out the kept cache rows of k and v, then
 * the chunk's, contiguously in the workspace, the prefill kernel runs over the
 * query blocks that hold chunk rows, reading q and writing out in place, and
 * the append kernel stores the chunk. */
SWA_API size_t swa_prefill_chunk_workspace_size(int B, int T, int Hq, int Hkv, int d, int w, int s,
                                                long long pos0);
SWA_API int swa_prefill_chunk(const void *q, const void *k_new, const void *v_new, void *kcache,
                              void *vcache, void *out, int B, int T, int Hq, int Hkv, int d, int w,
                              int s, long long pos0, float scale, void *workspace,
                              size_t workspace_bytes, swa_stream_t stream);

/* Bytes of device workspace swa_decode needs for these sizes (0 if none). */
SWA_API size_t swa_decode_workspace_size(int B, int Hq, int Hkv, int d, int w, int s);

/* Decode: one new query per head attends over the ring cache: the x_t of the
 * SWA(w, s) explainer (section "核心方法 / 1. 训练免费的 SWA(w, s)") for the
 * newest position, read from the rolling cache of the wiblog.cn article
 * (section "与 KV Cache 的配合：轮转替换策略").
 *   q   [B, Hq, d] bf16; out [B, Hq, d] bf16 (written)
 *   kcache, vcache [B, Hkv, s + w, d] bf16, already holding position pos[b]
 *   pos DEVICE int32[B]: position of the newest token of each sequence.
 * The cache then holds exactly K(pos) in its first min(pos + 1, s + w) slots,
 * so no masking is needed. workspace: caller-owned device memory of at least
 * swa_decode_workspace_size(...) bytes (may be NULL when that is 0). */
SWA_API int swa_decode(const void *q, const void *kcache, const void *vcache, const int *pos,
               void *out, int B, int Hq, int Hkv, int d, int w, int s, float scale,
               void *workspace, size_t workspace_bytes, swa_stream_t stream);

/* Append one new token per sequence, then decode it, in one launch: the same
 * result (and cache contents) as swa_cache_append with T = 1 at pos[b]
 * followed by swa_decode at pos[b] (the per-token step of the rolling cache,
 * wiblog.cn long-context SWA article, section "与 KV Cache 的配合：轮转替换策略").
 *   k_new, v_new [B, Hkv, d] bf16: the new token's key and value rows
 *   pos DEVICE int32[B]: the new token's position (the cache holds every
 *   earlier position); other arguments as swa_decode, same workspace size. */
SWA_API int swa_append_decode(const void *q, const void *k_new, const void *v_new, void *kcache,
                              void *vcache, const int *pos, void *out, int B, int Hq, int Hkv,
                              int d, int w, int s, float scale, void *workspace,
                              size_t workspace_bytes, swa_stream_t stream);

/* Maximum scratch bytes swa_decode_noalloc can use (see below). */
#define SWA_DECODE_NOALLOC_SCRATCH_BYTES (2u << 20)

/* Decode without any device allocation and without a caller workspace.
 *
 * (The pages have no counterpart: this is an interface convenience.)
 *
 * Same arguments, result and errors as swa_decode, minus the workspace. It is
 * for callers that cannot allocate device memory at the point of the call --
 * for example a serving loop whose engine owns all device memory in a fixed
 * pool and forbids allocation during a step (cudaMalloc can synchronise the
 * device and can fail under memory pressure), or plain C code that has no
 * allocator of its own for scratch buffers. When swa_decode would need a
 * split-KV workspace, this entry point uses a scratch array compiled into the
 * library instead: SWA_DECODE_NOALLOC_SCRATCH_BYTES (2 MiB) of device memory
 * that every GPU which loads libswa.so holds until the process exits.
 *  - Sizes whose workspace (swa_decode_workspace_size) exceeds that maximum
 *    are rejected with SWA_ERR_UNSUPPORTED before anything is launched.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - The first call on each device performs a one-time set-up (it looks up
 *    the scratch array's device address with that device current). Make that
 *    first call before any stream capture.
 *  - All calls share the one array, which keeps the previous call's contents;
 *    nothing in it needs to start at zero. Calls whose kernels overlap on the
 *    GPU (for example on two streams at once) race on it: order them on one
 *    stream, or use swa_decode with a workspace each. */
SWA_API int swa_decode_noalloc(const void *q, const void *kcache, const void *vcache,
                               const int *pos, void *out, int B, int Hq, int Hkv, int d, int w,
                               int s, float scale, swa_stream_t stream);

/* ------------------------------------------------------------------ paged layout
 * K and V of every layer can instead live in pages of page_size positions drawn
 * from one pool: kpool, vpool [n_pages, Hkv, page_size, d] bf16 (DEVICE, the
 * caller's). A sequence's page table, int32 [max_pages], maps logical page lp
 * (positions lp * page_size .. lp * page_size + page_size - 1) to a physical
 * page, or -1. A layer with window w and s sinks keeps exactly the pages that
 * hold a position of K(p): sliding-window layers recycle theirs as the window
 * moves, full-attention layers (w beyond every position) keep growing
 * ("Hybrid Sliding Window Attention (Hybrid SWA)", section
 * "三、1. vLLM 中的 Hybrid KV Cache 最佳实践"; the SWA(w, s) explainer, section
 * "工程落地与实践" item 1, route B: cache only the last w tokens and the sinks).
 * The page pool and the tables are HOST objects; the caller copies each table
 * to the device before a launch that reads it. */
typedef struct swa_page_pool swa_page_pool;

/* A pool of n_pages physical pages, all free. NULL on n_pages < 1. */
SWA_API swa_page_pool *swa_page_pool_create(int n_pages);
SWA_API void swa_page_pool_destroy(swa_page_pool *pool);
/* Free pages left in the pool (-1 for NULL). Thread-safe. */
SWA_API int swa_page_pool_free_pages(swa_page_pool *pool);

/* Prepare one sequence's HOST page table (int32 [max_pages], -1 = unmapped,
 * all -1 for a new sequence) for appending positions up to pos_hi and attending
 * at pos_hi: pages are taken from the pool for every logical page holding a
 * position of K(pos_hi) that is unmapped, and mapped pages that hold none are
 * returned. Call it with non-decreasing pos_hi. SWA_ERR_UNSUPPORTED (nothing
 * changed) when the pool has too few free pages or pos_hi lies beyond the
 * table; SWA_ERR_INVALID_ARG for a table entry this pool did not hand out.
 * Thread-safe per pool; the table is the caller's. */
SWA_API int swa_paged_reserve(swa_page_pool *pool, int *table, int max_pages, long long pos_hi,
                              int w, int s, int page_size);
/* swa_paged_reserve for a run of positions: the table then maps the pages of
 * every K(p) with pos_lo <= p <= pos_hi (the sink pages and the pages of
 * positions pos_lo - w + 1 .. pos_hi), which a chunk of prompt tokens at
 * pos_lo .. pos_hi reads and writes; other mapped pages are returned.
 * swa_paged_reserve(..., pos_hi, ...) is this call with pos_lo = pos_hi. Call it
 * with non-decreasing pos_lo. Same errors as swa_paged_reserve, plus
 * SWA_ERR_INVALID_ARG for pos_lo > pos_hi. */
SWA_API int swa_paged_reserve_range(swa_page_pool *pool, int *table, int max_pages,
                                    long long pos_lo, long long pos_hi, int w, int s,
                                    int page_size);
/* Return every page of a table to the pool and unmap it (end of a sequence). */
SWA_API int swa_paged_release(swa_page_pool *pool, int *table, int max_pages);

/* Paged swa_cache_append: the same survivors, stored in the pages of
 * page_table (DEVICE int32 [B, max_pages], prepared by swa_paged_reserve for the
 * last position of the call); n_pages is the pools' page count. An unmapped or
 * out-of-range page is skipped and flagged in the device error word. */
SWA_API int swa_paged_append(const void *k_new, const void *v_new, void *kpool, void *vpool,
                             const int *page_table, const int *pos_start, int B, int T, int Hkv,
                             int d, int page_size, int max_pages, int n_pages, int w, int s,
                             swa_stream_t stream);
/* Paged swa_decode: the same result, reading K(pos[b]) through page_table
 * (DEVICE int32 [B, max_pages]); workspace as swa_decode_workspace_size. A CTA
 * that meets an unmapped or out-of-range page issues no copy, writes nothing
 * and flags the device error word. */
SWA_API int swa_paged_decode(const void *q, const void *kpool, const void *vpool,
                             const int *page_table, const int *pos, void *out, int B, int Hq,
                             int Hkv, int d, int page_size, int max_pages, int n_pages, int w,
                             int s, float scale, void *workspace, size_t workspace_bytes,
                             swa_stream_t stream);

/* Paged swa_prefill_chunk: the chunk of T prompt tokens at positions
 * pos0 .. pos0 + T - 1 attends over the keys the pages still hold plus its
 * own, and is then appended to the pages (a long prompt prefilled in pieces,
 * wiblog.cn long-context SWA article, section "长 Prompt 的分块处理与工程实现",
 * into the paged hybrid layout of "Hybrid Sliding Window Attention (Hybrid
 * SWA)", section "三、1. vLLM 中的 Hybrid KV Cache 最佳实践").
 *   q, k_new, v_new, out as swa_prefill_chunk; kpool, vpool and n_pages as
 *   swa_paged_append; page_table DEVICE int32 [B, max_pages], prepared by
 *   swa_paged_reserve_range(pos0, pos0 + T - 1) so that every page the chunk
 *   reads or writes is mapped; every position < pos0 must already have been
 *   appended. workspace: swa_prefill_chunk_workspace_size(...) bytes.
 * A prefix row on an unmapped page is read as zeros and flagged in the device
 * error word; the append skips and flags unmapped pages as swa_paged_append. */
SWA_API int swa_paged_prefill_chunk(const void *q, const void *k_new, const void *v_new,
                                    void *kpool, void *vpool, const int *page_table, void *out,
                                    int B, int T, int Hq, int Hkv, int d, int page_size,
                                    int max_pages, int n_pages, int w, int s, long long pos0,
                                    float scale, void *workspace, size_t workspace_bytes,
                                    swa_stream_t stream);

/* Host helper: the cache slot of position pos (the formula above), or -1 for
 * pos < 0, w < 1 or s < 0. */
SWA_API long long swa_cache_slot(long long pos, int w, int s);

/* Host helper: bytes of ONE cache tensor (K or V) [B, Hkv, s + w, d] bf16. */
SWA_API size_t swa_cache_bytes(int B, int Hkv, int d, int w, int s);

/* Host helper: the prefill tiling the library picks for these sizes.
 * plan[0] query positions per block (Tq)      plan[1] tile rows (Tq * Hq/Hkv)
 * plan[2] keys per band tile (<= 192)         plan[3] keys per sink box (0: none)
 * plan[4] sink boxes (ceil(s / 128))          plan[5] K/V pipeline stages
 * plan[6] persistent CTAs on the current device (0 without a device)
 * plan[7] dynamic shared memory bytes per CTA */
SWA_API int swa_prefill_plan(int L, int Hq, int Hkv, int d, int w, int s, int plan[8]);

/* Test aid: which prefill kernel swa_prefill, swa_prefill_lse, the chunked
 * prefill and the key-mask aids below use, for the whole process: 0 = the
 * library's choice for the sizes (the default; currently always kernel 1,
 * the faster of the two on B300 at every size measured), 1 = the kernel that
 * computes one query block per work item, 2 = the kernel that computes two
 * consecutive query blocks per work item over one list of key tiles. Both
 * compute the same attention. Returns the previous mode, or -1 (nothing
 * changed) for a mode outside 0..2. Not thread-safe against concurrent
 * prefill calls that expect a different mode. */
SWA_API int swa_prefill_select(int mode);

/* Test aid: the (query, key) pairs that the prefill kernel's tile schedule and
 * in-tile masks admit, for rows row0 .. row0 + nrows - 1 of a prompt of length
 * L, with the same tiling as swa_prefill for these sizes.
 *   bits   DEVICE uint32 [nrows, ceil(L / 32)]: bit (j % 32) of word j / 32 of
 *          row r is set iff key j is admitted for query row0 + r
 *   counts DEVICE int32 [nrows]: admitted pairs counted over all tiles (equals
 *          the popcount of the row only if no key is admitted twice) */
SWA_API int swa_debug_keymask(int L, int Hq, int Hkv, int d, int w, int s, int row0, int nrows,
                      uint32_t *bits, int *counts, swa_stream_t stream);

/* Test aid: the same admitted-pair bitmask and counts as swa_debug_keymask,
 * computed on the host by the library's host copy of the schedule (no device
 * needed). bits and counts are HOST arrays of the same shapes. */
SWA_API int swa_keymask_host(int L, int Hq, int Hkv, int d, int w, int s, int row0, int nrows,
                     uint32_t *bits, int *counts);

/* Test aid: swa_decode (same arguments, workspace and result) with each wait
 * for the staged cache rows limited to wait_ns nanoseconds. With stall != 0 no
 * copy is issued at all, so every such wait runs out: the kernel then records
 * the wait timeout (code 1) in the device error word, writes nothing to out or
 * the workspace, and returns; the context stays usable. Used to exercise the
 * failure path without faulting the device. */
SWA_API int swa_debug_decode_timeout(const void *q, const void *kcache, const void *vcache,
                                     const int *pos, void *out, int B, int Hq, int Hkv, int d,
                                     int w, int s, float scale, void *workspace,
                                     size_t workspace_bytes, unsigned long long wait_ns, int stall,
                                     swa_stream_t stream);

/* (Outside this test aid, a decode whose wait runs out also records code 1 and
 * writes nothing from the CTAs concerned; when the cache is split over CTAs the
 * combine step still runs, so out is then undefined. Check the error word.) */

/* Read the device error word that kernels set instead of trapping (a bounded
 * wait that gave up, a negative position). *code receives 0 if no error was
 * recorded. Synchronises the current device. clear != 0 resets it to 0. */
SWA_API int swa_device_error(int *code, int clear);

SWA_API const char *swa_status_string(int status);
SWA_API const char *swa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SWA_H */
