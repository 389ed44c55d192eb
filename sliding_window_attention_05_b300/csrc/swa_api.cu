// swa_api.cu -- the C ABI of libswa.so (declared in include/swa.h).
//
// One translation unit holds every kernel so the device error word needs no
// relocatable device code. The library allocates no device memory: all
// tensors and the decode workspace are the caller's.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/swa.h"
#include "backward.cuh"
#include "chunk.cuh"
#include "decode.cuh"
#include "page_pool.h"
#include "prefill.cuh"
#include "prefill_pair.cuh"
#include "sm100_ptx.cuh"
#include "swa_index.cuh"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char *what) {
  return fail(SWA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_d(int d) { return d == 64 || d == 128; }

// ------------------------------------------------------------------ device info

struct DeviceInfo {
  int sms = 0;
  int max_smem_optin = 0;
  bool ok = false;
};

int current_device_info(DeviceInfo *info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static std::mutex mu;
  static DeviceInfo cache[64];
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return fail(SWA_ERR_DEVICE, "device ordinal %d out of range", dev);
  if (!cache[dev].ok) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(SWA_ERR_DEVICE, "libswa.so is built for sm_103a; device %d is sm_%d%d", dev,
                  major, minor);
    cudaDeviceGetAttribute(&cache[dev].sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&cache[dev].max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                           dev);
    cache[dev].ok = true;
  }
  *info = cache[dev];
  return SWA_OK;
}

// ------------------------------------------------------------------ launches

// The dynamic shared-memory limit of a kernel is a per-device attribute:
// raise it once per (kernel, device) that launches it.
cudaError_t ensure_max_dynamic_smem(const void *kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::pair<const void *, int>, int> raised;  // -> bytes
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kernel, dev);
  const auto it = raised.find(key);
  if (it != raised.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) raised[key] = bytes;
  return e;
}

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous kernel on the stream finishes; it waits for that kernel
// (griddepcontrol.wait) before touching global memory. In a captured CUDA
// graph this becomes a programmatic edge.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D bf16 map over a [B, L, H, d] tensor (dims listed innermost first) with
// a box of 64 x box_h x box_l x 1 and the 128-byte swizzle.
int make_map_bf16_4d(CUtensorMap *map, const void *base, int B, int L, int H, int d, int box_h,
                     int box_l) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return fail(SWA_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)L * H * d * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)box_h, (cuuint32_t)box_l, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SWA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SWA_OK;
}

// ------------------------------------------------------------------ prefill

// Which prefill kernel runs: 0 = by the rule in use_pair_kernel, 1 = the
// single-block kernel, 2 = the pair kernel (set by the test aid
// swa_prefill_select).
std::atomic<int> g_prefill_mode{0};

// The pair kernel (two query blocks per work item, prefill_pair.cuh) halves
// the key/value loads per block, but on this GPU it runs 25-40% slower than
// the single-block kernel at every window measured (64 to 2048; its MMA
// issue, with N = 128 tiles, is the limit), so the library runs the
// single-block kernel unless the pair kernel is selected explicitly.
bool use_pair_kernel(int d, int L, int Hq, int Hkv, int w, int s) {
  (void)d;
  (void)L;
  (void)Hq;
  (void)Hkv;
  (void)w;
  (void)s;
  return g_prefill_mode.load(std::memory_order_relaxed) == 2;
}

int pair_tile_keys(int d) {
  return d == 128 ? swa::PairSmem<128>::kTileKeys : swa::PairSmem<64>::kTileKeys;
}

// The tiling of the kernel swa_prefill runs for these sizes.
swa::PrefillPlan prefill_plan_for(int d, int L, int Hq, int Hkv, int w, int s) {
  if (use_pair_kernel(d, L, Hq, Hkv, w, s))
    return swa::make_plan(L, Hq, Hkv, w, s, pair_tile_keys(d), 2);
  return swa::make_plan(L, Hq, Hkv, w, s, swa::kMaxTileKeys, 1, /*allow_sink_last=*/1);
}

bool prefill_sep_stage(int d, const swa::PrefillPlan &plan, int max_smem) {
  return d == 64 ? swa::PrefillSmem<64>::use_sep_stage(plan, max_smem)
                 : swa::PrefillSmem<128>::use_sep_stage(plan, max_smem);
}

int prefill_stages(int d, const swa::PrefillPlan &plan, int max_smem) {
  if (plan.bpi == 2)
    return d == 64 ? swa::PairSmem<64>::stages(plan, max_smem)
                   : swa::PairSmem<128>::stages(plan, max_smem);
  const bool sep = prefill_sep_stage(d, plan, max_smem);
  return d == 64 ? swa::PrefillSmem<64>::stages(plan, max_smem, sep)
                 : swa::PrefillSmem<128>::stages(plan, max_smem, sep);
}

size_t prefill_smem_bytes(int d, const swa::PrefillPlan &plan, int stages, bool sep) {
  if (plan.bpi == 2)
    return d == 64 ? swa::PairSmem<64>::bytes(plan, stages)
                   : swa::PairSmem<128>::bytes(plan, stages);
  return d == 64 ? swa::PrefillSmem<64>::bytes(plan, stages, sep)
                 : swa::PrefillSmem<128>::bytes(plan, stages, sep);
}

// qb_first: query blocks below it are skipped (their rows of out are left
// unwritten). Work items run from the last query block down, so dropping the
// tail of the item range drops exactly those blocks.
// q_off: k and v hold L rows, q and out only the last L - q_off of them (a
// chunk after its staged prefix); query blocks wholly inside the first q_off
// rows must be skipped through qb_first.
template <int D>
int launch_prefill(const void *q, const void *k, const void *v, void *out, int B, int L, int Hq,
                   int Hkv, int w, int s, float scale, cudaStream_t stream,
                   const DeviceInfo &dev, int qb_first = 0, float *lse = nullptr, int q_off = 0) {
  const bool pair = use_pair_kernel(D, L, Hq, Hkv, w, s);
  const swa::PrefillPlan plan = prefill_plan_for(D, L, Hq, Hkv, w, s);
  CUtensorMap tq, tk, tv, tks, tvs, to;
  int rc;
  if ((rc = make_map_bf16_4d(&tq, q, B, L - q_off, Hq, D, plan.G, plan.Tq))) return rc;
  if ((rc = make_map_bf16_4d(&to, out, B, L - q_off, Hq, D, plan.G, plan.Tq))) return rc;
  if ((rc = make_map_bf16_4d(&tk, k, B, L, Hkv, D, 1, plan.n_band))) return rc;
  if ((rc = make_map_bf16_4d(&tv, v, B, L, Hkv, D, 1, plan.n_band))) return rc;
  if (plan.n_sink > 0) {
    if ((rc = make_map_bf16_4d(&tks, k, B, L, Hkv, D, 1, plan.s_box))) return rc;
    if ((rc = make_map_bf16_4d(&tvs, v, B, L, Hkv, D, 1, plan.s_box))) return rc;
  } else {
    tks = tk;
    tvs = tv;
  }
  // band boxes shortened by the sink box, for a block's last band tile that
  // carries the sinks at its end
  CUtensorMap tkb = tk, tvb = tv;
  if (plan.sink_last) {
    if ((rc = make_map_bf16_4d(&tkb, k, B, L, Hkv, D, 1, plan.n_band - plan.s_box))) return rc;
    if ((rc = make_map_bf16_4d(&tvb, v, B, L, Hkv, D, 1, plan.n_band - plan.s_box))) return rc;
  }
  const bool sep_stage = !pair && prefill_sep_stage(D, plan, dev.max_smem_optin);
  const int stages = prefill_stages(D, plan, dev.max_smem_optin);
  if (stages < 2) return fail(SWA_ERR_UNSUPPORTED, "not enough shared memory for the pipeline");
  const size_t smem = prefill_smem_bytes(D, plan, stages, sep_stage);
  const void *kernel =
      pair ? reinterpret_cast<const void *>(swa::swa_prefill_pair_kernel<D>)
           : plan.sink_last ? reinterpret_cast<const void *>(swa::swa_prefill_kernel<D, true>)
                            : reinterpret_cast<const void *>(swa::swa_prefill_kernel<D, false>);
  const cudaError_t attr_err = ensure_max_dynamic_smem(kernel, dev.max_smem_optin);
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(prefill)");

  swa::PrefillArgs a;
  a.out = reinterpret_cast<__nv_bfloat16 *>(out);
  a.lse = lse;
  a.B = B;
  a.L = L;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.w = w;
  a.s = s;
  a.q_off = q_off;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.plan = plan;
  a.qb_first = qb_first;
  a.n_items = B * Hkv * (pair ? swa::cdiv(plan.nqb - qb_first, 2) : plan.nqb - qb_first);
  a.stages = stages;
  a.kv_chunk = plan.slot_keys * 128;
  a.sep_stage = sep_stage ? 1 : 0;
  const int grid = swa::imin(a.n_items, dev.sms);
  cudaError_t e =
      pair ? launch_pdl(swa::swa_prefill_pair_kernel<D>, dim3(grid), dim3(swa::kPairThreads), smem,
                        stream, tq, tk, tv, tks, tvs, to, a)
           : plan.sink_last
               ? launch_pdl(swa::swa_prefill_kernel<D, true>, dim3(grid),
                            dim3(swa::kPrefillThreads), smem, stream, tq, tk, tv, tks, tvs, tkb,
                            tvb, to, a)
               : launch_pdl(swa::swa_prefill_kernel<D, false>, dim3(grid),
                            dim3(swa::kPrefillThreads), smem, stream, tq, tk, tv, tks, tvs, tkb,
                            tvb, to, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "swa_prefill launch");
  return SWA_OK;
}

// ------------------------------------------------------------------ decode

// SM count of the current device (the decode split policy depends on it), or
// 148 (a full B300) when no device is usable, so that a workspace-size query
// without a device still answers.
int decode_sms() {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 148;
  }
  DeviceInfo dev;
  if (current_device_info(&dev) != SWA_OK || dev.sms < 1) return 148;
  return dev.sms;
}

// Query heads one decode CTA packs: the largest of 4, 2, 1 that divides G.
// When the (sequence, KV head) pairs are too few to fill the GPU and the
// cache is short (cap = s + w slots, too few to split), one head per CTA
// instead: the K/V rows a group shares are then read again, from L2. A long
// cache is split over CTAs instead, and every K/V row is read once.
int head_group(int B, int Hq, int Hkv, long long cap, int sms) {
  const int G = Hq / Hkv;
  if ((long long)B * Hkv * 2 < sms && cap <= 512) return 1;
  if (G % 4 == 0) return 4;
  if (G % 2 == 0) return 2;
  return 1;
}

// The cache of each (sequence, KV head) is split over CTAs when it holds
// more slots than one CTA stages, or when there are too few (sequence, KV
// head, head group) units to fill the GPU and the cache is long. In the
// second case the splits hold at most 128 slots, so several CTAs share an SM
// and one CTA's copies overlap another's arithmetic, and there are at least
// two CTAs per SM where the cache allows 64 slots each. The count is fixed
// from the capacity s + w (positions are only known on the device).
int decode_splits(int B, int Hq, int Hkv, int w, int s, int sms) {
  const int G = Hq / Hkv;
  const long long cap = (long long)s + w;
  const long long units = (long long)B * Hkv * (G / head_group(B, Hq, Hkv, cap, sms));
  long long sp = (cap + swa::kDecodeMaxKeys - 1) / swa::kDecodeMaxKeys;
  if (units < sms && cap > 512) {
    const long long fine = (cap + 127) / 128;
    if (fine > sp) sp = fine;
    long long fill = (2LL * sms + units - 1) / units;
    const long long most = (cap + 63) / 64;
    if (fill > most) fill = most;
    if (fill > sp) sp = fill;
  }
  return (int)(sp < 1 ? 1 : sp);
}

int decode_max_keys(int w, int s, int splits) {
  return (int)(((long long)s + w + splits - 1) / splits);
}

size_t decode_workspace(int B, int Hq, int Hkv, int d, int w, int s, int sms) {
  const int sp = decode_splits(B, Hq, Hkv, w, s, sms);
  if (sp <= 1) return 0;
  const size_t n = (size_t)B * Hq * sp;
  return n * d * sizeof(float) + n * sizeof(float2);
}

template <int D, int HG, bool kPaged>
cudaError_t launch_decode_t(const swa::DecodeArgs &a, int B, cudaStream_t stream) {
  // (B * Hq * splits <= INT_MAX is checked by the caller)
  const int G = a.Hq / a.Hkv;
  const size_t smem = swa::DecodeSmem<D, HG>::bytes(a.max_keys);
  const cudaError_t attr_err = ensure_max_dynamic_smem(
      reinterpret_cast<const void *>(swa::swa_decode_kernel<D, HG, kPaged>),
      (int)swa::DecodeSmem<D, HG>::bytes(swa::kDecodeMaxKeys));
  if (attr_err != cudaSuccess) return attr_err;
  dim3 grid(a.splits, a.Hkv * (G / HG), B);
  cudaError_t e = launch_pdl(swa::swa_decode_kernel<D, HG, kPaged>, grid,
                             dim3(swa::kDecodeThreads), smem, stream, a);
  // (a stalled test launch writes no partials, so there is nothing to combine)
  if (e != cudaSuccess || a.splits == 1 || a.stall) return e;
  const unsigned combine_ctas = (unsigned)((long long)B * a.Hq);
  return launch_pdl(swa::swa_decode_combine_kernel<D>, dim3(combine_ctas),
                    dim3(swa::kCombineThreads), 0, stream, a.part_o, a.part_ml, a.out, a.splits);
}

template <int D, bool kPaged>
cudaError_t launch_decode_p(const swa::DecodeArgs &a, int B, int sms, cudaStream_t stream) {
  switch (head_group(B, a.Hq, a.Hkv, (long long)a.w + a.s, sms)) {
    case 4: return launch_decode_t<D, 4, kPaged>(a, B, stream);
    case 2: return launch_decode_t<D, 2, kPaged>(a, B, stream);
    default: return launch_decode_t<D, 1, kPaged>(a, B, stream);
  }
}

template <int D>
cudaError_t launch_decode_d(const swa::DecodeArgs &a, int B, int sms, cudaStream_t stream) {
  return a.page_table ? launch_decode_p<D, true>(a, B, sms, stream)
                      : launch_decode_p<D, false>(a, B, sms, stream);
}

int check_heads(int Hq, int Hkv) {
  if (Hq < 1 || Hkv < 1) return fail(SWA_ERR_INVALID_ARG, "Hq and Hkv must be >= 1");
  if (Hq % Hkv != 0) return fail(SWA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Hq / Hkv > 128) return fail(SWA_ERR_UNSUPPORTED, "group size Hq/Hkv > 128");
  return SWA_OK;
}

int check_scale(float scale) {
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(SWA_ERR_INVALID_ARG, "scale must be finite and > 0");
  return SWA_OK;
}

// Scratch of swa_decode_noalloc: the split-KV partial results live here
// instead of in a caller workspace. Every device that loads the library holds
// it until exit; calls that overlap on the GPU share (and race on) it.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[SWA_DECODE_NOALLOC_SCRATCH_BYTES];

// The current CUDA context's unique id (0 if there is none yet), through the
// driver entry points looked up at run time. The id changes whenever a
// context is created again (for example after cudaDeviceReset), so it tells a
// stale scratch address from a valid one.
unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext *);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current context. It is looked up
// once per context (cudaGetSymbolAddress needs the device current, and the
// array moves when the module is loaded again in a new context, e.g. after a
// device reset).
int noalloc_scratch_ptr(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static std::mutex mu;
  static std::map<unsigned long long, void *> ptrs;  // context id -> address
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = current_context_id();
  if (id != 0) {
    const auto it = ptrs.find(id);
    if (it != ptrs.end()) {
      *out = it->second;
      return SWA_OK;
    }
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);  // makes the primary context current
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
  if (id == 0) id = current_context_id();
  if (id != 0) ptrs[id] = p;
  *out = p;
  return SWA_OK;
}

// Device workspace of swa_prefill_chunk: the append's positions, then the
// staged keys and values over the prefix + chunk rows.
struct ChunkWorkspace {
  size_t pos, kx, vx, total;
};

ChunkWorkspace chunk_workspace(int B, int T, int Hkv, int d, int w, int s, long long pos0) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t Lx = (size_t)(swa::chunk_prefix_rows(pos0, w, s) + T);
  const size_t kvb = up((size_t)B * Lx * Hkv * d * 2);
  ChunkWorkspace c;
  c.pos = 0;
  c.kx = up((size_t)B * sizeof(int));
  c.vx = c.kx + kvb;
  c.total = c.vx + kvb;
  return c;
}

// Device workspace of swa_prefill_backward: D = dO . O per row (fp32
// [B, Hq, L]), then the sink keys' fp32 dK and dV accumulators ([B, Hkv,
// s_eff, d] each).
struct BwdWorkspace {
  size_t D, sink_dk, sink_dv, total;
};

BwdWorkspace bwd_workspace(int B, int L, int Hq, int Hkv, int d, int s) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t s_eff = (size_t)(s < L ? s : L);
  BwdWorkspace w;
  w.D = 0;
  w.sink_dk = up((size_t)B * Hq * L * sizeof(float));
  w.sink_dv = w.sink_dk + up((size_t)B * Hkv * s_eff * d * sizeof(float));
  w.total = w.sink_dv + up((size_t)B * Hkv * s_eff * d * sizeof(float));
  return w;
}

template <int D>
int launch_backward(const void *q, const void *k, const void *v, const void *out,
                    const void *dout, const float *lse, void *dq, void *dk, void *dv, int B, int L,
                    int Hq, int Hkv, int w, int s, float scale, void *workspace,
                    cudaStream_t stream, const DeviceInfo &dev) {
  const swa::PrefillPlan plan = swa::make_plan(L, Hq, Hkv, w, s);
  const BwdWorkspace ws = bwd_workspace(B, L, Hq, Hkv, D, s);
  uint8_t *base = reinterpret_cast<uint8_t *>(workspace);
  swa::BwdArgs a;
  a.out = reinterpret_cast<const __nv_bfloat16 *>(out);
  a.dout = reinterpret_cast<const __nv_bfloat16 *>(dout);
  a.lse = lse;
  a.D = reinterpret_cast<float *>(base + ws.D);
  a.sink_dk = reinterpret_cast<float *>(base + ws.sink_dk);
  a.sink_dv = reinterpret_cast<float *>(base + ws.sink_dv);
  a.dq = reinterpret_cast<__nv_bfloat16 *>(dq);
  a.dk = reinterpret_cast<__nv_bfloat16 *>(dk);
  a.dv = reinterpret_cast<__nv_bfloat16 *>(dv);
  a.B = B;
  a.L = L;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.w = w;
  a.s = s;
  a.s_eff = s < L ? s : L;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.plan = plan;
  a.n_band_tiles = L > s ? swa::cdiv(L - s, 128) : 0;
  a.n_sink_items = a.s_eff > 0 ? swa::cdiv(a.s_eff, 128) * swa::cdiv(plan.nqb, swa::kBwdSinkChunk) : 0;

  // 1. D = dO . O, sink accumulators cleared
  const long long n_rows = (long long)B * L * Hq;
  const long long n_sink = (long long)B * Hkv * a.s_eff * D;
  // a grid-stride kernel: 16 blocks of 256 threads per SM, fewer for small inputs
  const long long rows_per_block = 8LL * (32 / (D / 8)) * 4;  // warps x rows per pass x passes
  long long blocks = (n_rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 16LL * dev.sms) blocks = 16LL * dev.sms;
  if (blocks < 1) blocks = 1;
  cudaError_t e = launch_pdl(swa::swa_bwd_pre_kernel<D>, dim3((unsigned)blocks), dim3(256), 0,
                             stream, a, n_rows, n_sink);
  if (e != cudaSuccess) return cuda_fail(e, "swa_prefill_backward pre launch");

  // 2. dQ: one query block per work item, the forward's tiles
  {
    CUtensorMap tq, tdo, tk, tv, tks, tvs;
    int rc;
    if ((rc = make_map_bf16_4d(&tq, q, B, L, Hq, D, plan.G, plan.Tq))) return rc;
    if ((rc = make_map_bf16_4d(&tdo, dout, B, L, Hq, D, plan.G, plan.Tq))) return rc;
    if ((rc = make_map_bf16_4d(&tk, k, B, L, Hkv, D, 1, plan.n_band))) return rc;
    if ((rc = make_map_bf16_4d(&tv, v, B, L, Hkv, D, 1, plan.n_band))) return rc;
    if (plan.n_sink > 0) {
      if ((rc = make_map_bf16_4d(&tks, k, B, L, Hkv, D, 1, plan.s_box))) return rc;
      if ((rc = make_map_bf16_4d(&tvs, v, B, L, Hkv, D, 1, plan.s_box))) return rc;
    } else {
      tks = tk;
      tvs = tv;
    }
    const int stages = swa::BwdDqSmem<D>::stages(plan, dev.max_smem_optin);
    if (stages < 2) return fail(SWA_ERR_UNSUPPORTED, "not enough shared memory for the dQ pipeline");
    const size_t smem = swa::BwdDqSmem<D>::bytes(plan, stages);
    const cudaError_t attr = ensure_max_dynamic_smem(
        reinterpret_cast<const void *>(swa::swa_bwd_dq_kernel<D>), dev.max_smem_optin);
    if (attr != cudaSuccess) return cuda_fail(attr, "cudaFuncSetAttribute(backward dQ)");
    swa::BwdArgs ad = a;
    ad.n_items = B * Hkv * plan.nqb;
    ad.stages = stages;
    ad.kv_chunk = plan.slot_keys * 128;
    const int grid = swa::imin(ad.n_items, dev.sms);
    e = launch_pdl(swa::swa_bwd_dq_kernel<D>, dim3(grid), dim3(swa::kPrefillThreads), smem, stream,
                   tq, tdo, tk, tv, tks, tvs, ad);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "swa_prefill_backward dQ launch");
  }
  // 3. dK, dV: one key tile per CTA
  {
    CUtensorMap tq, tdo, tkt, tvt;
    int rc;
    if ((rc = make_map_bf16_4d(&tq, q, B, L, Hq, D, plan.G, plan.Tq))) return rc;
    if ((rc = make_map_bf16_4d(&tdo, dout, B, L, Hq, D, plan.G, plan.Tq))) return rc;
    if ((rc = make_map_bf16_4d(&tkt, k, B, L, Hkv, D, 1, 128))) return rc;
    if ((rc = make_map_bf16_4d(&tvt, v, B, L, Hkv, D, 1, 128))) return rc;
    const size_t smem = swa::BwdDkvSmem<D>::bytes();
    const cudaError_t attr = ensure_max_dynamic_smem(
        reinterpret_cast<const void *>(swa::swa_bwd_dkv_kernel<D>), (int)smem);
    if (attr != cudaSuccess) return cuda_fail(attr, "cudaFuncSetAttribute(backward dK dV)");
    const long long items = (long long)B * Hkv * (a.n_band_tiles + a.n_sink_items);
    if (items > 0x7FFFFFFFll) return fail(SWA_ERR_UNSUPPORTED, "too many key tiles");
    if (items > 0) {
      e = launch_pdl(swa::swa_bwd_dkv_kernel<D>, dim3((unsigned)items), dim3(swa::kPrefillThreads),
                     smem, stream, tq, tdo, tkt, tvt, a);
      if (e == cudaSuccess) e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "swa_prefill_backward dK/dV launch");
    }
  }
  // 4. the sink keys' rows of dK and dV
  if (n_sink > 0) {
    e = launch_pdl(swa::swa_bwd_sink_out_kernel, dim3((unsigned)((n_sink + 255) / 256)),
                   dim3(256), 0, stream, a, D);
    if (e != cudaSuccess) return cuda_fail(e, "swa_prefill_backward sink launch");
  }
  return SWA_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char *swa_status_string(int status) {
  switch (status) {
    case SWA_OK: return "ok";
    case SWA_ERR_INVALID_ARG: return "invalid argument";
    case SWA_ERR_UNSUPPORTED: return "unsupported configuration";
    case SWA_ERR_CUDA: return "CUDA error";
    case SWA_ERR_DEVICE: return "no usable sm_103a device";
    default: return "unknown status";
  }
}

const char *swa_last_error(void) { return g_last_error; }

long long swa_cache_slot(long long pos, int w, int s) {
  if (pos < 0 || w < 1 || s < 0) return -1;
  return swa::ring_slot(pos, w, s);
}

size_t swa_cache_bytes(int B, int Hkv, int d, int w, int s) {
  if (B < 0 || Hkv < 0 || d < 0 || w < 0 || s < 0) return 0;
  return (size_t)B * Hkv * ((size_t)s + w) * d * 2;
}

int swa_prefill_plan(int L, int Hq, int Hkv, int d, int w, int s, int plan[8]) {
  if (!plan) return fail(SWA_ERR_INVALID_ARG, "plan is NULL");
  if (L < 1 || w < 1 || s < 0) return fail(SWA_ERR_INVALID_ARG, "need L >= 1, w >= 1, s >= 0");
  int rc = check_heads(Hq, Hkv);
  if (rc) return rc;
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  const swa::PrefillPlan p = prefill_plan_for(d, L, Hq, Hkv, w, s);
  plan[0] = p.Tq;
  plan[1] = p.rows;
  plan[2] = p.n_band;
  plan[3] = p.s_box;
  plan[4] = p.n_sink;
  plan[5] = prefill_stages(d, p, 232448);
  plan[6] = 0;
  plan[7] = (int)prefill_smem_bytes(d, p, plan[5], prefill_sep_stage(d, p, 232448));
  int dev_count = 0;
  if (cudaGetDeviceCount(&dev_count) == cudaSuccess && dev_count > 0) {
    DeviceInfo dev;
    if (current_device_info(&dev) == SWA_OK) {
      plan[5] = prefill_stages(d, p, dev.max_smem_optin);
      plan[6] = dev.sms;
      plan[7] = (int)prefill_smem_bytes(d, p, plan[5], prefill_sep_stage(d, p, dev.max_smem_optin));
    }
  } else {
    cudaGetLastError();
  }
  return SWA_OK;
}

int swa_prefill(const void *q, const void *k, const void *v, void *out, int B, int L, int Hq,
                int Hkv, int d, int w, int s, float scale, swa_stream_t stream) {
  if (!q || !k || !v || !out) return fail(SWA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(SWA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (B < 1 || L < 1) return fail(SWA_ERR_INVALID_ARG, "B and L must be >= 1");
  if (w < 1) return fail(SWA_ERR_INVALID_ARG, "window w must be >= 1");
  if (s < 0) return fail(SWA_ERR_INVALID_ARG, "sink count s must be >= 0");
  int rc = check_heads(Hq, Hkv);
  if (rc) return rc;
  if ((rc = check_scale(scale))) return rc;
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  if ((long long)B * Hkv * swa::cdiv(L, 128 / (Hq / Hkv)) > 0x7FFFFFFFll)
    return fail(SWA_ERR_UNSUPPORTED, "too many query blocks");
  DeviceInfo dev;
  if ((rc = current_device_info(&dev))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d == 64) return launch_prefill<64>(q, k, v, out, B, L, Hq, Hkv, w, s, scale, st, dev);
  return launch_prefill<128>(q, k, v, out, B, L, Hq, Hkv, w, s, scale, st, dev);
}

int swa_prefill_lse(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                    int L, int Hq, int Hkv, int d, int w, int s, float scale,
                    swa_stream_t stream) {
  if (!lse) return fail(SWA_ERR_INVALID_ARG, "lse is NULL");
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(SWA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (!q || !k || !v || !out) return fail(SWA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(SWA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (B < 1 || L < 1) return fail(SWA_ERR_INVALID_ARG, "B and L must be >= 1");
  if (w < 1) return fail(SWA_ERR_INVALID_ARG, "window w must be >= 1");
  if (s < 0) return fail(SWA_ERR_INVALID_ARG, "sink count s must be >= 0");
  int rc = check_heads(Hq, Hkv);
  if (rc) return rc;
  if ((rc = check_scale(scale))) return rc;
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  if ((long long)B * Hkv * swa::cdiv(L, 128 / (Hq / Hkv)) > 0x7FFFFFFFll)
    return fail(SWA_ERR_UNSUPPORTED, "too many query blocks");
  DeviceInfo dev;
  if ((rc = current_device_info(&dev))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d == 64) return launch_prefill<64>(q, k, v, out, B, L, Hq, Hkv, w, s, scale, st, dev, 0, lse);
  return launch_prefill<128>(q, k, v, out, B, L, Hq, Hkv, w, s, scale, st, dev, 0, lse);
}

size_t swa_prefill_backward_workspace_size(int B, int L, int Hq, int Hkv, int d, int s) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || s < 0 || !supported_d(d)) return 0;
  return bwd_workspace(B, L, Hq, Hkv, d, s).total;
}

int swa_prefill_backward(const void *q, const void *k, const void *v, const void *out,
                         const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                         int L, int Hq, int Hkv, int d, int w, int s, float scale,
                         void *workspace, size_t workspace_bytes, swa_stream_t stream) {
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv)
    return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(SWA_ERR_INVALID_ARG, "pointers must be 16-byte aligned (lse 4-byte)");
  if (B < 1 || L < 1) return fail(SWA_ERR_INVALID_ARG, "B and L must be >= 1");
  if (w < 1) return fail(SWA_ERR_INVALID_ARG, "window w must be >= 1");
  if (s < 0) return fail(SWA_ERR_INVALID_ARG, "sink count s must be >= 0");
  int rc = check_heads(Hq, Hkv);
  if (rc) return rc;
  if ((rc = check_scale(scale))) return rc;
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  if (B > 65535) return fail(SWA_ERR_UNSUPPORTED, "B > 65535");
  if ((long long)B * Hkv * swa::cdiv(L, 128 / (Hq / Hkv)) > 0x7FFFFFFFll)
    return fail(SWA_ERR_UNSUPPORTED, "too many query blocks");
  const size_t need = bwd_workspace(B, L, Hq, Hkv, d, s).total;
  if (!workspace || workspace_bytes < need)
    return fail(SWA_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                workspace ? workspace_bytes : (size_t)0, need);
  DeviceInfo dev;
  if ((rc = current_device_info(&dev))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d == 64)
    return launch_backward<64>(q, k, v, out, dout, lse, dq, dk, dv, B, L, Hq, Hkv, w, s, scale,
                               workspace, st, dev);
  return launch_backward<128>(q, k, v, out, dout, lse, dq, dk, dv, B, L, Hq, Hkv, w, s, scale,
                              workspace, st, dev);
}

int swa_cache_append(const void *k_new, const void *v_new, void *kcache, void *vcache,
                     const int *pos_start, int B, int T, int Hkv, int d, int w, int s,
                     swa_stream_t stream) {
  if (!k_new || !v_new || !kcache || !vcache || !pos_start)
    return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kcache) || !aligned16(vcache))
    return fail(SWA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (B < 1 || T < 1 || Hkv < 1) return fail(SWA_ERR_INVALID_ARG, "B, T and Hkv must be >= 1");
  if (w < 1 || s < 0) return fail(SWA_ERR_INVALID_ARG, "need w >= 1 and s >= 0");
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  if (B > 65535) return fail(SWA_ERR_UNSUPPORTED, "B > 65535");
  DeviceInfo dev;
  int rc = current_device_info(&dev);
  if (rc) return rc;
  // only the tokens that survive the call are visited: at most s + w of them
  const int max_surv = (int)(T < (long long)s + w ? T : (long long)s + w);
  const long long n = (long long)max_surv * Hkv * (d / 8);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFll) return fail(SWA_ERR_UNSUPPORTED, "append too large");
  cudaError_t e = launch_pdl(
      swa::swa_append_kernel, dim3((unsigned)blocks, B), dim3(threads), 0,
      reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<const uint4 *>(k_new),
      reinterpret_cast<const uint4 *>(v_new), reinterpret_cast<uint4 *>(kcache),
      reinterpret_cast<uint4 *>(vcache), pos_start, T, Hkv, d, w, s, max_surv);
  if (e != cudaSuccess) return cuda_fail(e, "swa_cache_append launch");
  return SWA_OK;
}

size_t swa_prefill_chunk_workspace_size(int B, int T, int Hq, int Hkv, int d, int w, int s,
                                        long long pos0) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || w < 1 || s < 0 || pos0 < 0 ||
      !supported_d(d))
    return 0;
  return chunk_workspace(B, T, Hkv, d, w, s, pos0).total;
}

// The chunked prefill over a ring cache (src.table == nullptr) or a paged
// pool: stage the kept K/V rows and the chunk's, run the prefill kernel on
// the query blocks holding chunk rows (q read and out written in place), then
// append the chunk.
static int prefill_chunk_impl(const void *q, const void *k_new, const void *v_new, void *kcache,
                       void *vcache, const int *page_table, int page_size, int max_pages,
                       int n_pages, void *out, int B, int T, int Hq, int Hkv, int d, int w, int s,
                       long long pos0, float scale, void *workspace, size_t workspace_bytes,
                       swa_stream_t stream) {
  if (!q || !k_new || !v_new || !kcache || !vcache || !out)
    return fail(SWA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(kcache) ||
      !aligned16(vcache) || !aligned16(out) || !aligned16(workspace))
    return fail(SWA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (B < 1 || T < 1) return fail(SWA_ERR_INVALID_ARG, "B and T must be >= 1");
  if (w < 1) return fail(SWA_ERR_INVALID_ARG, "window w must be >= 1");
  if (s < 0) return fail(SWA_ERR_INVALID_ARG, "sink count s must be >= 0");
  if (pos0 < 0) return fail(SWA_ERR_INVALID_ARG, "pos0 must be >= 0");
  int rc = check_heads(Hq, Hkv);
  if (rc) return rc;
  if ((rc = check_scale(scale))) return rc;
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  if (pos0 + T > 0x7FFFFFFFll) return fail(SWA_ERR_UNSUPPORTED, "positions beyond int32");
  if (B > 65535) return fail(SWA_ERR_UNSUPPORTED, "B > 65535");
  const ChunkWorkspace ws = chunk_workspace(B, T, Hkv, d, w, s, pos0);
  if (!workspace || workspace_bytes < ws.total)
    return fail(SWA_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, ws.total);
  const int n_pre = (int)swa::chunk_prefix_rows(pos0, w, s);
  const int Lx = n_pre + T;
  const int Tq = 128 / (Hq / Hkv);  // query positions per prefill block
  if ((long long)B * Hkv * swa::cdiv(Lx, Tq) > 0x7FFFFFFFll)
    return fail(SWA_ERR_UNSUPPORTED, "too many query blocks");
  DeviceInfo dev;
  if ((rc = current_device_info(&dev))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *base = reinterpret_cast<uint8_t *>(workspace);
  int *wpos = reinterpret_cast<int *>(base + ws.pos);
  void *kx = base + ws.kx, *vx = base + ws.vx;

  // 1. stage the keys and values [kept cache rows | chunk] contiguously
  swa::ChunkSource src;
  src.kcache = reinterpret_cast<const uint4 *>(kcache);
  src.vcache = reinterpret_cast<const uint4 *>(vcache);
  src.table = page_table;
  src.page_size = page_size;
  src.max_pages = max_pages;
  src.n_pages = n_pages;
  const int threads = 256;
  long long n = (long long)Lx * 2 * Hkv * (d / 8);
  if (n < B) n = B;
  const long long blocks = (n + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFll) return fail(SWA_ERR_UNSUPPORTED, "chunk too large");
  cudaError_t e = launch_pdl(
      swa::swa_chunk_stage_kernel, dim3((unsigned)blocks, B), dim3(threads), 0, st,
      reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), src,
      reinterpret_cast<uint4 *>(kx), reinterpret_cast<uint4 *>(vx), wpos, B, T, Hkv, d, w, s,
      pos0, n_pre);
  if (e != cudaSuccess) return cuda_fail(e, "chunk stage launch");
  // 2. the prefill kernel over the staged rows, reading q and writing out in
  // place (query blocks made only of prefix rows are skipped)
  const int qb_first = n_pre / Tq;
  rc = d == 64 ? launch_prefill<64>(q, kx, vx, out, B, Lx, Hq, Hkv, w, s, scale, st, dev, qb_first,
                                    nullptr, n_pre)
               : launch_prefill<128>(q, kx, vx, out, B, Lx, Hq, Hkv, w, s, scale, st, dev,
                                     qb_first, nullptr, n_pre);
  if (rc) return rc;
  // 3. append the chunk (after the staging read every cache row it needs)
  if (page_table == nullptr)
    return swa_cache_append(k_new, v_new, kcache, vcache, wpos, B, T, Hkv, d, w, s, stream);
  return swa_paged_append(k_new, v_new, kcache, vcache, page_table, wpos, B, T, Hkv, d, page_size,
                          max_pages, n_pages, w, s, stream);
}

int swa_prefill_chunk(const void *q, const void *k_new, const void *v_new, void *kcache,
                      void *vcache, void *out, int B, int T, int Hq, int Hkv, int d, int w, int s,
                      long long pos0, float scale, void *workspace, size_t workspace_bytes,
                      swa_stream_t stream) {
  return prefill_chunk_impl(q, k_new, v_new, kcache, vcache, nullptr, 0, 0, 0, out, B, T, Hq, Hkv,
                            d, w, s, pos0, scale, workspace, workspace_bytes, stream);
}

int swa_paged_prefill_chunk(const void *q, const void *k_new, const void *v_new, void *kpool,
                            void *vpool, const int *page_table, void *out, int B, int T, int Hq,
                            int Hkv, int d, int page_size, int max_pages, int n_pages, int w,
                            int s, long long pos0, float scale, void *workspace,
                            size_t workspace_bytes, swa_stream_t stream) {
  if (!page_table) return fail(SWA_ERR_INVALID_ARG, "null page table");
  if (page_size < 1 || max_pages < 1 || n_pages < 1)
    return fail(SWA_ERR_INVALID_ARG, "page_size, max_pages and n_pages must be >= 1");
  return prefill_chunk_impl(q, k_new, v_new, kpool, vpool, page_table, page_size, max_pages,
                            n_pages, out, B, T, Hq, Hkv, d, w, s, pos0, scale, workspace,
                            workspace_bytes, stream);
}

size_t swa_decode_workspace_size(int B, int Hq, int Hkv, int d, int w, int s) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || w < 1 || s < 0 || !supported_d(d)) return 0;
  return decode_workspace(B, Hq, Hkv, d, w, s, decode_sms());
}

int decode_impl(const void *q, const void *k_new, const void *v_new, const void *kcache,
                const void *vcache, const int *pos, void *out, int B, int Hq, int Hkv, int d,
                int w, int s, float scale, void *workspace, size_t workspace_bytes,
                swa_stream_t stream, const int *page_table = nullptr, int page_size = 0,
                int max_pages = 0, int n_pages = 0,
                unsigned long long wait_ns = swa::kDecodeWaitNs, int stall = 0);

int swa_decode(const void *q, const void *kcache, const void *vcache, const int *pos, void *out,
               int B, int Hq, int Hkv, int d, int w, int s, float scale, void *workspace,
               size_t workspace_bytes, swa_stream_t stream) {
  return decode_impl(q, nullptr, nullptr, kcache, vcache, pos, out, B, Hq, Hkv, d, w, s, scale,
                     workspace, workspace_bytes, stream);
}

int swa_append_decode(const void *q, const void *k_new, const void *v_new, void *kcache,
                      void *vcache, const int *pos, void *out, int B, int Hq, int Hkv, int d,
                      int w, int s, float scale, void *workspace, size_t workspace_bytes,
                      swa_stream_t stream) {
  if (!k_new || !v_new) return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_new) || !aligned16(v_new))
    return fail(SWA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  return decode_impl(q, k_new, v_new, kcache, vcache, pos, out, B, Hq, Hkv, d, w, s, scale,
                     workspace, workspace_bytes, stream);
}

int decode_impl(const void *q, const void *k_new, const void *v_new, const void *kcache,
                const void *vcache, const int *pos, void *out, int B, int Hq, int Hkv, int d,
                int w, int s, float scale, void *workspace, size_t workspace_bytes,
                swa_stream_t stream, const int *page_table, int page_size, int max_pages,
                int n_pages, unsigned long long wait_ns, int stall) {
  if (!q || !kcache || !vcache || !pos || !out) return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
    return fail(SWA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (B < 1) return fail(SWA_ERR_INVALID_ARG, "B must be >= 1");
  if (w < 1 || s < 0) return fail(SWA_ERR_INVALID_ARG, "need w >= 1 and s >= 0");
  int rc = check_heads(Hq, Hkv);
  if (rc) return rc;
  if ((rc = check_scale(scale))) return rc;
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  if (B > 65535 || Hq > 65535) return fail(SWA_ERR_UNSUPPORTED, "B or Hq > 65535");
  // the split policy (and so the workspace) depends on the current device's SM count
  const int sms = decode_sms();
  const int splits = decode_splits(B, Hq, Hkv, w, s, sms);
  if ((long long)B * Hq * splits > 0x7FFFFFFFLL)
    return fail(SWA_ERR_UNSUPPORTED, "B * Hq * splits (%d * %d * %d) is beyond the grid limit", B,
                Hq, splits);
  const size_t need = decode_workspace(B, Hq, Hkv, d, w, s, sms);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return fail(SWA_ERR_INVALID_ARG, "workspace of %zu bytes (16-byte aligned) required, got %zu",
                need, workspace ? workspace_bytes : (size_t)0);
  DeviceInfo dev;
  if ((rc = current_device_info(&dev))) return rc;
  swa::DecodeArgs a;
  a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
  a.kc = reinterpret_cast<const __nv_bfloat16 *>(kcache);
  a.vc = reinterpret_cast<const __nv_bfloat16 *>(vcache);
  a.k_new = reinterpret_cast<const __nv_bfloat16 *>(k_new);
  a.v_new = reinterpret_cast<const __nv_bfloat16 *>(v_new);
  a.kc_w = const_cast<__nv_bfloat16 *>(a.kc);
  a.vc_w = const_cast<__nv_bfloat16 *>(a.vc);
  a.pos = pos;
  a.out = reinterpret_cast<__nv_bfloat16 *>(out);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.w = w;
  a.s = s;
  a.splits = splits;
  a.max_keys = decode_max_keys(w, s, a.splits);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.page_table = page_table;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.n_pages = n_pages;
  a.wait_ns = wait_ns;
  a.stall = stall;
  const size_t n = (size_t)B * Hq * a.splits;
  a.part_o = a.splits > 1 ? reinterpret_cast<float *>(workspace) : nullptr;
  a.part_ml = a.splits > 1 ? reinterpret_cast<float2 *>(reinterpret_cast<char *>(workspace) +
                                                        n * d * sizeof(float))
                           : nullptr;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = d == 64 ? launch_decode_d<64>(a, B, sms, st)
                          : launch_decode_d<128>(a, B, sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "swa_decode launch");
  return SWA_OK;
}

int swa_decode_noalloc(const void *q, const void *kcache, const void *vcache, const int *pos,
                       void *out, int B, int Hq, int Hkv, int d, int w, int s, float scale,
                       swa_stream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || w < 1 || s < 0 || !supported_d(d))
    return swa_decode(q, kcache, vcache, pos, out, B, Hq, Hkv, d, w, s, scale, nullptr, 0,
                      stream);  // let swa_decode report the argument error
  const size_t need = decode_workspace(B, Hq, Hkv, d, w, s, decode_sms());
  if (need > SWA_DECODE_NOALLOC_SCRATCH_BYTES)
    return fail(SWA_ERR_UNSUPPORTED,
                "swa_decode_noalloc: these sizes need %zu bytes of scratch, above its fixed "
                "maximum of %u bytes; use swa_decode with a workspace",
                need, (unsigned)SWA_DECODE_NOALLOC_SCRATCH_BYTES);
  void *scratch = nullptr;
  if (need > 0) {
    int rc = noalloc_scratch_ptr(&scratch);
    if (rc) return rc;
  }
  return swa_decode(q, kcache, vcache, pos, out, B, Hq, Hkv, d, w, s, scale, scratch,
                    need > 0 ? (size_t)SWA_DECODE_NOALLOC_SCRATCH_BYTES : 0, stream);
}

// ------------------------------------------------------------ paged layout

swa_page_pool *swa_page_pool_create(int n_pages) {
  if (n_pages < 1) {
    fail(SWA_ERR_INVALID_ARG, "n_pages must be >= 1");
    return nullptr;
  }
  swa_page_pool *pool = new (std::nothrow) swa_page_pool;
  if (!pool) {
    fail(SWA_ERR_INVALID_ARG, "out of host memory");
    return nullptr;
  }
  pool->n_pages = n_pages;
  pool->used.assign((size_t)n_pages, 0);
  pool->free_pages.reserve((size_t)n_pages);
  for (int i = n_pages - 1; i >= 0; --i) pool->free_pages.push_back(i);  // hands out 0, 1, ...
  return pool;
}

void swa_page_pool_destroy(swa_page_pool *pool) { delete pool; }

int swa_page_pool_free_pages(swa_page_pool *pool) {
  if (!pool) return -1;
  std::lock_guard<std::mutex> lock(pool->mu);
  return (int)pool->free_pages.size();
}

int swa_paged_reserve(swa_page_pool *pool, int *table, int max_pages, long long pos_hi, int w,
                      int s, int page_size) {
  return swa_paged_reserve_range(pool, table, max_pages, pos_hi, pos_hi, w, s, page_size);
}

// The pages of the union of K(p) over pos_lo <= p <= pos_hi: the sink pages
// and those of positions pos_lo - w + 1 .. pos_hi.
int swa_paged_reserve_range(swa_page_pool *pool, int *table, int max_pages, long long pos_lo,
                            long long pos_hi, int w, int s, int page_size) {
  if (!pool || !table) return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (max_pages < 1 || pos_lo < 0 || pos_hi < pos_lo || w < 1 || s < 0 || page_size < 1)
    return fail(SWA_ERR_INVALID_ARG,
                "need max_pages, w, page_size >= 1, s >= 0 and 0 <= pos_lo <= pos_hi");
  const long long last = pos_hi / page_size;
  if (last >= max_pages)
    return fail(SWA_ERR_UNSUPPORTED, "position %lld is beyond the %d-page table", pos_hi,
                max_pages);
  const long long sink_pages = ((long long)s + page_size - 1) / page_size;
  const long long win_lo = (pos_lo - w + 1 > 0 ? pos_lo - w + 1 : 0) / page_size;
  const long long sink_top = sink_pages < last + 1 ? sink_pages : last + 1;  // sink pages in use
  const long long keep_lo = win_lo > sink_pages ? win_lo : sink_pages;      // window pages
  std::lock_guard<std::mutex> lock(pool->mu);
  auto valid = [&](int pg) { return pg >= 0 && pg < pool->n_pages && pool->used[(size_t)pg]; };
  // Past the sink pages, the mapped pages form one run (pages are mapped and
  // released in position order). Find it from the top: the unmapped pages
  // above it, then the run itself. This costs the window plus whatever the
  // positions moved since the last call, not the whole table.
  long long lp = last;
  while (lp >= sink_pages && table[lp] < 0) --lp;
  const long long run_top = lp;
  while (lp >= sink_pages && table[lp] >= 0) {
    if (!valid(table[lp]))
      return fail(SWA_ERR_INVALID_ARG, "page table entry %lld was not handed out by this pool", lp);
    --lp;
  }
  const long long run_bot = lp + 1;  // run = [run_bot, run_top], possibly empty
  // leaving: the run below the window; coming: unmapped sink and window pages
  const long long rel_lo = run_bot, rel_hi = run_top < keep_lo - 1 ? run_top : keep_lo - 1;
  const long long n_rel = rel_hi >= rel_lo ? rel_hi - rel_lo + 1 : 0;
  // window pages outside the run: below it (only if it starts inside the
  // window) and above it
  const long long a_lo = keep_lo, a_hi = run_bot - 1 < last ? run_bot - 1 : last;
  const long long b_lo = run_top + 1 > keep_lo ? run_top + 1 : keep_lo, b_hi = last;
  long long need = 0;
  for (long long i = 0; i < sink_top; ++i) need += table[i] < 0;
  for (long long i = a_lo; i <= a_hi; ++i) need += table[i] < 0;
  for (long long i = b_lo; i <= b_hi; ++i) need += table[i] < 0;
  if (need > (long long)pool->free_pages.size() + n_rel)
    return fail(SWA_ERR_UNSUPPORTED, "page pool exhausted: %lld pages needed, %zu free", need,
                pool->free_pages.size());
  for (long long i = rel_lo; i <= rel_hi; ++i) {
    pool->used[(size_t)table[i]] = 0;
    pool->free_pages.push_back(table[i]);
    table[i] = -1;
  }
  auto take = [&](long long i) {
    const int pg = pool->free_pages.back();
    pool->free_pages.pop_back();
    pool->used[(size_t)pg] = 1;
    table[i] = pg;
  };
  for (long long i = 0; i < sink_top; ++i)
    if (table[i] < 0) take(i);
  for (long long i = a_lo; i <= a_hi; ++i)
    if (table[i] < 0) take(i);
  for (long long i = b_lo; i <= b_hi; ++i)
    if (table[i] < 0) take(i);
  return SWA_OK;
}

int swa_paged_release(swa_page_pool *pool, int *table, int max_pages) {
  if (!pool || !table) return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (max_pages < 1) return fail(SWA_ERR_INVALID_ARG, "max_pages must be >= 1");
  std::lock_guard<std::mutex> lock(pool->mu);
  for (int lp = 0; lp < max_pages; ++lp) {
    const int pg = table[lp];
    if (pg < 0) continue;
    if (pg >= pool->n_pages || !pool->used[(size_t)pg])
      return fail(SWA_ERR_INVALID_ARG, "page table entry %d was not handed out by this pool", lp);
    pool->used[(size_t)pg] = 0;
    pool->free_pages.push_back(pg);
    table[lp] = -1;
  }
  return SWA_OK;
}

int swa_paged_append(const void *k_new, const void *v_new, void *kpool, void *vpool,
                     const int *page_table, const int *pos_start, int B, int T, int Hkv, int d,
                     int page_size, int max_pages, int n_pages, int w, int s,
                     swa_stream_t stream) {
  if (!k_new || !v_new || !kpool || !vpool || !page_table || !pos_start)
    return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kpool) || !aligned16(vpool))
    return fail(SWA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (B < 1 || T < 1 || Hkv < 1) return fail(SWA_ERR_INVALID_ARG, "B, T and Hkv must be >= 1");
  if (w < 1 || s < 0) return fail(SWA_ERR_INVALID_ARG, "need w >= 1 and s >= 0");
  if (page_size < 1 || max_pages < 1 || n_pages < 1)
    return fail(SWA_ERR_INVALID_ARG, "page_size, max_pages and n_pages must be >= 1");
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  if (B > 65535) return fail(SWA_ERR_UNSUPPORTED, "B > 65535");
  DeviceInfo dev;
  int rc = current_device_info(&dev);
  if (rc) return rc;
  const int max_surv = (int)(T < (long long)s + w ? T : (long long)s + w);
  const long long n = (long long)max_surv * Hkv * (d / 8);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFll) return fail(SWA_ERR_UNSUPPORTED, "append too large");
  cudaError_t e = launch_pdl(
      swa::swa_paged_append_kernel, dim3((unsigned)blocks, B), dim3(threads), 0,
      reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<const uint4 *>(k_new),
      reinterpret_cast<const uint4 *>(v_new), reinterpret_cast<uint4 *>(kpool),
      reinterpret_cast<uint4 *>(vpool), page_table, pos_start, T, Hkv, d, w, s, max_surv,
      page_size, max_pages, n_pages);
  if (e != cudaSuccess) return cuda_fail(e, "swa_paged_append launch");
  return SWA_OK;
}

int swa_paged_decode(const void *q, const void *kpool, const void *vpool, const int *page_table,
                     const int *pos, void *out, int B, int Hq, int Hkv, int d, int page_size,
                     int max_pages, int n_pages, int w, int s, float scale, void *workspace,
                     size_t workspace_bytes, swa_stream_t stream) {
  if (!page_table) return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (page_size < 1 || max_pages < 1 || n_pages < 1)
    return fail(SWA_ERR_INVALID_ARG, "page_size, max_pages and n_pages must be >= 1");
  return decode_impl(q, nullptr, nullptr, kpool, vpool, pos, out, B, Hq, Hkv, d, w, s, scale,
                     workspace, workspace_bytes, stream, page_table, page_size, max_pages,
                     n_pages);
}

int swa_debug_decode_timeout(const void *q, const void *kcache, const void *vcache,
                             const int *pos, void *out, int B, int Hq, int Hkv, int d, int w,
                             int s, float scale, void *workspace, size_t workspace_bytes,
                             unsigned long long wait_ns, int stall, swa_stream_t stream) {
  return decode_impl(q, nullptr, nullptr, kcache, vcache, pos, out, B, Hq, Hkv, d, w, s, scale,
                     workspace, workspace_bytes, stream, nullptr, 0, 0, 0, wait_ns, stall);
}

int swa_debug_keymask(int L, int Hq, int Hkv, int d, int w, int s, int row0, int nrows,
                      uint32_t *bits, int *counts, swa_stream_t stream) {
  if (!bits || !counts) return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (L < 1 || w < 1 || s < 0) return fail(SWA_ERR_INVALID_ARG, "need L >= 1, w >= 1, s >= 0");
  if (row0 < 0 || nrows < 1 || (long long)row0 + nrows > L)
    return fail(SWA_ERR_INVALID_ARG, "rows [%d, %d) outside [0, %d)", row0, row0 + nrows, L);
  int rc = check_heads(Hq, Hkv);
  if (rc) return rc;
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  DeviceInfo dev;
  if ((rc = current_device_info(&dev))) return rc;
  const swa::PrefillPlan plan = prefill_plan_for(d, L, Hq, Hkv, w, s);
  swa::swa_keymask_kernel<<<nrows, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      plan, L, w, s, row0, nrows, bits, counts);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "swa_debug_keymask launch");
  return SWA_OK;
}

int swa_keymask_host(int L, int Hq, int Hkv, int d, int w, int s, int row0, int nrows,
                     uint32_t *bits, int *counts) {
  if (!bits || !counts) return fail(SWA_ERR_INVALID_ARG, "null pointer");
  if (L < 1 || w < 1 || s < 0) return fail(SWA_ERR_INVALID_ARG, "need L >= 1, w >= 1, s >= 0");
  if (row0 < 0 || nrows < 1 || (long long)row0 + nrows > L)
    return fail(SWA_ERR_INVALID_ARG, "rows [%d, %d) outside [0, %d)", row0, row0 + nrows, L);
  int rc = check_heads(Hq, Hkv);
  if (rc) return rc;
  if (!supported_d(d)) return fail(SWA_ERR_UNSUPPORTED, "head dimension %d (supported: 64, 128)", d);
  const swa::PrefillPlan plan = prefill_plan_for(d, L, Hq, Hkv, w, s);
  const int words = swa::cdiv(L, 32);
  for (int r = 0; r < nrows; ++r) {
    const int t = row0 + r;
    uint32_t *row_bits = bits + (size_t)r * words;
    for (int i = 0; i < words; ++i) row_bits[i] = 0u;
    int cnt = 0;
    const int qb = t / plan.Tq;
    const swa::BlockTiles bt =
        swa::block_tiles(plan, plan.bpi == 2 ? (qb & ~1) : qb, L, w, s);
    for (int i = 0; i < bt.n_tiles; ++i) {
      const swa::Tile tl = swa::tile_at(plan, bt, i, w, s);
      const bool full = swa::tile_full_for(tl, qb * plan.Tq, plan.Tq, w);
      const swa::ColRanges cr = swa::tile_ranges(tl, t, w, s);
      for (int c = 0; c < tl.ncols; ++c) {
        const int j = swa::tile_key(tl, c);
        const bool ok =
            full || (c >= cr.a_lo && c < cr.a_hi) || (c >= cr.b_lo && c < cr.b_hi);
        if (ok && j >= 0 && j < L) {
          row_bits[j / 32] |= 1u << (j % 32);
          ++cnt;
        }
      }
    }
    counts[r] = cnt;
  }
  return SWA_OK;
}

int swa_device_error(int *code, int clear) {
  if (!code) return fail(SWA_ERR_INVALID_ARG, "code is NULL");
  DeviceInfo dev;
  int rc = current_device_info(&dev);
  if (rc) return rc;
  cudaError_t e = cudaMemcpyFromSymbol(code, swa::g_device_error, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (clear) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(swa::g_device_error, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  }
  return SWA_OK;
}

int swa_prefill_select(int mode) {
  if (mode < 0 || mode > 2) return -1;
  return g_prefill_mode.exchange(mode);
}

}  // extern "C"
