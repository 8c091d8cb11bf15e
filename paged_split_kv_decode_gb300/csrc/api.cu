// The C ABI: context, argument validation, work-list upload, kernel dispatch and
// the cascade orchestration (mlxcel PR #1004, "compute shared prompt prefixes once
// per decode batch": Decomposition, Merge contract, Task items 2-5, Path
// attribution).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "context.h"

namespace psd {

static thread_local std::string g_error;

void clear_error() { g_error.clear(); }

void longest_first(const psd_work_item *items, int32_t n, int32_t *order) {
  for (int32_t i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order, order + n,
                   [items](int32_t a, int32_t b) { return items[a].n_tokens > items[b].n_tokens; });
}

psd_status fail(psd_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_error = buf;
  return st;
}

}  // namespace psd

using namespace psd;

namespace psd {

static const float kLog2e = 1.4426950408889634f;
static const int kLevel0Tcgen05MinRows = 32;
// Longest wait a test may set (about 1 s at 2 GHz): below the default limit.
static const long long kMaxTestWaitCycles = 2000000000LL;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

psd_status validate_args(const psd_decode_args *a) {
  if (!a) return fail(PSD_ERR_INVALID_ARG, "args: NULL");
  if ((a->batch > 0 && !a->q) || !a->k_pool || !a->v_pool || !a->page_indices_dev)
    return fail(PSD_ERR_INVALID_ARG, "args: NULL device pointer");
  if (!aligned16(a->q) || !aligned16(a->k_pool) || !aligned16(a->v_pool))
    return fail(PSD_ERR_INVALID_ARG, "args: q / k_pool / v_pool must be 16-byte aligned");
  if (a->batch < 0 || a->Hq < 1 || a->Hkv < 1 || a->Hq % a->Hkv != 0)
    return fail(PSD_ERR_INVALID_ARG, "args: need Hq %% Hkv == 0 (Hq %d, Hkv %d)", a->Hq, a->Hkv);
  if (a->Dqk < 8 || a->Dv < 8 || a->Dqk % 8 || a->Dv % 8)
    return fail(PSD_ERR_INVALID_ARG, "args: head dims must be positive multiples of 8");
  if (a->page_size < 1 || a->num_pages < 1 || a->num_page_indices < 0)
    return fail(PSD_ERR_INVALID_ARG, "args: page_size / num_pages / num_page_indices");
  if (a->num_pages > 0x7fffffffLL) return fail(PSD_ERR_INVALID_ARG, "args: num_pages > 2^31-1");
  if (a->kv_dtype != PSD_BF16 && a->kv_dtype != PSD_FP8_E4M3)
    return fail(PSD_ERR_INVALID_ARG, "args: kv_dtype %d", a->kv_dtype);
  if (!std::isfinite(a->sm_scale) || !std::isfinite(a->k_scale) || !std::isfinite(a->v_scale))
    return fail(PSD_ERR_INVALID_ARG, "args: scales must be finite");
  if (a->v_pool == a->k_pool && (a->Hkv != 1 || a->Dv > a->Dqk))
    return fail(PSD_ERR_INVALID_ARG, "args: a shared latent (v_pool == k_pool) needs Hkv == 1, Dv <= Dqk");
  return PSD_OK;
}

psd_status validate_items(const psd_decode_args *a, const psd_work_item *items, int32_t n,
                          int64_t out_rows, bool stacked, int32_t num_members) {
  const int P = a->page_size;
  for (int32_t i = 0; i < n; ++i) {
    const psd_work_item &it = items[i];
    if (stacked ? it.q_index != -1 : (it.q_index < 0 || it.q_index >= a->batch))
      return fail(PSD_ERR_INVALID_ARG, "item %d: q_index %d", i, it.q_index);
    if (it.n_tokens < 1 || it.page_off < 0 ||
        int64_t(it.page_off) + (it.n_tokens + P - 1) / P > a->num_page_indices)
      return fail(PSD_ERR_INVALID_ARG, "item %d: page_off %d / n_tokens %d outside the page table", i,
                  it.page_off, it.n_tokens);
    if (it.out_row < 0 || (!stacked && it.out_row >= out_rows))
      return fail(PSD_ERR_INVALID_ARG, "item %d: out_row %d outside [0, %lld)", i, it.out_row,
                  (long long)out_rows);
  }
  (void)num_members;
  return PSD_OK;
}

PartialLaunch base_launch(const psd_decode_args *a) {
  PartialLaunch L;
  L.q = a->q;
  L.k_pool = a->k_pool;
  L.v_pool = a->v_pool;
  L.page_indices = a->page_indices_dev;
  L.num_pages = a->num_pages;
  L.q_batch = a->batch;
  L.Hq_req = a->Hq;
  L.Hkv = a->Hkv;
  L.Dqk = a->Dqk;
  L.Dv = a->Dv;
  L.page_size = a->page_size;
  L.Gm = a->Hq / a->Hkv;
  L.G_cta = L.Gm;
  L.kv_dtype = a->kv_dtype;
  L.latent_v = a->v_pool == a->k_pool;
  const float ks = a->kv_dtype == PSD_FP8_E4M3 ? a->k_scale : 1.f;
  L.q_scale = a->sm_scale * kLog2e * ks;
  L.v_scale = a->kv_dtype == PSD_FP8_E4M3 ? a->v_scale : 1.f;
  return L;
}

bool dispatchable(const PartialLaunch &L) {
  return partial_tcs_supports(L) || partial_cc_supports(L) || partial_mla_supports(L) ||
         partial_tc_supports(L) || (L.stacked && partial_l0_supports(L));
}

// Stacked level-0 rows take the tcgen05 kernel (persistent, one CTA per SM over
// (chunk, KV head, 128-row block) tasks) when it applies and the context allows it.
// By default: from 32 rows per KV head, where the 16-row-group form reads every tile
// two or more times, and when level 0 has at least two tasks per SM.  With fewer,
// the single launch that runs level 0 beside level 1 is faster (cascade batch with
// an 8192-token prefix, 128 tasks: 0.097 ms against 0.105 ms a step), because the
// tcgen05 kernel holds whole SMs that level 1 could share.
static bool use_level0_tcgen05(const PartialLaunch &L, const DeviceInfo &dev) {
  if (!L.stacked || !partial_l0_supports(L) || dev.level0_kernel == PSD_LEVEL0_MMA_SYNC) return false;
  if (dev.level0_kernel == PSD_LEVEL0_TCGEN05) return true;
  const int64_t tasks = int64_t(L.num_items) * L.Hkv * ((L.G_cta + 127) / 128);
  return dev.partial_kernel != PSD_KERNEL_CUDA_CORE && L.G_cta >= kLevel0Tcgen05MinRows &&
         tasks >= 2 * int64_t(dev.num_sms > 0 ? dev.num_sms : 1);
}

// bf16 pools with separate K and V: the 16-row-group tensor-core kernel (or, for
// G <= 8 when the context asks for it, the CUDA-core kernel); the fp8 MLA latent
// (128 heads, 576/512): the tcgen05 kernel; other fp8 or latent shapes: the
// 64-row mma.sync kernel (also used for MLA when the context asks for CUDA_CORE,
// as the legacy-tensor-path reference).
PartialKind select_partial(const PartialLaunch &L, const DeviceInfo &dev) {
  if (use_level0_tcgen05(L, dev)) return PartialKind::kTensorL0;
  if (dev.partial_kernel == PSD_KERNEL_CUDA_CORE && partial_cc_supports(L)) return PartialKind::kCudaCore;
  if (partial_tcs_supports(L)) return PartialKind::kTensorSmall;
  if (partial_cc_supports(L)) return PartialKind::kCudaCore;
  if (partial_mla_supports(L) && dev.partial_kernel != PSD_KERNEL_CUDA_CORE) return PartialKind::kMLA;
  if (partial_tc_supports(L)) return PartialKind::kTensorLegacy;
  return PartialKind::kNone;
}

// The MLA kernel and the tcgen05 level-0 kernel accumulate runs of items
// (PartialLaunch::merge_runs) and leave the other rows of a run empty.
bool writes_empty_rows(const PartialLaunch &L, const DeviceInfo &dev) {
  const PartialKind k = select_partial(L, dev);
  return L.merge_runs && (k == PartialKind::kMLA || k == PartialKind::kTensorL0);
}

psd_status launch_partial(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s) {
  switch (select_partial(L, dev)) {
    case PartialKind::kCudaCore: return launch_partial_cc(L, dev, s);
    case PartialKind::kTensorSmall: return launch_partial_tcs(L, dev, s);
    case PartialKind::kMLA: return launch_partial_mla(L, dev, s);
    case PartialKind::kTensorLegacy: return launch_partial_tc(L, dev, s);
    case PartialKind::kTensorL0: return launch_partial_l0(L, dev, s);
    case PartialKind::kNone: break;
  }
  return fail(PSD_ERR_UNSUPPORTED, "no kernel for Dqk %d, Dv %d, rows/KV head %d, dtype %d, latent %d",
              L.Dqk, L.Dv, L.G_cta, L.kv_dtype, int(L.latent_v));
}

}  // namespace psd

namespace psd {

// Both cascade levels can share one launch when the 16-row-group tensor-core
// kernel serves both and level 1 fits one row group.
bool dispatch_fused(const PartialLaunch &L0, const PartialLaunch &L1, const DeviceInfo &dev) {
  if (dev.partial_kernel == PSD_KERNEL_CUDA_CORE || select_partial(L0, dev) == PartialKind::kTensorL0) return false;
  return partial_tcs_supports(L0) && partial_tcs_supports(L1) && L1.G_cta <= 16;
}

// Kernels that take their work lists from the launch parameters.
bool inline_lists_kernel(PartialKind k) { return k == PartialKind::kTensorSmall || k == PartialKind::kTensorL0; }

}  // namespace psd

namespace {

// Work lists of one call, placed either in the workspace by one H2D copy or, when
// they fit and every launch of the call reads them from its parameters, in `block`
// (the items, order, members and row bases; the merge takes o_indptr the same way).
struct CallLists {
  bool inl = false;
  InlineLists block;
  const uint8_t *base = nullptr;  // device address of the lists' first byte (the items)
  // Points L's list pointers (device addresses inside the workspace's lists) at the
  // same offsets of the parameter block.
  void apply(PartialLaunch &L) const {
    if (!inl) return;
    auto off = [&](const void *ptr) -> uint32_t {
      return ptr ? uint32_t(static_cast<const uint8_t *>(ptr) - base) : 0u;
    };
    L.inline_lists = &block;
    L.inl_items = off(L.items);
    L.inl_order = off(L.order);
    L.inl_members = off(L.members);
    L.inl_row_base = off(L.member_row_base);
  }
};

psd_status upload(psd_ctx *ctx, void *dst, const void *src, size_t bytes, cudaStream_t s);

// Inline lists when they fit and every launch takes them; otherwise one upload of the
// host copy of the workspace's list region.
psd_status place_lists(psd_ctx *ctx, CallLists &cl, uint8_t *ws, const WorkspaceLayout &lay,
                       const std::vector<uint8_t> &host, int32_t batch, bool all_inline_kernels,
                       cudaStream_t s) {
  const size_t used = lay.indptr_off - lay.items_off;
  cl.base = ws + lay.items_off;
  cl.inl = all_inline_kernels && used <= kInlineListBytes && batch + 1 <= kInlineIndptr;
  if (!cl.inl) {
    ctx->counters.lists_uploaded += 1;
    return upload(ctx, ws, host.data(), host.size(), s);
  }
  ctx->counters.lists_inline += 1;
  cl.block.used = used;
  std::memcpy(cl.block.bytes, host.data() + lay.items_off, used);
  return PSD_OK;
}

// Copies `bytes` of host data into a pinned staging buffer and enqueues one H2D
// copy to `dst` on `s`.
psd_status upload(psd_ctx *ctx, void *dst, const void *src, size_t bytes, cudaStream_t s) {
  const int i = ctx->next;
  ctx->next ^= 1;
  if (ctx->staging_pending[i]) {
    cudaError_t e = cudaEventSynchronize(ctx->staging_done[i]);
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "staging event: %s", cudaGetErrorString(e));
    ctx->staging_pending[i] = false;
  }
  if (ctx->staging_cap[i] < bytes) {
    if (ctx->staging[i]) cudaFreeHost(ctx->staging[i]);
    ctx->staging[i] = nullptr;
    size_t cap = bytes < 65536 ? 65536 : bytes * 2;
    cudaError_t e = cudaHostAlloc(&ctx->staging[i], cap, cudaHostAllocDefault);
    if (e != cudaSuccess) {
      ctx->staging_cap[i] = 0;
      return fail(PSD_ERR_CUDA, "pinned staging buffer: %s", cudaGetErrorString(e));
    }
    ctx->staging_cap[i] = cap;
  }
  std::memcpy(ctx->staging[i], src, bytes);
  cudaError_t e = cudaMemcpyAsync(dst, ctx->staging[i], bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "work-list upload: %s", cudaGetErrorString(e));
  e = cudaEventRecord(ctx->staging_done[i], s);
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "staging event record: %s", cudaGetErrorString(e));
  ctx->staging_pending[i] = true;
  return PSD_OK;
}

}  // namespace

extern "C" const char *psd_last_error(void) { return g_error.c_str(); }

extern "C" psd_status psd_create(psd_ctx **out, int device) {
  clear_error();
  if (!out) return fail(PSD_ERR_INVALID_ARG, "psd_create: NULL out");
  *out = nullptr;
  int n = 0;
  cudaError_t e = cudaGetDeviceCount(&n);
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cudaGetDeviceCount: %s", cudaGetErrorString(e));
  if (device < 0 || device >= n) return fail(PSD_ERR_INVALID_ARG, "device %d of %d", device, n);
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  if (major != 10 || minor != 3)
    return fail(PSD_ERR_UNSUPPORTED, "built for sm_103a (GB300); device %d is sm_%d%d", device, major,
                minor);
  psd_ctx *c = new psd_ctx();
  std::memset(&c->counters, 0, sizeof(c->counters));
  c->dev.device = device;
  cudaDeviceGetAttribute(&c->dev.num_sms, cudaDevAttrMultiProcessorCount, device);
  cudaDeviceGetAttribute(&c->dev.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  DeviceGuard g(device);
  cudaDriverEntryPointQueryResult q;
  void *fn = nullptr;
  e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    delete c;
    return fail(PSD_ERR_CUDA, "driver entry point cuTensorMapEncodeTiled unavailable");
  }
  c->dev.encode_tiled = fn;
  for (int i = 0; i < 2; ++i) {
    e = cudaEventCreateWithFlags(&c->staging_done[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      psd_destroy(c);
      return fail(PSD_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(e));
    }
  }
  e = cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    psd_destroy(c);
    return fail(PSD_ERR_CUDA, "side stream / events: %s", cudaGetErrorString(e));
  }
  *out = c;
  return PSD_OK;
}

extern "C" psd_status psd_destroy(psd_ctx *c) {
  clear_error();
  if (!c) return PSD_OK;
  DeviceGuard g(c->dev.device);
  for (int i = 0; i < 2; ++i) {
    if (c->staging_pending[i]) cudaEventSynchronize(c->staging_done[i]);
    if (c->staging_done[i]) cudaEventDestroy(c->staging_done[i]);
    if (c->staging[i]) cudaFreeHost(c->staging[i]);
  }
  if (c->side) {
    cudaStreamSynchronize(c->side);
    cudaStreamDestroy(c->side);
  }
  if (c->fork) cudaEventDestroy(c->fork);
  if (c->join) cudaEventDestroy(c->join);
  for (auto &ev : c->tev)
    if (ev) cudaEventDestroy(ev);
  if (c->flush) cudaFree(c->flush);
  delete c;
  return PSD_OK;
}

extern "C" psd_status psd_set_partial_kernel(psd_ctx *c, int32_t kind) {
  clear_error();
  if (!c) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  if (kind != PSD_KERNEL_AUTO && kind != PSD_KERNEL_CUDA_CORE && kind != PSD_KERNEL_TENSOR_CORE)
    return fail(PSD_ERR_INVALID_ARG, "partial kernel kind %d", kind);
  c->dev.partial_kernel = kind;
  return PSD_OK;
}

extern "C" psd_status psd_set_level0_kernel(psd_ctx *c, int32_t kind) {
  clear_error();
  if (!c) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  if (kind != PSD_LEVEL0_AUTO && kind != PSD_LEVEL0_MMA_SYNC && kind != PSD_LEVEL0_TCGEN05)
    return fail(PSD_ERR_INVALID_ARG, "level-0 kernel kind %d", kind);
  c->dev.level0_kernel = kind;
  return PSD_OK;
}

extern "C" psd_status psd_test_withhold_loads(psd_ctx *c, int32_t from_tile, int64_t wait_limit_cycles) {
  clear_error();
  if (!c) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  if (from_tile >= 0 && (wait_limit_cycles < 100000 || wait_limit_cycles > kMaxTestWaitCycles))
    return fail(PSD_ERR_INVALID_ARG, "psd_test_withhold_loads: wait limit %lld outside [1e5, %lld] cycles",
                (long long)wait_limit_cycles, (long long)kMaxTestWaitCycles);
  c->dev.test_withhold_from = from_tile >= 0 ? from_tile : -1;
  c->dev.test_wait_limit = from_tile >= 0 ? wait_limit_cycles : 0;
  return PSD_OK;
}

extern "C" psd_status psd_set_timing(psd_ctx *c, int32_t enable) {
  clear_error();
  if (!c) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  if (enable) {
    DeviceGuard g(c->dev.device);
    for (auto &ev : c->tev)
      if (!ev) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "timing events: %s", cudaGetErrorString(e));
      }
  }
  c->timing = enable != 0;
  return PSD_OK;
}

extern "C" psd_status psd_get_kernel_times(psd_ctx *c, float *level0_ms, float *partial_ms,
                                           float *merge_ms) {
  clear_error();
  if (!c) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  if (!c->timing) return fail(PSD_ERR_INVALID_ARG, "timing is off (psd_set_timing)");
  DeviceGuard g(c->dev.device);
  float *out[3] = {level0_ms, partial_ms, merge_ms};
  for (int k = 0; k < 3; ++k) {
    if (!out[k]) continue;
    *out[k] = 0.f;
    if (!c->tev_used[k]) continue;
    cudaError_t e = cudaEventSynchronize(c->tev[2 * k + 1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(out[k], c->tev[2 * k], c->tev[2 * k + 1]);
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "kernel times: %s", cudaGetErrorString(e));
  }
  return PSD_OK;
}

extern "C" psd_status psd_get_counters(const psd_ctx *c, psd_counters *out) {
  clear_error();
  if (!c || !out) return fail(PSD_ERR_INVALID_ARG, "NULL");
  *out = c->counters;
  return PSD_OK;
}

extern "C" size_t psd_workspace_bytes(int32_t batch, int32_t num_items, int64_t num_rows, int32_t Hq,
                                      int32_t Dv) {
  if (batch < 0 || num_items < 0 || num_rows < 0 || Hq < 0 || Dv < 0) return 0;
  return workspace_layout(batch, num_items, num_rows, Hq, Dv).total;
}

extern "C" psd_status paged_decode_partial(psd_ctx *ctx, const psd_decode_args *args,
                                           const psd_work_item *items, int32_t num_items,
                                           float *v_out, float *lse_out, int64_t out_rows,
                                           void *workspace, size_t workspace_bytes,
                                           psd_stream_t stream) {
  clear_error();
  if (!ctx) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  psd_status st = validate_args(args);
  if (st != PSD_OK) return st;
  if (num_items < 0 || (num_items > 0 && (!items || !v_out || !lse_out)) || !workspace)
    return fail(PSD_ERR_INVALID_ARG, "paged_decode_partial: NULL items / outputs / workspace");
  if (!aligned16(workspace) || !aligned16(v_out))
    return fail(PSD_ERR_INVALID_ARG, "paged_decode_partial: workspace and v_out must be 16-byte aligned");
  st = validate_items(args, items, num_items, out_rows, false, 0);
  if (st != PSD_OK) return st;
  const WorkspaceLayout lay = workspace_layout(0, num_items, 0, args->Hq, args->Dv);
  if (workspace_bytes < lay.total)
    return fail(PSD_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, lay.total);
  PartialLaunch L = base_launch(args);
  if (!dispatchable(L))
    return launch_partial(L, ctx->dev, reinterpret_cast<cudaStream_t>(stream));
  DeviceGuard g(ctx->dev.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<uint8_t> host(lay.lists_bytes, 0);
  if (num_items) std::memcpy(host.data() + lay.items_off, items, sizeof(psd_work_item) * num_items);
  longest_first(items, num_items, reinterpret_cast<int32_t *>(host.data() + lay.order_off));
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  st = upload(ctx, ws, host.data(), host.size(), s);
  if (st != PSD_OK) return st;
  L.items = reinterpret_cast<const psd_work_item *>(ws + lay.items_off);
  L.items_host = items;
  L.order = reinterpret_cast<const int32_t *>(ws + lay.order_off);
  L.num_items = num_items;
  L.v_out = v_out;
  L.lse_out = lse_out;
  L.fault = next_fault(ctx, ws);
  ctx->tev_used[0] = false;
  ctx->tev_used[1] = ctx->timing;
  ctx->tev_used[2] = false;
  time_mark(ctx, 2, s);
  st = launch_partial(L, ctx->dev, s);
  time_mark(ctx, 3, s);
  return st;
}

extern "C" psd_status merge_states(psd_ctx *ctx, const float *v_in, const float *lse_in,
                                   const int32_t *o_indptr_dev, int64_t num_out, int32_t H, int32_t D,
                                   float *v_out, float *lse_out, psd_stream_t stream) {
  clear_error();
  if (!ctx) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  if (num_out < 0 || H < 0 || D < 4 || D % 4 || D > 1024)
    return fail(PSD_ERR_INVALID_ARG, "merge_states: need num_out >= 0, H >= 0, D %% 4 == 0, D <= 1024");
  if (num_out == 0 || H == 0) return PSD_OK;
  if (!v_in || !lse_in || !o_indptr_dev || !v_out)
    return fail(PSD_ERR_INVALID_ARG, "merge_states: NULL pointer");
  if (!aligned16(v_in) || !aligned16(v_out))
    return fail(PSD_ERR_INVALID_ARG, "merge_states: v_in / v_out must be 16-byte aligned");
  DeviceGuard g(ctx->dev.device);
  return launch_merge(v_in, lse_in, o_indptr_dev, num_out, H, D, v_out, lse_out, ctx->dev,
                      reinterpret_cast<cudaStream_t>(stream));
}

extern "C" psd_status cascade_decode(psd_ctx *ctx, const psd_decode_args *args,
                                     const psd_cascade_plan *plan, float *o, float *lse,
                                     void *workspace, size_t workspace_bytes,
                                     psd_cascade_stats *stats, psd_stream_t stream) {
  clear_error();
  if (!ctx) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  psd_status st = validate_args(args);
  if (st != PSD_OK) return st;
  if (!plan || (!o && args->batch > 0) || !workspace)
    return fail(PSD_ERR_INVALID_ARG, "cascade_decode: NULL plan / o / workspace");
  if (!aligned16(workspace) || !aligned16(o))
    return fail(PSD_ERR_INVALID_ARG, "cascade_decode: workspace and o must be 16-byte aligned");
  const int32_t B = args->batch;
  if (plan->batch != B || plan->page_size != args->page_size)
    return fail(PSD_ERR_INVALID_ARG, "cascade_decode: plan batch/page_size (%d/%d) != args (%d/%d)",
                plan->batch, plan->page_size, B, args->page_size);
  const int32_t M = plan->num_members, n0 = plan->l0_num_items, n1 = plan->l1_num_items;
  if (M < 0 || M > B || n0 < 0 || n1 < 0 || (M == 0) != (n0 == 0) || plan->num_rows < 0 ||
      plan->o_indptr[0] != 0 || plan->o_indptr[B] != plan->num_rows)
    return fail(PSD_ERR_INVALID_ARG, "cascade_decode: inconsistent plan");
  for (int32_t b = 0; b < B; ++b)
    if (plan->o_indptr[b + 1] < plan->o_indptr[b])
      return fail(PSD_ERR_INVALID_ARG, "cascade_decode: o_indptr decreasing at %d", b);
  for (int32_t m = 0; m < M; ++m) {
    if (plan->members[m] < 0 || plan->members[m] >= B ||
        plan->member_row_base[m] != plan->o_indptr[plan->members[m]])
      return fail(PSD_ERR_INVALID_ARG, "cascade_decode: member %d", m);
    if (plan->o_indptr[plan->members[m] + 1] - plan->member_row_base[m] < n0)
      return fail(PSD_ERR_INVALID_ARG, "cascade_decode: member %d has fewer rows than level 0", m);
  }
  st = validate_items(args, plan->l0_items, n0, plan->num_rows, true, M);
  if (st == PSD_OK) st = validate_items(args, plan->l1_items, n1, plan->num_rows, false, M);
  if (st != PSD_OK) return st;
  for (int32_t i = 0; i < n0; ++i)
    if (plan->l0_items[i].out_row >= n0) return fail(PSD_ERR_INVALID_ARG, "level-0 item %d: chunk index", i);

  const WorkspaceLayout lay = workspace_layout(B, n0 + n1, plan->num_rows, args->Hq, args->Dv);
  if (workspace_bytes < lay.total)
    return fail(PSD_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, lay.total);

  PartialLaunch L1 = base_launch(args);
  L1.merge_runs = true;  // the partial rows feed the merge below
  PartialLaunch L0 = L1;
  L0.G_cta = M * L1.Gm;
  L0.stacked = true;
  L0.num_items = n0;
  if (!dispatchable(L1)) return launch_partial(L1, ctx->dev, nullptr);
  if (M > 0 && !dispatchable(L0)) return launch_partial(L0, ctx->dev, nullptr);

  DeviceGuard g(ctx->dev.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<uint8_t> host(lay.lists_bytes, 0);
  psd_work_item *hi = reinterpret_cast<psd_work_item *>(host.data() + lay.items_off);
  if (n0) std::memcpy(hi, plan->l0_items, sizeof(psd_work_item) * n0);
  if (n1) std::memcpy(hi + n0, plan->l1_items, sizeof(psd_work_item) * n1);
  int32_t *ho = reinterpret_cast<int32_t *>(host.data() + lay.order_off);
  longest_first(plan->l0_items, n0, ho);
  longest_first(plan->l1_items, n1, ho + n0);
  if (M) {
    std::memcpy(host.data() + lay.members_off, plan->members, sizeof(int32_t) * M);
    std::memcpy(host.data() + lay.row_base_off, plan->member_row_base, sizeof(int32_t) * M);
  }
  std::memcpy(host.data() + lay.indptr_off, plan->o_indptr, sizeof(int32_t) * (B + 1));
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const bool fused = M > 0 && dispatch_fused(L0, L1, ctx->dev);
  const bool tcs_only = select_partial(L1, ctx->dev) == PartialKind::kTensorSmall &&
                        (M == 0 || fused || inline_lists_kernel(select_partial(L0, ctx->dev)));
  CallLists cl;
  st = place_lists(ctx, cl, ws, lay, host, B, tcs_only, s);
  if (st != PSD_OK) return st;

  float *vpart = reinterpret_cast<float *>(ws + lay.vpart_off);
  float *lpart = reinterpret_cast<float *>(ws + lay.lpart_off);
  const FaultRef fault = next_fault(ctx, ws);
  const psd_work_item *ditems = reinterpret_cast<const psd_work_item *>(ws + lay.items_off);
  if (fused) {  // both levels in one launch of the 16-row-group tensor-core kernel
    L1.items = ditems;
    L1.order = reinterpret_cast<const int32_t *>(ws + lay.order_off) + n0;
    L1.num_items = n1;
    L1.members = reinterpret_cast<const int32_t *>(ws + lay.members_off);
    L1.member_row_base = reinterpret_cast<const int32_t *>(ws + lay.row_base_off);
    L1.fused_segments = 1;
    L1.fused_l0_items = n0;
    L1.seg_items[0] = n0;
    L1.seg_rows[0] = L0.G_cta;
    L1.seg_member0[0] = 0;
  } else if (M > 0) {  // level 0 on the side stream, after the lists are placed
    L0.items = ditems;
    L0.order = reinterpret_cast<const int32_t *>(ws + lay.order_off);
    L0.num_items = n0;
    L0.members = reinterpret_cast<const int32_t *>(ws + lay.members_off);
    L0.member_row_base = reinterpret_cast<const int32_t *>(ws + lay.row_base_off);
    L0.v_out = vpart;
    L0.lse_out = lpart;
    L0.fault = fault;
    cudaError_t e = cudaEventRecord(ctx->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->side, ctx->fork, 0);
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cascade fork: %s", cudaGetErrorString(e));
    time_mark(ctx, 0, ctx->side);
    cl.apply(L0);
    st = launch_partial(L0, ctx->dev, ctx->side);
    time_mark(ctx, 1, ctx->side);
    if (st != PSD_OK) return st;
    e = cudaEventRecord(ctx->join, ctx->side);
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cascade join: %s", cudaGetErrorString(e));
  }
  if (!fused) {
    L1.items = ditems + n0;
    L1.items_host = plan->l1_items;
    L1.order = reinterpret_cast<const int32_t *>(ws + lay.order_off) + n0;
    L1.num_items = n1;
  }
  L1.v_out = vpart;
  L1.lse_out = lpart;
  L1.fault = fault;
  cl.apply(L1);
  time_mark(ctx, 2, s);
  st = launch_partial(L1, ctx->dev, s);
  time_mark(ctx, 3, s);
  if (st != PSD_OK) return st;
  if (M > 0 && !fused) {
    cudaError_t e = cudaStreamWaitEvent(s, ctx->join, 0);
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "cascade join: %s", cudaGetErrorString(e));
  }
  time_mark(ctx, 4, s);
  const bool merge_follows_partial = !(M > 0 && !fused) && !ctx->timing;
  const bool empty_rows = writes_empty_rows(L1, ctx->dev) || (M > 0 && !fused && writes_empty_rows(L0, ctx->dev));
  st = launch_merge(vpart, lpart, reinterpret_cast<const int32_t *>(ws + lay.indptr_off), B, args->Hq,
                    args->Dv, o, lse, ctx->dev, s, merge_follows_partial, empty_rows,
                    cl.inl ? plan->o_indptr : nullptr);
  time_mark(ctx, 5, s);
  ctx->tev_used[0] = ctx->timing && M > 0 && !fused;
  ctx->tev_used[1] = ctx->timing;
  ctx->tev_used[2] = ctx->timing;
  if (st != PSD_OK) return st;

  if (M > 0) {
    ctx->counters.launches_cascade += 1;
    ctx->counters.cascade_shared_tokens += int64_t(plan->shared_pages) * args->page_size;
    ctx->counters.cascade_member_sequences += M;
  } else {
    ctx->counters.launches_flat += 1;
    if (plan->decline_reason != PSD_DECLINE_NONE && plan->decline_reason != PSD_DECLINE_DISABLED)
      ctx->counters.cascade_failures += 1;
  }
  if (stats) {
    stats->path = M > 0 ? 1 : 0;
    stats->decline_reason = plan->decline_reason;
    stats->batch = B;
    stats->members = M;
    stats->shared_pages = plan->shared_pages;
    stats->shared_tokens = plan->shared_pages * args->page_size;
    stats->prefix_chunks = n0;
    stats->suffix_chunks = n1;
  }
  return PSD_OK;
}

extern "C" size_t psd_nested_workspace_bytes(const psd_nested_plan *plan, int32_t Hq, int32_t Dv) {
  if (!plan) return 0;
  return workspace_layout(plan->batch, plan->l0_num_items + plan->l1_num_items, plan->num_rows, Hq, Dv,
                          plan->num_entries)
      .total;
}

extern "C" psd_status cascade_decode_nested(psd_ctx *ctx, const psd_decode_args *args,
                                            const psd_nested_plan *plan, float *o, float *lse,
                                            void *workspace, size_t workspace_bytes,
                                            psd_cascade_stats *stats, psd_stream_t stream) {
  clear_error();
  if (!ctx || !plan || !workspace) return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: NULL");
  psd_status st = validate_args(args);
  if (st != PSD_OK) return st;
  if (args->batch > 0 && (!o || !lse)) return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: NULL o / lse");
  if (!aligned16(workspace)) return fail(PSD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  const int32_t B = plan->batch, S = plan->num_segments, E = plan->num_entries;
  const int32_t n0 = plan->l0_num_items, n1 = plan->l1_num_items;
  if (B != args->batch) return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: plan batch %d != %d", B, args->batch);
  if (S < 0 || E < 0 || n0 < 0 || n1 < 0 || (S == 0) != (n0 == 0) || plan->o_indptr[0] != 0 ||
      plan->o_indptr[B] != plan->num_rows)
    return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: inconsistent plan");
  for (int32_t b = 0; b < B; ++b)
    if (plan->o_indptr[b + 1] < plan->o_indptr[b])
      return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: o_indptr decreasing at %d", b);
  int32_t covered_entries = 0, covered_items = 0;
  for (int32_t s = 0; s < S; ++s) {
    const psd_segment &g = plan->segments[s];
    if (g.first_member != covered_entries || g.num_members < 1 || g.first_item != covered_items ||
        g.num_items < 1 || g.start_page < 0 || g.shared_pages < 1)
      return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: segment %d", s);
    covered_entries += g.num_members;
    covered_items += g.num_items;
    for (int32_t k = 0; k < g.num_members; ++k) {
      const int32_t e = g.first_member + k, b = plan->members[e];
      if (b < 0 || b >= B || (k > 0 && b <= plan->members[e - 1]))
        return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: segment %d members", s);
      if (plan->member_row_base[e] < plan->o_indptr[b] ||
          int64_t(plan->member_row_base[e]) + g.num_items > plan->o_indptr[b + 1])
        return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: segment %d rows of request %d", s, b);
    }
    for (int32_t i = g.first_item; i < g.first_item + g.num_items; ++i)
      if (plan->l0_items[i].out_row != i - g.first_item)
        return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: level-0 item %d: chunk index", i);
  }
  if (covered_entries != E || covered_items != n0)
    return fail(PSD_ERR_INVALID_ARG, "cascade_decode_nested: segments do not cover the lists");
  st = validate_items(args, plan->l0_items, n0, plan->num_rows, true, E);
  if (st == PSD_OK) st = validate_items(args, plan->l1_items, n1, plan->num_rows, false, E);
  if (st != PSD_OK) return st;

  const WorkspaceLayout lay = workspace_layout(B, n0 + n1, plan->num_rows, args->Hq, args->Dv, E);
  if (workspace_bytes < lay.total)
    return fail(PSD_ERR_WORKSPACE_TOO_SMALL, "workspace %zu < %zu bytes", workspace_bytes, lay.total);
  PartialLaunch L1 = base_launch(args);
  L1.merge_runs = true;  // the partial rows feed the merge below
  if (!dispatchable(L1)) return launch_partial(L1, ctx->dev, nullptr);
  for (int32_t s = 0; s < S; ++s) {
    PartialLaunch L0 = L1;
    L0.G_cta = plan->segments[s].num_members * L1.Gm;
    L0.stacked = true;
    L0.num_items = plan->segments[s].num_items;
    if (!dispatchable(L0)) return launch_partial(L0, ctx->dev, nullptr);
  }

  DeviceGuard g(ctx->dev.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<uint8_t> host(lay.lists_bytes, 0);
  psd_work_item *hi = reinterpret_cast<psd_work_item *>(host.data() + lay.items_off);
  if (n0) std::memcpy(hi, plan->l0_items, sizeof(psd_work_item) * n0);
  if (n1) std::memcpy(hi + n0, plan->l1_items, sizeof(psd_work_item) * n1);
  int32_t *ho = reinterpret_cast<int32_t *>(host.data() + lay.order_off);
  for (int32_t i = 0; i < n0; ++i) ho[i] = i;  // level 0: one launch per segment, in item order
  longest_first(plan->l1_items, n1, ho + n0);
  if (E) {
    std::memcpy(host.data() + lay.members_off, plan->members, sizeof(int32_t) * E);
    std::memcpy(host.data() + lay.row_base_off, plan->member_row_base, sizeof(int32_t) * E);
  }
  std::memcpy(host.data() + lay.indptr_off, plan->o_indptr, sizeof(int32_t) * (B + 1));
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  // Every segment's level 0 and level 1 in one launch when the 16-row-group
  // tensor-core kernel serves all of them.
  bool fused = S > 0 && S <= PartialLaunch::kMaxFusedSegments;
  for (int32_t k = 0; fused && k < S; ++k) {
    PartialLaunch L0 = L1;
    L0.G_cta = plan->segments[k].num_members * L1.Gm;
    L0.stacked = true;
    L0.num_items = plan->segments[k].num_items;
    fused = dispatch_fused(L0, L1, ctx->dev);
  }
  bool tcs_only = select_partial(L1, ctx->dev) == PartialKind::kTensorSmall;
  for (int32_t k = 0; tcs_only && !fused && k < S; ++k) {
    PartialLaunch L0 = L1;
    L0.G_cta = plan->segments[k].num_members * L1.Gm;
    L0.stacked = true;
    L0.num_items = plan->segments[k].num_items;
    tcs_only = inline_lists_kernel(select_partial(L0, ctx->dev));
  }
  CallLists cl;
  st = place_lists(ctx, cl, ws, lay, host, B, tcs_only, s);
  if (st != PSD_OK) return st;

  float *vpart = reinterpret_cast<float *>(ws + lay.vpart_off);
  float *lpart = reinterpret_cast<float *>(ws + lay.lpart_off);
  const FaultRef fault = next_fault(ctx, ws);
  const psd_work_item *ditems = reinterpret_cast<const psd_work_item *>(ws + lay.items_off);
  const int32_t *dmembers = reinterpret_cast<const int32_t *>(ws + lay.members_off);
  const int32_t *drow_base = reinterpret_cast<const int32_t *>(ws + lay.row_base_off);
  if (fused) {
    L1.fused_segments = S;
    L1.fused_l0_items = n0;
    for (int32_t k = 0; k < S; ++k) {
      L1.seg_items[k] = plan->segments[k].num_items;
      L1.seg_rows[k] = plan->segments[k].num_members * L1.Gm;
      L1.seg_member0[k] = plan->segments[k].first_member;
    }
    L1.members = dmembers;
    L1.member_row_base = drow_base;
  } else if (S > 0) {  // every segment's level 0 on the side stream, after the lists are placed
    cudaError_t e = cudaEventRecord(ctx->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->side, ctx->fork, 0);
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "nested fork: %s", cudaGetErrorString(e));
    time_mark(ctx, 0, ctx->side);
    for (int32_t k = 0; k < S; ++k) {
      const psd_segment &gk = plan->segments[k];
      PartialLaunch L0 = L1;
      L0.G_cta = gk.num_members * L1.Gm;
      L0.stacked = true;
      L0.items = ditems + gk.first_item;
      L0.order = nullptr;
      L0.num_items = gk.num_items;
      L0.members = dmembers + gk.first_member;
      L0.member_row_base = drow_base + gk.first_member;
      L0.v_out = vpart;
      L0.lse_out = lpart;
      L0.fault = fault;
      cl.apply(L0);
      st = launch_partial(L0, ctx->dev, ctx->side);
      if (st != PSD_OK) return st;
    }
    time_mark(ctx, 1, ctx->side);
    e = cudaEventRecord(ctx->join, ctx->side);
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "nested join: %s", cudaGetErrorString(e));
  }
  L1.items = fused ? ditems : ditems + n0;
  if (!fused) L1.items_host = plan->l1_items;
  L1.order = reinterpret_cast<const int32_t *>(ws + lay.order_off) + n0;
  L1.num_items = n1;
  L1.v_out = vpart;
  L1.lse_out = lpart;
  L1.fault = fault;
  cl.apply(L1);
  time_mark(ctx, 2, s);
  st = launch_partial(L1, ctx->dev, s);
  time_mark(ctx, 3, s);
  if (st != PSD_OK) return st;
  const bool joined = S > 0 && !fused;
  if (joined) {
    cudaError_t e = cudaStreamWaitEvent(s, ctx->join, 0);
    if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "nested join: %s", cudaGetErrorString(e));
  }
  time_mark(ctx, 4, s);
  bool empty_rows = writes_empty_rows(L1, ctx->dev);
  for (int32_t k = 0; !fused && k < S; ++k) {
    PartialLaunch L0 = L1;
    L0.G_cta = plan->segments[k].num_members * L1.Gm;
    L0.stacked = true;
    L0.num_items = plan->segments[k].num_items;
    empty_rows = empty_rows || writes_empty_rows(L0, ctx->dev);
  }
  st = launch_merge(vpart, lpart, reinterpret_cast<const int32_t *>(ws + lay.indptr_off), B, args->Hq, args->Dv, o,
                    lse, ctx->dev, s, !joined && !ctx->timing, empty_rows, cl.inl ? plan->o_indptr : nullptr);
  time_mark(ctx, 5, s);
  ctx->tev_used[0] = ctx->timing && joined;
  ctx->tev_used[1] = ctx->timing;
  ctx->tev_used[2] = ctx->timing;
  if (st != PSD_OK) return st;

  int64_t shared_pages = 0;
  for (int32_t k = 0; k < S; ++k) shared_pages += plan->segments[k].shared_pages;
  if (S > 0) {
    ctx->counters.launches_cascade += 1;
    ctx->counters.cascade_shared_tokens += shared_pages * args->page_size;
    ctx->counters.cascade_member_sequences += E;
  } else {
    ctx->counters.launches_flat += 1;
    if (plan->decline_reason != PSD_DECLINE_NONE && plan->decline_reason != PSD_DECLINE_DISABLED)
      ctx->counters.cascade_failures += 1;
  }
  if (stats) {
    stats->path = S > 0 ? 1 : 0;
    stats->decline_reason = plan->decline_reason;
    stats->batch = B;
    stats->members = E;
    stats->shared_pages = int32_t(shared_pages);
    stats->shared_tokens = int32_t(shared_pages * args->page_size);
    stats->prefix_chunks = n0;
    stats->suffix_chunks = n1;
  }
  return PSD_OK;
}

extern "C" psd_status rope_append_kv(psd_ctx *ctx, const psd_rope_append_args *a, psd_stream_t stream) {
  clear_error();
  if (!ctx || !a) return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: NULL");
  if (a->num_tokens < 0 || a->Hq < 0 || a->Hkv < 1 || a->Dk_nope < 0 || a->Dk_rope < 1 || a->Dv < 0)
    return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: bad sizes");
  if (a->num_tokens == 0) return PSD_OK;  // nothing is read or written (pointers may be NULL)
  if (a->rot_dim < 2 || a->rot_dim % 2 || a->rot_dim > a->Dk_rope)
    return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: rot_dim %d must be even, >= 2 and <= Dk_rope %d",
                a->rot_dim, a->Dk_rope);
  if (a->Hq > 0 && (!a->q || a->q_rope_col < 0 || a->q_rope_col + a->rot_dim > a->Dq))
    return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: q rope columns outside Dq");
  if ((a->Dk_nope > 0) != (a->k_nope != nullptr) || (a->Dv > 0) != (a->v != nullptr) ||
      (a->Dv > 0) != (a->v_pool != nullptr))
    return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: k_nope / v / v_pool must be given exactly when their width > 0");
  if (!a->k_rope || !a->cos_sin || !a->positions || !a->slot_mapping || !a->k_pool || !a->fault_dev)
    return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: NULL pointer");
  if (a->max_position < 1 || a->page_size < 1 || a->num_pages < 0)
    return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: bad pool or table sizes");
  if (a->kv_dtype != PSD_BF16 && a->kv_dtype != PSD_FP8_E4M3)
    return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: kv_dtype %d", a->kv_dtype);
  if (a->kv_dtype == PSD_FP8_E4M3 && !(std::isfinite(a->k_scale) && a->k_scale > 0.f &&
                                       std::isfinite(a->v_scale) && a->v_scale > 0.f))
    return fail(PSD_ERR_INVALID_ARG, "rope_append_kv: fp8 scales must be finite and > 0");
  DeviceGuard g(ctx->dev.device);
  return launch_rope_append(a, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" psd_status psd_check_device_error(psd_ctx *ctx, void *workspace, psd_stream_t stream,
                                             int32_t *fault_bits) {
  clear_error();
  if (!ctx || !workspace) return fail(PSD_ERR_INVALID_ARG, "NULL");
  DeviceGuard g(ctx->dev.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned long long word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(PSD_ERR_CUDA, "psd_check_device_error: %s", cudaGetErrorString(e));
  // only the bits of this context's latest call on the workspace count
  const int slot = ctx->epoch_slot(workspace);
  const bool latest = slot >= 0 && ctx->ws_epoch[slot] == uint32_t(word >> 32);
  const int32_t flag = latest ? int32_t(uint32_t(word)) : 0;
  if (fault_bits) *fault_bits = flag;
  if (flag) {
    e = cudaMemsetAsync(workspace, 0, sizeof(word), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return fail(PSD_ERR_DEVICE_FAULT, "kernel fault flag 0x%x (1 = page id out of range, 2 = wait timeout)", flag);
  }
  return PSD_OK;
}
