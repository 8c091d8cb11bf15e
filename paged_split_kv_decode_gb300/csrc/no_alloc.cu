// cascade_decode_no_alloc: cascade_decode for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they
// decode: code running inside another framework's memory pool that forbids
// foreign allocations, plugins handed only the tensors they read and write, or
// runtimes that reserve all device memory up front.  They cannot provide the
// workspace cascade_decode needs, so this entry point keeps its scratch (work
// lists, the fault word and the partial rows) in one fixed array in the library's
// own device memory instead.  It calls no allocating routine.
//
// The array lives for the life of the process on every GPU that loads the
// library and is shared by every call on that GPU: calls whose device work
// overlaps (different streams, or host threads without ordering) race on it and
// produce garbage.  Each call clears the part that must start at zero (the fault
// word); the rest keeps the previous call's contents until overwritten.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "context.h"

namespace {

// 16 MiB: the flat and cascade decode batches need about 3 and 6 MiB.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

}  // namespace

static __device__ __align__(256) uint8_t g_no_alloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The first call on a
// device looks it up with cudaGetSymbolAddress (host code only sees a host-side
// stand-in under the array's name, never a usable device address) and keeps it for
// the life of the process; a cudaDeviceReset would invalidate the kept address.
psd_status scratch_address(int device, uint8_t **out) {
  if (device < 0 || device >= kMaxDevices)
    return psd::fail(PSD_ERR_UNSUPPORTED, "cascade_decode_no_alloc: device %d out of range", device);
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[device]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess || !p)
      return psd::fail(PSD_ERR_CUDA, "cascade_decode_no_alloc: cudaGetSymbolAddress: %s",
                       cudaGetErrorString(e));
    g_scratch_addr[device] = p;
  }
  *out = static_cast<uint8_t *>(g_scratch_addr[device]);
  return PSD_OK;
}

}  // namespace

using namespace psd;

extern "C" psd_status cascade_decode_no_alloc(psd_ctx *ctx, const psd_decode_args *args,
                                              const psd_cascade_plan *plan, float *o, float *lse,
                                              int32_t *fault_bits_dev, psd_cascade_stats *stats,
                                              psd_stream_t stream) {
  clear_error();
  if (!ctx) return fail(PSD_ERR_INVALID_ARG, "NULL context");
  psd_status st = validate_args(args);
  if (st != PSD_OK) return st;
  if (!plan || (!o && args->batch > 0)) return fail(PSD_ERR_INVALID_ARG, "cascade_decode_no_alloc: NULL plan / o");
  if (!aligned16(o)) return fail(PSD_ERR_INVALID_ARG, "cascade_decode_no_alloc: o must be 16-byte aligned");
  const int32_t B = args->batch;
  if (plan->batch != B || plan->page_size != args->page_size)
    return fail(PSD_ERR_INVALID_ARG, "cascade_decode_no_alloc: plan batch/page_size (%d/%d) != args (%d/%d)",
                plan->batch, plan->page_size, B, args->page_size);
  const int32_t M = plan->num_members, n0 = plan->l0_num_items, n1 = plan->l1_num_items;
  if (M < 0 || M > B || n0 < 0 || n1 < 0 || (M == 0) != (n0 == 0) || plan->num_rows < 0 ||
      plan->o_indptr[0] != 0 || plan->o_indptr[B] != plan->num_rows)
    return fail(PSD_ERR_INVALID_ARG, "cascade_decode_no_alloc: inconsistent plan");
  for (int32_t b = 0; b < B; ++b)
    if (plan->o_indptr[b + 1] < plan->o_indptr[b])
      return fail(PSD_ERR_INVALID_ARG, "cascade_decode_no_alloc: o_indptr decreasing at %d", b);
  for (int32_t m = 0; m < M; ++m) {
    if (plan->members[m] < 0 || plan->members[m] >= B ||
        plan->member_row_base[m] != plan->o_indptr[plan->members[m]] ||
        plan->o_indptr[plan->members[m] + 1] - plan->member_row_base[m] < n0)
      return fail(PSD_ERR_INVALID_ARG, "cascade_decode_no_alloc: member %d", m);
  }
  st = validate_items(args, plan->l0_items, n0, plan->num_rows, true, M);
  if (st == PSD_OK) st = validate_items(args, plan->l1_items, n1, plan->num_rows, false, M);
  if (st != PSD_OK) return st;
  for (int32_t i = 0; i < n0; ++i)
    if (plan->l0_items[i].out_row >= n0)
      return fail(PSD_ERR_INVALID_ARG, "cascade_decode_no_alloc: level-0 item %d chunk index", i);

  const WorkspaceLayout lay = workspace_layout(B, n0 + n1, plan->num_rows, args->Hq, args->Dv);
  if (lay.total > kNoAllocScratchBytes)
    return fail(PSD_ERR_WORKSPACE_TOO_SMALL,
                "cascade_decode_no_alloc: this plan needs %zu bytes of scratch but the library's "
                "static scratch holds %zu bytes; use cascade_decode with a workspace",
                lay.total, kNoAllocScratchBytes);

  PartialLaunch L1 = base_launch(args);
  L1.merge_runs = true;  // the partial rows feed the merge below
  PartialLaunch L0 = L1;
  L0.G_cta = M * L1.Gm;
  L0.stacked = true;
  L0.num_items = n0;
  if (!dispatchable(L1)) return launch_partial(L1, ctx->dev, nullptr);
  if (M > 0 && !dispatchable(L0)) return launch_partial(L0, ctx->dev, nullptr);

  DeviceGuard g(ctx->dev.device);
  uint8_t *ws = nullptr;
  st = scratch_address(ctx->dev.device, &ws);
  if (st != PSD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // The lists as cascade_decode lays them out: items (level 0, then level 1), the
  // longest-first CTA order of each level, members, member row bases, o_indptr.
  std::vector<uint8_t> host(lay.lists_bytes, 0);  // the header (fault word) stays 0
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

  // Both levels in one launch where the 16-row-group tensor-core kernel serves them;
  // the lists then travel in the launch parameters when they fit, and only the fault
  // word is cleared on the device.  Otherwise one copy from this host buffer (the
  // runtime stages pageable memory before the call returns) places the lists and the
  // cleared header in the scratch.
  const bool fused = M > 0 && dispatch_fused(L0, L1, ctx->dev);
  const bool tcs_only = select_partial(L1, ctx->dev) == PartialKind::kTensorSmall &&
                        (M == 0 || fused || inline_lists_kernel(select_partial(L0, ctx->dev)));
  const size_t used = lay.indptr_off - lay.items_off;
  const bool inl = tcs_only && used <= kInlineListBytes && B + 1 <= kInlineIndptr;
  InlineLists block;
  cudaError_t e;
  if (inl) {
    block.used = used;
    std::memcpy(block.bytes, host.data() + lay.items_off, used);
    e = cudaMemsetAsync(ws, 0, sizeof(unsigned long long), s);
  } else {
    e = cudaMemcpyAsync(ws, host.data(), host.size(), cudaMemcpyHostToDevice, s);
  }
  if (e != cudaSuccess)
    return fail(PSD_ERR_CUDA, "cascade_decode_no_alloc: lists: %s", cudaGetErrorString(e));
  auto place = [&](PartialLaunch &L) {  // list pointers into the parameter block
    if (!inl) return;
    auto off = [&](const void *ptr) -> uint32_t {
      return ptr ? uint32_t(static_cast<const uint8_t *>(ptr) - (ws + lay.items_off)) : 0u;
    };
    L.inline_lists = &block;
    L.inl_items = off(L.items);
    L.inl_order = off(L.order);
    L.inl_members = off(L.members);
    L.inl_row_base = off(L.member_row_base);
  };

  float *vpart = reinterpret_cast<float *>(ws + lay.vpart_off);
  float *lpart = reinterpret_cast<float *>(ws + lay.lpart_off);
  // The scratch's fault word was cleared above, so its low 32 bits are this call's
  // fault bits whatever the epoch.
  const FaultRef fault = next_fault(ctx, ws);
  const psd_work_item *ditems = reinterpret_cast<const psd_work_item *>(ws + lay.items_off);
  const int32_t *dorder = reinterpret_cast<const int32_t *>(ws + lay.order_off);
  const int32_t *dmembers = reinterpret_cast<const int32_t *>(ws + lay.members_off);
  const int32_t *drow_base = reinterpret_cast<const int32_t *>(ws + lay.row_base_off);
  if (fused) {
    L1.items = ditems;
    L1.members = dmembers;
    L1.member_row_base = drow_base;
    L1.fused_segments = 1;
    L1.fused_l0_items = n0;
    L1.seg_items[0] = n0;
    L1.seg_rows[0] = L0.G_cta;
    L1.seg_member0[0] = 0;
  } else {
    if (M > 0) {  // level 0 first, on the same stream
      L0.items = ditems;
      L0.order = dorder;
      L0.num_items = n0;
      L0.members = dmembers;
      L0.member_row_base = drow_base;
      L0.v_out = vpart;
      L0.lse_out = lpart;
      L0.fault = fault;
      place(L0);
      if ((st = launch_partial(L0, ctx->dev, s)) != PSD_OK) return st;
    }
    L1.items = ditems + n0;
    L1.items_host = plan->l1_items;
  }
  L1.order = dorder + n0;
  L1.num_items = n1;
  L1.v_out = vpart;
  L1.lse_out = lpart;
  L1.fault = fault;
  place(L1);
  if ((st = launch_partial(L1, ctx->dev, s)) != PSD_OK) return st;
  const bool empty_rows = writes_empty_rows(L1, ctx->dev) || (M > 0 && !fused && writes_empty_rows(L0, ctx->dev));
  st = launch_merge(vpart, lpart, reinterpret_cast<const int32_t *>(ws + lay.indptr_off), B, args->Hq,
                    args->Dv, o, lse, ctx->dev, s, true, empty_rows, inl ? plan->o_indptr : nullptr);
  if (st != PSD_OK) return st;
  if (fault_bits_dev) {
    e = cudaMemcpyAsync(fault_bits_dev, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess)
      return fail(PSD_ERR_CUDA, "cascade_decode_no_alloc: fault word: %s", cudaGetErrorString(e));
  }

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
