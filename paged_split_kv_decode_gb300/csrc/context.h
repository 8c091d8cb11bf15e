// The context object and the host-side helpers shared by the entry points.
#pragma once

#include <cuda_runtime.h>

#include <array>
#include <map>

#include "kernels.h"
#include "psd_internal.h"

struct psd_ctx {
  psd::DeviceInfo dev;
  psd_counters counters;
  // Two pinned staging buffers for the per-call H2D upload of work lists (when they
  // do not travel in the launch parameters); an event per buffer tells when its
  // previous copy has finished reading it.
  void *staging[2] = {nullptr, nullptr};
  size_t staging_cap[2] = {0, 0};
  cudaEvent_t staging_done[2] = {nullptr, nullptr};
  bool staging_pending[2] = {false, false};
  int next = 0;
  // Level 0 of a cascade runs on `side`, concurrently with level 1 on the caller's
  // stream: fork once the lists are placed, join before the merge.
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  // Optional kernel timing: events around level 0, level 1 / flat, and merge.
  bool timing = false;
  cudaEvent_t tev[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  bool tev_used[3] = {false, false, false};
  // Chunk sizes chosen by psd_autotune_tile, by shape bucket, and the cold-L2 flush
  // buffer it writes between timed calls (allocated on its first use).
  std::map<std::array<int64_t, 9>, int32_t> tuned;
  void *flush = nullptr;
  size_t flush_bytes = 0;
  // Fault-word epochs: a counter advanced by every decode call, and the epoch of the
  // latest call on each of the last kEpochSlots workspaces used (what
  // psd_check_device_error compares against; an older workspace reads as clean).
  static constexpr int kEpochSlots = 64;
  uint32_t epoch = 0;
  const void *ws_ptr[kEpochSlots] = {};
  uint32_t ws_epoch[kEpochSlots] = {};
  int ws_next = 0;
  // the slot of workspace `ws`, or -1
  int epoch_slot(const void *ws) const {
    for (int i = 0; i < kEpochSlots; ++i)
      if (ws_ptr[i] == ws) return i;
    return -1;
  }
};

namespace psd {
// The fault word of a new decode call on workspace `ws`: a fresh epoch, recorded as
// the workspace's latest.
inline FaultRef next_fault(psd_ctx *c, void *ws) {
  if (++c->epoch == 0) c->epoch = 1;
  int i = c->epoch_slot(ws);
  if (i < 0) {
    i = c->ws_next;
    c->ws_next = (c->ws_next + 1) % psd_ctx::kEpochSlots;
    c->ws_ptr[i] = ws;
  }
  c->ws_epoch[i] = c->epoch;
  return FaultRef{static_cast<unsigned long long *>(ws), c->epoch};
}
// Records timing event `i` (0..5) of the context on stream `s` when timing is on.
inline void time_mark(psd_ctx *c, int i, cudaStream_t s) {
  if (c->timing && c->tev[i]) cudaEventRecord(c->tev[i], s);
}
}  // namespace psd

namespace psd {

struct DeviceGuard {  // make a device current for one call, restore the caller's after
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
    else prev = -1;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

bool aligned16(const void *p);
psd_status validate_args(const psd_decode_args *a);
psd_status validate_items(const psd_decode_args *a, const psd_work_item *items, int32_t n,
                          int64_t out_rows, bool stacked, int32_t num_members);
PartialLaunch base_launch(const psd_decode_args *a);
bool dispatchable(const PartialLaunch &L);
enum class PartialKind { kNone, kCudaCore, kTensorSmall, kMLA, kTensorLegacy, kTensorL0 };
// The kernel launch_partial runs for L on dev.
PartialKind select_partial(const PartialLaunch &L, const DeviceInfo &dev);
// The launch may leave empty partial rows (LSE -inf, v not written) for the merge.
bool writes_empty_rows(const PartialLaunch &L, const DeviceInfo &dev);
psd_status launch_partial(const PartialLaunch &L, const DeviceInfo &dev, cudaStream_t s);
// Both cascade levels can share one launch of the 16-row-group tensor-core kernel.
bool dispatch_fused(const PartialLaunch &L0, const PartialLaunch &L1, const DeviceInfo &dev);
// Kernels of this kind take their work lists from the launch parameters.
bool inline_lists_kernel(PartialKind k);

}  // namespace psd
