// Host-side launch interfaces of the CUDA kernels.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "psd_internal.h"

namespace psd {

struct DeviceInfo {
  int device = 0;
  int num_sms = 0;
  int smem_optin = 0;
  void *encode_tiled = nullptr;  // driver cuTensorMapEncodeTiled
  int partial_kernel = 0;        // psd_partial_kernel preference for G <= 16
  int level0_kernel = 0;         // psd_level0_kernel preference for stacked level-0 rows
  // Testing aid for the bounded waits (psd_test_withhold_loads): the 16-row-group
  // tensor-core, CUDA-core, tcgen05 level-0 and MLA partial kernels issue no loads
  // for tiles at index test_withhold_from and later of any item, and the streaming
  // merge none for input rows from that index of a CTA's range on (-1: off); they
  // give up a wait after test_wait_limit cycles (0: the default limit).
  int32_t test_withhold_from = -1;
  int64_t test_wait_limit = 0;
};

// The workspace's fault word: 64 bits at its start, (epoch << 32) | fault bits.  The
// kernels of one call carry that call's epoch; a kernel that flags a fault ORs its
// bits in when the word holds its epoch and replaces the word otherwise, so the word
// needs no clearing before a call, and bits left by an earlier call (or whatever a
// fresh workspace holds) never read as a fault of the current one.
struct FaultRef {
  unsigned long long *word = nullptr;
  uint32_t epoch = 0;
};

// Per-call work lists carried in a launch's parameter space.  A small H2D copy in
// front of the kernels costs about 5 us of device time on GB300; parameters of up to
// a few KB arrive with the launch at no measurable cost.  Only kernels whose CTAs read
// a few warp-uniform entries take them (parameter loads go through the constant cache).
// A launch carries the smallest of these block sizes that holds its lists (the
// parameter copy grows with the declared size, about 0.1 us per KB).
constexpr size_t kInlineListBytes = 16384;
template <int CAP> struct ListBlock {
  alignas(16) unsigned char bytes[CAP];
};
struct InlineLists {  // host side: `used` bytes of lists
  size_t used = 0;
  alignas(16) unsigned char bytes[kInlineListBytes];
};
constexpr int kInlineIndptr = 1024;  // o_indptr entries carried by a merge launch
struct InlineIndptr {
  int32_t v[kInlineIndptr];
};
struct NoInline {  // stands in for the blocks above in launches that do not use them
  alignas(16) unsigned char bytes[16];
  int32_t v[4];
};
template <int CAP> using ListParam = std::conditional_t<CAP != 0, ListBlock<CAP != 0 ? CAP : 16>, NoInline>;
template <bool INL> using IndptrParam = std::conditional_t<INL, InlineIndptr, NoInline>;

// One partial-attention launch over a device work list.
//   Items with q_index >= 0 use query rows q[q_index, kv*Gm + g] (g < Gm) and
//   write rows out_row.  Items with q_index < 0 are the stacked level-0 request:
//   CTA row j (< G_cta = M*Gm) is member m = j / Gm, head kv*Gm + j % Gm, reading
//   q[members[m], .] and writing row member_row_base[m] + out_row.
struct PartialLaunch {
  const void *q = nullptr;
  const void *k_pool = nullptr;
  const void *v_pool = nullptr;  // == k_pool for a shared latent
  const int32_t *page_indices = nullptr;
  const psd_work_item *items = nullptr;  // device
  const psd_work_item *items_host = nullptr;  // host copy of `items`, when the caller has one
  const int32_t *order = nullptr;        // device, CTA -> item index (longest first), or NULL
  int32_t num_items = 0;
  const int32_t *members = nullptr;          // device, stacked items only
  const int32_t *member_row_base = nullptr;  // device, stacked items only
  float *v_out = nullptr;
  float *lse_out = nullptr;
  FaultRef fault;
  int64_t num_pages = 0;
  int32_t q_batch = 0;  // requests in q
  int32_t Hq_req = 0;  // query heads per request in q and in the outputs
  int32_t Hkv = 0, Dqk = 0, Dv = 0, page_size = 0;
  int32_t Gm = 0;      // query heads per KV head of one request
  int32_t G_cta = 0;   // query rows per CTA (Gm, or M*Gm when stacked)
  int32_t kv_dtype = PSD_BF16;
  bool latent_v = false;
  bool stacked = false;  // a stacked level-0 launch (items with q_index < 0)
  int32_t max_item_tokens = 0;
  // The partial rows feed this library's merge: a kernel may accumulate a run of
  // consecutive items of one request into one partial, written to the run's last
  // row, and mark the other rows empty (LSE -inf, v unused by the merge).
  bool merge_runs = false;
  // When set, items / order / members / member_row_base are not read from the device
  // pointers above but from this host block, copied into the launch's parameters, at
  // the given byte offsets (order may still be NULL: identity).  Honoured by the
  // 16-row-group tensor-core kernel only.
  const InlineLists *inline_lists = nullptr;
  uint32_t inl_items = 0, inl_order = 0, inl_members = 0, inl_row_base = 0;
  float q_scale = 1.f;  // sm_scale * log2(e) * k_scale
  float v_scale = 1.f;
  // Fused cascade launch (16-row-group tensor-core kernel only): `items` starts
  // with the level-0 items of `fused_segments` segments, in segment order (segment s:
  // seg_items[s] items of seg_rows[s] stacked rows whose members are the entries
  // from seg_member0[s] of `members` / `member_row_base`), followed by the
  // num_items level-1 items (order indexes those).
  static constexpr int kMaxFusedSegments = 8;
  int32_t fused_segments = 0;
  int32_t fused_l0_items = 0;  // sum of seg_items
  int32_t seg_items[kMaxFusedSegments] = {}, seg_rows[kMaxFusedSegments] = {}, seg_member0[kMaxFusedSegments] = {};
};

bool partial_cc_supports(const PartialLaunch &p);
psd_status launch_partial_cc(const PartialLaunch &p, const DeviceInfo &dev, cudaStream_t s);
bool partial_tcs_supports(const PartialLaunch &p);
psd_status launch_partial_tcs(const PartialLaunch &p, const DeviceInfo &dev, cudaStream_t s);
bool partial_mla_supports(const PartialLaunch &p);
psd_status launch_partial_mla(const PartialLaunch &p, const DeviceInfo &dev, cudaStream_t s);
bool partial_tc_supports(const PartialLaunch &p);
psd_status launch_partial_tc(const PartialLaunch &p, const DeviceInfo &dev, cudaStream_t s);
bool partial_l0_supports(const PartialLaunch &p);
psd_status launch_partial_l0(const PartialLaunch &p, const DeviceInfo &dev, cudaStream_t s);

psd_status launch_rope_append(const psd_rope_append_args *a, cudaStream_t s);

// after_partial: the launch directly follows a partial kernel on stream s (no event
// or copy between them), so it may start early and wait for that grid on the device.
// skip_empty: many rows are empty (LSE -inf); each row's LSE is read before its v,
// and an empty row's v is not loaded.  Without it the rows of a batch are loaded
// with the LSE values (one round trip fewer) and an empty row's v is ignored.
psd_status launch_merge(const float *v_in, const float *lse_in, const int32_t *o_indptr,
                        int64_t num_out, int32_t H, int32_t D, float *v_out, float *lse_out,
                        const DeviceInfo &dev, cudaStream_t s, bool after_partial = false,
                        bool skip_empty = false, const int32_t *o_indptr_host = nullptr);
// o_indptr_host: when not NULL and num_out + 1 <= kInlineIndptr, the group bounds are
// taken from this host array, copied into the launch's parameters; o_indptr is unused.

}  // namespace psd
