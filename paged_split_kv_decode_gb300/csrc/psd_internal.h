// Internal declarations shared by the host-side translation units.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "../../include/psd.h"

namespace psd {

// Item visiting order for a launch: indices of items[0, n) by decreasing token
// count (stable), so the longest tiles start first and short ones fill the tail.
void longest_first(const psd_work_item *items, int32_t n, int32_t *order);

// Thread-local error message (psd_last_error).
void clear_error();
psd_status fail(psd_status st, const char *fmt, ...);

psd_status validate_table(const psd_page_table *t, int64_t num_pages);

// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)        header: int32 fault flag at offset 0
//   lists           work items, CTA order, members, member_row_base, o_indptr
//                   (one H2D copy)
//   v partials      [num_rows, Hq, Dv] f32
//   lse partials    [num_rows, Hq] f32
struct WorkspaceLayout {
  size_t lists_off, lists_bytes;
  size_t items_off, order_off, members_off, row_base_off, indptr_off;
  size_t vpart_off, lpart_off;
  size_t total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// member_entries: length of the members / member_row_base lists (the batch for a
// two-level plan, the (segment, member) entries for a nested one).
inline WorkspaceLayout workspace_layout(int32_t batch, int32_t num_items, int64_t num_rows,
                                        int32_t Hq, int32_t Dv, int32_t member_entries = -1) {
  if (member_entries < 0) member_entries = batch;
  WorkspaceLayout L;
  L.lists_off = 0;  // the header travels with the lists in the same copy
  L.items_off = 256;
  const size_t n = size_t(num_items > 0 ? num_items : 0);
  L.order_off = L.items_off + sizeof(psd_work_item) * n;
  L.members_off = L.order_off + sizeof(int32_t) * n;
  L.row_base_off = L.members_off + sizeof(int32_t) * size_t(member_entries);
  L.indptr_off = L.row_base_off + sizeof(int32_t) * size_t(member_entries);
  L.lists_bytes = L.indptr_off + sizeof(int32_t) * size_t(batch + 1);
  L.vpart_off = align256(L.lists_bytes);
  L.lpart_off = L.vpart_off + align256(sizeof(float) * size_t(num_rows) * size_t(Hq) * size_t(Dv));
  L.total = L.lpart_off + align256(sizeof(float) * size_t(num_rows) * size_t(Hq));
  return L;
}

}  // namespace psd
