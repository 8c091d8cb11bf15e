// Host planning: split-KV work lists, shared-prefix detection, cascade plans.
//
// mlxcel PR #1004, "compute shared prompt prefixes once per decode batch":
//   Decomposition  - the partial kernel's unit is one (request, page tile);
//   Detection      - equal page ids at the same CSR position are one shared block;
//   Task item 1    - group by first page, longest common page prefix per group,
//                    best subgroup by saved reads shared_pages * (members - 1);
//   Task item 2    - level-0 view over the span, level-1 view without it;
//   Task item 4    - kill switch, thresholds, the last-page cap;
//   Left out / unsure - early divergers shorten the span; defaults 16 pages, 2
//                    members.
// All passes are O(nnz) over the host page table.
#include <algorithm>
#include <cctype>
#include <cstdlib>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "psd_internal.h"

namespace psd {

static inline int32_t pages_of(const psd_page_table *t, int32_t b) {
  return t->page_indptr[b + 1] - t->page_indptr[b];
}

static inline int64_t tokens_of(const psd_page_table *t, int32_t b) {
  return int64_t(pages_of(t, b) - 1) * t->page_size + t->last_page_len[b];
}

psd_status validate_table(const psd_page_table *t, int64_t num_pages) {
  if (!t || !t->page_indptr || !t->last_page_len)
    return fail(PSD_ERR_INVALID_ARG, "page table: NULL pointer");
  if (t->batch < 0) return fail(PSD_ERR_INVALID_ARG, "page table: batch < 0");
  if (t->page_size < 1) return fail(PSD_ERR_INVALID_ARG, "page table: page_size < 1");
  if (t->page_indptr[0] != 0) return fail(PSD_ERR_INVALID_ARG, "page table: page_indptr[0] != 0");
  if (t->batch > 0 && !t->page_indices)
    return fail(PSD_ERR_INVALID_ARG, "page table: page_indices is NULL");
  for (int32_t b = 0; b < t->batch; ++b) {
    int32_t n = pages_of(t, b);
    if (n < 1) return fail(PSD_ERR_INVALID_ARG, "page table: request %d has %d pages", b, n);
    int32_t last = t->last_page_len[b];
    if (last < 1 || last > t->page_size)
      return fail(PSD_ERR_INVALID_ARG, "page table: last_page_len[%d] = %d outside [1, %d]", b,
                  last, t->page_size);
  }
  if (num_pages >= 0) {
    const int32_t nnz = t->page_indptr[t->batch];
    for (int32_t i = 0; i < nnz; ++i) {
      int32_t p = t->page_indices[i];
      if (p < 0 || int64_t(p) >= num_pages)
        return fail(PSD_ERR_INVALID_ARG, "page table: page_indices[%d] = %d outside [0, %lld)", i,
                    p, (long long)num_pages);
    }
  }
  return PSD_OK;
}

// Appends the T-token chunks of `n_tok` tokens whose first page sits at position
// `page_off`; rows start at `row0`.  Returns the number of chunks.
static int32_t emit_chunks(int32_t q_index, int32_t page_off, int64_t n_tok, int32_t tile_tokens,
                           int32_t page_size, int32_t row0, psd_work_item *out, int32_t cap,
                           int32_t *count) {
  const int32_t ppt = tile_tokens / page_size;
  int32_t c = 0;
  for (int64_t t0 = 0; t0 < n_tok; t0 += tile_tokens, ++c) {
    if (*count >= cap) return -1;
    psd_work_item &it = out[(*count)++];
    it.q_index = q_index;
    it.page_off = page_off + c * ppt;
    it.n_tokens = int32_t(std::min<int64_t>(tile_tokens, n_tok - t0));
    it.out_row = row0 + c;
  }
  return c;
}

}  // namespace psd

using namespace psd;

extern "C" psd_status psd_split_plan(const psd_page_table *host, int32_t tile_tokens,
                                     psd_work_item *items, int32_t item_capacity,
                                     int32_t *num_items, int32_t *o_indptr) {
  clear_error();
  psd_status st = validate_table(host, -1);
  if (st != PSD_OK) return st;
  if (tile_tokens < 1 || tile_tokens % host->page_size != 0)
    return fail(PSD_ERR_INVALID_ARG, "tile_tokens %d is not a positive multiple of page_size %d",
                tile_tokens, host->page_size);
  if (!items || !num_items || !o_indptr) return fail(PSD_ERR_INVALID_ARG, "NULL output");
  int32_t count = 0;
  o_indptr[0] = 0;
  for (int32_t b = 0; b < host->batch; ++b) {
    int32_t c = emit_chunks(b, host->page_indptr[b], tokens_of(host, b), tile_tokens,
                            host->page_size, o_indptr[b], items, item_capacity, &count);
    if (c < 0) return fail(PSD_ERR_INVALID_ARG, "item_capacity %d too small", item_capacity);
    o_indptr[b + 1] = o_indptr[b] + c;
  }
  *num_items = count;
  return PSD_OK;
}

extern "C" psd_status detect_shared_prefix(const psd_page_table *host, int32_t min_shared_pages,
                                           int32_t min_members, int32_t *members,
                                           int32_t *num_members, int32_t *shared_pages,
                                           int32_t *decline_reason) {
  clear_error();
  psd_status st = validate_table(host, -1);
  if (st != PSD_OK) return st;
  if (!members || !num_members || !shared_pages || !decline_reason)
    return fail(PSD_ERR_INVALID_ARG, "NULL output");
  *num_members = 0;
  *shared_pages = 0;
  const int32_t *ip = host->page_indptr;
  const int32_t *ix = host->page_indices;

  // Groups keyed by first page id, members in increasing batch order; groups in
  // order of their first member.
  std::unordered_map<int32_t, int32_t> slot;
  std::vector<std::vector<int32_t>> groups;
  slot.reserve(size_t(host->batch) * 2);
  for (int32_t b = 0; b < host->batch; ++b) {
    if (pages_of(host, b) < 2) continue;  // needs a page before its last one
    auto ins = slot.emplace(ix[ip[b]], int32_t(groups.size()));
    if (ins.second) groups.emplace_back();
    groups[ins.first->second].push_back(b);
  }
  bool any_pair = false;
  for (auto &g : groups) any_pair |= g.size() >= 2;
  if (!any_pair) {
    *decline_reason = PSD_DECLINE_NO_SHARED_PAGES;
    return PSD_OK;
  }
  const size_t need = size_t(std::max(2, min_members));
  const int32_t min_span = std::max(1, min_shared_pages);
  bool any_eligible = false;
  int64_t best_score = -1;
  int32_t best_group = -1, best_span = 0;
  for (size_t gi = 0; gi < groups.size(); ++gi) {
    const auto &g = groups[gi];
    if (g.size() < need) continue;
    any_eligible = true;
    int32_t cap = pages_of(host, g[0]);
    for (int32_t b : g) cap = std::min(cap, pages_of(host, b));
    cap -= 1;
    int32_t span = 0;
    const int32_t *lead = ix + ip[g[0]];
    for (; span < cap; ++span) {
      bool same = true;
      for (size_t k = 1; k < g.size() && same; ++k) same = ix[ip[g[k]] + span] == lead[span];
      if (!same) break;
    }
    if (span < min_span) continue;
    int64_t score = int64_t(span) * int64_t(g.size() - 1);
    // groups are visited in order of their first member, so a strict '>' keeps
    // the smallest first member on ties
    if (score > best_score) {
      best_score = score;
      best_group = int32_t(gi);
      best_span = span;
    }
  }
  if (!any_eligible) {
    *decline_reason = PSD_DECLINE_MEMBERS_BELOW_THRESHOLD;
    return PSD_OK;
  }
  if (best_group < 0) {
    *decline_reason = PSD_DECLINE_SPAN_BELOW_THRESHOLD;
    return PSD_OK;
  }
  const auto &g = groups[best_group];
  for (size_t k = 0; k < g.size(); ++k) members[k] = g[k];
  *num_members = int32_t(g.size());
  *shared_pages = best_span;
  *decline_reason = PSD_DECLINE_NONE;
  return PSD_OK;
}

extern "C" psd_status build_cascade_plan(const psd_page_table *host, const int32_t *members,
                                         int32_t num_members, int32_t shared_pages,
                                         int32_t tile_tokens, psd_cascade_plan *plan) {
  clear_error();
  psd_status st = validate_table(host, -1);
  if (st != PSD_OK) return st;
  if (!plan || !plan->o_indptr || !plan->l1_items || !plan->l0_items ||
      !plan->member_row_base || !plan->members)
    return fail(PSD_ERR_INVALID_ARG, "plan: NULL array");
  const int32_t B = host->batch, P = host->page_size;
  if (tile_tokens < 1 || tile_tokens % P != 0)
    return fail(PSD_ERR_INVALID_ARG, "tile_tokens %d is not a positive multiple of page_size %d",
                tile_tokens, P);
  if (plan->batch_capacity < B) return fail(PSD_ERR_INVALID_ARG, "plan: batch_capacity < batch");
  if (num_members < 0 || num_members > B || (num_members > 0 && (!members || shared_pages < 1)))
    return fail(PSD_ERR_INVALID_ARG, "plan: bad members (%d) / shared_pages (%d)", num_members,
                shared_pages);
  std::vector<char> is_member(size_t(B), 0);
  for (int32_t m = 0; m < num_members; ++m) {
    int32_t b = members[m];
    if (b < 0 || b >= B || (m > 0 && b <= members[m - 1]))
      return fail(PSD_ERR_INVALID_ARG, "plan: members must be increasing batch indices");
    if (pages_of(host, b) <= shared_pages)
      return fail(PSD_ERR_INVALID_ARG, "plan: shared span reaches the last page of request %d", b);
    for (int32_t p = 0; p < shared_pages; ++p)
      if (host->page_indices[host->page_indptr[b] + p] !=
          host->page_indices[host->page_indptr[members[0]] + p])
        return fail(PSD_ERR_INVALID_ARG, "plan: request %d does not share page position %d", b, p);
    is_member[b] = 1;
  }
  int32_t n0 = 0, n1 = 0;
  int32_t C0 = 0;
  if (num_members > 0) {
    C0 = emit_chunks(-1, host->page_indptr[members[0]], int64_t(shared_pages) * P, tile_tokens, P,
                     0, plan->l0_items, plan->item_capacity, &n0);
    if (C0 < 0) return fail(PSD_ERR_INVALID_ARG, "plan: item_capacity too small");
  }
  plan->o_indptr[0] = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t skip = is_member[b] ? shared_pages : 0;
    const int32_t base = plan->o_indptr[b] + (is_member[b] ? C0 : 0);
    int32_t c = emit_chunks(b, host->page_indptr[b] + skip, tokens_of(host, b) - int64_t(skip) * P,
                            tile_tokens, P, base, plan->l1_items, plan->item_capacity, &n1);
    if (c < 0) return fail(PSD_ERR_INVALID_ARG, "plan: item_capacity too small");
    plan->o_indptr[b + 1] = base + c;
  }
  for (int32_t m = 0; m < num_members; ++m) {
    plan->members[m] = members[m];
    plan->member_row_base[m] = plan->o_indptr[members[m]];
  }
  plan->batch = B;
  plan->page_size = P;
  plan->tile_tokens = tile_tokens;
  plan->num_members = num_members;
  plan->shared_pages = num_members > 0 ? shared_pages : 0;
  plan->l0_num_items = n0;
  plan->l1_num_items = n1;
  plan->num_rows = plan->o_indptr[B];
  return PSD_OK;
}

extern "C" int32_t psd_cascade_env_enabled(int32_t fallback) {
  const char *v = std::getenv("PSD_CASCADE_ATTENTION");
  if (!v) return fallback;
  std::string s(v);
  size_t a = s.find_first_not_of(" \t\r\n"), e = s.find_last_not_of(" \t\r\n");
  s = a == std::string::npos ? std::string() : s.substr(a, e - a + 1);
  for (auto &ch : s) ch = char(std::tolower((unsigned char)ch));
  if (s == "0" || s == "false" || s == "off" || s == "no") return 0;
  if (s == "1" || s == "true" || s == "on" || s == "yes") return 1;
  return fallback;
}

extern "C" psd_status psd_plan_decode(const psd_page_table *host, int32_t tile_tokens,
                                      int32_t enable, int32_t min_shared_pages,
                                      int32_t min_members, psd_cascade_plan *plan) {
  clear_error();
  if (!plan || !plan->members) return fail(PSD_ERR_INVALID_ARG, "plan: NULL");
  if (enable < 0) enable = psd_cascade_env_enabled(0);
  int32_t nm = 0, span = 0, reason = PSD_DECLINE_DISABLED;
  if (enable) {
    psd_status st = detect_shared_prefix(host, min_shared_pages, min_members, plan->members, &nm,
                                         &span, &reason);
    if (st != PSD_OK) return st;
  }
  std::vector<int32_t> mem(plan->members, plan->members + nm);
  psd_status st = build_cascade_plan(host, mem.data(), nm, span, tile_tokens, plan);
  if (st != PSD_OK) return st;
  plan->decline_reason = reason;
  return PSD_OK;
}

extern "C" psd_status psd_plan_capacity(const psd_page_table *host, int32_t *batch_capacity,
                                        int32_t *item_capacity) {
  clear_error();
  psd_status st = validate_table(host, -1);
  if (st != PSD_OK) return st;
  if (batch_capacity) *batch_capacity = std::max(host->batch, 1);
  if (item_capacity) *item_capacity = std::max(host->page_indptr[host->batch], 1);
  return PSD_OK;
}

// ------------------------------------------------ several and nested shared spans
// (An extension the pages scope out: mlxcel PR #1004, Task item 1 keeps to a single
// shared level; Left out / unsure lists nested sharing of a system prompt plus a
// per-tenant sub-prefix as not attempted.)  Every first-page group passing the thresholds becomes a
// segment; inside a segment the members regroup by their page at its end and the
// same rules apply from there, up to max_levels; segments depth first, groups in
// order of their lowest batch index.
namespace psd {
namespace {

struct Seg {
  std::vector<int32_t> members;
  int32_t start, span;
};

void find_segments(const psd_page_table *t, const std::vector<int32_t> &cands, int32_t start,
                   int32_t level, int32_t max_levels, size_t need, int32_t min_span, std::vector<Seg> &out) {
  const int32_t *ip = t->page_indptr, *ix = t->page_indices;
  std::unordered_map<int32_t, int32_t> slot;
  std::vector<std::vector<int32_t>> groups;
  for (int32_t b : cands) {
    if (pages_of(t, b) - 1 - start < 1) continue;  // no shareable page at `start`
    auto ins = slot.emplace(ix[ip[b] + start], int32_t(groups.size()));
    if (ins.second) groups.emplace_back();
    groups[ins.first->second].push_back(b);
  }
  for (auto &g : groups) {
    if (g.size() < need) continue;
    int32_t cap = pages_of(t, g[0]);
    for (int32_t b : g) cap = std::min(cap, pages_of(t, b));
    cap -= 1 + start;
    int32_t span = 0;
    const int32_t *lead = ix + ip[g[0]];
    for (; span < cap; ++span) {
      bool same = true;
      for (size_t k = 1; k < g.size() && same; ++k) same = ix[ip[g[k]] + start + span] == lead[start + span];
      if (!same) break;
    }
    if (span < min_span) continue;
    out.push_back(Seg{g, start, span});
    if (level < max_levels) find_segments(t, g, start + span, level + 1, max_levels, need, min_span, out);
  }
}

}  // namespace
}  // namespace psd

using psd::clear_error;
using psd::fail;

extern "C" psd_status psd_plan_nested_capacity(const psd_page_table *host, int32_t max_levels,
                                               int32_t *batch_capacity, int32_t *entry_capacity,
                                               int32_t *segment_capacity, int32_t *item_capacity) {
  clear_error();
  psd_status st = psd::validate_table(host, -1);
  if (st != PSD_OK) return st;
  if (max_levels < 1 || max_levels > 8) return fail(PSD_ERR_INVALID_ARG, "max_levels %d outside [1, 8]", max_levels);
  const int32_t B = std::max(host->batch, 1);
  if (batch_capacity) *batch_capacity = B;
  if (entry_capacity) *entry_capacity = B * max_levels;
  if (segment_capacity) *segment_capacity = B * max_levels;
  if (item_capacity) *item_capacity = std::max(host->page_indptr[host->batch], 1);
  return PSD_OK;
}

extern "C" psd_status psd_plan_nested(const psd_page_table *host, int32_t tile_tokens, int32_t enable,
                                      int32_t min_shared_pages, int32_t min_members, int32_t max_levels,
                                      psd_nested_plan *plan) {
  clear_error();
  psd_status st = psd::validate_table(host, -1);
  if (st != PSD_OK) return st;
  if (!plan || !plan->segments || !plan->members || !plan->member_row_base || !plan->l0_items ||
      !plan->l1_items || !plan->o_indptr)
    return fail(PSD_ERR_INVALID_ARG, "nested plan: NULL array");
  if (max_levels < 1 || max_levels > 8) return fail(PSD_ERR_INVALID_ARG, "max_levels %d outside [1, 8]", max_levels);
  const int32_t B = host->batch, P = host->page_size;
  if (tile_tokens < 1 || tile_tokens % P != 0)
    return fail(PSD_ERR_INVALID_ARG, "tile_tokens %d is not a positive multiple of page_size %d", tile_tokens, P);
  if (plan->batch_capacity < B) return fail(PSD_ERR_INVALID_ARG, "nested plan: batch_capacity < batch");
  if (enable < 0) enable = psd_cascade_env_enabled(0);

  std::vector<psd::Seg> segs;
  if (enable) {
    std::vector<int32_t> all(static_cast<size_t>(B));
    for (int32_t b = 0; b < B; ++b) all[size_t(b)] = b;
    psd::find_segments(host, all, 0, 1, max_levels, size_t(std::max(2, min_members)),
                       std::max(1, min_shared_pages), segs);
  }
  int32_t reason = PSD_DECLINE_NONE;
  if (!enable) {
    reason = PSD_DECLINE_DISABLED;
  } else if (segs.empty()) {  // the top level applies the two-level tests: same reason
    std::vector<int32_t> tmp(static_cast<size_t>(std::max(B, 1)));
    int32_t nm = 0, span = 0;
    st = detect_shared_prefix(host, min_shared_pages, min_members, tmp.data(), &nm, &span, &reason);
    if (st != PSD_OK) return st;
  }
  if (int32_t(segs.size()) > plan->segment_capacity)
    return fail(PSD_ERR_INVALID_ARG, "nested plan: segment_capacity too small");

  // level-0 items and member lists by segment
  int32_t n0 = 0, entries = 0;
  std::vector<int32_t> seg_chunks(static_cast<size_t>(segs.size()));
  for (size_t s = 0; s < segs.size(); ++s) {
    const psd::Seg &g = segs[s];
    psd_segment &d = plan->segments[s];
    d.first_member = entries;
    d.num_members = int32_t(g.members.size());
    d.start_page = g.start;
    d.shared_pages = g.span;
    d.first_item = n0;
    const int32_t c = psd::emit_chunks(-1, host->page_indptr[g.members[0]] + g.start, int64_t(g.span) * P,
                                       tile_tokens, P, 0, plan->l0_items, plan->item_capacity, &n0);
    if (c < 0) return fail(PSD_ERR_INVALID_ARG, "nested plan: item_capacity too small");
    d.num_items = c;
    seg_chunks[s] = c;
    if (entries + d.num_members > plan->entry_capacity)
      return fail(PSD_ERR_INVALID_ARG, "nested plan: entry_capacity too small");
    for (int32_t b : g.members) plan->members[entries++] = b;
  }
  // rows: each request's segments in segment order, then its level-1 chunks
  std::vector<std::vector<std::pair<int32_t, int32_t>>> of_request(static_cast<size_t>(B));  // (segment, entry)
  for (size_t s = 0; s < segs.size(); ++s)
    for (int32_t k = 0; k < plan->segments[s].num_members; ++k) {
      const int32_t e = plan->segments[s].first_member + k;
      of_request[size_t(plan->members[e])].push_back({int32_t(s), e});
    }
  int32_t n1 = 0;
  plan->o_indptr[0] = 0;
  for (int32_t b = 0; b < B; ++b) {
    int32_t r = plan->o_indptr[b], deepest = 0;
    for (auto &se : of_request[size_t(b)]) {
      plan->member_row_base[se.second] = r;
      r += seg_chunks[size_t(se.first)];
      deepest = std::max(deepest, segs[size_t(se.first)].start + segs[size_t(se.first)].span);
    }
    const int32_t c = psd::emit_chunks(b, host->page_indptr[b] + deepest,
                                       psd::tokens_of(host, b) - int64_t(deepest) * P, tile_tokens, P, r,
                                       plan->l1_items, plan->item_capacity, &n1);
    if (c < 0) return fail(PSD_ERR_INVALID_ARG, "nested plan: item_capacity too small");
    plan->o_indptr[b + 1] = r + c;
  }
  plan->batch = B;
  plan->page_size = P;
  plan->tile_tokens = tile_tokens;
  plan->max_levels = max_levels;
  plan->num_segments = int32_t(segs.size());
  plan->num_entries = entries;
  plan->decline_reason = reason;
  plan->l0_num_items = n0;
  plan->l1_num_items = n1;
  plan->num_rows = plan->o_indptr[B];
  return PSD_OK;
}
