"""Split-KV work lists, shared-prefix detection and the cascade plan, in plain
Python integers (oracle; test infrastructure only).

Source: mlxcel PR #1004, "compute shared prompt prefixes once per decode batch".
  * Decomposition: the partial kernel's unit is one (request, page tile); level 0 is
    the shared span as one request with M*G query heads per KV head, stacked
    h0 = kv_head * (M * G) + m * G + g; level 1 is each request's private suffix.
  * Merge contract: o_indptr groups contiguous partial rows per output row.
  * Detection: equal page ids at the same position mean one shared block.
  * Task items 1, 2, 4: group by first page, longest common page prefix per group,
    pick the subgroup with the most saved reads shared_pages * (members - 1); one
    shared level; spans that would reach a member's last page, sub-threshold spans
    and sub-threshold member counts fall back to flat.
  * Left out / unsure: a member that diverges early shortens the group's span
    rather than being dropped; thresholds default to 16 pages and 2 members.

Readings where the page leaves a rule open (each pinned by a hand-made case):
  R1  candidates are requests with at least two pages (one page before the last);
  R2  the span is capped at min(n_b - 1) over members before the page threshold is
      applied, so every shared page is full and no member's last page is shared;
  R3  ties in saved reads go to the group whose lowest batch index is smallest;
  R4  members are ordered by increasing batch index;
  R5  each member's level-0 chunk rows precede its level-1 chunk rows in the final
      merge group.

Work item tuples are (q_index, page_off, n_tokens, out_row): q_index is the
request whose query rows are used (-1 for the stacked level-0 request), page_off
the absolute position in page_indices of the chunk's first page, n_tokens the
chunk's token count, out_row its partial row (for level 0: the chunk index).
"""
from __future__ import annotations

DECLINE_NONE = 0
DECLINE_DISABLED = 1
DECLINE_NO_SHARED_PAGES = 2
DECLINE_MEMBERS_BELOW_THRESHOLD = 3
DECLINE_SPAN_BELOW_THRESHOLD = 4

DEFAULT_MIN_SHARED_PAGES = 16
DEFAULT_MIN_MEMBERS = 2


def num_pages(page_indptr, b) -> int:
    return int(page_indptr[b + 1]) - int(page_indptr[b])


def request_length(page_indptr, last_page_len, page_size, b) -> int:
    return (num_pages(page_indptr, b) - 1) * page_size + int(last_page_len[b])


def chunks_of(n_tokens_total: int, tile_tokens: int) -> list:
    """Token ranges [cT, min((c+1)T, L)) of a request split into T-token tiles."""
    out = []
    c = 0
    while c * tile_tokens < n_tokens_total:
        out.append((c * tile_tokens, min((c + 1) * tile_tokens, n_tokens_total)))
        c += 1
    return out


def split_plan(page_indptr, last_page_len, page_size: int, tile_tokens: int):
    """Flat split-KV work list (Decomposition: one unit per (request, page tile)).

    Request b gets C_b = ceil(L_b / T) chunks; chunk c starts at page position
    page_indptr[b] + c * T / P and holds min(T, L_b - c T) tokens; its partial row
    is o_indptr[b] + c with o_indptr[b + 1] = o_indptr[b] + C_b.
    Returns (items, o_indptr).
    """
    assert tile_tokens % page_size == 0
    ppt = tile_tokens // page_size
    B = len(page_indptr) - 1
    items, o_indptr = [], [0]
    for b in range(B):
        L = request_length(page_indptr, last_page_len, page_size, b)
        ch = chunks_of(L, tile_tokens)
        for c, (t0, t1) in enumerate(ch):
            items.append((b, int(page_indptr[b]) + c * ppt, t1 - t0, o_indptr[-1] + c))
        o_indptr.append(o_indptr[-1] + len(ch))
    return items, o_indptr


def detect_shared_prefix(page_indptr, page_indices, min_shared_pages=DEFAULT_MIN_SHARED_PAGES,
                         min_members=DEFAULT_MIN_MEMBERS):
    """Pick one subgroup of requests sharing a whole-page prompt prefix.

    Returns (members, shared_pages, decline_reason); members is empty on decline.
    Steps (Task item 1, Detection, Left out / unsure; readings R1-R4 above):
      1. candidates: requests with n_b >= 2;
      2. group candidates by their first page id;
      3. groups with fewer than max(2, min_members) requests are not eligible;
      4. span = longest positional common page prefix over all group members,
         capped at min(n_b - 1);
      5. keep groups with span >= min_shared_pages;
      6. highest span * (members - 1) wins; ties to the smallest first member.
    """
    B = len(page_indptr) - 1
    groups = {}
    for b in range(B):
        if num_pages(page_indptr, b) >= 2:
            groups.setdefault(int(page_indices[int(page_indptr[b])]), []).append(b)
    multi = [g for g in groups.values() if len(g) >= 2]
    if not multi:
        return [], 0, DECLINE_NO_SHARED_PAGES
    need = max(2, int(min_members))
    eligible = [g for g in multi if len(g) >= need]
    if not eligible:
        return [], 0, DECLINE_MEMBERS_BELOW_THRESHOLD
    best = None
    for g in eligible:
        cap = min(num_pages(page_indptr, b) for b in g) - 1
        span = 0
        while span < cap:
            p0 = int(page_indices[int(page_indptr[g[0]]) + span])
            if all(int(page_indices[int(page_indptr[b]) + span]) == p0 for b in g[1:]):
                span += 1
            else:
                break
        if span < max(1, int(min_shared_pages)):
            continue
        key = (span * (len(g) - 1), -g[0])
        if best is None or key > best[0]:
            best = (key, sorted(g), span)
    if best is None:
        return [], 0, DECLINE_SPAN_BELOW_THRESHOLD
    return best[1], best[2], DECLINE_NONE


def build_cascade_plan(page_indptr, last_page_len, page_size, members, shared_pages,
                       tile_tokens):
    """Level-0 and level-1 work lists and the final merge groups (Task item 2).

    Level 0: one request over the first ``shared_pages`` pages of the members (all
    full pages), split into T-token chunks; its items have q_index -1 and
    out_row = chunk index c.  Level 1: every request; members start after the span
    and keep their last_page_len, non-members keep their whole range.  Final merge
    group of request b: its level-0 chunk rows (members only) then its level-1 rows.
    Returns dict(l0_items, l1_items, o_indptr, member_row_base, num_rows).
    """
    ppt = tile_tokens // page_size
    B = len(page_indptr) - 1
    mset = set(members)
    l0 = []
    if members:
        for c, (t0, t1) in enumerate(chunks_of(shared_pages * page_size, tile_tokens)):
            l0.append((-1, int(page_indptr[members[0]]) + c * ppt, t1 - t0, c))
    C0 = len(l0)
    l1, o_indptr = [], [0]
    for b in range(B):
        L = request_length(page_indptr, last_page_len, page_size, b)
        skip = shared_pages if b in mset else 0
        base = o_indptr[-1] + (C0 if b in mset else 0)
        ch = chunks_of(L - skip * page_size, tile_tokens)
        for c, (t0, t1) in enumerate(ch):
            l1.append((b, int(page_indptr[b]) + skip + c * ppt, t1 - t0, base + c))
        o_indptr.append(base + len(ch))
    member_row_base = [o_indptr[m] for m in members]
    return dict(l0_items=l0, l1_items=l1, o_indptr=o_indptr,
                member_row_base=member_row_base, num_rows=o_indptr[-1])


def plan_decode(page_indptr, page_indices, last_page_len, page_size, tile_tokens,
                enable=True, min_shared_pages=DEFAULT_MIN_SHARED_PAGES,
                min_members=DEFAULT_MIN_MEMBERS):
    """Cascade plan when detection accepts, else the flat plan with the reason."""
    if enable:
        members, span, reason = detect_shared_prefix(page_indptr, page_indices,
                                                     min_shared_pages, min_members)
    else:
        members, span, reason = [], 0, DECLINE_DISABLED
    plan = build_cascade_plan(page_indptr, last_page_len, page_size, members, span,
                              tile_tokens)
    plan.update(members=members, shared_pages=span, decline_reason=reason)
    return plan


def stacked_head(kv: int, m: int, g: int, M: int, G: int) -> int:
    """KV-head-major stacking of level-0 query heads (Decomposition section):
    h0 = kv_head * (M * G) + m * G + g."""
    return kv * (M * G) + m * G + g


def member_major_head(kv: int, m: int, g: int, Hkv: int, G: int) -> int:
    """The wrong, member-major order h0 = m * (Hkv * G) + kv * G + g (negative
    control named on the page)."""
    return m * (Hkv * G) + kv * G + g


def env_switch(value, default: bool) -> bool:
    """Kill-switch parsing of Task item 4: 0/false/off/no disable, 1/true/on/yes
    enable, anything else (or unset) takes the default."""
    if value is None:
        return default
    v = value.strip().lower()
    if v in ("0", "false", "off", "no"):
        return False
    if v in ("1", "true", "on", "yes"):
        return True
    return default


# ------------------------------------------------ several and nested shared spans
# An extension the pages scope out (Task item 1 keeps to a single shared level; Left
# out / unsure names nested sharing, a system prompt common to all plus a per-tenant
# sub-prefix, as not attempted, since it needs one more level).  Readings, each
# pinned by a hand-made case:
#   N1  every first-page group that passes the thresholds becomes a segment (the
#       groups are disjoint), not only the one with the most saved reads;
#   N2  inside a segment [start, start + span), the members are grouped again by
#       their page at start + span, and each group gets the same rules from there
#       (span over all its members, capped so no member's last page is shared, both
#       thresholds), up to max_levels levels in all;
#   N3  segments are listed depth first, groups in order of their lowest batch index;
#   N4  a request's final merge group holds the chunk rows of its segments in that
#       order, then its level-1 rows, which start after its deepest segment.
# With max_levels = 1 and one qualifying group the result is the two-level plan.

def detect_segments(page_indptr, page_indices, min_shared_pages=DEFAULT_MIN_SHARED_PAGES,
                    min_members=DEFAULT_MIN_MEMBERS, max_levels=2):
    """Shared spans as (members, start_page, shared_pages), readings N1-N3."""
    B = len(page_indptr) - 1
    need, msp = max(2, int(min_members)), max(1, int(min_shared_pages))

    def page(b, pos):
        return int(page_indices[int(page_indptr[b]) + pos])

    segs = []

    def recurse(cands, start, level):
        groups = {}
        for b in cands:
            if num_pages(page_indptr, b) - 1 - start >= 1:
                groups.setdefault(page(b, start), []).append(b)
        for g in groups.values():
            if len(g) < need:
                continue
            cap = min(num_pages(page_indptr, b) for b in g) - 1 - start
            span = 0
            while span < cap and all(page(b, start + span) == page(g[0], start + span) for b in g[1:]):
                span += 1
            if span < msp:
                continue
            segs.append((list(g), start, span))
            if level < max_levels:
                recurse(g, start + span, level + 1)

    recurse(list(range(B)), 0, 1)
    return segs


def build_nested_plan(page_indptr, last_page_len, page_size, segments, tile_tokens):
    """Level-0 items per segment, level-1 items and the final merge groups (N4).

    Returns dict(segments=[(first_member, num_members, start_page, shared_pages,
    first_item, num_items)], members, member_row_base (one entry per (segment,
    member)), l0_items (out_row = chunk index within the segment), l1_items, o_indptr,
    num_rows)."""
    ppt = tile_tokens // page_size
    B = len(page_indptr) - 1
    seg_chunks = [chunks_of(span * page_size, tile_tokens) for _, _, span in segments]
    l0, seg_rows, members = [], [], []
    for (g, start, span), ch in zip(segments, seg_chunks):
        first_item = len(l0)
        for c, (t0, t1) in enumerate(ch):
            l0.append((-1, int(page_indptr[g[0]]) + start + c * ppt, t1 - t0, c))
        seg_rows.append((len(members), len(g), start, span, first_item, len(ch)))
        members.extend(g)
    # rows of each request: its segments' chunks (segment order), then level 1
    row_base = [0] * len(members)
    l1, o_indptr = [], [0]
    for b in range(B):
        r = o_indptr[-1]
        deepest = 0
        for s, (g, start, span) in enumerate(segments):
            if b in g:
                row_base[seg_rows[s][0] + g.index(b)] = r
                r += len(seg_chunks[s])
                deepest = max(deepest, start + span)
        L = request_length(page_indptr, last_page_len, page_size, b)
        ch = chunks_of(L - deepest * page_size, tile_tokens)
        for c, (t0, t1) in enumerate(ch):
            l1.append((b, int(page_indptr[b]) + deepest + c * ppt, t1 - t0, r + c))
        o_indptr.append(r + len(ch))
    return dict(segments=seg_rows, members=members, member_row_base=row_base, l0_items=l0,
                l1_items=l1, o_indptr=o_indptr, num_rows=o_indptr[-1])


def plan_nested(page_indptr, page_indices, last_page_len, page_size, tile_tokens, enable=True,
                min_shared_pages=DEFAULT_MIN_SHARED_PAGES, min_members=DEFAULT_MIN_MEMBERS,
                max_levels=2):
    """Nested plan when any segment qualifies, else the flat plan with the
    two-level planner's decline reason (the top level applies the same tests)."""
    segs = detect_segments(page_indptr, page_indices, min_shared_pages, min_members,
                           max_levels) if enable else []
    if enable and not segs:
        reason = detect_shared_prefix(page_indptr, page_indices, min_shared_pages, min_members)[2]
    else:
        reason = DECLINE_NONE if segs else DECLINE_DISABLED
    plan = build_nested_plan(page_indptr, last_page_len, page_size, segs, tile_tokens)
    plan.update(decline_reason=reason)
    return plan
