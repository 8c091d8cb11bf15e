"""Pins of the oracle planner and cascade: hand-derived golden cases, page
conservation between the two levels and the flat view, the cascade = flat
invariant, and the member-major stacking negative control (mlxcel PR #1004,
Decomposition, Task items 1-2 and 4, Correctness coverage)."""
import json
import os
from collections import Counter

import numpy as np
import pytest

from oracle import attention as A
from oracle import cascade as C
from oracle import planner as PL
import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "planner_cases.json")))


@pytest.mark.parametrize("case", GOLDEN["detect"], ids=lambda c: c["name"])
def test_detect_golden(case):
    members, span, reason = PL.detect_shared_prefix(
        case["page_indptr"], case["page_indices"], case["min_shared_pages"], case["min_members"])
    e = case["expect"]
    assert (members, span, reason) == (e["members"], e["shared_pages"], e["decline_reason"])


@pytest.mark.parametrize("case", GOLDEN["plan"], ids=lambda c: c["name"])
def test_cascade_plan_golden(case):
    p = PL.build_cascade_plan(case["page_indptr"], case["last_page_len"], case["page_size"],
                              case["members"], case["shared_pages"], case["tile_tokens"])
    e = case["expect"]
    assert [list(x) for x in p["l0_items"]] == e["l0_items"]
    assert [list(x) for x in p["l1_items"]] == e["l1_items"]
    assert p["o_indptr"] == e["o_indptr"]
    assert p["member_row_base"] == e["member_row_base"]
    assert p["num_rows"] == e["num_rows"]


@pytest.mark.parametrize("case", GOLDEN["split"], ids=lambda c: c["name"])
def test_split_golden(case):
    items, o_indptr = PL.split_plan(case["page_indptr"], case["last_page_len"],
                                    case["page_size"], case["tile_tokens"])
    assert [list(x) for x in items] == case["expect"]["items"]
    assert o_indptr == case["expect"]["o_indptr"]


def test_env_switch_golden():
    for value, default, expect in GOLDEN["env_switch"]["cases"]:
        assert PL.env_switch(value, default) is expect


def _random_table(rng, B=12, P=4):
    """Random page table with a few planted shared prefixes of random depth."""
    lengths = rng.integers(1, 60, size=B)
    indptr, indices, last = synth.page_table(lengths, P, 2000, rng)
    indices = indices.copy()
    for _ in range(3):
        grp = rng.choice(B, size=int(rng.integers(2, 5)), replace=False)
        depth = int(rng.integers(1, 8))
        src = grp[0]
        for b in grp[1:]:
            n = min(depth, indptr[b + 1] - indptr[b], indptr[src + 1] - indptr[src])
            indices[indptr[b]:indptr[b] + n] = indices[indptr[src]:indptr[src] + n]
    return indptr, indices, last, P


def _page_multiset(items, page_indices, P, indptr):
    """Pool pages each request's items touch (level-0 items count once per member)."""
    out = Counter()
    for qi, off, n, _ in items:
        npages = (n + P - 1) // P
        for k in range(npages):
            out[(qi, int(page_indices[off + k]))] += 1
    return out


@pytest.mark.parametrize("seed", range(25))
def test_plan_conserves_pages_between_levels_and_flat(seed):
    rng = np.random.default_rng(seed)
    indptr, indices, last, P = _random_table(rng)
    T = P * int(rng.integers(1, 4))
    plan = PL.plan_decode(indptr, indices, last, P, T, True, 1, 2)
    flat_items, flat_indptr = PL.split_plan(indptr, last, P, T)
    flat = _page_multiset(flat_items, indices, P, indptr)
    casc = _page_multiset(plan["l1_items"], indices, P, indptr)
    for m in plan["members"]:
        for qi, off, n, c in plan["l0_items"]:
            for k in range((n + P - 1) // P):
                casc[(m, int(indices[off + k]))] += 1
    assert casc == flat
    # level-0 pages are the members' common prefix, read once instead of M times
    span = plan["shared_pages"]
    for m in plan["members"]:
        assert list(indices[indptr[m]:indptr[m] + span]) == \
            list(indices[indptr[plan["members"][0]]:indptr[plan["members"][0]] + span])
        assert indptr[m + 1] - indptr[m] > span
    # every partial row is written exactly once and groups are contiguous
    rows = sorted([r for *_, r in plan["l1_items"]] +
                  [base + c for base in plan["member_row_base"] for *_, c in plan["l0_items"]])
    assert rows == list(range(plan["num_rows"]))
    assert plan["o_indptr"][-1] == plan["num_rows"]
    # token conservation per request
    for b in range(len(indptr) - 1):
        L = PL.request_length(indptr, last, P, b)
        got = sum(n for qi, _, n, _ in plan["l1_items"] if qi == b)
        if b in plan["members"]:
            got += sum(n for *_, n, _ in plan["l0_items"])
        assert got == L


def _oracle_case(w):
    return A.workload_arrays(w)


def test_cascade_levels_equal_flat_on_tiny_cascade():
    w = synth.tiny_cascade(seed=0)
    a = _oracle_case(w)
    plan = PL.plan_decode(w.page_indptr, w.page_indices, w.last_page_len, w.page_size,
                          w.tile_tokens, True, w.min_shared_pages, w.min_members)
    assert plan["members"] == [0, 1, 2] and plan["shared_pages"] == 4
    o, lse, _, _ = C.cascade_levels(a, plan, w.tile_tokens)
    fo, fl = A.decode_attention(a)
    assert np.abs(o - fo).max() < 1e-12 and np.abs(lse - fl).max() < 1e-12
    # the flat plan (partials + merge) agrees too
    items, o_indptr = PL.split_plan(w.page_indptr, w.last_page_len, w.page_size, w.tile_tokens)
    chunks = [(b, (off - int(w.page_indptr[b])) * w.page_size,
               (off - int(w.page_indptr[b])) * w.page_size + n, row) for b, off, n, row in items]
    vp, lp = A.partial_attention(a, chunks)
    mo, ml = A.merge_states(vp, lp, o_indptr)
    assert np.abs(mo - fo).max() < 1e-12 and np.abs(ml - fl).max() < 1e-12


def test_tiny_cascade_declines_at_default_thresholds():
    w = synth.tiny_cascade(seed=1)
    members, span, reason = PL.detect_shared_prefix(w.page_indptr, w.page_indices)
    assert members == [] and reason == PL.DECLINE_SPAN_BELOW_THRESHOLD


def test_member_major_stacking_reads_the_wrong_kv_head():
    """Negative control named on the page: with member-major stacking the level-0
    partials no longer match the per-member attention over the span."""
    w = synth.tiny_cascade(seed=2)
    a = _oracle_case(w)
    members, span = [0, 1, 2], 4
    q = A.bf16_bits_to_f64(a["q_raw"])
    G = w.Hq // w.Hkv
    good0, _ = C.level0_partials(a, members, span, span * w.page_size)
    bad0, _ = C.level0_partials(a, members, span, span * w.page_size, member_major=True)
    vo, _ = C.unstack(good0, good0[..., 0], len(members), w.Hkv, G)
    vb, _ = C.unstack(bad0, bad0[..., 0], len(members), w.Hkv, G)
    for m, b in enumerate(members):
        K, V = A.gather_kv(a, b)
        ref, _ = A.attend(q[b], K[:span * w.page_size], V[:span * w.page_size], w.sm_scale)
        assert np.abs(vo[m, 0] - ref).max() < 1e-12
        assert np.abs(vb[m, 0] - ref).max() > 1e-2


def test_cascade_equals_flat_on_reduced_cascade_workload():
    w = synth.cascade_decode(seed=0, members=4, others=4, shared_tokens=512)
    a = _oracle_case(w)
    plan = PL.plan_decode(w.page_indptr, w.page_indices, w.last_page_len, w.page_size,
                          w.tile_tokens, True, 16, 2)
    assert len(plan["members"]) == 4 and plan["shared_pages"] == 32
    o, lse, _, _ = C.cascade_levels(a, plan, w.tile_tokens)
    fo, fl = A.decode_attention(a)
    assert np.abs(o - fo).max() < 1e-11 and np.abs(lse - fl).max() < 1e-11
