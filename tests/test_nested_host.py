"""CPU tests of the C ABI's nested planner (psd_plan_nested): bit for bit equal to the
oracle planner on the hand-derived cases, on random nested and general tables at one
to three levels and on the nested decode batch; bounds and capacities are checked."""
import json
import os

import numpy as np
import pytest

from oracle import planner as PL
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = json.load(open(os.path.join(ROOT, "tests", "golden", "nested_cases.json")))["nested"]


@pytest.fixture(scope="module")
def api():
    import paged_split_kv_decode_gb300.api as api
    api.L.load()
    return api


def _csr(pages):
    indptr, idx = [0], []
    for p in pages:
        idx += p
        indptr.append(len(idx))
    return np.array(indptr, dtype=np.int32), np.array(idx, dtype=np.int32)


def _assert_equal(p, r):
    assert [tuple(s) for s in p.segments] == [tuple(s) for s in r["segments"]]
    assert p.members == r["members"] and p.member_row_base == r["member_row_base"]
    assert p.l0_items.tolist() == [list(x) for x in r["l0_items"]]
    assert p.l1_items.tolist() == [list(x) for x in r["l1_items"]]
    assert p.o_indptr == r["o_indptr"] and p.num_rows == r["num_rows"]
    assert p.decline_reason == r["decline_reason"]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"])
def test_golden_cases(api, case):
    indptr, idx = _csr(case["pages"])
    last = np.array(case["last_page_len"], dtype=np.int32)
    t = api.HostTable(indptr, idx, last, case["page_size"])
    args = (case["tile_tokens"], 1, case["min_shared_pages"], case["min_members"], case["max_levels"])
    p = api.plan_nested(t, *args)
    r = PL.plan_nested(indptr, idx, last, case["page_size"], *args)
    _assert_equal(p, r)


def _nested_table(rng, B, P):
    base = list(rng.choice(np.arange(1000, 2000), size=int(rng.integers(1, 7)), replace=False))
    tenants = [list(rng.choice(np.arange(2000 + 300 * t, 2300 + 300 * t), size=int(rng.integers(1, 5)),
                               replace=False)) for t in range(3)]
    sub = [list(rng.choice(np.arange(3000 + 100 * t, 3100 + 100 * t), size=int(rng.integers(1, 3)),
                           replace=False)) for t in range(3)]
    nxt, pages = 5000, []
    for b in range(B):
        kind = int(rng.integers(0, 5))
        pre = [] if kind == 4 else base + (tenants[kind % 3] if kind < 3 else [])
        if kind < 3 and rng.random() < 0.5:
            pre = pre + sub[kind]
        own = int(rng.integers(1, 4))
        pages.append(pre + list(range(nxt, nxt + own)))
        nxt += own
    return pages, rng.integers(1, P + 1, size=B).astype(np.int32)


@pytest.mark.parametrize("seed", range(50))
def test_random_nested_tables_bit_exact(api, seed):
    rng = np.random.default_rng(300 + seed)
    P = int(rng.choice([1, 4, 16]))
    B = int(rng.integers(1, 20))
    pages, last = _nested_table(rng, B, P)
    indptr, idx = _csr(pages)
    t = api.HostTable(indptr, idx, last, P)
    T = P * int(rng.integers(1, 4))
    for levels in (1, 2, 3):
        for msp, mm in ((1, 2), (2, 2), (1, 3)):
            p = api.plan_nested(t, T, 1, msp, mm, levels)
            r = PL.plan_nested(indptr, idx, last, P, T, True, msp, mm, levels)
            _assert_equal(p, r)


@pytest.mark.parametrize("seed", range(20))
def test_random_general_tables_bit_exact(api, seed):
    rng = np.random.default_rng(400 + seed)
    B, P = int(rng.integers(1, 24)), 4
    lengths = rng.integers(1, 80, size=B)
    indptr, indices, last = synth.page_table(lengths, P, 4000, rng)
    indices = indices.copy()
    for _ in range(int(rng.integers(0, 4)) if B >= 2 else 0):
        grp = rng.choice(B, size=int(rng.integers(2, min(6, B) + 1)), replace=False)
        depth = int(rng.integers(1, 10))
        for b in grp[1:]:
            n = min(depth, indptr[b + 1] - indptr[b], indptr[grp[0] + 1] - indptr[grp[0]])
            indices[indptr[b]:indptr[b] + n] = indices[indptr[grp[0]]:indptr[grp[0]] + n]
    t = api.HostTable(indptr, indices, last, P)
    for enable in (0, 1):
        p = api.plan_nested(t, 8, enable, 1, 2, 2)
        r = PL.plan_nested(indptr, indices, last, P, 8, bool(enable), 1, 2, 2)
        _assert_equal(p, r)


def test_nested_decode_batch(api):
    w = synth.nested_decode(0, canary=False)
    t = api.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
    p = api.plan_nested(t, w.tile_tokens, 1, 16, 2, 2)
    r = PL.plan_nested(w.page_indptr, w.page_indices, w.last_page_len, w.page_size, w.tile_tokens, True, 16, 2, 2)
    _assert_equal(p, r)
    assert [s[1] for s in p.segments] == [16, 8, 8] and [s[3] for s in p.segments] == [256, 128, 128]


@pytest.mark.parametrize("levels", [0, 9, -1])
def test_max_levels_bounds(api, levels):
    w = synth.tiny_cascade(0, canary=False)
    t = api.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
    with pytest.raises(api.L.PsdError):
        api.plan_nested(t, w.tile_tokens, 1, 4, 2, levels)


def test_entry_capacity_too_small_is_rejected(api):
    w = synth.nested_decode(1, canary=False)
    t = api.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
    plan = api.NestedPlan(t, 2)
    plan.c.entry_capacity = 3
    with pytest.raises(api.L.PsdError):
        api.L.check(api.L.load().psd_plan_nested(api.C.byref(t.c), w.tile_tokens, 1, 16, 2, 2,
                                                 api.C.byref(plan.c)))
