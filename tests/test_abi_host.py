"""CPU tests of the C ABI: the library loads and exports every declared symbol, and
its host planning (split work list, shared-prefix detection, cascade plan, kill
switch) agrees bit for bit with the oracle planner."""
import ctypes as C
import json
import os
import re

import numpy as np
import pytest

from oracle import planner as PL
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "planner_cases.json")))


@pytest.fixture(scope="module")
def api():
    import paged_split_kv_decode_gb300.api as api
    api.L.load()
    return api


def declared_functions():
    text = open(os.path.join(ROOT, "include", "psd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^(?:psd_status|size_t|int32_t|const char \*)\s*\**(\w+)\s*\(",
                                 text, flags=re.M)))


def test_library_exports_every_declared_symbol(api):
    names = declared_functions()
    assert len(names) >= 15
    lib = api.L.load()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(api.L.EXPORTS)


def _table(api, case):
    indices = case.get("page_indices")
    if indices is None:
        indices = list(range(case["page_indptr"][-1]))
    return api.HostTable(case["page_indptr"], indices, case["last_page_len"], case["page_size"])


@pytest.mark.parametrize("case", GOLDEN["detect"], ids=lambda c: c["name"])
def test_detect_matches_golden(api, case):
    t = _table(api, case)
    got = api.detect_shared_prefix(t, case["min_shared_pages"], case["min_members"])
    e = case["expect"]
    assert got == (e["members"], e["shared_pages"], e["decline_reason"])


@pytest.mark.parametrize("case", GOLDEN["plan"], ids=lambda c: c["name"])
def test_cascade_plan_matches_golden(api, case):
    t = _table(api, case)
    p = api.build_cascade_plan(t, case["members"], case["shared_pages"], case["tile_tokens"])
    e = case["expect"]
    assert p.l0_items.tolist() == e["l0_items"]
    assert p.l1_items.tolist() == e["l1_items"]
    assert p.o_indptr == e["o_indptr"]
    assert p.member_row_base == e["member_row_base"]
    assert p.num_rows == e["num_rows"]


@pytest.mark.parametrize("case", GOLDEN["split"], ids=lambda c: c["name"])
def test_split_matches_golden(api, case):
    t = _table(api, case)
    items, o_indptr = api.split_plan(t, case["tile_tokens"])
    assert items.tolist() == case["expect"]["items"]
    assert o_indptr.tolist() == case["expect"]["o_indptr"]


def _random_table(rng, B, P):
    lengths = rng.integers(1, 80, size=B)
    indptr, indices, last = synth.page_table(lengths, P, 4000, rng)
    indices = indices.copy()
    for _ in range(int(rng.integers(0, 4)) if B >= 2 else 0):
        grp = rng.choice(B, size=int(rng.integers(2, min(6, B) + 1)), replace=False)
        depth = int(rng.integers(1, 10))
        src = grp[0]
        for b in grp[1:]:
            n = min(depth, indptr[b + 1] - indptr[b], indptr[src + 1] - indptr[src])
            indices[indptr[b]:indptr[b] + n] = indices[indptr[src]:indptr[src] + n]
    return indptr, indices, last


@pytest.mark.parametrize("seed", range(60))
def test_planner_bit_exact_against_oracle_on_random_tables(api, seed):
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice([1, 4, 16]))
    B = int(rng.integers(1, 24))
    indptr, indices, last = _random_table(rng, B, P)
    T = P * int(rng.integers(1, 5))
    msp = int(rng.integers(0, 6))
    mm = int(rng.integers(0, 4))
    t = api.HostTable(indptr, indices, last, P)
    assert api.detect_shared_prefix(t, msp, mm) == tuple(PL.detect_shared_prefix(indptr, indices, msp, mm))
    items, o_indptr = api.split_plan(t, T)
    ritems, ro = PL.split_plan(indptr, last, P, T)
    assert items.tolist() == [list(x) for x in ritems] and o_indptr.tolist() == ro
    for enable in (0, 1):
        p = api.plan_decode(t, T, enable, msp, mm)
        r = PL.plan_decode(indptr, indices, last, P, T, bool(enable), msp, mm)
        assert p.members == r["members"]
        assert p.shared_pages == r["shared_pages"]
        assert p.decline_reason == r["decline_reason"]
        assert p.l0_items.tolist() == [list(x) for x in r["l0_items"]]
        assert p.l1_items.tolist() == [list(x) for x in r["l1_items"]]
        assert p.o_indptr == r["o_indptr"]
        assert p.member_row_base == r["member_row_base"]
        assert p.num_rows == r["num_rows"]


@pytest.mark.parametrize("maker,kw", [(synth.tiny_cascade, {}), (synth.flat_decode, {}),
                                      (synth.cascade_decode, {}),
                                      (synth.mla_decode, dict(batch=16, lo=4096, hi=8192, num_pages=2048))])
def test_planner_bit_exact_on_config_shapes(api, maker, kw):
    w = maker(seed=0, canary=False, **kw)
    t = api.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
    p = api.plan_decode(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    r = PL.plan_decode(w.page_indptr, w.page_indices, w.last_page_len, w.page_size, w.tile_tokens,
                       True, w.min_shared_pages, w.min_members)
    assert (p.members, p.shared_pages, p.decline_reason) == (r["members"], r["shared_pages"], r["decline_reason"])
    assert p.l0_items.tolist() == [list(x) for x in r["l0_items"]]
    assert p.l1_items.tolist() == [list(x) for x in r["l1_items"]]
    assert p.o_indptr == r["o_indptr"]
    if maker is synth.cascade_decode:
        assert len(p.members) == 16 and p.shared_pages == 512
    if maker is synth.tiny_cascade:
        assert p.members == [0, 1, 2] and p.shared_pages == 4


def test_env_kill_switch_parsing(api, monkeypatch):
    for value, default, expect in GOLDEN["env_switch"]["cases"]:
        if value is None:
            monkeypatch.delenv("PSD_CASCADE_ATTENTION", raising=False)
        else:
            monkeypatch.setenv("PSD_CASCADE_ATTENTION", value)
        assert api.cascade_env_enabled(int(default)) == int(expect), (value, default)


def test_plan_decode_env_disable(api, monkeypatch):
    w = synth.tiny_cascade(seed=0, canary=False)
    t = api.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
    monkeypatch.setenv("PSD_CASCADE_ATTENTION", "off")
    p = api.plan_decode(t, w.tile_tokens, -1, 4, 2)
    assert p.num_members == 0 and p.decline_reason == PL.DECLINE_DISABLED
    monkeypatch.setenv("PSD_CASCADE_ATTENTION", "on")
    p = api.plan_decode(t, w.tile_tokens, -1, 4, 2)
    assert p.members == [0, 1, 2]


@pytest.mark.parametrize("bad", [
    dict(page_indptr=[0, 2], page_indices=[1, 2], last_page_len=[0], page_size=4),       # last 0
    dict(page_indptr=[0, 2], page_indices=[1, 2], last_page_len=[5], page_size=4),       # last > P
    dict(page_indptr=[0, 0], page_indices=[1], last_page_len=[1], page_size=4),          # empty request
    dict(page_indptr=[1, 2], page_indices=[1, 2], last_page_len=[1], page_size=4),       # indptr[0] != 0
])
def test_host_validation_rejects_bad_tables(api, bad):
    t = api.HostTable(**bad)
    with pytest.raises(api.L.PsdError) as e:
        api.detect_shared_prefix(t)
    assert e.value.status == 1
    with pytest.raises(api.L.PsdError):
        api.split_plan(t, 4)


def test_tile_must_be_multiple_of_page(api):
    t = api.HostTable([0, 3], [0, 1, 2], [3], 4)
    with pytest.raises(api.L.PsdError) as e:
        api.split_plan(t, 6)
    assert "multiple of page_size" in str(e.value)


def test_cascade_plan_rejects_span_reaching_last_page(api):
    t = api.HostTable([0, 2, 4], [5, 6, 5, 6], [1, 1], 4)
    with pytest.raises(api.L.PsdError):
        api.build_cascade_plan(t, [0, 1], 2, 4)


def test_workspace_bytes_grows_with_rows(api):
    a = api.workspace_bytes(4, 10, 10, 8, 64)
    b = api.workspace_bytes(4, 10, 20, 8, 64)
    assert b - a >= 10 * 8 * 64 * 4 and a % 256 == 0
