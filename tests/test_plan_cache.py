"""CPU tests of the plan cache (psd_plan_cache_*): every lookup returns exactly the
oracle planner's plan for its table, hits happen exactly when the same key is still
cached (least recently used eviction), and the key covers KV lengths, not only the
page rows (FreeToken issue #750, Attention batching section: a cache keyed by rows
was a bug, because split-KV also depends on KV length)."""
import numpy as np
import pytest

from oracle import planner as PL
import synth


@pytest.fixture(scope="module")
def api():
    import paged_split_kv_decode_gb300.api as api
    api.L.load()
    return api


def _assert_plan_equals_oracle(p, indptr, indices, last, P, T, enable, msp, mm):
    r = PL.plan_decode(indptr, indices, last, P, T, bool(enable), msp, mm)
    assert p.members == r["members"]
    assert p.shared_pages == r["shared_pages"]
    assert p.decline_reason == r["decline_reason"]
    assert p.l0_items.tolist() == [list(x) for x in r["l0_items"]]
    assert p.l1_items.tolist() == [list(x) for x in r["l1_items"]]
    assert p.o_indptr == r["o_indptr"]
    assert p.member_row_base == r["member_row_base"]
    assert p.num_rows == r["num_rows"]


def _variants(rng, n):
    """n page tables: a few bases plus near-copies that differ in one KV length, one
    page id, or nothing."""
    out = []
    for _ in range(3):
        B = int(rng.integers(2, 12))
        lengths = rng.integers(1, 120, size=B)
        indptr, indices, last = synth.page_table(lengths, 4, 2000, rng)
        indices = indices.copy()
        if B >= 3:  # a shared prefix so some plans cascade
            n_sh = int(min(indptr[1] - indptr[0], indptr[2] - indptr[1]))
            indices[indptr[1]:indptr[1] + n_sh] = indices[indptr[0]:indptr[0] + n_sh]
        out.append((indptr, indices, last))
    while len(out) < n:
        indptr, indices, last = out[int(rng.integers(0, 3))]
        kind = int(rng.integers(0, 3))
        indices, last = indices.copy(), last.copy()
        b = int(rng.integers(0, len(last)))
        if kind == 0:
            last[b] = 1 + (last[b] % 4)        # another KV length, same page rows
        elif kind == 1:
            indices[int(rng.integers(0, len(indices)))] = 1999  # one page id differs
        out.append((indptr, indices, last))
    return out


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("capacity", [1, 3, 8])
def test_lookups_equal_the_oracle_plan_and_hits_follow_lru(api, seed, capacity):
    rng = np.random.default_rng(seed)
    tables = _variants(rng, 8)
    plan_args = [(4, 1, 2, 2), (8, 1, 2, 2), (4, 0, 2, 2), (4, 1, 1, 3)]  # (tile, enable, msp, mm)
    pc = api.PlanCache(capacity)
    model = []  # keys, most recently used last
    hits = misses = 0
    for step in range(60):
        ti = int(rng.integers(0, len(tables)))
        ci = int(rng.integers(0, len(plan_args)))
        indptr, indices, last = tables[ti]
        T, enable, msp, mm = plan_args[ci]
        key = (indptr.tobytes(), indices.tobytes(), last.tobytes(), plan_args[ci])
        expect_hit = key in model
        t = api.HostTable(indptr, indices, last, 4)
        p = pc.lookup(t, T, enable, msp, mm)
        assert p.hit == expect_hit, f"step {step}"
        _assert_plan_equals_oracle(p, indptr, indices, last, 4, T, enable, msp, mm)
        if expect_hit:
            model.remove(key)
            hits += 1
        else:
            if len(model) == capacity:
                model.pop(0)
            misses += 1
        model.append(key)
    assert pc.stats() == {"hits": hits, "misses": misses, "entries": len(model)}


def test_kv_length_is_part_of_the_key(api):
    """Same page rows, one request's last page one token longer: the split changes
    (the request crosses a tile boundary), so a rows-only key would return a wrong
    plan.  The cache must miss and return the new plan."""
    P, T = 4, 8
    indptr = np.array([0, 3, 5], dtype=np.int32)
    indices = np.array([10, 11, 12, 20, 21], dtype=np.int32)
    last_a = np.array([4, 4], dtype=np.int32)   # request 0: 12 tokens -> chunks of 8 + 4
    last_b = np.array([1, 4], dtype=np.int32)   # request 0: 9 tokens  -> chunks of 8 + 1
    ra = PL.plan_decode(indptr, indices, last_a, P, T, False, 16, 2)
    rb = PL.plan_decode(indptr, indices, last_b, P, T, False, 16, 2)
    assert ra["l1_items"] != rb["l1_items"]      # the control is meaningful
    pc = api.PlanCache(4)
    pa = pc.lookup(api.HostTable(indptr, indices, last_a, P), T, 0)
    assert not pa.hit
    _assert_plan_equals_oracle(pa, indptr, indices, last_a, P, T, 0, 16, 2)
    pb = pc.lookup(api.HostTable(indptr, indices, last_b, P), T, 0)
    assert not pb.hit
    _assert_plan_equals_oracle(pb, indptr, indices, last_b, P, T, 0, 16, 2)
    pa2 = pc.lookup(api.HostTable(indptr, indices, last_a, P), T, 0)
    assert pa2.hit
    _assert_plan_equals_oracle(pa2, indptr, indices, last_a, P, T, 0, 16, 2)


def test_env_switch_is_resolved_before_keying(api, monkeypatch):
    w = synth.tiny_cascade(seed=0, canary=False)
    t = api.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
    pc = api.PlanCache(4)
    monkeypatch.setenv("PSD_CASCADE_ATTENTION", "on")
    p_on = pc.lookup(t, w.tile_tokens, -1, 4, 2)
    assert not p_on.hit and p_on.num_members == 3
    monkeypatch.setenv("PSD_CASCADE_ATTENTION", "off")
    p_off = pc.lookup(t, w.tile_tokens, -1, 4, 2)
    assert not p_off.hit and p_off.num_members == 0
    monkeypatch.setenv("PSD_CASCADE_ATTENTION", "on")
    assert pc.lookup(t, w.tile_tokens, -1, 4, 2).hit


def test_config_shapes_hit_on_the_second_layer(api):
    for w in (synth.flat_decode(seed=0, canary=False), synth.cascade_decode(seed=0, canary=False)):
        t = api.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
        pc = api.PlanCache(2)
        first = pc.lookup(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
        second = pc.lookup(t, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
        assert not first.hit and second.hit
        _assert_plan_equals_oracle(second, w.page_indptr, w.page_indices, w.last_page_len, w.page_size,
                                   w.tile_tokens, 1, w.min_shared_pages, w.min_members)


@pytest.mark.parametrize("bad", ["decreasing_indptr", "last_page_len_zero", "batch_negative"])
def test_invalid_tables_are_rejected(api, bad):
    indptr = np.array([0, 2, 3], dtype=np.int32)
    indices = np.array([0, 1, 2], dtype=np.int32)
    last = np.array([2, 1], dtype=np.int32)
    if bad == "decreasing_indptr":
        indptr = np.array([0, 2, 1], dtype=np.int32)
    elif bad == "last_page_len_zero":
        last = np.array([0, 1], dtype=np.int32)
    t = api.HostTable(indptr, indices, last, 4)
    if bad == "batch_negative":
        t.c.batch = -1
    pc = api.PlanCache(2)
    with pytest.raises(api.L.PsdError):
        pc.lookup(t, 4, 0)
    assert pc.stats() == {"hits": 0, "misses": 0, "entries": 0}


@pytest.mark.parametrize("capacity", [0, -3, 1025])
def test_capacity_bounds(api, capacity):
    with pytest.raises(api.L.PsdError):
        api.PlanCache(capacity)


def test_generation_hits_skip_reading_the_table(api):
    """Under one generation the cache trusts the caller: the second lookup returns the
    stored plan without reading the (here deliberately changed) arrays.  A new
    generation reads them again and plans the changed table."""
    w = synth.cascade_decode(seed=1, canary=False, members=4, others=4, shared_tokens=512)
    args = (w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    t = api.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)
    pc = api.PlanCache(4)
    p1 = pc.lookup(t, *args, generation=7)
    assert not p1.hit
    first = (p1.members, p1.l1_items.tolist(), p1.o_indptr)
    last2 = w.last_page_len.copy()
    last2[0] = 1 if last2[0] != 1 else 2
    t2 = api.HostTable(w.page_indptr, w.page_indices, last2, w.page_size)
    p2 = pc.lookup(t2, *args, generation=7)
    assert p2.hit and (p2.members, p2.l1_items.tolist(), p2.o_indptr) == first
    p3 = pc.lookup(t2, *args, generation=8)
    assert not p3.hit
    _assert_plan_equals_oracle(p3, w.page_indptr, w.page_indices, last2, w.page_size, *args)
    # a different tile or threshold under the same generation is a different entry
    p4 = pc.lookup(t2, w.tile_tokens * 2, 1, w.min_shared_pages, w.min_members, generation=8)
    assert not p4.hit
    _assert_plan_equals_oracle(p4, w.page_indptr, w.page_indices, last2, w.page_size, w.tile_tokens * 2, 1,
                               w.min_shared_pages, w.min_members)
    # a generation lookup whose contents match an entry planned without one is a hit
    p5 = pc.lookup(t, *args)
    assert p5.hit
    assert pc.lookup(t, *args, generation=9).hit
