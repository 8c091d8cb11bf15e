"""Nested / several-subgroup cascade decode on the GPU against the float64 oracle's
dense attention (the decomposition is exact up to rounding: mlxcel PR #1004,
Decomposition and Merge contract), plus agreement with the two-level decode where
the plans coincide."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
from oracle import attention as A
import synth
from _gpu_util import Dev, assert_close, ctx, use_kernel, use_level0

pytestmark = pytest.mark.gpu


def _nested_small(seed):
    """10 requests: a 4-page system prompt for 8 of them, two tenants of 4 with a
    3-page and a 2-page sub-prefix, private suffixes; 2 strangers."""
    rng = np.random.default_rng(seed)
    P = 16
    mem = list(range(8))
    lengths = [4 * P + (3 if b < 4 else 2) * P + int(rng.integers(1, 70)) for b in mem] + \
              [int(x) for x in rng.integers(20, 300, size=2)]
    prefixes = [(mem, 4), (mem[:4], 3), (mem[4:], 2)]
    return synth._make("nested_small", rng, lengths, Hq=8, Hkv=2, Dqk=64, Dv=64, page_size=P, num_pages=400,
                       tile_tokens=32, prefixes=prefixes, min_shared_pages=2, min_members=2)


def _decode_nested(w, levels, msp, mm):
    d = Dev(w)
    plan = psd.plan_nested(d.table, w.tile_tokens, 1, msp, mm, levels)
    o = torch.empty((w.batch, w.Hq, w.Dv), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.batch, w.Hq), dtype=torch.float32, device="cuda")
    ws = psd.nested_workspace_for(plan, w.Hq, w.Dv, "cuda")
    stats = psd.cascade_decode_nested(ctx(), d.args(), plan, o, lse, ws)
    assert psd.check_device_error(ctx(), ws) == 0
    return o.cpu().double().numpy(), lse.cpu().double().numpy(), stats, plan


@pytest.mark.parametrize("level0", ["auto", "tcgen05"])
@pytest.mark.parametrize("kernel", ["auto", "cuda_core"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_small_nested_matches_dense_attention(seed, kernel, level0):
    """level0 'tcgen05': every segment's stacked rows on the tcgen05 kernel, one
    launch per segment on the side stream, runs of chunks leaving empty rows."""
    w = _nested_small(seed)
    with use_kernel(kernel), use_level0(level0):
        o, lse, stats, plan = _decode_nested(w, 3, 2, 2)
    assert plan.num_segments == 3 and [s[1] for s in plan.segments] == [8, 4, 4]
    assert stats["path"] == 1 and stats["members"] == 16 and stats["shared_pages"] == 4 + 3 + 2
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, f"nested seed {seed}")


@pytest.mark.parametrize("seed", [0, 1])
def test_nested_batch_full_size(seed):
    w = synth.nested_decode(seed)
    o, lse, stats, plan = _decode_nested(w, 2, 16, 2)
    assert stats["members"] == 32 and stats["shared_pages"] == 512
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, "nested batch")


def test_one_level_agrees_with_two_level_decode():
    w = synth.cascade_decode(seed=2, members=4, others=4, shared_tokens=1024)
    o1, l1, stats, plan = _decode_nested(w, 1, 16, 2)
    assert plan.num_segments == 1
    o2, l2 = Dev(w).decode(enable=1)
    assert np.abs(o1 - o2).max() < 1e-5 and np.abs(l1 - l2).max() < 1e-5


def test_no_segment_is_the_flat_decode():
    w = synth.flat_decode(seed=3, batch=8)
    o, lse, stats, plan = _decode_nested(w, 2, 16, 2)
    assert plan.num_segments == 0 and stats["path"] == 0
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, "flat through the nested entry")


def test_more_segments_than_one_launch_holds():
    """A system prompt for 18 requests and nine two-request tenants with their own
    sub-prefix: ten segments, more than one fused launch carries, so every
    segment's level 0 runs on the side stream (its work lists in the launch
    parameters) before the level-1 launch and the merge."""
    rng = np.random.default_rng(31)
    P = 16
    mem = list(range(18))
    lengths = [4 * P + 2 * P + int(rng.integers(1, 60)) for _ in mem] + [int(x) for x in rng.integers(20, 200, size=3)]
    prefixes = [(mem, 4)] + [([2 * k, 2 * k + 1], 2) for k in range(9)]
    w = synth._make("nested_wide", rng, lengths, Hq=8, Hkv=2, Dqk=64, Dv=64, page_size=P, num_pages=600,
                    tile_tokens=32, prefixes=prefixes, min_shared_pages=2, min_members=2)
    before = ctx().counters()["lists_inline"]
    o, lse, stats, plan = _decode_nested(w, 2, 2, 2)
    assert plan.num_segments == 10 and stats["path"] == 1
    assert ctx().counters()["lists_inline"] - before == 1
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, "ten segments")
    with use_level0("tcgen05"):   # ten tcgen05 level-0 launches, lists still inline
        o, lse, stats, plan = _decode_nested(w, 2, 2, 2)
    assert_close(o, lse, ro, rl, w.kv_dtype, "ten segments, level 0 on tcgen05")
