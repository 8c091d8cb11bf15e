"""cascade_decode_no_alloc through the C ABI: the entry point for callers that may
not allocate device memory (it keeps its scratch in the library's fixed 16 MiB
device array instead of a caller workspace).  Its results must equal those of
cascade_decode with a workspace, call after call on the shared array.

This file is collected last on purpose, so a run that stops at the first failure
has already run every other test."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
import synth
from _gpu_util import LSE_TOL, OUT_TOL, Dev, ctx

pytestmark = pytest.mark.gpu


def _with_workspace(d, plan):
    w = d.w
    o = torch.empty((w.batch, w.Hq, w.Dv), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.batch, w.Hq), dtype=torch.float32, device="cuda")
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    psd.cascade_decode(ctx(), d.args(), plan, o, lse, ws)
    assert psd.check_device_error(ctx(), ws) == 0
    return o.cpu().double().numpy(), lse.cpu().double().numpy()


def _no_alloc(d, plan):
    w = d.w
    o = torch.full((w.batch, w.Hq, w.Dv), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((w.batch, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    fault = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    stats = psd.cascade_decode_no_alloc(ctx(), d.args(), plan, o, lse, fault)
    torch.cuda.synchronize()
    assert int(fault.item()) == 0
    return o.cpu().double().numpy(), lse.cpu().double().numpy(), stats


@pytest.mark.parametrize("maker,enable", [(synth.tiny_cascade, 1), (synth.cascade_decode, 1),
                                          (synth.flat_decode, 0)])
def test_no_alloc_matches_workspace_entry_point_twice(maker, enable):
    w = maker(seed=0)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, enable, w.min_shared_pages, w.min_members)
    ro, rl = _with_workspace(d, plan)
    for _ in range(2):  # the second call runs on the array the first call left behind
        o, lse, stats = _no_alloc(d, plan)
        assert np.abs(o - ro).max() <= OUT_TOL[w.kv_dtype]
        assert np.abs(lse - rl).max() <= LSE_TOL
        assert stats["path"] == (1 if plan.num_members else 0)


def test_no_alloc_rejects_plans_beyond_its_scratch():
    w = synth.flat_decode(seed=1)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.page_size, 0)          # one chunk per page: ~70 MB of rows
    o = torch.empty((w.batch, w.Hq, w.Dv), dtype=torch.float32, device="cuda")
    with pytest.raises(psd.PsdError) as e:
        psd.cascade_decode_no_alloc(ctx(), d.args(), plan, o)
    assert e.value.status == 5 and "static scratch holds 16777216 bytes" in str(e.value)


def test_no_alloc_smaller_plan_after_larger_plan_against_oracle():
    """A large cascade plan and then the tiny one on the same array: stale partial rows
    or LSE values the first call left behind must not reach the second call's
    outputs.  Both are checked against the float64 oracle."""
    from oracle import attention as A
    from _gpu_util import assert_close
    for w in (synth.cascade_decode(seed=1), synth.tiny_cascade(seed=1)):
        d = Dev(w)
        plan = psd.plan_decode(d.table, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
        assert plan.num_members > 0
        o, lse, _ = _no_alloc(d, plan)
        ro, rl = A.decode_attention(A.workload_arrays(w))
        assert_close(o, lse, ro, rl, w.kv_dtype, f"no_alloc {w.name}")


def _small_fp8(latent):
    rng = np.random.default_rng(77 + int(latent))
    if latent:
        lengths = [int(x) for x in rng.integers(1, 4000, size=3)]
        return synth._make("mla_small", rng, lengths, Hq=128, Hkv=1, Dqk=576, Dv=512, page_size=64,
                           num_pages=sum((L + 63) // 64 for L in lengths) + 2, tile_tokens=2048,
                           kv_dtype="fp8_e4m3", latent_v=True)
    lengths = [int(x) for x in rng.integers(1, 1500, size=6)]
    for m in (0, 1, 4):
        lengths[m] = max(lengths[m], 4 * 16 + 5)
    return synth._make("fp8_small", rng, lengths, Hq=16, Hkv=2, Dqk=128, Dv=128, page_size=16,
                       num_pages=sum((L + 15) // 16 for L in lengths) + 2, tile_tokens=128,
                       kv_dtype="fp8_e4m3", shared=([0, 1, 4], 4), min_shared_pages=1, min_members=2)


@pytest.mark.parametrize("latent", [False, True], ids=["fp8_separate_kv_cascade", "fp8_mla_latent"])
def test_no_alloc_fp8_and_mla_plans(latent):
    """fp8 pools: separate K and V with a shared prefix (the 64-row kernel for both
    levels, lists copied into the array), and the MLA latent (the tcgen05 kernel with
    runs of items and the merge that skips empty rows).  Against the oracle, and
    equal within tolerance to cascade_decode with a workspace, twice in a row."""
    from oracle import attention as A
    from _gpu_util import assert_close
    w = _small_fp8(latent)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    assert (plan.num_members > 0) == (not latent)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    wo, wl = _with_workspace(d, plan)
    for _ in range(2):
        o, lse, _ = _no_alloc(d, plan)
        assert_close(o, lse, ro, rl, "fp8_e4m3", f"no_alloc {w.name}")
        assert np.abs(o - wo).max() <= OUT_TOL["fp8_e4m3"] and np.abs(lse - wl).max() <= LSE_TOL


def test_no_alloc_tcgen05_level0_runs_of_chunks():
    """Level 0 on the tcgen05 kernel with more tasks than SMs (160 chunks x 2 KV heads
    over one CTA per SM): runs of chunks accumulate into one partial and leave the
    run's other rows empty (LSE -inf), which the merge must skip.  In the shared
    array, twice, against the oracle and against cascade_decode with a workspace."""
    from oracle import attention as A
    from _gpu_util import assert_close, use_level0
    rng = np.random.default_rng(7)
    lengths = [int(x) for x in rng.integers(1, 700, size=11)]
    mem = sorted(int(m) for m in rng.choice(11, size=8, replace=False))
    for m in mem:
        lengths[m] = 640 * 16 + int(rng.integers(1, 48))
    w = synth._make("no_alloc_l0_runs", rng, lengths, Hq=8, Hkv=2, Dqk=128, Dv=128, page_size=16,
                    num_pages=sum((n + 15) // 16 for n in lengths) + 8, tile_tokens=64,
                    shared=(mem, 640), min_shared_pages=1, min_members=2)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    assert plan.num_members == 8
    ro, rl = A.decode_attention(A.workload_arrays(w))
    with use_level0("tcgen05"):
        wo, wl = _with_workspace(d, plan)
        for _ in range(2):
            o, lse, stats = _no_alloc(d, plan)
            assert stats["path"] == 1 and stats["prefix_chunks"] == 160
            assert_close(o, lse, ro, rl, "bf16", "no_alloc, tcgen05 level 0 with runs")
            assert np.abs(o - wo).max() <= OUT_TOL["bf16"] and np.abs(lse - wl).max() <= LSE_TOL
