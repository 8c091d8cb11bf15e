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
