"""Error behaviour through the C ABI on the GPU: host validation rejects bad
arguments before any launch; an out-of-range page id in the device page table is
caught by the kernels' bounds checks, skipped, and reported through the workspace
fault flag (no trap)."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
import synth
from _gpu_util import Dev, ctx

pytestmark = pytest.mark.gpu


def _run_partial(d, indices_dev):
    w = d.w
    items, o_indptr = psd.split_plan(d.table, w.tile_tokens)
    N = int(o_indptr[-1])
    v = torch.empty((N, w.Hq, w.Dv), device="cuda")
    l = torch.empty((N, w.Hq), device="cuda")
    ws = torch.empty(psd.workspace_bytes(0, len(items), 0, w.Hq, w.Dv), dtype=torch.uint8, device="cuda")
    args = psd.decode_args(d.q, d.k, d.v, indices_dev, num_pages=w.num_pages, page_size=w.page_size,
                           Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale)
    psd.paged_decode_partial(ctx(), args, items, v, l, ws)
    return ws


@pytest.mark.parametrize("which", ["cuda_core", "tensor_core"])
def test_out_of_range_page_id_sets_fault_flag(which):
    w = synth.tiny_cascade(seed=0)
    d = Dev(w)
    bad = d.indices.clone()
    bad[3] = w.num_pages + 7
    if which == "cuda_core":
        ws = _run_partial(d, bad)
    else:
        plan = psd.plan_decode(d.table, w.tile_tokens, 1, 4, 2)
        assert plan.num_members == 3
        o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
        ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
        args = psd.decode_args(d.q, d.k, d.v, bad, num_pages=w.num_pages, page_size=w.page_size,
                               Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale)
        psd.cascade_decode(ctx(), args, plan, o, None, ws)
    with pytest.raises(psd.PsdError) as e:
        psd.check_device_error(ctx(), ws)
    assert e.value.status == 4
    # the flag is cleared by the check and the context stays usable
    assert psd.check_device_error(ctx(), ws) == 0
    ws2 = _run_partial(d, d.indices)
    assert psd.check_device_error(ctx(), ws2) == 0


def test_invalid_arguments_are_rejected_before_launch():
    w = synth.tiny_cascade(seed=0)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 1, 4, 2)
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    args = d.args()
    args.Hkv = 3                                    # Hq % Hkv != 0
    with pytest.raises(psd.PsdError) as e:
        psd.cascade_decode(ctx(), args, plan, o, None, ws)
    assert e.value.status == 1
    small = ws[: ws.numel() // 2]
    with pytest.raises(psd.PsdError) as e:
        psd.cascade_decode(ctx(), d.args(), plan, o, None, small)
    assert e.value.status == 5
    mis = torch.empty(ws.numel() + 16, dtype=torch.uint8, device="cuda")[4:4 + ws.numel()]
    with pytest.raises(psd.PsdError) as e:
        psd.cascade_decode(ctx(), d.args(), plan, o, None, mis)
    assert e.value.status == 1
    items = np.array([[0, int(w.page_indptr[-1]) - 1, 10 * w.page_size, 0]], dtype=np.int32)
    v = torch.empty((1, w.Hq, w.Dv), device="cuda")
    l = torch.empty((1, w.Hq), device="cuda")
    with pytest.raises(psd.PsdError) as e:                # item runs past the page table
        psd.paged_decode_partial(ctx(), d.args(), items, v, l, ws)
    assert e.value.status == 1
    torch.cuda.synchronize()


def test_unsupported_head_dim_is_reported():
    rng = np.random.default_rng(0)
    w = synth._make("d40", rng, [40, 50], Hq=2, Hkv=1, Dqk=40, Dv=40, page_size=16, num_pages=16,
                    tile_tokens=32)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 0)
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    with pytest.raises(psd.PsdError) as e:
        psd.cascade_decode(ctx(), d.args(), plan, o, None, psd.workspace_for(plan, w.Hq, w.Dv, "cuda"))
    assert e.value.status == 2


def test_counters_track_paths():
    w = synth.tiny_cascade(seed=1)
    d = Dev(w)
    before = ctx().counters()
    d.decode(enable=1)
    d.decode(enable=0)
    after = ctx().counters()
    assert after["launches_cascade"] == before["launches_cascade"] + 1
    assert after["launches_flat"] == before["launches_flat"] + 1
    assert after["cascade_member_sequences"] == before["cascade_member_sequences"] + 3


def test_fresh_workspace_garbage_is_not_a_fault():
    """A workspace whose first bytes hold garbage (all ones, as a reused allocation
    might) reads as no fault after a clean call: the fault word's epoch is not the
    call's."""
    w = synth.tiny_cascade(seed=0)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 1, 4, 2)
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    ws.fill_(255)
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    psd.cascade_decode(ctx(), d.args(), plan, o, None, ws)
    assert psd.check_device_error(ctx(), ws) == 0


PSD_FAULT_WAIT_TIMEOUT = 2


def _wide_level0_cascade():
    """16 members sharing an 8192-token prefix split into 128-token chunks: 64 chunks x
    8 KV heads of 64 stacked rows, enough 64-row blocks to fill a wave, so level 0 runs
    in the shared-tile form."""
    import dataclasses
    w = synth.cascade_decode(seed=4, members=16, others=4, shared_tokens=8192)
    return dataclasses.replace(w, tile_tokens=128)


@pytest.mark.parametrize("case", ["cuda_core_flat", "tensor_core_cascade", "tensor_core_shared_tiles",
                                  "tcgen05_level0_cascade", "tcgen05_level0_wide"])
def test_bounded_wait_runs_out_and_is_reported(case):
    """A wait that nothing completes gives up after its limit: the partial kernels are
    told to withhold the loads of every tile from index 1 on, so the waits for those
    tiles run out (about 1 ms limit), every warp stops, the call completes, and
    psd_check_device_error reports PSD_FAULT_WAIT_TIMEOUT.  The next decode on the
    same context is clean and matches the oracle.  The tcgen05 level-0 cases give up
    with a level-0 tile's stage landed and its S MMAs complete, and free their tensor
    memory after the issued MMAs have drained."""
    from oracle import attention as A
    from _gpu_util import assert_close, use_kernel, use_level0
    wide = case in ("tensor_core_shared_tiles", "tcgen05_level0_wide")
    w = _wide_level0_cascade() if wide else synth.tiny_cascade(seed=2)
    d = Dev(w)
    enable = 0 if case == "cuda_core_flat" else 1
    kind = "cuda_core" if case == "cuda_core_flat" else "auto"
    level0 = "tcgen05" if case.startswith("tcgen05") else "mma_sync"
    with use_kernel(kind), use_level0(level0):
        plan = psd.plan_decode(d.table, w.tile_tokens, enable, w.min_shared_pages, w.min_members)
        assert (plan.num_members > 0) == bool(enable)
        o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
        lse = torch.empty((w.batch, w.Hq), device="cuda")
        ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
        ctx().test_withhold_loads(1, 2_000_000)
        try:
            psd.cascade_decode(ctx(), d.args(), plan, o, lse, ws)
            with pytest.raises(psd.PsdError) as e:
                psd.check_device_error(ctx(), ws)
        finally:
            ctx().test_withhold_loads(-1)
        assert e.value.status == 4 and e.value.fault_bits == PSD_FAULT_WAIT_TIMEOUT
        psd.cascade_decode(ctx(), d.args(), plan, o, lse, ws)
        assert psd.check_device_error(ctx(), ws) == 0
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), ro, rl, "bf16", case)


def test_withhold_loads_rejects_a_limit_outside_its_range():
    for bad in (10, 5_000_000_000):
        with pytest.raises(psd.PsdError):
            ctx().test_withhold_loads(1, bad)
    ctx().test_withhold_loads(-1)


@pytest.mark.parametrize("case,from_tile", [("long_items", 1), ("query_switches", 0)])
def test_mla_bounded_wait_runs_out_and_is_reported(case, from_tile):
    """The same aid on the tcgen05 MLA partial.  long_items: four requests in
    2048-token items, every item's tiles from index 1 on withheld, so the CTAs give up
    with a tile's S and softmax done and its PV never issued.  query_switches: 300
    requests of 1 to 130 tokens in 64-token items with no tile loaded, so the
    producer gives up at its first query switch while the control warp waits for a
    tile.  Each CTA waits for the copies it issued and for its issued MMAs before
    freeing its tensor memory; the call reports PSD_FAULT_WAIT_TIMEOUT, and the next
    decode on the same context is clean and matches the oracle."""
    from oracle import attention as A
    from _gpu_util import assert_close
    if case == "long_items":
        w = synth.mla_decode(seed=1, batch=4, lo=4096, hi=9000, num_pages=1024)
    else:
        rng = np.random.default_rng(7)
        lengths = [int(x) for x in rng.integers(1, 131, size=300)]
        w = synth._make("mla_small", rng, lengths, Hq=128, Hkv=1, Dqk=576, Dv=512, page_size=64,
                        num_pages=1024, tile_tokens=64, kv_dtype="fp8_e4m3", latent_v=True)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 0, w.min_shared_pages, w.min_members)
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    lse = torch.empty((w.batch, w.Hq), device="cuda")
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    ctx().test_withhold_loads(from_tile, 2_000_000)
    try:
        psd.cascade_decode(ctx(), d.args(), plan, o, lse, ws)
        with pytest.raises(psd.PsdError) as e:
            psd.check_device_error(ctx(), ws)
    finally:
        ctx().test_withhold_loads(-1)
    assert e.value.status == 4 and e.value.fault_bits == PSD_FAULT_WAIT_TIMEOUT
    psd.cascade_decode(ctx(), d.args(), plan, o, lse, ws)
    assert psd.check_device_error(ctx(), ws) == 0
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), ro, rl, "fp8_e4m3", f"MLA after {case}")
