"""Split-KV partials, flat decode and the two-level cascade on the GPU against the
float64 oracle (mlxcel PR #1004: Decomposition, Merge contract, Task item 2,
Correctness coverage)."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
import synth
from oracle import attention as A
from oracle import cascade as OC
from oracle import planner as PL
from _gpu_util import Dev, assert_close, ctx, oracle_partials, use_kernel, use_level0

pytestmark = pytest.mark.gpu

KERNELS = ["auto", "cuda_core"]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("maker,seed", [(synth.tiny_cascade, 0), (synth.tiny_cascade, 1),
                                        (synth.flat_decode, 0)])
def test_partials_match_oracle_chunk_by_chunk(maker, seed, kernel):
    w = maker(seed=seed)
    with use_kernel(kernel):
        v, l, items, o_indptr = Dev(w).partials()
    rv, rl, ro = oracle_partials(w)
    assert o_indptr.tolist() == ro
    assert_close(v, l, rv, rl, w.kv_dtype, "partials")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_flat_decode_full_size(seed, kernel):
    """Flat config at full size (32 requests, 16384-page pool, tile 512), every output."""
    w = synth.flat_decode(seed=seed)
    d = Dev(w)
    with use_kernel(kernel):
        o, lse, stats, plan = d.decode(enable=1, with_stats=True)
    assert stats["path"] == 0 and stats["decline_reason"] == PL.DECLINE_NO_SHARED_PAGES
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, "flat")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_cascade_matches_oracle(seed):
    w = synth.tiny_cascade(seed=seed)
    d = Dev(w)
    o, lse, stats, plan = d.decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == 3 and stats["shared_pages"] == 4
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, "tiny cascade")
    fo, fl = d.decode(enable=0)
    assert np.abs(o - fo).max() < 1e-3 and np.abs(lse - fl).max() < 1e-4


def test_tiny_cascade_declines_at_default_thresholds():
    w = synth.tiny_cascade(seed=0)
    o, lse, stats, _ = Dev(w).decode(enable=1, min_shared_pages=16, min_members=2, with_stats=True)
    assert stats["path"] == 0 and stats["decline_reason"] == PL.DECLINE_SPAN_BELOW_THRESHOLD
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, "declined")


@pytest.mark.parametrize("level0", ["mma_sync", "tcgen05"])
@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("seed", [0, 1])
def test_cascade_config_full_size(seed, kernel, level0):
    """Cascade config at full size: 64 requests, 16 members share 8192 tokens; the
    cascade arm, the flat arm and the oracle agree, with level 0 (64 stacked rows per
    KV head) in either kernel."""
    w = synth.cascade_decode(seed=seed)
    d = Dev(w)
    with use_kernel(kernel), use_level0(level0):
        o, lse, stats, plan = d.decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == 16 and stats["shared_pages"] == 512
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, "cascade")
    fo, fl = d.decode(enable=0)
    assert_close(fo, fl, ro, rl, w.kv_dtype, "flat arm")
    assert np.abs(o - fo).max() < 2e-3


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("members", [2, 4])
def test_cascade_with_small_group_uses_stacked_small_kernels(kernel, members):
    """2 members x G=4 = 8 stacked rows per KV head (either small-group kernel's
    stacked mode) and 4 x 4 = 16 rows (small-group tensor-core kernel)."""
    w = synth.cascade_decode(seed=3, members=members, others=3, shared_tokens=512)
    with use_kernel(kernel):
        o, lse, stats, _ = Dev(w).decode(enable=1, with_stats=True)
    assert stats["members"] == members
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype, f"{members}-member cascade")


def test_cascade_level_partials_match_oracle_levels():
    """The composite partial rows of a cascade equal the oracle's level-0 (unstacked)
    and level-1 rows."""
    w = synth.cascade_decode(seed=4, members=4, others=4, shared_tokens=1024)
    a = A.workload_arrays(w)
    plan = PL.plan_decode(w.page_indptr, w.page_indices, w.last_page_len, w.page_size,
                          w.tile_tokens, True, 16, 2)
    o, lse, vref, lref = OC.cascade_levels(a, plan, w.tile_tokens)
    fo, fl = A.decode_attention(a)
    assert np.abs(o - fo).max() < 1e-11
    go, gl = Dev(w).decode(enable=1)
    assert_close(go, gl, fo, fl, w.kv_dtype, "4-member cascade")


def _stacked_level0(w, member_major):
    members = [0, 1, 2]
    M, G = len(members), w.Hq // w.Hkv
    d = Dev(w)
    qm = d.q[members]                                            # [M, Hq, D]
    if member_major:
        q0 = qm.reshape(1, M * w.Hq, w.Dqk).contiguous()
    else:
        q0 = qm.reshape(M, w.Hkv, G, w.Dqk).permute(1, 0, 2, 3).reshape(1, M * w.Hq, w.Dqk).contiguous()
    span = 4
    items = np.array([[0, int(w.page_indptr[0]), span * w.page_size, 0]], dtype=np.int32)
    v = torch.empty((1, M * w.Hq, w.Dv), device="cuda")
    l = torch.empty((1, M * w.Hq), device="cuda")
    ws = torch.empty(psd.workspace_bytes(0, 1, 0, M * w.Hq, w.Dv), dtype=torch.uint8, device="cuda")
    psd.paged_decode_partial(ctx(), d.args(q=q0), items, v, l, ws)
    return v.cpu().double().numpy(), l.cpu().double().numpy()


def test_kv_head_major_stacking_matches_and_member_major_reads_wrong_kv_head():
    """Negative control named on the page: member-major stacking through the kernel's
    h / (M*G) mapping reads the wrong KV head."""
    w = synth.tiny_cascade(seed=2)
    a = A.workload_arrays(w)
    rv, rl = OC.level0_partials(a, [0, 1, 2], 4, 4 * w.page_size)
    gv, gl = _stacked_level0(w, member_major=False)
    assert_close(gv, gl, rv, rl, "bf16", "kv-major level 0")
    bv, bl = _stacked_level0(w, member_major=True)
    assert np.abs(bv - rv).max() > 0.1


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("D,Hq,Hkv", [(256, 8, 1), (64, 6, 3), (128, 2, 2), (128, 16, 1)])
def test_other_head_dims_and_group_sizes(D, Hq, Hkv, kernel):
    rng = np.random.default_rng(D + Hq)
    lengths = synth.lengths_with_partial_last_page(rng, 5, 20, 700, 16)
    w = synth._make("shape", rng, lengths, Hq=Hq, Hkv=Hkv, Dqk=D, Dv=D, page_size=16,
                    num_pages=400, tile_tokens=64)
    with use_kernel(kernel):
        o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", f"D={D} G={Hq // Hkv}")


def test_fp8_pool_with_separate_k_and_v():
    rng = np.random.default_rng(21)
    lengths = synth.lengths_with_partial_last_page(rng, 6, 30, 900, 16)
    w = synth._make("fp8gqa", rng, lengths, Hq=8, Hkv=2, Dqk=128, Dv=128, page_size=16,
                    num_pages=512, tile_tokens=128, kv_dtype="fp8_e4m3")
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "fp8_e4m3", "fp8 GQA")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("P", [64, 8])
def test_page_sizes_and_single_token_requests(kernel, P):
    rng = np.random.default_rng(22)
    lengths = [1, 2, 63, 64, 65, 300]
    w = synth._make("edge", rng, lengths, Hq=8, Hkv=2, Dqk=128, Dv=128, page_size=P,
                    num_pages=512 // P * 8, tile_tokens=128)
    with use_kernel(kernel):
        o, lse = Dev(w).decode(enable=0)
        v, l, items, o_indptr = Dev(w).partials()
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", f"page {P}")
    rv, rl2, _ = oracle_partials(w)
    assert_close(v, l, rv, rl2, "bf16", "page 64 partials")


def test_outputs_ignore_nan_canaries():
    """Unused pool pages and slots past last_page_len are NaN; any stray read would
    surface as NaN in the outputs."""
    w = synth.flat_decode(seed=5, batch=8)
    assert torch.isnan(w.k_pool.float()).any()
    o, lse = Dev(w).decode(enable=0)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("tile,inline", [(2048, True), (256, True), (128, False)])
def test_work_lists_inline_or_uploaded(tile, inline):
    """80 requests of 512-4096 tokens: at tiles of 2048 and 256 the work lists (about
    4 KB and 15 KB) travel in the launches' parameters, at 128 (about 29 KB) by one
    upload into the workspace; outputs match the oracle either way."""
    rng = np.random.default_rng(12)
    lengths = synth.lengths_with_partial_last_page(rng, 80, 512, 4096, 16)
    w = synth._make("flat80", rng, lengths, Hq=32, Hkv=8, Dqk=128, Dv=128, page_size=16,
                    num_pages=16384, tile_tokens=tile)
    before = ctx().counters()
    o, lse = Dev(w).decode(enable=0)
    after = ctx().counters()
    assert after["lists_inline"] - before["lists_inline"] == int(inline)
    assert after["lists_uploaded"] - before["lists_uploaded"] == int(not inline)
    req = [0, 17, 45, 79]
    ro, rl = A.decode_attention(A.workload_arrays(w), requests=req)
    assert_close(o[req], lse[req], ro[req], rl[req], "bf16", f"flat, tile {tile}")


def test_fault_word_reports_only_the_latest_call():
    """A call whose page table holds an out-of-range id flags the workspace's fault
    word; after a later clean call on the same workspace the check reports nothing
    (the word carries the epoch of the call that wrote it, and no call clears it), and
    a fault of the latest call is reported again."""
    w = synth.tiny_cascade(seed=0)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 1, 4, 2)
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    bad = d.indices.clone()
    bad[5] = w.num_pages + 3
    before = ctx().counters()["lists_inline"]
    psd.cascade_decode(ctx(), d.args(), plan, o, None, ws)          # clean
    args_bad = psd.decode_args(d.q, d.k, d.v, bad, num_pages=w.num_pages, page_size=w.page_size,
                               Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale)
    psd.cascade_decode(ctx(), args_bad, plan, o, None, ws)          # flags
    psd.cascade_decode(ctx(), d.args(), plan, o, None, ws)          # clean again
    assert ctx().counters()["lists_inline"] - before == 3
    assert psd.check_device_error(ctx(), ws) == 0
    psd.cascade_decode(ctx(), args_bad, plan, o, None, ws)
    with pytest.raises(psd.PsdError):
        psd.check_device_error(ctx(), ws)


@pytest.mark.slow
def test_cascade_prefix_beyond_l2_sampled():
    """The cascade batch with a 65536-token shared prefix (268 MB of K/V, more than
    L2) that the bench times beside the configured batch: cascade and flat outputs of
    sampled members and non-members against the oracle, and against each other."""
    w = synth.cascade_decode(seed=0, shared_tokens=65536)
    d = Dev(w)
    o, lse, stats, _ = d.decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == 16 and stats["shared_pages"] == 4096
    of, lf = d.decode(enable=0)
    members = [int(b) for b in np.where(w.lengths > 65536)[0]]
    others = [int(b) for b in np.where(w.lengths <= 65536)[0]]
    req = sorted({members[0], members[-1], others[0], others[-1]})
    ro, rl = A.decode_attention(A.workload_arrays(w), requests=req)
    assert_close(o[req], lse[req], ro[req], rl[req], "bf16", "cascade, prefix beyond L2")
    assert_close(of[req], lf[req], ro[req], rl[req], "bf16", "flat, prefix beyond L2")
    assert np.abs(o - of).max() < 2e-3 and np.abs(lse - lf).max() < 1e-3


def test_empty_batch_is_a_no_op():
    """A decode step with no requests: planning gives an empty flat plan, and
    cascade_decode, paged_decode_partial and merge_states return without device work
    (q and the outputs are empty tensors)."""
    w = synth.tiny_cascade(seed=0)
    d = Dev(w)
    empty = np.zeros(0, dtype=np.int32)
    t = psd.HostTable(np.zeros(1, dtype=np.int32), empty, empty, w.page_size)
    plan = psd.plan_decode(t, w.tile_tokens, 1, 4, 2)
    assert plan.num_members == 0 and plan.num_rows == 0
    q0 = torch.empty((0, w.Hq, w.Dqk), dtype=torch.bfloat16, device="cuda")
    args = psd.decode_args(q0, d.k, d.v, d.indices, num_pages=w.num_pages, page_size=w.page_size,
                           Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale)
    o = torch.empty((0, w.Hq, w.Dv), device="cuda")
    lse = torch.empty((0, w.Hq), device="cuda")
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    stats = psd.cascade_decode(ctx(), args, plan, o, lse, ws)
    assert stats["path"] == 0 and stats["batch"] == 0
    assert psd.check_device_error(ctx(), ws) == 0
    items, o_indptr = psd.split_plan(t, w.tile_tokens)
    assert len(items) == 0 and list(o_indptr) == [0]
    psd.paged_decode_partial(ctx(), args, items, o, lse, ws)
    psd.merge_states(ctx(), torch.empty((0, w.Hq, w.Dv), device="cuda"), torch.empty((0, w.Hq), device="cuda"),
                     torch.zeros(1, dtype=torch.int32, device="cuda"), o, lse)
    torch.cuda.synchronize()


def test_one_long_request_merges_hundreds_of_chunks():
    """One 131072-token request split into 256 chunks of 512: one merge group of 256
    rows (eight 32-row LSE windows), plus a one-token request beside it."""
    rng = np.random.default_rng(23)
    w = synth._make("long", rng, [131072, 1], Hq=8, Hkv=2, Dqk=128, Dv=128, page_size=16,
                    num_pages=8200, tile_tokens=512)
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", "long request")


def test_largest_stacked_group_per_kv_head():
    """256 query rows on one KV head (the most the 16-row-group kernel takes), D=128."""
    rng = np.random.default_rng(24)
    lengths = synth.lengths_with_partial_last_page(rng, 3, 100, 1500, 16)
    w = synth._make("g256", rng, lengths, Hq=256, Hkv=1, Dqk=128, Dv=128, page_size=16,
                    num_pages=512, tile_tokens=256)
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", "G=256")


@pytest.mark.parametrize("maker", [synth.tiny_cascade, synth.flat_decode])
def test_outputs_into_pinned_host_memory(maker):
    """cascade_decode with o and lse in pinned host memory: the merge kernel stores
    them over the host link; after a stream sync they equal the device outputs bit
    for bit."""
    w = maker(seed=3)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    lse = torch.empty((w.batch, w.Hq), device="cuda")
    psd.cascade_decode(ctx(), d.args(), plan, o, lse, ws)
    oh = torch.full((w.batch, w.Hq, w.Dv), float("nan")).pin_memory()
    lh = torch.full((w.batch, w.Hq), float("nan")).pin_memory()
    psd.cascade_decode(ctx(), d.args(), plan, oh, lh, ws)
    torch.cuda.synchronize()
    assert psd.check_device_error(ctx(), ws) == 0
    assert torch.equal(oh, o.cpu()) and torch.equal(lh, lse.cpu())


@pytest.mark.parametrize("kernel,level0", [(k, "auto") for k in KERNELS] + [("auto", "tcgen05")])
@pytest.mark.parametrize("maker", [synth.tiny_cascade, synth.flat_decode, synth.cascade_decode])
def test_inputs_from_pinned_host_memory(maker, kernel, level0):
    """cascade_decode with q and page_indices in pinned host memory (read by the
    partial kernels over the host link, the tcgen05 level-0 kernel included) and the
    outputs in pinned host memory: equal bit for bit to the all-device call, on flat
    and cascade plans."""
    w = maker(seed=5)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    lse = torch.empty((w.batch, w.Hq), device="cuda")
    qh = w.q.contiguous().pin_memory()
    ih = d.indices.cpu().pin_memory()
    args_h = psd.decode_args(qh, d.k, d.v, ih, num_pages=w.num_pages, page_size=w.page_size,
                             Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale, k_scale=w.k_scale,
                             v_scale=w.v_scale)
    oh = torch.full((w.batch, w.Hq, w.Dv), float("nan")).pin_memory()
    lh = torch.full((w.batch, w.Hq), float("nan")).pin_memory()
    with use_kernel(kernel), use_level0(level0):
        psd.cascade_decode(ctx(), d.args(), plan, o, lse, ws)
        psd.cascade_decode(ctx(), args_h, plan, oh, lh, ws)
    torch.cuda.synchronize()
    assert psd.check_device_error(ctx(), ws) == 0
    assert (plan.num_members > 0) == (maker is not synth.flat_decode)
    assert torch.equal(oh, o.cpu()) and torch.equal(lh, lse.cpu())


@pytest.mark.parametrize("G,D", [(20, 128), (24, 64), (40, 128), (64, 128), (80, 64), (132, 128)])
def test_large_query_groups_share_each_tile(G, D):
    """More than 16 query rows per KV head.  Up to 48 rows (20, 24, 40 here) take a
    CTA per 16-row group; more rows (64, 80, 132) take blocks of 64 rows whose warps
    own a group each and read every tile from one shared ring, with a partly filled
    last warp and blocks with idle warps.  Ragged lengths with single-token and tail
    tiles, NaN canaries in every unused slot, against the oracle."""
    rng = np.random.default_rng(G + D)
    lengths = [1, 15, 16, 17, 300, 515, 1024, 1300]
    w = synth._make(f"gqa{G}", rng, lengths, Hq=2 * G, Hkv=2, Dqk=D, Dv=D, page_size=16,
                    num_pages=sum((n + 15) // 16 for n in lengths) + 8, tile_tokens=256)
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", f"G={G}, D={D}")


@pytest.mark.parametrize("level0", ["mma_sync", "tcgen05"])
@pytest.mark.parametrize("members", [5, 9, 17, 33])
def test_cascade_stacked_rows_in_shared_tile_blocks(members, level0):
    """Level-0 stacks members x G rows per KV head (20, 36, 68, 132 here).  mma_sync:
    CTAs per 16-row group below 49 rows, blocks of 64 rows with partly filled and idle
    warps above, through the fused launch.  tcgen05: one CTA per 128 rows (two row
    blocks at 132, the second with 4 live rows).  Against the oracle and the flat
    arm."""
    rng = np.random.default_rng(70 + members)
    B = members + 3
    P, sp = 16, 40
    lengths = [int(x) for x in rng.integers(1, 900, size=B)]
    mem = sorted(int(m) for m in rng.choice(B, size=members, replace=False))
    for m in mem:
        lengths[m] = sp * P + int(rng.integers(1, 200))
    w = synth._make(f"casc{members}", rng, lengths, Hq=8, Hkv=2, Dqk=128, Dv=128, page_size=P,
                    num_pages=sum((n + P - 1) // P for n in lengths) + 8, tile_tokens=128,
                    shared=(mem, sp), min_shared_pages=1, min_members=2)
    d = Dev(w)
    with use_level0(level0):
        o, lse, stats, plan = d.decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == members
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", f"cascade, {members} members, level 0 {level0}")
    fo, fl = d.decode(enable=0)
    assert np.abs(o - fo).max() < 2e-3


def _wave():
    """Resident CTAs of the tensor-core partial kernel per wave (three per SM)."""
    return 3 * torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("G", [64, 80])
def test_large_groups_in_shared_tile_blocks(G):
    """64-row blocks take the shared-tile form once they fill a wave of resident
    CTAs.  This batch has enough work items for 1.25 waves of blocks (80 rows: a
    full block and one with a single live warp per item).  Ragged lengths, NaN
    canaries in every unused slot, every output against the oracle."""
    rng = np.random.default_rng(300 + G)
    Hkv, D, P, tile = 8, 128, 16, 64
    need = -(-_wave() * 5 // 4 // (Hkv * ((G + 63) // 64)))
    lengths = []
    while sum(-(-n // tile) for n in lengths) < need:
        lengths.append(int(rng.integers(1, 700)))
    lengths[0] = 1
    w = synth._make(f"gqa{G}_blocks", rng, lengths, Hq=Hkv * G, Hkv=Hkv, Dqk=D, Dv=D, page_size=P,
                    num_pages=sum((n + P - 1) // P for n in lengths) + 8, tile_tokens=tile)
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", f"G={G}, shared-tile blocks")


def test_cascade_level0_in_shared_tile_blocks():
    """16 members x 4 rows = 64 stacked rows per KV head, with enough prefix chunks
    (tile 64) for 1.25 waves of level-0 blocks, so the fused launch takes the
    shared-tile form for level 0 (the mma_sync level-0 kernel): every output against
    the oracle and the flat arm."""
    rng = np.random.default_rng(77)
    Hkv, P, tile, members = 8, 16, 64, 16
    chunks = -(-_wave() * 5 // 4 // Hkv)
    sp = chunks * tile // P
    B = members + 4
    lengths = [int(x) for x in rng.integers(1, 900, size=B)]
    mem = sorted(int(m) for m in rng.choice(B, size=members, replace=False))
    for m in mem:
        lengths[m] = sp * P + int(rng.integers(1, 300))
    w = synth._make("casc_blocks", rng, lengths, Hq=4 * Hkv, Hkv=Hkv, Dqk=128, Dv=128, page_size=P,
                    num_pages=sum((n + P - 1) // P for n in lengths) + 8, tile_tokens=tile,
                    shared=(mem, sp), min_shared_pages=1, min_members=2)
    d = Dev(w)
    with use_level0("mma_sync"):
        o, lse, stats, plan = d.decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == members and stats["prefix_chunks"] >= chunks
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", "cascade, level-0 blocks")
    fo, fl = d.decode(enable=0)
    assert np.abs(o - fo).max() < 2e-3


def test_pageable_host_query_is_rejected_by_the_binding():
    w = synth.tiny_cascade(seed=0)
    d = Dev(w)
    with pytest.raises(ValueError):
        psd.decode_args(w.q.contiguous(), d.k, d.v, d.indices, num_pages=w.num_pages,
                        page_size=w.page_size, Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale)


@pytest.mark.slow
def test_flat_decode_128_requests_sampled():
    """The flat workload with 128 requests (the bench's large-batch arm, 1.2 GB of
    K/V): sampled requests against the oracle, every output finite."""
    w = synth.flat_decode(seed=0, batch=128, num_pages=65536)
    o, lse = Dev(w).decode(enable=0)
    req = [0, 37, 90, 127, int(np.argmax(w.lengths))]
    ro, rl = A.decode_attention(A.workload_arrays(w), requests=req)
    assert_close(o[req], lse[req], ro[req], rl[req], "bf16", "flat, 128 requests")
    assert np.isfinite(o).all() and np.isfinite(lse).all()
