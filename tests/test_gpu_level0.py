"""The stacked level-0 rows of the cascade on the tcgen05 kernel (persistent, one CTA
per SM over (level-0 chunk, KV head, block of 128 stacked rows) tasks; mlxcel PR
#1004, Decomposition: the M members' G query heads of a KV head stacked KV-head
major).  Edge cases of its 64-token tiles against the float64 oracle: spans that end
inside a tile (page positions past the chunk's pages load as zeros), page sizes from
16 to 128, head dims 64 and 128, a page id out of range, lists uploaded or in the
launch parameters, runs of chunks accumulated into one partial, and the same results
as the 16-row-group kernel."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
import synth
from oracle import attention as A
from _gpu_util import Dev, assert_close, ctx, use_level0

pytestmark = pytest.mark.gpu


def _cascade(seed, P, span_pages, tile, D, G, members, Hkv=2, others=3):
    rng = np.random.default_rng(seed)
    B = members + others
    lengths = [int(x) for x in rng.integers(1, 700, size=B)]
    mem = sorted(int(m) for m in rng.choice(B, size=members, replace=False))
    for m in mem:
        lengths[m] = span_pages * P + int(rng.integers(1, 3 * P))
    return synth._make(f"l0_{P}_{span_pages}_{D}_{G}_{members}", rng, lengths, Hq=G * Hkv, Hkv=Hkv, Dqk=D, Dv=D,
                       page_size=P, num_pages=sum((n + P - 1) // P for n in lengths) + 8, tile_tokens=tile,
                       shared=(mem, span_pages), min_shared_pages=1, min_members=2)


CASES = [
    # P, span pages, tile, D, G, members: stacked rows = G * members
    (16, 5, 128, 128, 4, 8),     # 80-token span: a 64-token tile, then 16 tokens and three zero-filled boxes
    (32, 3, 64, 128, 4, 8),      # chunks of 64 and 32 tokens; the second tile half zero-filled
    (64, 3, 128, 64, 8, 5),      # D = 64, 40 rows, a 192-token span in chunks of 128 and 64
    (128, 2, 256, 128, 2, 20),   # P = 128: a 64-token tile is half a page
    (16, 33, 512, 128, 4, 40),   # 160 rows: two row blocks, the second with 32 live rows
]


@pytest.mark.parametrize("case", CASES, ids=[f"P{c[0]}_span{c[1]}_tile{c[2]}_D{c[3]}_rows{c[4] * c[5]}"
                                              for c in CASES])
def test_level0_tcgen05_against_oracle(case):
    P, sp, tile, D, G, members = case
    w = _cascade(500 + P + sp, P, sp, tile, D, G, members)
    d = Dev(w)
    with use_level0("tcgen05"):
        o, lse, stats, _ = d.decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == members and stats["shared_pages"] == sp
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", f"level 0 tcgen05 {case}")
    with use_level0("mma_sync"):
        mo, ml = d.decode(enable=1)
    assert np.abs(o - mo).max() < 2e-3 and np.abs(lse - ml).max() < 1e-3


def test_level0_tcgen05_on_the_tiny_cascade():
    """The tiny cascade (3 members x G = 4: 12 stacked rows, D = 64) forced onto the
    tcgen05 kernel: 116 of its 128 TMEM lanes are padding rows."""
    w = synth.tiny_cascade(seed=5)
    with use_level0("tcgen05"):
        o, lse, stats, _ = Dev(w).decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == 3
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", "tiny cascade, level 0 tcgen05")


def test_level0_tcgen05_flags_an_out_of_range_page_id():
    """A shared-span page id past the pool: the kernel loads the zero fill in its place
    and flags PSD_FAULT_PAGE_ID; the next clean call on the context is correct."""
    w = _cascade(71, 16, 6, 128, 128, 4, 8)
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 1, w.min_shared_pages, w.min_members)
    m0 = int(plan.members[0])
    bad = d.indices.clone()
    bad[int(w.page_indptr[m0]) + 2] = w.num_pages + 11         # inside the shared span
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    lse = torch.empty((w.batch, w.Hq), device="cuda")
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    args_bad = psd.decode_args(d.q, d.k, d.v, bad, num_pages=w.num_pages, page_size=w.page_size,
                               Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale)
    with use_level0("tcgen05"):
        psd.cascade_decode(ctx(), args_bad, plan, o, lse, ws)
        with pytest.raises(psd.PsdError) as e:
            psd.check_device_error(ctx(), ws)
        assert e.value.fault_bits == 1
        psd.cascade_decode(ctx(), d.args(), plan, o, lse, ws)
        assert psd.check_device_error(ctx(), ws) == 0
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), ro, rl, "bf16", "after the fault")


@pytest.mark.parametrize("tile,inline", [(512, True), (128, False)])
def test_level0_tcgen05_lists_inline_or_uploaded(tile, inline):
    """The cascade batch at tile 512 (lists in the launch parameters of both partial
    kernels) and tile 128 (about 34 KB of lists, uploaded): sampled members and
    non-members against the oracle."""
    import dataclasses
    w = dataclasses.replace(synth.cascade_decode(seed=2), tile_tokens=tile)
    before = ctx().counters()
    with use_level0("tcgen05"):
        o, lse, stats, _ = Dev(w).decode(enable=1, with_stats=True)
    after = ctx().counters()
    assert stats["path"] == 1 and stats["members"] == 16
    assert after["lists_inline"] - before["lists_inline"] == int(inline)
    assert after["lists_uploaded"] - before["lists_uploaded"] == int(not inline)
    members = [int(b) for b in np.where(w.lengths > 8192)[0]]
    others = [int(b) for b in np.where(w.lengths <= 8192)[0]]
    req = sorted({members[0], members[7], members[-1], others[0], others[-1]})
    ro, rl = A.decode_attention(A.workload_arrays(w), requests=req)
    assert_close(o[req], lse[req], ro[req], rl[req], "bf16", f"cascade, tile {tile}")


def test_level0_tcgen05_runs_of_chunks():
    """400 level-0 tasks (100 chunks x 2 KV heads x 2 row blocks of 160 stacked rows)
    over one CTA per SM: each CTA takes a contiguous range of about 2.6 tasks, whose
    chunks of one KV head and row block accumulate into one partial (a run) and leave
    the run's other chunk rows empty; runs end where the KV head or the row block
    changes inside a CTA's range.  Against the oracle and the mma.sync form."""
    w = _cascade(91, 16, 400, 64, 128, 4, 40)
    d = Dev(w)
    with use_level0("tcgen05"):
        o, lse, stats, _ = d.decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == 40 and stats["prefix_chunks"] == 100
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", "level 0 tcgen05 runs")
    with use_level0("mma_sync"):
        mo, ml = d.decode(enable=1)
    assert np.abs(o - mo).max() < 2e-3 and np.abs(lse - ml).max() < 1e-3
