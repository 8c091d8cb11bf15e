"""Chunk-size autotuning per shape bucket (mlxcel PR #1004, Left out / unsure: the
shape-bucketed autotuner with cold-L2 methodology is not wired to the cascade
geometries): the tuner times every candidate, keeps the fastest for the batch's
bucket, answers it back for that bucket only, and decoding with it stays exact."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
from oracle import attention as A
import synth
from _gpu_util import Dev, assert_close, ctx

pytestmark = pytest.mark.gpu


def _buffers(w, d, smallest_tile):
    items, o_indptr = psd.split_plan(d.table, smallest_tile)
    rows = int(o_indptr[-1])
    ws = torch.empty(psd.workspace_bytes(w.batch, max(len(items), 1), rows, w.Hq, w.Dv), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty((w.batch, w.Hq, w.Dv), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.batch, w.Hq), dtype=torch.float32, device="cuda")
    return o, lse, ws


def test_tuner_picks_the_fastest_and_answers_its_bucket():
    w = synth.flat_decode(seed=0, canary=False)
    d = Dev(w)
    tiles = [256, 512, 1024]
    o, lse, ws = _buffers(w, d, min(tiles))
    c = psd.Context(0)
    assert c.tuned_tile(d.args(), d.table, 512, 1, w.min_shared_pages, w.min_members) == 512
    best, ms = c.autotune_tile(d.args(), d.table, tiles, o, lse, ws, 1, w.min_shared_pages, w.min_members, reps=3)
    assert best in tiles and len(ms) == 3 and all(m > 0 for m in ms)
    assert best == tiles[int(np.argmin(ms))]
    assert c.tuned_tile(d.args(), d.table, 512, 1, w.min_shared_pages, w.min_members) == best
    # another bucket (8 requests) keeps the default
    w8 = synth.flat_decode(seed=1, canary=False, batch=8)
    d8 = Dev(w8)
    assert c.tuned_tile(d8.args(), d8.table, 512, 1, w8.min_shared_pages, w8.min_members) == 512
    # decoding with the tuned tile is still the attention result
    plan = psd.plan_decode(d.table, best, 1, w.min_shared_pages, w.min_members)
    psd.cascade_decode(c, d.args(), plan, o, lse, ws)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), ro, rl, w.kv_dtype, "tuned tile")


def test_tiles_must_be_page_multiples():
    w = synth.flat_decode(seed=2, canary=False, batch=4)
    d = Dev(w)
    o, lse, ws = _buffers(w, d, 16)
    with pytest.raises(psd.PsdError):
        ctx().autotune_tile(d.args(), d.table, [24], o, lse, ws, reps=1)
