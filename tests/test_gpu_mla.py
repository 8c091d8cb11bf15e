"""MLA-shaped decode (128 query heads over one 576-wide fp8-e4m3 latent, V = its
first 512 columns) on the tensor-core partial kernel, against the float64 oracle
(ROCm ATOM PR #1701 section 3.2 for the fp8 latent; mlxcel PR #1004 Merge contract
for the split-KV merge)."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
import synth
from oracle import attention as A
from _gpu_util import Dev, assert_close, ctx, oracle_partials

pytestmark = pytest.mark.gpu


def test_mla_reduced_batch_every_output():
    w = synth.mla_decode(seed=1, batch=4, lo=4096, hi=9000, num_pages=1024)
    o, lse = Dev(w).decode(enable=1)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "fp8_e4m3", "MLA reduced")


def test_mla_partials_chunk_by_chunk():
    w = synth.mla_decode(seed=2, batch=2, lo=2000, hi=5000, num_pages=256)
    v, l, _, o_indptr = Dev(w).partials()
    rv, rl, ro = oracle_partials(w)
    assert o_indptr.tolist() == ro
    assert_close(v, l, rv, rl, "fp8_e4m3", "MLA partials")


def test_mla_bf16_latent():
    rng = np.random.default_rng(3)
    w = synth._make("mla_bf16", rng, [700, 2100], Hq=128, Hkv=1, Dqk=576, Dv=512, page_size=64,
                    num_pages=64, tile_tokens=512, latent_v=True)
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "bf16", "MLA bf16 latent")


@pytest.mark.slow
def test_mla_full_size_sampled_requests():
    """Full MLA config (128 requests, 4K-32K tokens, 65536-page pool) in the launch
    configuration the bench times; six seeded requests checked against the oracle."""
    w = synth.mla_decode(seed=0)
    o, lse = Dev(w).decode(enable=1)
    rng = np.random.default_rng(9)
    req = sorted(set(rng.choice(w.batch, size=5, replace=False).tolist()) |
                 {int(np.argmax(w.lengths))})
    ro, rl = A.decode_attention(A.workload_arrays(w), requests=req)
    assert_close(o[req], lse[req], ro[req], rl[req], "fp8_e4m3", "MLA full")
    assert np.isfinite(o).all()


def _mla_small(seed, lengths, page_size=64, num_pages=512, tile=2048):
    rng = np.random.default_rng(seed)
    return synth._make("mla_small", rng, lengths, Hq=128, Hkv=1, Dqk=576, Dv=512, page_size=page_size,
                       num_pages=num_pages, tile_tokens=tile, kv_dtype="fp8_e4m3", latent_v=True)


def test_mla_takes_device_query_only():
    """The MLA kernel loads q by TMA: pinned host q is refused with
    PSD_ERR_UNSUPPORTED before any launch, and the same call with device q and host
    page ids runs and matches the oracle."""
    w = _mla_small(12, [300, 2500])
    d = Dev(w)
    plan = psd.plan_decode(d.table, w.tile_tokens, 0, w.min_shared_pages, w.min_members)
    ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
    o = torch.empty((w.batch, w.Hq, w.Dv), device="cuda")
    lse = torch.empty((w.batch, w.Hq), device="cuda")
    ih = d.indices.cpu().pin_memory()
    mk = lambda q: psd.decode_args(q, d.k, d.v, ih, num_pages=w.num_pages, page_size=w.page_size,
                                   Hkv=w.Hkv, Dv=w.Dv, sm_scale=w.sm_scale, k_scale=w.k_scale,
                                   v_scale=w.v_scale)
    with pytest.raises(psd.PsdError) as e:
        psd.cascade_decode(ctx(), mk(w.q.contiguous().pin_memory()), plan, o, lse, ws)
    assert e.value.status == 2 and "device memory" in str(e.value)
    psd.cascade_decode(ctx(), mk(d.q), plan, o, lse, ws)
    torch.cuda.synchronize()
    assert psd.check_device_error(ctx(), ws) == 0
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), ro, rl, "fp8_e4m3",
                 "MLA, host page ids")


@pytest.mark.parametrize("page_size", [64, 128])
def test_mla_ragged_tails_and_short_items(page_size):
    """Items of 1 to 2049 tokens: single-token and one-short tiles, whole pages, an
    item that ends one token into a tile; NaN canaries fill every unused slot."""
    w = _mla_small(4, [1, 63, 64, 65, 127, 128, 700, 2049], page_size=page_size)
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "fp8_e4m3", f"MLA ragged, page {page_size}")


def test_mla_query_rows_far_outside_the_f16_range():
    """A query row is split into two e4m3 terms after scaling by a power of two, so
    any finite bf16 magnitude works: q * 2^40 with sm_scale * 2^-40 and q * 2^-60 with
    sm_scale * 2^60 give the same scores and the same outputs as q itself."""
    w = _mla_small(5, [900, 1500, 64])
    d = Dev(w)
    o0, l0 = d.decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o0, l0, ro, rl, "fp8_e4m3", "MLA q")
    base_scale = w.sm_scale
    for e in (40, -60):
        d.q = (w.q.float() * 2.0 ** e).to(torch.bfloat16).to("cuda")
        w.sm_scale = base_scale * 2.0 ** -e
        o, l = d.decode(enable=0)
        assert np.abs(o - o0).max() <= 1e-6 and np.abs(l - l0).max() <= 1e-6, f"2^{e}"
    w.sm_scale = base_scale


def test_mla_heads_of_different_magnitude():
    """Head h scaled by 2^((h % 9) - 4): rows from flat to sharp softmax in one CTA."""
    w = _mla_small(6, [3000, 777])
    scale = torch.tensor([2.0 ** ((h % 9) - 4) for h in range(128)], dtype=torch.float32)
    w.q = (w.q.float() * scale[None, :, None]).to(torch.bfloat16)
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "fp8_e4m3", "MLA mixed head magnitudes")


def test_mla_many_short_requests_switch_queries_inside_a_cta():
    """300 requests of 1 to 130 tokens, 64-token items: every CTA pair of the
    persistent launch walks several requests (a query split per switch) and many
    ragged last tiles."""
    rng = np.random.default_rng(7)
    lengths = [int(x) for x in rng.integers(1, 131, size=300)]
    w = _mla_small(7, lengths, num_pages=1024, tile=64)
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "fp8_e4m3", "MLA many short requests")


def test_mla_many_items_per_request_keep_the_query():
    """Three long requests in 256-token items: a CTA pair runs consecutive items of
    one request on the query it split once; partials checked chunk by chunk."""
    w = _mla_small(8, [20000, 18001, 9999], num_pages=1024, tile=256)
    v, l, _, o_indptr = Dev(w).partials()
    rv, rl, ro = oracle_partials(w)
    assert o_indptr.tolist() == ro
    assert_close(v, l, rv, rl, "fp8_e4m3", "MLA partials, many items per request")


def test_mla_decode_accumulates_runs_of_items():
    """Decode through the merge: a CTA pair adds consecutive items of one request into
    one partial and marks the others empty, and the runs of the persistent launch end
    mid-request.  Against the oracle, and beside merge_states over the per-item
    partials of the same work list."""
    w = _mla_small(9, [20000, 18001, 9999, 64, 1, 130, 4097, 2047], num_pages=1024, tile=256)
    d = Dev(w)
    o, lse = d.decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "fp8_e4m3", "MLA runs of items")
    v, l, _, o_indptr = d.partials()
    vo = torch.empty((w.batch, w.Hq, w.Dv), dtype=torch.float32, device="cuda")
    lo_ = torch.empty((w.batch, w.Hq), dtype=torch.float32, device="cuda")
    psd.merge_states(ctx(), torch.from_numpy(v).float().cuda(), torch.from_numpy(l).float().cuda(),
                     torch.from_numpy(np.asarray(o_indptr, dtype=np.int32)).cuda(), vo, lo_)
    # Both within the fp8 bounds of the oracle.  They are not bit-equal: a run carries
    # one running max across items, so P's two e4m3 terms round differently.
    assert_close(vo.cpu().double().numpy(), lo_.cpu().double().numpy(), ro, rl, "fp8_e4m3",
                 "MLA per-item partials merged")
    assert np.abs(vo.cpu().double().numpy() - o).max() < 2e-3


def test_mla_cascade_level1_runs():
    """A shared whole-page prefix: level 0 (stacked rows) on the 64-row kernel, level 1
    on the persistent kernel with runs of items accumulated, one merge over both."""
    rng = np.random.default_rng(10)
    lengths = [4096 + 1500, 4096 + 3000, 4096 + 70, 6000, 2500]
    w = synth._make("mla_cascade", rng, lengths, Hq=128, Hkv=1, Dqk=576, Dv=512, page_size=64,
                    num_pages=1024, tile_tokens=512, kv_dtype="fp8_e4m3", latent_v=True,
                    shared=([0, 1, 2], 4096 // 64), min_shared_pages=16, min_members=2)
    o, lse, stats, _ = Dev(w).decode(enable=1, with_stats=True)
    assert stats["path"] == 1 and stats["members"] == 3
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "fp8_e4m3", "MLA cascade")
