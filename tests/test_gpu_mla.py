"""MLA-shaped decode (128 query heads over one 576-wide fp8-e4m3 latent, V = its
first 512 columns) on the tensor-core partial kernel, against the float64 oracle
(ROCm ATOM PR #1701 section 3.2 for the fp8 latent; mlxcel PR #1004 Merge contract
for the split-KV merge)."""
import math

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


# ---------------------------------------------------------------------------------
# Precision of the two-term e4m3 query split inside a row.  The kernel scales each
# query row by a power of two (its largest element to [128, 256)) and splits it into
# hi = e4m3(x) and lo = e4m3(x - hi): exact down to about 2^-10 of the row's largest
# element; below that each element carries an absolute error of up to about 2^-17 of
# it (e4m3's subnormal step), so a score's absolute error grows with the row's
# largest element.  These rows spread their magnitudes over 2^20.
#   * Scores with a spread of a few log2 units (every token weighs in): the bf16
#     level of accuracy, 2e-3 on outputs and 1e-3 on LSE.
#   * The default scale 1/sqrt(576) on these rows gives scores of several hundred
#     log2 units, a softmax that is nearly one-hot: the score errors (about 1e-5 of
#     the scores) move near-tied weights, and outputs stay within the 1e-2 bound of an
#     fp8 pool (measured up to 7.8e-3), and the LSE within the bound the split gives:
#     a score's error is at most sm_scale * log2(e) * 576 * 2^-17 * max|q_row| *
#     max|K| (measured 1.3e-2 with scores up to about 1500).
BF16_LEVEL_OUT = 2e-3


def _wide_range_rows(w, seed, kind):
    rng = np.random.default_rng(seed)
    B, H, D = w.q.shape
    if kind == "log_uniform":          # |q| log-uniform over [2^-10, 2^10], random signs
        q = 2.0 ** rng.uniform(-10, 10, size=(B, H, D)) * rng.choice([-1.0, 1.0], size=(B, H, D))
    elif kind == "spike":              # N(0,1) * 2^-10 with one element per row at +-2^10
        q = rng.standard_normal((B, H, D)) * 2.0 ** -10
        col = rng.integers(0, D, size=(B, H))
        np.put_along_axis(q, col[..., None], rng.choice([-1.0, 1.0], size=(B, H, 1)) * 2.0 ** 10, axis=2)
    elif kind == "rope_heavy":         # the 64 rope columns 2^8 larger than the 512 latent ones
        q = rng.standard_normal((B, H, D)) * 2.0 ** -6
        q[..., 512:] *= 2.0 ** 14
    else:
        raise ValueError(kind)
    return torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("kind", ["log_uniform", "spike", "rope_heavy"])
@pytest.mark.parametrize("scores", ["normalised", "default"])
def test_mla_query_rows_spanning_2_to_the_20(kind, scores):
    """Rows whose elements span 2^20 in magnitude, with the softmax scale either set so
    the log2 scores have a spread of about 2 (every token matters: the bf16 level of
    accuracy) or left at 1/sqrt(576) (a nearly one-hot softmax over scores of several
    hundred: the fp8-pool output bound, the LSE relative to its magnitude)."""
    import dataclasses
    w = _mla_small(31 + len(kind), [1100, 2049, 300, 64])
    q = _wide_range_rows(w, 40 + len(kind), kind)
    w = dataclasses.replace(w, q=q)
    if scores == "normalised":
        a = A.workload_arrays(w)
        K, _ = A.gather_kv(a, 0)
        s = A.bf16_bits_to_f64(a["q_raw"])[0] @ K[:, 0, :].T          # raw scores of request 0
        w = dataclasses.replace(w, sm_scale=float(2.0 / math.log2(math.e) / s.std()))
    o, lse = Dev(w).decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    eo = np.abs(o - ro).max()
    el = np.abs(lse - rl).max()
    print(f"{kind} {scores}: out {eo:.3g} lse {el:.3g} (|lse| up to {np.abs(rl).max():.4g})")
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    if scores == "normalised":
        assert eo <= BF16_LEVEL_OUT and el <= 1e-3, (kind, scores, eo, el)
    else:
        assert eo <= 1e-2, (kind, scores, eo)
        a = A.workload_arrays(w)
        qmax = np.abs(A.bf16_bits_to_f64(a["q_raw"])).max(axis=2)                 # [B, Hq]
        kmax = np.array([np.abs(A.gather_kv(a, b)[0]).max() for b in range(w.batch)])
        bound = w.sm_scale * math.log2(math.e) * 576 * 2.0 ** -17 * qmax * kmax[:, None]
        assert (np.abs(lse - rl) <= np.maximum(1e-3, bound)).all(), (kind, scores, el)
