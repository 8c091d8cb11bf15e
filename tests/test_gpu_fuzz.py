"""Seeded random configurations of the decode path on the GPU against the float64
oracle: batch, head counts, head dims, page size, tile, pool dtype, ragged lengths
and optional shared prefixes (mlxcel PR #1004, Decomposition, Merge contract and
Detection sections; ROCm ATOM PR #1701 section 3.2 for the fp8 pool).  Every case
goes through psd_plan_decode and cascade_decode, flat or cascade as the planner
decides."""
import numpy as np
import pytest

import synth
from oracle import attention as A
from _gpu_util import Dev, assert_close

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    D = int(rng.choice([64, 128, 256]))
    P = int(rng.choice([16, 32, 64]))
    tile = P * int(rng.choice([1, 2, 4, 8]))
    kv_dtype = "fp8_e4m3" if rng.random() < 0.3 else "bf16"
    B = int(rng.integers(1, 13))
    lengths = [int(x) for x in rng.integers(1, 1500, size=B)]
    shared = None
    if B >= 3 and rng.random() < 0.5:
        members = sorted(int(m) for m in rng.choice(B, size=int(rng.integers(2, B + 1)), replace=False))
        sp = int(rng.integers(1, 6))
        for m in members:                       # a member needs a page after the shared span
            lengths[m] = max(lengths[m], sp * P + int(rng.integers(1, 3 * P)))
        shared = (members, sp)
    pages = sum((L + P - 1) // P for L in lengths) + 8
    w = synth._make(f"fuzz{seed}", rng, lengths, Hq=Hkv * G, Hkv=Hkv, Dqk=D, Dv=D, page_size=P,
                    num_pages=pages, tile_tokens=tile, kv_dtype=kv_dtype, shared=shared,
                    min_shared_pages=1, min_members=2)
    return w


@pytest.mark.parametrize("seed", list(range(48)))
def test_random_decode_configurations(seed):
    w = _case(seed)
    o, lse, stats, plan = Dev(w).decode(enable=1, with_stats=True)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, w.kv_dtype,
                 f"seed {seed}: B={w.batch} Hkv={w.Hkv} G={w.Hq // w.Hkv} D={w.Dqk} P={w.page_size} "
                 f"tile={w.tile_tokens} {w.kv_dtype} path={stats['path']}")


def _mla_case(seed):
    rng = np.random.default_rng(2000 + seed)
    P = int(rng.choice([64, 128]))
    tile = int(rng.choice([64, 128, 256, 512, 2048]))
    tile = max(tile, P)
    B = int(rng.integers(1, 13))
    lengths = [int(x) for x in rng.integers(1, 6000, size=B)]
    pages = sum((L + P - 1) // P for L in lengths) + 4
    return synth._make(f"mla_fuzz{seed}", rng, lengths, Hq=128, Hkv=1, Dqk=576, Dv=512, page_size=P,
                       num_pages=pages, tile_tokens=tile, kv_dtype="fp8_e4m3", latent_v=True)


@pytest.mark.parametrize("seed", list(range(12)))
def test_random_mla_configurations(seed):
    """MLA decode over random batches, lengths, tiles and page sizes: the persistent
    kernel's runs are planned on the host and split inside items at tile boundaries
    (rows feed the merge), so both the merged outputs and the per-chunk partials are
    checked against the oracle."""
    from _gpu_util import oracle_partials
    w = _mla_case(seed)
    d = Dev(w)
    o, lse = d.decode(enable=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    assert_close(o, lse, ro, rl, "fp8_e4m3",
                 f"MLA seed {seed}: B={w.batch} P={w.page_size} tile={w.tile_tokens}")
    if w.batch <= 4:
        v, l, _, o_indptr = d.partials()
        rv, rlp, rind = oracle_partials(w)
        assert o_indptr.tolist() == rind
        assert_close(v, l, rv, rlp, "fp8_e4m3", f"MLA partials seed {seed}")


def _distinct_scales_case(seed, latent, shared):
    import dataclasses
    rng = np.random.default_rng(3000 + seed)
    if latent:
        Hq, Hkv, Dqk, Dv, P, tile = 128, 1, 576, 512, 64, 256
        lengths = [int(x) for x in rng.integers(1, 3000, size=5)]
    else:
        Hq, Hkv, Dqk, Dv, P, tile = 16, 2, 128, 128, 16, 64
        lengths = [int(x) for x in rng.integers(1, 1500, size=6)]
    sh = None
    if shared:
        members, sp = [0, 2, 3], 3
        for m in members:
            lengths[m] = max(lengths[m], sp * P + int(rng.integers(1, 2 * P)))
        sh = (members, sp)
    pages = sum((L + P - 1) // P for L in lengths) + 4
    w = synth._make(f"scales{seed}", rng, lengths, Hq=Hq, Hkv=Hkv, Dqk=Dqk, Dv=Dv, page_size=P,
                    num_pages=pages, tile_tokens=tile, kv_dtype="fp8_e4m3", latent_v=latent, shared=sh,
                    min_shared_pages=1, min_members=2)
    # the same codes with K's and V's scales far apart (V dequantises with v_scale only)
    return dataclasses.replace(w, k_scale=w.k_scale * 0.5, v_scale=w.k_scale * 4.0)


@pytest.mark.parametrize("latent", [False, True], ids=["separate_kv", "latent"])
@pytest.mark.parametrize("shared", [False, True], ids=["flat", "cascade"])
def test_fp8_distinct_k_and_v_scales(latent, shared):
    """fp8 pools whose K and V scales differ by 8x (ROCm ATOM PR #1701, 3.2: each
    tensor dequantises with its own scale), flat and cascade, against the oracle.  The
    oracle with V dequantised by K's scale misses by far more than the tolerance, so
    a kernel that swapped the scales would fail here."""
    w = _distinct_scales_case(int(latent) * 2 + int(shared), latent, shared)
    a = A.workload_arrays(w)
    ro, rl = A.decode_attention(a)
    slip, _ = A.decode_attention(dict(a, v_scale=a["k_scale"]))
    assert np.abs(slip - ro).max() > 0.1
    o, lse, stats, _ = Dev(w).decode(enable=1, with_stats=True)
    assert stats["path"] == int(shared)
    assert_close(o, lse, ro, rl, "fp8_e4m3", f"distinct scales latent={latent} shared={shared}")
