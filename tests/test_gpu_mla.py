"""MLA-shaped decode (128 query heads over one 576-wide fp8-e4m3 latent, V = its
first 512 columns) on the tensor-core partial kernel, against the float64 oracle
(ROCm ATOM PR #1701 section 3.2 for the fp8 latent; mlxcel PR #1004 Merge contract
for the split-KV merge)."""
import numpy as np
import pytest

import synth
from oracle import attention as A
from _gpu_util import Dev, assert_close, oracle_partials

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
