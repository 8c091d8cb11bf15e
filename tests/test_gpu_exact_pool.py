"""The pages' own tolerance for an exact pool (mlxcel PR #1004, Correctness
coverage: cascade against a host f64 reference and against the flat launch, 2e-5
when the pool is exact f32).  A bf16 pool, bf16 queries and the f32 arithmetic of
the kernels make an exact pool in that sense: every input value is represented
without rounding, so what separates the kernels from the float64 oracle is their own
f32 arithmetic (and P entering the tensor-core MMAs as two bf16 terms, about 16
significant bits).  Both few-row partial kernels, both level-0 kernels, flat and
cascade, against the oracle and against each other at 2e-5, output and LSE."""
import numpy as np
import pytest

import synth
from oracle import attention as A
from _gpu_util import Dev, use_kernel, use_level0

pytestmark = pytest.mark.gpu

EXACT_TOL = 2e-5


def _small_cascade(seed):
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(1, 900, size=10)]
    mem = [0, 3, 4, 7, 8, 9]
    for m in mem:
        lengths[m] = 24 * 16 + int(rng.integers(1, 300))
    return synth._make(f"exact_{seed}", rng, lengths, Hq=32, Hkv=8, Dqk=128, Dv=128, page_size=16,
                       num_pages=sum((n + 15) // 16 for n in lengths) + 8, tile_tokens=128,
                       shared=(mem, 24), min_shared_pages=1, min_members=2)


def _check(o, lse, ro, rl, what):
    do, dl = np.abs(o - ro).max(), np.abs(lse - rl).max()
    assert do <= EXACT_TOL and dl <= EXACT_TOL, f"{what}: max|o - oracle| {do:.3g}, max|lse - oracle| {dl:.3g}"


def test_tiny_cascade_at_the_exact_pool_tolerance():
    w = synth.tiny_cascade(seed=3)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    d = Dev(w)
    for level0 in ("mma_sync", "tcgen05"):
        with use_level0(level0):
            o, lse, stats, _ = d.decode(enable=1, with_stats=True)
        assert stats["path"] == 1
        _check(o, lse, ro, rl, f"tiny cascade, level 0 {level0}")
    _check(*d.decode(enable=0), ro, rl, "tiny workload, flat")


@pytest.mark.parametrize("seed", [0, 1])
def test_cascade_and_flat_at_the_exact_pool_tolerance(seed):
    w = _small_cascade(seed)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    d = Dev(w)
    outs = {}
    for kernel in ("auto", "cuda_core"):
        with use_kernel(kernel):
            outs[("flat", kernel)] = d.decode(enable=0)
            for level0 in ("mma_sync", "tcgen05"):
                with use_level0(level0):
                    o, lse, stats, _ = d.decode(enable=1, with_stats=True)
                assert stats["path"] == 1 and stats["members"] == 6
                outs[("cascade " + level0, kernel)] = (o, lse)
    for key, (o, lse) in outs.items():
        _check(o, lse, ro, rl, f"{key}")
    # cascade against the flat launch, as the pages compare them
    fo, fl = outs[("flat", "auto")]
    for key, (o, lse) in outs.items():
        _check(o, lse, fo, fl, f"{key} against the flat launch")


@pytest.mark.parametrize("maker", [synth.flat_decode, synth.cascade_decode], ids=["flat", "cascade"])
def test_full_size_batches_at_the_exact_pool_tolerance(maker):
    """The bench's flat batch (contexts up to 4096 tokens) and its cascade batch
    (8192-token shared prefix), every output, in the launch configuration the bench
    times."""
    w = maker(seed=0)
    ro, rl = A.decode_attention(A.workload_arrays(w))
    o, lse = Dev(w).decode(enable=1)
    _check(o, lse, ro, rl, w.name)
