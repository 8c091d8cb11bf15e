"""merge_states (K3) on the GPU against the float64 oracle merge (mlxcel PR #1004,
Merge contract section)."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
import synth
from oracle import attention as A
from _gpu_util import ctx

pytestmark = pytest.mark.gpu

TOL_O, TOL_L = 2e-5, 2e-5  # f32 arithmetic on f32 inputs


def _gpu_merge(v_in, lse_in, o_indptr, lse_out=True):
    M = len(o_indptr) - 1
    H, D = v_in.shape[1], v_in.shape[2]
    dv = v_in.cuda() if not v_in.is_cuda else v_in
    dl = lse_in.cuda() if not lse_in.is_cuda else lse_in
    ind = torch.from_numpy(np.asarray(o_indptr, dtype=np.int32)).cuda()
    vo = torch.full((M, H, D), float("nan"), device="cuda")
    lo = torch.full((M, H), float("nan"), device="cuda") if lse_out else None
    psd.merge_states(ctx(), dv, dl, ind, vo, lo)
    torch.cuda.synchronize()
    return vo, lo


@pytest.mark.parametrize("num_out,seed", [(1, 0), (1000, 1), (16384, 2)])
def test_merge_parity_full_check(num_out, seed):
    v_in, lse_in, o_indptr = synth.merge_inputs(seed, num_out)
    ro, rl = A.merge_states(v_in.numpy(), lse_in.numpy(), o_indptr)
    vo, lo = _gpu_merge(v_in, lse_in, o_indptr)
    assert np.abs(vo.cpu().double().numpy() - ro).max() < TOL_O
    assert np.abs(lo.cpu().double().numpy() - rl).max() < TOL_L


@pytest.mark.parametrize("H,D", [(128, 512), (8, 64), (4, 1024), (3, 12)])
def test_merge_parity_other_shapes(H, D):
    rng = np.random.default_rng(H + D)
    o_indptr = synth.merge_groups(rng, 300, 1, 40)
    N = int(o_indptr[-1])
    v_in = torch.from_numpy(rng.standard_normal((N, H, D), dtype=np.float32))
    lse_in = torch.from_numpy(rng.uniform(-5, 20, size=(N, H)).astype(np.float32))
    ro, rl = A.merge_states(v_in.numpy(), lse_in.numpy(), o_indptr)
    vo, lo = _gpu_merge(v_in, lse_in, o_indptr)
    assert np.abs(vo.cpu().double().numpy() - ro).max() < TOL_O
    assert np.abs(lo.cpu().double().numpy() - rl).max() < TOL_L


def test_group_of_one_is_bit_exact_identity():
    v_in, lse_in, _ = synth.merge_inputs(3, 64)
    N = v_in.shape[0]
    vo, lo = _gpu_merge(v_in, lse_in, np.arange(N + 1))
    assert torch.equal(vo.cpu(), v_in) and torch.equal(lo.cpu(), lse_in)


def test_merge_is_associative_across_regroupings():
    rng = np.random.default_rng(4)
    v_in = torch.from_numpy(rng.standard_normal((9, 32, 128), dtype=np.float32))
    lse_in = torch.from_numpy(rng.uniform(-5, 20, size=(9, 32)).astype(np.float32))
    direct, dl = _gpu_merge(v_in, lse_in, [0, 9])
    sub, sl = _gpu_merge(v_in, lse_in, [0, 2, 5, 9])
    two, tl = _gpu_merge(sub, sl, [0, 3])
    assert (two - direct).abs().max().item() < 1e-5 and (tl - dl).abs().max().item() < 1e-5


def test_natural_log_lse_fails_parity():
    """Negative control: LSEs in natural-log units fed to the log2 merge."""
    v_in, lse_in, o_indptr = synth.merge_inputs(5, 500)
    ro, _ = A.merge_states(v_in.numpy(), lse_in.numpy(), o_indptr)
    vo, _ = _gpu_merge(v_in, lse_in * float(np.log(2.0)), o_indptr)
    assert np.abs(vo.cpu().double().numpy() - ro).max() > 1e-2


def test_empty_and_neg_inf_groups():
    v_in = torch.ones((3, 2, 8))
    lse_in = torch.tensor([[0.0, 1.0], [-float("inf"), -float("inf")], [-float("inf"), 2.0]])
    vo, lo = _gpu_merge(v_in, lse_in, [0, 0, 1, 2, 3])
    assert torch.equal(vo[0].cpu(), torch.zeros(2, 8)) and torch.all(lo[0].cpu() == -float("inf"))
    assert torch.equal(vo[1].cpu(), v_in[0]) and torch.equal(lo[1].cpu(), lse_in[0])
    assert torch.equal(vo[2].cpu(), torch.zeros(2, 8))           # one row, lse -inf
    assert torch.equal(vo[3, 1].cpu(), v_in[2, 1]) and torch.equal(vo[3, 0].cpu(), torch.zeros(8))


def test_empty_partials_in_groups_are_ignored():
    """Rows with LSE -inf inside larger groups (v NaN) contribute nothing, against the
    oracle (which ignores them too), over groups of 1 to 40 rows."""
    rng = np.random.default_rng(11)
    o_indptr = synth.merge_groups(rng, 400, 1, 40)
    N = int(o_indptr[-1])
    v_in = torch.from_numpy(rng.standard_normal((N, 8, 64), dtype=np.float32))
    lse_in = torch.from_numpy(rng.uniform(-5, 20, size=(N, 8)).astype(np.float32))
    empty = torch.from_numpy(rng.random((N, 8)) < 0.4)
    for r in range(len(o_indptr) - 1):      # keep one live row per (group, head)
        empty[int(o_indptr[r])] = False
    lse_in[empty] = -float("inf")
    v_in[empty] = float("nan")
    ro, rl = A.merge_states(v_in.numpy(), lse_in.numpy(), o_indptr)
    assert np.isfinite(ro).all()
    vo, lo = _gpu_merge(v_in, lse_in, o_indptr)
    assert np.abs(vo.cpu().double().numpy() - ro).max() < TOL_O
    assert np.abs(lo.cpu().double().numpy() - rl).max() < TOL_L


def test_lse_out_may_be_null():
    v_in, lse_in, o_indptr = synth.merge_inputs(6, 100)
    ro, _ = A.merge_states(v_in.numpy(), lse_in.numpy(), o_indptr)
    vo, _ = _gpu_merge(v_in, lse_in, o_indptr, lse_out=False)
    assert np.abs(vo.cpu().double().numpy() - ro).max() < TOL_O


@pytest.mark.parametrize("num_out", [262144, 1048576])
def test_merge_sweep_large_sampled(num_out):
    """Large sweep points: inputs drawn on the device; 4096 seeded output rows are
    checked against the oracle on their own input rows."""
    v_in, lse_in, o_indptr = synth.merge_inputs_device(7, num_out)
    vo, lo = _gpu_merge(v_in, lse_in, o_indptr)
    rng = np.random.default_rng(8)
    rows = np.sort(rng.choice(num_out, size=4096, replace=False))
    rows[0] = 0  # includes the forced group of one
    src = np.concatenate([np.arange(o_indptr[r], o_indptr[r + 1]) for r in rows])
    sizes = o_indptr[rows + 1] - o_indptr[rows]
    sub_indptr = np.concatenate([[0], np.cumsum(sizes)])
    idx = torch.from_numpy(src).cuda()
    ro, rl = A.merge_states(v_in[idx].cpu().numpy(), lse_in[idx].cpu().numpy(), sub_indptr)
    ridx = torch.from_numpy(rows).cuda()
    assert np.abs(vo[ridx].cpu().double().numpy() - ro).max() < TOL_O
    assert np.abs(lo[ridx].cpu().double().numpy() - rl).max() < TOL_L
    del v_in, lse_in, vo, lo
    torch.cuda.empty_cache()


@pytest.mark.parametrize("H,misaligned", [(6, False), (6, True), (5, False)])
def test_two_heads_per_warp_and_its_fallbacks(H, misaligned):
    """Large grids merge two heads per warp when H is even and the LSE rows are 8-byte
    aligned; odd H, or an LSE buffer that starts one float past an 8-byte boundary,
    take the one-head form.  Each matches the oracle, with an empty group, a group of
    one, an all -inf group and empty rows (v NaN) included, and the two forms agree
    bit for bit."""
    rng = np.random.default_rng(40 + H)
    sizes = rng.integers(1, 21, size=900)
    sizes[3], sizes[4] = 0, 1
    o_indptr = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    N = int(o_indptr[-1])
    v_in = torch.from_numpy(rng.standard_normal((N, H, 128), dtype=np.float32))
    lse_in = torch.from_numpy(rng.uniform(-5, 20, size=(N, H)).astype(np.float32))
    a, b = int(o_indptr[7]), int(o_indptr[8])
    lse_in[a:b, 0] = -float("inf")                       # group 7, head 0: all -inf
    empty = torch.from_numpy(rng.random((N, H)) < 0.2)
    empty[torch.from_numpy(o_indptr[:-1][sizes > 0].astype(np.int64))] = False
    lse_in[empty] = -float("inf")
    v_in[empty] = float("nan")
    ro, rl = A.merge_states(v_in.numpy(), lse_in.numpy(), o_indptr)
    if misaligned:
        store = torch.empty(N * H + 1, device="cuda")
        dl = store[1:].view(N, H)
        dl.copy_(lse_in.cuda())
        assert dl.data_ptr() % 8 == 4
    else:
        dl = lse_in
    vo, lo = _gpu_merge(v_in, dl, o_indptr)
    assert np.abs(vo.cpu().double().numpy() - ro).max() < TOL_O
    assert np.array_equal(np.isneginf(lo.cpu().numpy()), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(lo.cpu().double().numpy()[fin] - rl[fin]).max() < TOL_L
    if H % 2 == 0 and not misaligned:   # the other form on the same rows
        store = torch.empty(N * H + 1, device="cuda")
        dl1 = store[1:].view(N, H)
        dl1.copy_(lse_in.cuda())
        vo1, lo1 = _gpu_merge(v_in, dl1, o_indptr)
        assert torch.equal(vo1, vo) and torch.equal(lo1, lo)


@pytest.mark.parametrize("H", [8, 16, 32])
def test_streaming_form_for_large_merges(H):
    """Large merges with 16-byte LSE rows and H * D / 4 a multiple of 256 stream whole
    input rows through shared memory (three CTAs per SM, 1, 2 or 4 float4 chunks per
    thread here).  Groups of one (bit-exact identity), an empty group, an all -inf
    group and empty rows whose v is NaN, against the oracle; and against the
    two-heads-per-warp form on the same rows (an LSE buffer 8 bytes past a 16-byte
    boundary takes that form), which sums in another order."""
    rng = np.random.default_rng(70 + H)
    sizes = rng.integers(1, 17, size=4000)
    sizes[3], sizes[4], sizes[5] = 0, 1, 1
    o_indptr = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    N = int(o_indptr[-1])
    v_in = torch.from_numpy(rng.standard_normal((N, H, 128), dtype=np.float32))
    lse_in = torch.from_numpy(rng.uniform(-5, 20, size=(N, H)).astype(np.float32))
    a, b = int(o_indptr[7]), int(o_indptr[8])
    lse_in[a:b, 0] = -float("inf")                       # group 7, head 0: all -inf
    empty = torch.from_numpy(rng.random((N, H)) < 0.2)
    empty[torch.from_numpy(o_indptr[:-1][sizes > 0].astype(np.int64))] = False
    lse_in[empty] = -float("inf")
    v_in[empty] = float("nan")
    ro, rl = A.merge_states(v_in.numpy(), lse_in.numpy(), o_indptr)
    dl = lse_in.cuda()
    assert dl.data_ptr() % 16 == 0
    vo, lo = _gpu_merge(v_in, dl, o_indptr)
    assert np.abs(vo.cpu().double().numpy() - ro).max() < TOL_O
    assert np.array_equal(np.isneginf(lo.cpu().numpy()), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(lo.cpu().double().numpy()[fin] - rl[fin]).max() < TOL_L
    for g in (4, 5):   # groups of one: v and lse bit for bit
        row = int(o_indptr[g])
        assert torch.equal(vo[g].cpu(), v_in[row]) and torch.equal(lo[g].cpu(), lse_in[row])
    store = torch.empty(N * H + 2, device="cuda")
    dl2 = store[2:].view(N, H)
    dl2.copy_(dl)
    assert dl2.data_ptr() % 16 == 8
    vo2, lo2 = _gpu_merge(v_in, dl2, o_indptr)
    assert (vo2 - vo).abs().max().item() < TOL_O
    both = torch.isfinite(lo2) & torch.isfinite(lo)
    assert torch.equal(torch.isneginf(lo2), torch.isneginf(lo)) and (lo2[both] - lo[both]).abs().max().item() < TOL_L


def test_streaming_form_offset_indptr_and_trailing_empty_groups():
    """The streaming form's split of output rows over its CTAs (each the range whose
    first input row falls in its equal share): o_indptr starting past row 0, one large
    group, and the last 300 groups empty, every output row against the oracle."""
    rng = np.random.default_rng(81)
    sizes = rng.integers(1, 17, size=4000)
    sizes[-300:] = 0
    sizes[1000] = 700
    o_indptr = np.concatenate([[37], 37 + np.cumsum(sizes)]).astype(np.int32)
    N = int(o_indptr[-1]) + 5
    v_in = torch.from_numpy(rng.standard_normal((N, 32, 128), dtype=np.float32))
    lse_in = torch.from_numpy(rng.uniform(-5, 20, size=(N, 32)).astype(np.float32))
    ro, rl = A.merge_states(v_in.numpy(), lse_in.numpy(), o_indptr)
    vo, lo = _gpu_merge(v_in, lse_in, o_indptr)
    assert np.abs(vo.cpu().double().numpy() - ro).max() < TOL_O
    assert np.array_equal(np.isneginf(lo.cpu().numpy()), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(lo.cpu().double().numpy()[fin] - rl[fin]).max() < TOL_L


def test_streaming_merge_gives_up_into_nan_rows():
    """The bounded waits of the streaming form: with the withheld-loads aid its
    producers copy only the first three input rows of each CTA's range, so the
    consumers' wait for the fourth runs out (about 1 ms limit).  Each CTA fills the
    output rows from the first one that needs a withheld input to the end of its range
    with NaN (v and LSE), every earlier row equals the clean merge bit for bit, and
    the next merge on the same context is clean.  The expected NaN rows follow from
    the kernel's partition of the input rows (equal shares of them, each CTA starting
    at the group that holds its share's first row)."""
    rng = np.random.default_rng(91)
    H, D = 32, 128
    sizes = rng.integers(1, 17, size=4000)
    o_indptr = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    N, M = int(o_indptr[-1]), 4000
    v_in = torch.from_numpy(rng.standard_normal((N, H, D), dtype=np.float32)).cuda()
    lse_in = torch.from_numpy(rng.uniform(-5, 20, size=(N, H)).astype(np.float32)).cuda()
    assert lse_in.data_ptr() % 16 == 0
    ind = torch.from_numpy(o_indptr).cuda()

    def run():
        vo = torch.full((M, H, D), 7.0, device="cuda")
        lo = torch.full((M, H), 7.0, device="cuda")
        psd.merge_states(ctx(), v_in, lse_in, ind, vo, lo)
        torch.cuda.synchronize()
        return vo, lo

    clean_v, clean_l = run()
    assert torch.isfinite(clean_v).all() and torch.isfinite(clean_l).all()
    ctx().test_withhold_loads(3, 2_000_000)
    try:
        vo, lo = run()
    finally:
        ctx().test_withhold_loads(-1)
    grid = 3 * torch.cuda.get_device_properties(0).multi_processor_count
    assert M >= 8 * grid   # the streaming form applies
    expect_nan = np.zeros(M, dtype=bool)
    starts = [int(np.searchsorted(o_indptr[:M], N * b // grid, side="left")) for b in range(grid)] + [M]
    for b in range(grid):
        r0, r1 = starts[b], starts[b + 1]
        if r1 <= r0:
            continue
        g0 = int(o_indptr[r0])
        for r in range(r0, r1):
            expect_nan[r] = int(o_indptr[r + 1]) > g0 + 3
    nan_v = torch.isnan(vo).all(dim=2).all(dim=1).cpu().numpy()
    nan_l = torch.isnan(lo).all(dim=1).cpu().numpy()
    fin = ~expect_nan
    assert expect_nan.sum() > M // 2 and fin.sum() > 0
    assert np.array_equal(nan_v, expect_nan) and np.array_equal(nan_l, expect_nan)
    fin_t = torch.from_numpy(fin).cuda()
    assert torch.equal(vo[fin_t], clean_v[fin_t]) and torch.equal(lo[fin_t], clean_l[fin_t])
    again_v, again_l = run()
    assert torch.equal(again_v, clean_v) and torch.equal(again_l, clean_l)
