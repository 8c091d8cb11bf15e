"""Pins of the oracle's log2-LSE merge: the invariants of the Merge contract section
of mlxcel PR #1004 (disjoint key ranges merge to the flat result, regrouping is
associative, a group of one is the identity) and its negative control (natural-log
LSEs must not reproduce the flat result)."""
import numpy as np
import pytest

from oracle import attention as A


def _request(rng, L=53, Hkv=2, G=3, D=16):
    q = rng.standard_normal((Hkv * G, D))
    K = rng.standard_normal((L, Hkv, D)) * 1.5
    V = rng.standard_normal((L, Hkv, D))
    return q, K, V


@pytest.mark.parametrize("cuts", [[20], [1, 2, 40], [7, 14, 21, 28, 35, 42, 49]])
def test_merge_of_disjoint_ranges_equals_flat(cuts):
    rng = np.random.default_rng(len(cuts))
    q, K, V = _request(rng)
    o, lse = A.attend(q, K, V, 0.3)
    bounds = [0] + cuts + [K.shape[0]]
    parts = [A.attend(q, K[a:b], V[a:b], 0.3) for a, b in zip(bounds[:-1], bounds[1:])]
    v_in = np.stack([p[0] for p in parts])
    lse_in = np.stack([p[1] for p in parts])
    mo, ml = A.merge_states(v_in, lse_in, [0, len(parts)])
    assert np.abs(mo[0] - o).max() < 1e-13
    assert np.abs(ml[0] - lse).max() < 1e-13


def test_merge_is_associative_across_regroupings():
    rng = np.random.default_rng(1)
    N, H, D = 9, 4, 8
    v = rng.standard_normal((N, H, D))
    l = rng.uniform(-5, 20, size=(N, H))
    direct = A.merge_states(v, l, [0, N])
    left = A.merge_states(v, l, [0, 2, 5, 9])           # (0,1) (2,3,4) (5..8)
    two = A.merge_states(left[0], left[1], [0, 3])
    right = A.merge_states(v, l, [0, 4, 6, 9])
    two_r = A.merge_states(right[0], right[1], [0, 3])
    for o, ll in (two, two_r):
        assert np.abs(o - direct[0]).max() < 1e-13
        assert np.abs(ll - direct[1]).max() < 1e-12


def test_group_of_one_is_the_identity_bit_exact():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((5, 3, 7))
    l = rng.uniform(-5, 20, size=(5, 3))
    o, lo = A.merge_states(v, l, [0, 1, 2, 3, 4, 5])
    assert np.array_equal(o, v) and np.array_equal(lo, l)


def test_natural_log_lse_does_not_reproduce_flat():
    """Negative control: chunks of unequal length have unequal LSEs, and a merge
    that reads them as natural logs misweights them."""
    rng = np.random.default_rng(3)
    q, K, V = _request(rng, L=80)
    o, _ = A.attend(q, K, V, 0.5)
    parts = [A.attend(q, K[a:b], V[a:b], 0.5) for a, b in ((0, 5), (5, 80))]
    v_in = np.stack([p[0] for p in parts])
    lse_in = np.stack([p[1] for p in parts])
    good = A.merge_states(v_in, lse_in, [0, 2])[0][0]
    bad = A.merge_states_natural_log(v_in, lse_in, [0, 2])[0]
    assert np.abs(good - o).max() < 1e-13
    assert np.abs(bad - o).max() > 1e-2


def test_empty_and_all_neg_inf_groups_are_zero_with_neg_inf_lse():
    v = np.ones((2, 1, 4))
    l = np.full((2, 1), -np.inf)
    o, lo = A.merge_states(v, l, [0, 0, 2])
    assert np.array_equal(o, np.zeros((2, 1, 4))) and np.all(lo == -np.inf)


def test_two_row_merge_weights_by_powers_of_two():
    """Closed form with lse = (0, 1): weights 1 and 2 (log2 units), so the result is
    (v0 + 2 v1) / 3 and lse = log2 3."""
    v = np.array([[[3.0]], [[6.0]]])
    o, lo = A.merge_states(v, np.array([[0.0], [1.0]]), [0, 2])
    assert abs(o[0, 0, 0] - 5.0) < 1e-15 and abs(lo[0, 0] - np.log2(3.0)) < 1e-15


def test_empty_partials_are_ignored_whatever_their_v():
    """A row with LSE = -inf is an empty partial (a chunk with no tokens): merging a
    group with such rows (v NaN or huge) equals merging the group without them, and
    equals attention over the union of the non-empty chunks."""
    rng = np.random.default_rng(4)
    q, K, V = _request(rng, L=60)
    o, lse = A.attend(q, K, V, 0.4)
    parts = [A.attend(q, K[a:b], V[a:b], 0.4) for a, b in ((0, 25), (25, 60))]
    H, D = parts[0][0].shape
    empty_v = np.full((H, D), np.nan)
    rows_v = [parts[0][0], empty_v, parts[1][0], np.full((H, D), 1e300)]
    rows_l = [parts[0][1], np.full(H, -np.inf), parts[1][1], np.full(H, -np.inf)]
    mo, ml = A.merge_states(np.stack(rows_v), np.stack(rows_l), [0, 4])
    assert np.abs(mo[0] - o).max() < 1e-13 and np.abs(ml[0] - lse).max() < 1e-13
    # mixed: head 0 of a row empty, the other heads live
    l2 = np.stack([parts[0][1], parts[1][1]]).copy()
    v2 = np.stack([parts[0][0], parts[1][0]]).copy()
    l2[1, 0], v2[1, 0] = -np.inf, np.nan
    mo2, ml2 = A.merge_states(v2, l2, [0, 2])
    assert np.array_equal(mo2[0, 0], parts[0][0][0]) and ml2[0, 0] == parts[0][1][0]
    assert np.abs(mo2[0, 1:] - o[1:]).max() < 1e-13
