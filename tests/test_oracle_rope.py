"""Pins of the RoPE + KV-append oracle against things other than itself: library
casts (torch bf16 and float8_e4m3fn), the E4M3 code table, the defining properties of
a rotary embedding (a basis vector lands on (cos, sin); position 0 is the identity;
pair norms are kept; dot products depend only on the relative position), the exact
float64 rotation, and the append contract (ROCm ATOM PR #1701, 3.3: rope every query,
write KV only for owned slots; [latent | roped part] row order)."""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import rope_append as R
import synth


# ----------------------------------------------------------------- rounding
def test_bf16_rounding_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * np.float32(1e3),
                        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-38),
                        np.array([0.0, -0.0, np.inf, -np.inf, 3.0e38, -3.4e38], dtype=np.float32)])
    # exact ties: low half 0x8000 with even and odd top halves
    ties = (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties])
    ours = R.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    nan = R.f32_to_bf16_bits(np.array([np.nan, -np.nan], dtype=np.float32))
    assert np.isnan(A.bf16_bits_to_f64(nan)).all()


def test_e4m3_round_trip_of_every_finite_code():
    codes = np.arange(256)
    vals = A.e4m3_to_f64(codes)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254
    assert np.array_equal(R.encode_e4m3(vals[finite]), codes[finite].astype(np.uint8))


def test_e4m3_encoding_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    pos_vals = np.sort(A.e4m3_to_f64(np.arange(0x7F)))
    mids = (pos_vals[1:] + pos_vals[:-1]) / 2            # exact ties, even code wins
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 0.01,
                        mids, -mids, pos_vals, [0.0, -0.0]]).astype(np.float32)
    ours = R.encode_e4m3(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_and_keeps_nan():
    codes = R.encode_e4m3(np.array([448.0, 449.0, 464.0, 1e6, -1e6, np.nan, -np.nan]))
    assert codes.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F, 0xFF]


# -------------------------------------------------------------- RoPE itself
@pytest.mark.parametrize("neox", [True, False])
def test_basis_vector_lands_on_cos_sin(neox):
    r, D = 16, 24
    cs = synth.rope_cos_sin_table(100, r)
    a, b = R.rope_pair_index(r, neox)
    for i in range(r // 2):
        for p in (0, 1, 37, 99):
            v = np.zeros((1, 1, D), dtype=np.float32)
            v[0, 0, a[i]] = 1.0
            out = R.rope_f32(v, np.array([p]), cs, r, neox)[0, 0]
            theta = 10000.0 ** (-2.0 * i / r)
            assert abs(out[a[i]] - np.cos(p * theta)) < 1e-6
            assert abs(out[b[i]] - np.sin(p * theta)) < 1e-6
            others = np.delete(out, [a[i], b[i]])
            assert np.all(others == 0)


def test_pairing_layouts_by_hand():
    assert [list(x) for x in R.rope_pair_index(8, True)] == [[0, 1, 2, 3], [4, 5, 6, 7]]
    assert [list(x) for x in R.rope_pair_index(8, False)] == [[0, 2, 4, 6], [1, 3, 5, 7]]


@pytest.mark.parametrize("neox", [True, False])
def test_position_zero_is_identity_and_tail_columns_untouched(neox):
    rng = np.random.default_rng(2)
    v = rng.standard_normal((3, 4, 40)).astype(np.float32)
    cs = synth.rope_cos_sin_table(10, 32)
    out = R.rope_f32(v, np.zeros(3, dtype=np.int64), cs, 32, neox)
    assert np.array_equal(out, v)
    out = R.rope_f32(v, np.array([3, 5, 7]), cs, 32, neox)
    assert np.array_equal(out[..., 32:], v[..., 32:])


@pytest.mark.parametrize("neox", [True, False])
def test_float32_rotation_is_the_exact_rotation_to_rounding(neox):
    rng = np.random.default_rng(3)
    r = 64
    v = rng.standard_normal((50, 4, r)).astype(np.float32)
    pos = rng.integers(0, 4096, size=50)
    cs = synth.rope_cos_sin_table(4096, r)
    got = R.rope_f32(v, pos, cs, r, neox).astype(np.float64)
    theta = 10000.0 ** (-2.0 * np.arange(r // 2) / r)
    exact = R.rope_f64(v.astype(np.float64), pos[:, None] * theta[None, :], r, neox)
    # table entries carry a float32 rounding, products and sums one each
    assert np.abs(got - exact).max() < 4e-6 * np.abs(v).max() * 4
    # pair norms are kept
    a, b = R.rope_pair_index(r, neox)
    n_in = v[..., a].astype(np.float64) ** 2 + v[..., b].astype(np.float64) ** 2
    n_out = got[..., a] ** 2 + got[..., b] ** 2
    assert np.abs(n_out - n_in).max() < 1e-5 * n_in.max()


@pytest.mark.parametrize("neox", [True, False])
def test_scores_depend_only_on_relative_position(neox):
    """<rope(q, m), rope(k, n)> = <rope(q, m + s), rope(k, n + s)>: the defining
    property of a rotary embedding (exact float64 rotation)."""
    rng = np.random.default_rng(4)
    r = 32
    q, k = rng.standard_normal((1, 1, r)), rng.standard_normal((1, 1, r))
    theta = 10000.0 ** (-2.0 * np.arange(r // 2) / r)
    for m, n, s in [(5, 2, 11), (100, 7, 900), (0, 30, 3)]:
        d1 = np.sum(R.rope_f64(q, m * theta[None], r, neox) * R.rope_f64(k, n * theta[None], r, neox))
        d2 = np.sum(R.rope_f64(q, (m + s) * theta[None], r, neox) * R.rope_f64(k, (n + s) * theta[None], r, neox))
        assert abs(d1 - d2) < 1e-9
    # and a different relative position gives a different score
    d3 = np.sum(R.rope_f64(q, 6 * theta[None], r, neox) * R.rope_f64(k, 2 * theta[None], r, neox))
    assert abs(d3 - np.sum(R.rope_f64(q, 5 * theta[None], r, neox) * R.rope_f64(k, 2 * theta[None], r, neox))) > 1e-6


# ------------------------------------------------------------- the append op
def _run(step):
    return R.rope_append(
        synth.bf16_bits(step.q), None if step.k_nope is None else synth.bf16_bits(step.k_nope),
        synth.bf16_bits(step.k_rope), None if step.v is None else synth.bf16_bits(step.v),
        step.cos_sin, step.positions, step.slot_mapping, rot_dim=step.rot_dim, neox=step.neox,
        q_rope_col=step.q_rope_col,
        k_pool=synth.bf16_bits(step.k_pool) if step.kv_dtype == "bf16" else synth.u8_codes(step.k_pool),
        v_pool=None if step.v_pool is None else (synth.bf16_bits(step.v_pool) if step.kv_dtype == "bf16"
                                                 else synth.u8_codes(step.v_pool)),
        page_size=step.page_size, kv_dtype=step.kv_dtype, k_scale=step.k_scale, v_scale=step.v_scale)


def test_append_writes_owned_slots_only_and_copies_unroped_columns():
    st = synth.append_step(5, "mla", T=24, kv_dtype="bf16", skip_every=3, num_pages=64)
    q_out, k_out, v_out = _run(st)
    assert v_out is None
    k_in = synth.bf16_bits(st.k_pool)
    written = np.zeros(k_in.shape[:2], dtype=bool)
    for t, s in enumerate(st.slot_mapping):
        if s < 0:
            continue
        page, slot = divmod(int(s), st.page_size)
        written[page, slot] = True
        # [latent | roped part]: the latent is copied bit for bit
        assert np.array_equal(k_out[page, slot, 0, :512], synth.bf16_bits(st.k_nope)[t, 0])
        assert not np.array_equal(k_out[page, slot, 0, 512:], synth.bf16_bits(st.k_rope)[t, 0]) or st.positions[t] == 0
    assert np.array_equal(k_out[~written], k_in[~written])     # untouched (NaN canaries)
    assert written.sum() == np.sum(st.slot_mapping >= 0)
    # queries: every token roped, only the rope columns change
    qb = synth.bf16_bits(st.q)
    assert np.array_equal(q_out[..., :512], qb[..., :512])
    changed = np.any(q_out[..., 512:] != qb[..., 512:], axis=(1, 2))
    assert changed[st.positions != 0].all()


def test_fp8_codes_dequantise_to_the_stored_values():
    st = synth.append_step(6, "gqa", T=16, kv_dtype="fp8_e4m3", num_pages=64)
    _, k_out, v_out = _run(st)
    kr = R.rope_f32(R.bf16_bits_to_f32(synth.bf16_bits(st.k_rope)), st.positions, st.cos_sin, st.rot_dim,
                    st.neox).astype(np.float64)
    vv = R.bf16_bits_to_f32(synth.bf16_bits(st.v)).astype(np.float64)
    for t, s in enumerate(st.slot_mapping):
        page, slot = divmod(int(s), st.page_size)
        kd = A.e4m3_to_f64(k_out[page, slot]) * st.k_scale
        vd = A.e4m3_to_f64(v_out[page, slot]) * st.v_scale
        # E4M3 keeps 3 mantissa bits: half an ulp is 2^-4 of the value (plus the
        # subnormal step 2^-10 * scale near zero)
        assert np.all(np.abs(kd - kr[t]) <= np.abs(kr[t]) * 2 ** -4 + 2 ** -10 * st.k_scale)
        assert np.all(np.abs(vd - vv[t]) <= np.abs(vv[t]) * 2 ** -4 + 2 ** -10 * st.v_scale)
