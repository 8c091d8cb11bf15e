"""RoPE + KV append on the GPU against the oracle, bit for bit: the roped queries,
and every byte of the K and V pools (written rows, untouched rows and skipped
slots) for the GQA and MLA shapes, bf16 and fp8 pools, both pairings (ROCm ATOM PR
#1701, 3.3: rope every query, write KV only for owned slots)."""
import numpy as np
import pytest
import torch

import paged_split_kv_decode_gb300 as psd
from oracle import rope_append as R
import synth
from _gpu_util import ctx

pytestmark = pytest.mark.gpu


def _pool_codes(t):
    return synth.bf16_bits(t) if t.dtype == torch.bfloat16 else synth.u8_codes(t)


def _run_gpu(st, fault=None):
    dev = lambda t: None if t is None else t.cuda().contiguous()
    q, kn, kr, v = dev(st.q), dev(st.k_nope), dev(st.k_rope), dev(st.v)
    kp, vp = dev(st.k_pool), dev(st.v_pool)
    cs = torch.from_numpy(st.cos_sin).cuda()
    pos = torch.from_numpy(st.positions).cuda()
    slots = torch.from_numpy(st.slot_mapping).cuda()
    f = psd.rope_append_kv(ctx(), q, kn, kr, v, cs, pos, slots, kp, vp, rot_dim=st.rot_dim, neox=st.neox,
                           q_rope_col=st.q_rope_col, page_size=st.page_size, k_scale=st.k_scale,
                           v_scale=st.v_scale, fault=fault)
    torch.cuda.synchronize()
    return q.cpu(), kp.cpu(), (vp.cpu() if vp is not None else None), int(f.cpu().item())


def _run_oracle(st):
    return R.rope_append(
        synth.bf16_bits(st.q), None if st.k_nope is None else synth.bf16_bits(st.k_nope),
        synth.bf16_bits(st.k_rope), None if st.v is None else synth.bf16_bits(st.v), st.cos_sin, st.positions,
        st.slot_mapping, rot_dim=st.rot_dim, neox=st.neox, q_rope_col=st.q_rope_col,
        k_pool=_pool_codes(st.k_pool), v_pool=None if st.v_pool is None else _pool_codes(st.v_pool),
        page_size=st.page_size, kv_dtype=st.kv_dtype, k_scale=st.k_scale, v_scale=st.v_scale)


def _compare(st):
    gq, gk, gv, fault = _run_gpu(st)
    rq, rk, rv = _run_oracle(st)
    assert fault == 0
    assert np.array_equal(synth.bf16_bits(gq), rq)
    assert np.array_equal(_pool_codes(gk), rk)
    if rv is not None:
        assert np.array_equal(_pool_codes(gv), rv)


@pytest.mark.parametrize("kind", ["gqa", "mla"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("skip_every", [0, 3])
def test_bit_exact_against_oracle(kind, kv_dtype, neox, skip_every):
    st = synth.append_step(seed=hash((kind, kv_dtype, neox, skip_every)) % 1000, kind=kind, T=48,
                           kv_dtype=kv_dtype, neox=neox, skip_every=skip_every, num_pages=128)
    _compare(st)


def test_decode_batch_sizes_and_a_prefill_chunk():
    for T in (1, 128, 1024):
        _compare(synth.append_step(seed=T, kind="gqa", T=T, num_pages=max(128, T // 16 + 64)))


def test_partial_rotary_copies_the_tail_columns():
    st = synth.append_step(seed=9, kind="gqa", T=32, num_pages=128)
    st.rot_dim = 64
    st.cos_sin = synth.rope_cos_sin_table(st.cos_sin.shape[0], 64)
    _compare(st)


def test_saturating_fp8_scale():
    st = synth.append_step(seed=10, kind="mla", T=16, kv_dtype="fp8_e4m3", num_pages=64)
    st.k_scale = st.k_scale / 8.0          # many values above 448 * scale: saturate to 448
    _compare(st)


def test_zero_tokens_is_a_no_op():
    st = synth.append_step(seed=11, kind="gqa", T=1, num_pages=64)
    st.q, st.k_rope, st.v = st.q[:0], st.k_rope[:0], st.v[:0]
    st.positions, st.slot_mapping = st.positions[:0], st.slot_mapping[:0]
    gq, gk, gv, fault = _run_gpu(st)
    assert fault == 0 and np.array_equal(_pool_codes(gk), _pool_codes(st.k_pool))


def test_out_of_range_position_and_slot_are_flagged_and_skipped():
    st = synth.append_step(seed=12, kind="gqa", T=8, num_pages=64)
    st.positions = st.positions.copy()
    st.slot_mapping = st.slot_mapping.copy()
    st.positions[2] = st.cos_sin.shape[0]            # no table row
    st.slot_mapping[5] = 64 * st.page_size           # one past the pool
    gq, gk, gv, fault = _run_gpu(st)
    assert fault == (psd._lib.PSD_OK | 4 | 1)        # PSD_FAULT_RANGE | PSD_FAULT_PAGE_ID
    assert np.array_equal(synth.bf16_bits(gq)[2], synth.bf16_bits(st.q)[2])   # token 2 untouched
    # the other tokens are as the oracle writes them when tokens 2 and 5 write nothing
    ok = np.ones(8, dtype=bool)
    ok[[2, 5]] = False
    st2 = synth.append_step(seed=12, kind="gqa", T=8, num_pages=64)
    st2.slot_mapping = st.slot_mapping.copy()
    st2.slot_mapping[[2, 5]] = -1
    st2.positions = st.positions.copy()
    st2.positions[2] = 0
    rq, rk, rv = _run_oracle(st2)
    assert np.array_equal(synth.bf16_bits(gq)[ok], rq[ok])
    assert np.array_equal(_pool_codes(gk), rk) and np.array_equal(_pool_codes(gv), rv)


@pytest.mark.parametrize("bad", ["odd_rot", "rot_too_wide", "missing_v_pool", "zero_scale"])
def test_host_validation(bad):
    st = synth.append_step(seed=13, kind="gqa", T=4, kv_dtype="fp8_e4m3", num_pages=16)
    kw = dict(rot_dim=st.rot_dim, neox=st.neox, q_rope_col=0, page_size=st.page_size, k_scale=st.k_scale,
              v_scale=st.v_scale)
    vp = st.v_pool.cuda()
    if bad == "odd_rot":
        kw["rot_dim"] = 63
    elif bad == "rot_too_wide":
        kw["rot_dim"] = 130
    elif bad == "missing_v_pool":
        vp = None
    else:
        kw["k_scale"] = 0.0
    with pytest.raises(psd.PsdError):
        psd.rope_append_kv(ctx(), st.q.cuda(), None, st.k_rope.cuda(), st.v.cuda(),
                           torch.from_numpy(st.cos_sin).cuda(), torch.from_numpy(st.positions).cuda(),
                           torch.from_numpy(st.slot_mapping).cuda(), st.k_pool.cuda(), vp, **kw)


@pytest.mark.parametrize("neox", [True, False])
def test_scalar_form_for_narrow_rotary(neox):
    """rot_dim 8 is not a multiple of 16: the scalar kernel serves it, same bits."""
    st = synth.append_step(seed=14, kind="gqa", T=32, kv_dtype="fp8_e4m3", neox=neox, num_pages=128)
    st.rot_dim = 8
    st.cos_sin = synth.rope_cos_sin_table(st.cos_sin.shape[0], 8)
    _compare(st)
