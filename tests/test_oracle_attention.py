"""Pins of the float64 oracle's gather, dequantisation and attention against things
other than itself: torch's fp8/bf16 casts, brute force over a dense copy of each
request's keys, closed forms, and torch's scaled_dot_product_attention."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from synth import bf16_bits, page_table


def test_fp8_e4m3_decode_all_256_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = A.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2                      # S.1111.111 for both signs
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_bf16_widening_matches_torch():
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal(4096).astype(np.float32) * 100).to(torch.bfloat16)
    ours = A.bf16_bits_to_f64(bf16_bits(x))
    assert np.array_equal(ours, x.double().numpy())


def _dense_then_paged(rng, lengths, Hq, Hkv, D, P, num_pages):
    """Dense per-request K/V first, then scattered into a pool through a random
    page permutation.  The brute force below only ever reads the dense copy."""
    indptr, indices, last = page_table(lengths, P, num_pages, rng)
    dense_k = [torch.from_numpy(rng.standard_normal((L, Hkv, D), dtype=np.float32)).to(torch.bfloat16)
               for L in lengths]
    dense_v = [torch.from_numpy(rng.standard_normal((L, Hkv, D), dtype=np.float32)).to(torch.bfloat16)
               for L in lengths]
    kpool = torch.full((num_pages, P, Hkv, D), float("nan"), dtype=torch.bfloat16)
    vpool = kpool.clone()
    for b, L in enumerate(lengths):
        for j in range(L):
            page = int(indices[indptr[b] + j // P])
            kpool[page, j % P] = dense_k[b][j]
            vpool[page, j % P] = dense_v[b][j]
    q = torch.from_numpy(rng.standard_normal((len(lengths), Hq, D), dtype=np.float32)).to(torch.bfloat16)
    a = dict(q_raw=bf16_bits(q), k_raw=bf16_bits(kpool), v_raw=bf16_bits(vpool), kv_dtype="bf16",
             k_scale=1.0, v_scale=1.0, page_indptr=indptr, page_indices=indices,
             last_page_len=last, page_size=P, Dv=D, sm_scale=1.0 / math.sqrt(D), Hq=Hq, Hkv=Hkv)
    return a, q, dense_k, dense_v


def _brute(q, dense_k, dense_v, sm_scale):
    """Scalar Python softmax attention on the dense copies (no numpy, no page table)."""
    B, Hq, D = q.shape
    out, lse = [], []
    for b in range(B):
        K, V = dense_k[b].double().tolist(), dense_v[b].double().tolist()
        Hkv = len(K[0])
        G = Hq // Hkv
        ob, lb = [], []
        for h in range(Hq):
            qh = q[b, h].double().tolist()
            kv = h // G
            s = [sm_scale * math.fsum(qh[d] * K[j][kv][d] for d in range(D)) for j in range(len(K))]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            den = math.fsum(e)
            ob.append([math.fsum(e[j] * V[j][kv][d] for j in range(len(K))) / den for d in range(D)])
            lb.append((mx + math.log(den)) / math.log(2.0))
        out.append(ob)
        lse.append(lb)
    return np.array(out), np.array(lse)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 3), (8, 1)])
def test_gather_attention_matches_brute_force_on_dense_copy(Hq, Hkv):
    rng = np.random.default_rng(11 + Hq)
    a, q, dk, dv = _dense_then_paged(rng, [5, 9, 1, 16, 17], Hq, Hkv, 8, 4, 40)
    o, lse = A.decode_attention(a)
    ob, lb = _brute(q, dk, dv, a["sm_scale"])
    assert np.abs(o - ob).max() < 1e-12
    assert np.abs(lse - lb).max() < 1e-12


def test_gather_reads_wrong_values_if_slots_transposed():
    """A plausible gather bug (page and slot roles swapped) must change the result:
    the brute-force pin above is sensitive to the gather indexing."""
    rng = np.random.default_rng(5)
    a, q, dk, dv = _dense_then_paged(rng, [9, 12], 4, 2, 8, 4, 40)
    good = A.decode_attention(a)[0]
    k = a["k_raw"]
    bad = dict(a, k_raw=np.ascontiguousarray(k[:, ::-1]))      # slot order reversed
    assert np.nanmax(np.abs(A.decode_attention(bad)[0] - good)) > 1e-3 or \
        np.isnan(A.decode_attention(bad)[0]).any()


def test_equal_keys_give_uniform_weights_closed_form():
    """All keys of a request equal: s_j = c for every j, so o = mean(V) and
    lse2 = log2 L + c * log2 e."""
    rng = np.random.default_rng(7)
    L, Hkv, D, Hq = 37, 2, 16, 4
    k1 = rng.standard_normal((Hkv, D))
    K = np.broadcast_to(k1, (L, Hkv, D)).copy()
    V = rng.standard_normal((L, Hkv, D))
    q = rng.standard_normal((Hq, D))
    sm = 0.25
    o, lse = A.attend(q, K, V, sm)
    G = Hq // Hkv
    for h in range(Hq):
        c = sm * math.fsum(q[h, d] * k1[h // G, d] for d in range(D))
        assert abs(lse[h] - (math.log2(L) + c / math.log(2.0))) < 1e-12
        assert np.abs(o[h] - V[:, h // G].mean(axis=0)).max() < 1e-13


def test_constant_values_give_constant_output():
    rng = np.random.default_rng(8)
    K = rng.standard_normal((50, 1, 8)) * 3
    V = np.full((50, 1, 8), 1.75)
    o, _ = A.attend(rng.standard_normal((4, 8)), K, V, 0.5)
    assert np.abs(o - 1.75).max() < 1e-14


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (8, 2)])
def test_attention_matches_torch_sdpa_float64(Hq, Hkv):
    """Textbook MHA (G = 1) and GQA via repeated KV heads, as computed by torch's
    scaled_dot_product_attention in float64 on the CPU."""
    rng = np.random.default_rng(9)
    L, D = 29, 16
    q = rng.standard_normal((Hq, D))
    K = rng.standard_normal((L, Hkv, D))
    V = rng.standard_normal((L, Hkv, D))
    o, lse = A.attend(q, K, V, 1.0 / math.sqrt(D))
    G = Hq // Hkv
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq, L, D]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, :], kt, vt)[:, 0, :].numpy()
    assert np.abs(o - ref).max() < 1e-12
    s = torch.einsum("hd,hld->hl", torch.from_numpy(q), kt) / math.sqrt(D)
    assert np.abs(lse - (torch.logsumexp(s, dim=1).numpy() / math.log(2))).max() < 1e-12


def test_fp8_pool_dequant_uses_scale_and_latent_v():
    """fp8 latent pool: K = code * scale, V = first Dv columns of the same rows."""
    rng = np.random.default_rng(4)
    P, Dqk, Dv = 4, 12, 8
    indptr, indices, last = page_table([7, 3], P, 10, rng)
    vals = rng.standard_normal((10, P, 1, Dqk)).astype(np.float32)
    scale = float(np.abs(vals).max() / 448.0)
    codes = torch.from_numpy(vals / scale).to(torch.float8_e4m3fn)
    q = torch.from_numpy(rng.standard_normal((2, 4, Dqk), dtype=np.float32)).to(torch.bfloat16)
    a = dict(q_raw=bf16_bits(q), k_raw=codes.view(torch.uint8).numpy(), v_raw=None,
             kv_dtype="fp8_e4m3", k_scale=scale, v_scale=scale, page_indptr=indptr,
             page_indices=indices, last_page_len=last, page_size=P, Dv=Dv, sm_scale=0.3,
             Hq=4, Hkv=1)
    o, lse = A.decode_attention(a)
    deq = codes.to(torch.float32).double().numpy() * scale           # library cast
    for b in range(2):
        L = (indptr[b + 1] - indptr[b] - 1) * P + last[b]
        j = np.arange(L)
        rows = deq[indices[indptr[b] + j // P], j % P]                # [L, 1, Dqk]
        oo, ll = A.attend(q[b].double().numpy(), rows, rows[..., :Dv], 0.3)
        assert np.abs(o[b] - oo).max() < 1e-12 and np.abs(lse[b] - ll).max() < 1e-12


# ------------------------------------------------------------------------------
# workload_arrays and separate K / V scales, pinned against torch computing the same
# attention straight from a synth.Workload's own tensors: pages gathered by torch
# indexing, fp8 codes decoded by torch's float8_e4m3fn cast and scaled by their own
# tensor's scale (ROCm ATOM PR #1701, 3.2: value = code * scale), request lengths
# taken from the generator's lengths (not last_page_len), softmax by torch SDPA.

def _torch_decode(w, k_scale=None, v_scale=None):
    """o [B, Hq, Dv], lse2 [B, Hq] by torch in float64 from the Workload's tensors."""
    ks = w.k_scale if k_scale is None else k_scale
    vs = w.v_scale if v_scale is None else v_scale
    G = w.Hq // w.Hkv

    def dq(raw, scale):
        if w.kv_dtype == "bf16":
            return raw.double()
        return raw.view(torch.float8_e4m3fn).to(torch.float32).double() * scale

    o = torch.empty((w.batch, w.Hq, w.Dv), dtype=torch.float64)
    lse = torch.empty((w.batch, w.Hq), dtype=torch.float64)
    for b in range(w.batch):
        pages = torch.as_tensor(w.page_indices[w.page_indptr[b]:w.page_indptr[b + 1]].astype(np.int64))
        L = int(w.lengths[b])
        kraw = w.k_pool[pages].reshape(-1, w.Hkv, w.Dqk)[:L]
        k = dq(kraw, ks)
        if w.v_pool is None:
            v = dq(kraw[..., :w.Dv].contiguous(), vs)
        else:
            v = dq(w.v_pool[pages].reshape(-1, w.Hkv, w.Dv)[:L], vs)
        kt = k.permute(1, 0, 2).repeat_interleave(G, dim=0)     # [Hq, L, Dqk]
        vt = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
        qb = w.q[b].double()[:, None, :]
        o[b] = torch.nn.functional.scaled_dot_product_attention(qb, kt, vt, scale=w.sm_scale)[:, 0]
        s = torch.einsum("hd,hld->hl", w.q[b].double(), kt) * w.sm_scale
        lse[b] = torch.logsumexp(s, dim=1) / math.log(2.0)
    return o.numpy(), lse.numpy()


def _small_fp8_kv(seed, kv_scale_ratio=None):
    import synth
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(1, 120, size=4)]
    w = synth._make("fp8_kv_small", rng, lengths, Hq=8, Hkv=2, Dqk=64, Dv=64, page_size=16,
                    num_pages=40, tile_tokens=32, kv_dtype="fp8_e4m3")
    if kv_scale_ratio is not None:          # same codes, V's scale far from K's
        import dataclasses
        w = dataclasses.replace(w, v_scale=w.k_scale * kv_scale_ratio)
    return w


def _small_fp8_latent(seed):
    import synth
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(1, 300, size=3)]
    return synth._make("fp8_latent_small", rng, lengths, Hq=16, Hkv=1, Dqk=576, Dv=512, page_size=64,
                       num_pages=20, tile_tokens=128, kv_dtype="fp8_e4m3", latent_v=True)


def _synth_case(kind):
    import synth
    if kind == "bf16_tiny_cascade":
        return synth.tiny_cascade(seed=1)
    if kind == "fp8_separate_kv":
        return _small_fp8_kv(21)
    if kind == "fp8_latent":
        return _small_fp8_latent(22)
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["bf16_tiny_cascade", "fp8_separate_kv", "fp8_latent"])
def test_workload_arrays_decode_matches_torch_on_synth_workloads(kind):
    """The adapter every GPU parity test uses (bit views, scales, Dv, sm_scale, a
    latent's missing V pool) feeds decode_attention the same attention torch computes
    from the Workload directly."""
    w = _synth_case(kind)
    o, lse = A.decode_attention(A.workload_arrays(w))
    ro, rl = _torch_decode(w)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert np.abs(o - ro).max() < 1e-10
    assert np.abs(lse - rl).max() < 1e-10


def test_fp8_separate_k_and_v_scales_are_applied_independently():
    """fp8 pool with separate K and V and v_scale = 4 * k_scale: K dequantises with
    k_scale and V with v_scale.  gather_kv matches torch's cast times each tensor's
    own scale; decode_attention matches torch; and the slip of dequantising V with
    k_scale (planted in the inputs, on the CPU) misses torch by far more than the
    fp8 tolerance."""
    w = _small_fp8_kv(23, kv_scale_ratio=4.0)
    a = A.workload_arrays(w)
    assert a["v_scale"] == 4.0 * a["k_scale"]
    for b in range(w.batch):
        K, V = A.gather_kv(a, b)
        pages = torch.as_tensor(w.page_indices[w.page_indptr[b]:w.page_indptr[b + 1]].astype(np.int64))
        L = int(w.lengths[b])
        kt = w.k_pool[pages].reshape(-1, w.Hkv, w.Dqk)[:L].view(torch.float8_e4m3fn).double() * w.k_scale
        vt = w.v_pool[pages].reshape(-1, w.Hkv, w.Dv)[:L].view(torch.float8_e4m3fn).double() * w.v_scale
        assert np.array_equal(K, kt.numpy()) and np.array_equal(V, vt.numpy())
    o, lse = A.decode_attention(a)
    ro, rl = _torch_decode(w)
    assert np.abs(o - ro).max() < 1e-10 and np.abs(lse - rl).max() < 1e-10
    slip, _ = A.decode_attention(dict(a, v_scale=a["k_scale"]))
    assert np.abs(slip - ro).max() > 10 * 1e-2
    # and K's scale moves the scores: the same slip on K (k_scale := v_scale) fails too
    slip_k, slip_kl = A.decode_attention(dict(a, k_scale=a["v_scale"]))
    assert np.abs(slip_kl - rl).max() > 10 * 1e-3
