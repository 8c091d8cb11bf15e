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
