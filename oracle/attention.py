"""Float64 attention, partials and merge (oracle; test infrastructure only).

Source: mlxcel PR #1004, "compute shared prompt prefixes once per decode batch".
  * Decomposition section: one threadgroup owns all query heads of one KV head for
    one (request, page tile); query head h reads KV head h / NRep.
  * Merge contract section: v_in [N, H, D] already normalised per row, lse_in [N, H]
    in log2 units (m + log2 l), o_indptr [M + 1] groups contiguous rows; a group of
    one row is the identity (l = 1, out = v).
  * Detection section: a CSR page table; one block id is one physical pool row.
ROCm ATOM PR #1701, section 3.2: fp8 latent KV is dequantised as value * k_scale.

The Decomposition section states that the two key ranges of the cascade are
disjoint, so its merge reproduces dense attention apart from f32 rounding.  The
oracle is therefore that definition: gather a request's pages into contiguous K/V,
then plain softmax attention in float64.
"""
from __future__ import annotations

import math

import numpy as np

LN2 = math.log(2.0)


# --------------------------------------------------------------------------- dtypes
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns: a bf16 is the top half of an IEEE f32."""
    b = np.ascontiguousarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode OCP FP8 E4M3FN codes by the format's definition.

    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.  Exponent field 0
    holds subnormals m/8 * 2^-6; there are no infinities; S.1111.111 is NaN; the
    largest finite magnitude is 1.75 * 2^8 = 448.
    """
    c = np.ascontiguousarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = (m / 8.0) * 2.0 ** -6
    mag = np.where(e == 0, subnormal, normal)
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def dequant(raw: np.ndarray, kv_dtype: str, scale: float) -> np.ndarray:
    """K/V element values in float64.  bf16 widens exactly.  fp8-e4m3 is the
    decoded code times the per-tensor scale (ATOM PR #1701, 3.2: ag_kv.to(bf16) *
    k_scale); the oracle keeps the exact float64 product."""
    if kv_dtype == "bf16":
        return bf16_bits_to_f64(raw)
    if kv_dtype == "fp8_e4m3":
        return e4m3_to_f64(raw) * float(scale)
    raise ValueError(kv_dtype)


# ---------------------------------------------------------------------- page table
def request_length(page_indptr, last_page_len, page_size, b) -> int:
    """L_b = (n_b - 1) * page_size + last_page_len[b]: every page but the last is
    full (CSR page-table convention of the Detection section)."""
    n = int(page_indptr[b + 1]) - int(page_indptr[b])
    return (n - 1) * int(page_size) + int(last_page_len[b])


def gather_tokens(pool_raw: np.ndarray, page_indptr, page_indices, last_page_len,
                  page_size: int, b: int) -> np.ndarray:
    """Raw pool rows of request b in token order, [L_b, Hkv, D].

    Token j of request b lives in pool page page_indices[page_indptr[b] + j // P]
    at slot j % P.
    """
    L = request_length(page_indptr, last_page_len, page_size, b)
    j = np.arange(L)
    pages = np.asarray(page_indices)[int(page_indptr[b]) + j // page_size]
    slots = j % page_size
    return pool_raw[pages, slots]


def gather_kv(w_arrays: dict, b: int):
    """Dequantised K [L, Hkv, Dqk] and V [L, Hkv, Dv] of request b (float64).

    When ``v_raw`` is None the V rows are the first Dv columns of the K rows (a
    shared MLA latent, MLA decode of the mlxcel epic #907 as cited on the page)."""
    a = w_arrays
    kraw = gather_tokens(a["k_raw"], a["page_indptr"], a["page_indices"],
                         a["last_page_len"], a["page_size"], b)
    K = dequant(kraw, a["kv_dtype"], a["k_scale"])
    if a["v_raw"] is None:
        V = dequant(kraw[..., :a["Dv"]], a["kv_dtype"], a["v_scale"])
    else:
        vraw = gather_tokens(a["v_raw"], a["page_indptr"], a["page_indices"],
                             a["last_page_len"], a["page_size"], b)
        V = dequant(vraw, a["kv_dtype"], a["v_scale"])
    return K, V


# ----------------------------------------------------------------------- attention
def attend(q_b: np.ndarray, K: np.ndarray, V: np.ndarray, sm_scale: float):
    """Softmax attention of one request's query heads over its keys (float64).

    q_b [Hq, Dqk], K [L, Hkv, Dqk], V [L, Hkv, Dv].  Query head h reads KV head
    h // G with G = Hq / Hkv (the head mapping of the Decomposition section, whose
    NRep is this G).  Returns o [Hq, Dv] and the log-sum-exp in log2 units
        lse2 = log2 sum_j 2^(s_j * log2 e) = (ln sum_j e^(s_j)) / ln 2,
    i.e. the partial kernel's m + log2(l) with m taken on log2-scaled scores
    (Merge contract section).  An empty key set gives o = 0, lse2 = -inf.
    """
    Hq, Dqk = q_b.shape
    L, Hkv, _ = K.shape
    Dv = V.shape[2]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    o = np.zeros((Hq, Dv), dtype=np.float64)
    lse2 = np.full(Hq, -np.inf, dtype=np.float64)
    if L == 0:
        return o, lse2
    for kv in range(Hkv):
        heads = slice(kv * G, (kv + 1) * G)
        s = sm_scale * (q_b[heads] @ K[:, kv, :].T)          # [G, L]
        mx = s.max(axis=1, keepdims=True)
        e = np.exp(s - mx)
        den = e.sum(axis=1)
        o[heads] = (e @ V[:, kv, :]) / den[:, None]
        lse2[heads] = (mx[:, 0] + np.log(den)) / LN2
    return o, lse2


def workload_arrays(w) -> dict:
    """Plain numpy views of a ``synth.Workload`` (raw bit patterns / codes)."""
    import torch  # only for reading the workload's CPU tensors

    def raw(t):
        if t is None:
            return None
        if t.dtype == torch.bfloat16:
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)
        return t.contiguous().view(torch.uint8).numpy()

    return dict(
        q_raw=raw(w.q), k_raw=raw(w.k_pool), v_raw=raw(w.v_pool), kv_dtype=w.kv_dtype,
        k_scale=w.k_scale, v_scale=w.v_scale, page_indptr=np.asarray(w.page_indptr),
        page_indices=np.asarray(w.page_indices), last_page_len=np.asarray(w.last_page_len),
        page_size=w.page_size, Dv=w.Dv, sm_scale=w.sm_scale, Hq=w.Hq, Hkv=w.Hkv)


def decode_attention(a: dict, requests=None):
    """Flat decode: full softmax attention of every request over all its tokens.

    Returns o [B, Hq, Dv] and lse2 [B, Hq] (rows of requests not listed stay NaN).
    """
    q = bf16_bits_to_f64(a["q_raw"])
    B = len(a["page_indptr"]) - 1
    o = np.full((B, a["Hq"], a["Dv"]), np.nan)
    lse = np.full((B, a["Hq"]), np.nan)
    for b in (range(B) if requests is None else requests):
        K, V = gather_kv(a, b)
        o[b], lse[b] = attend(q[b], K, V, a["sm_scale"])
    return o, lse


def partial_attention(a: dict, chunks):
    """Split-KV partials: attention restricted to each chunk's token range.

    ``chunks`` is a list of (b, token_begin, token_end, out_row) and the result
    rows v_part[out_row] [Hq, Dv], lse_part[out_row] [Hq] follow the Decomposition
    section's per-(request, page tile) partial.  Returns (v_part, lse_part).
    """
    q = bf16_bits_to_f64(a["q_raw"])
    n_rows = 1 + max(c[3] for c in chunks) if chunks else 0
    v_part = np.full((n_rows, a["Hq"], a["Dv"]), np.nan)
    lse_part = np.full((n_rows, a["Hq"]), np.nan)
    cache = {}
    for b, t0, t1, row in chunks:
        if b not in cache:
            cache = {b: gather_kv(a, b)}
        K, V = cache[b]
        v_part[row], lse_part[row] = attend(q[b], K[t0:t1], V[t0:t1], a["sm_scale"])
    return v_part, lse_part


# --------------------------------------------------------------------------- merge
def merge_states(v_in: np.ndarray, lse_in: np.ndarray, o_indptr) -> tuple:
    """Log2-LSE merge of contiguous row groups (Merge contract section).

    For output row r and head h over rows i in [o_indptr[r], o_indptr[r+1]):
        M = max_i lse_i,  w_i = 2^(lse_i - M),
        out = sum_i w_i v_i / sum_i w_i,  lse_out = M + log2 sum_i w_i.
    A one-row group gives w = 1, out = v, lse_out = lse.  A row whose LSE is -inf is
    an empty partial (no tokens): its weight 2^(-inf - M) is zero and its v is not
    used, whatever it holds (the pages define no V for an empty partial).  An empty
    group, or one whose LSEs are all -inf, gives out = 0 and lse_out = -inf (the
    pages leave this open).
    """
    v_in = np.asarray(v_in, dtype=np.float64)
    lse_in = np.asarray(lse_in, dtype=np.float64)
    M = len(o_indptr) - 1
    N, H, D = v_in.shape if v_in.ndim == 3 else (0, lse_in.shape[1], 0)
    out = np.zeros((M, H, v_in.shape[2]), dtype=np.float64)
    lse_out = np.full((M, H), -np.inf, dtype=np.float64)
    for r in range(M):
        lo, hi = int(o_indptr[r]), int(o_indptr[r + 1])
        if hi <= lo:
            continue
        l = lse_in[lo:hi]                                     # [n, H]
        mx = l.max(axis=0)                                    # [H]
        ok = np.isfinite(mx)
        mx_safe = np.where(ok, mx, 0.0)
        w = np.exp2(l - mx_safe)                              # [n, H]
        sw = w.sum(axis=0)
        live = ~np.isneginf(l)                                # empty rows contribute nothing
        acc = np.where(live[:, :, None], w[:, :, None] * np.where(live[:, :, None], v_in[lo:hi], 0.0),
                       0.0).sum(axis=0)
        out[r] = np.where(ok[:, None], acc / np.where(ok, sw, 1.0)[:, None], 0.0)
        lse_out[r] = np.where(ok, mx_safe + np.log2(np.where(ok, sw, 1.0)), -np.inf)
    return out, lse_out


def merge_states_natural_log(v_in, lse_in, o_indptr):
    """The wrong-units merge the Merge contract section warns about: LSEs taken as
    natural logs (w = e^(lse - M)).  Used only as a negative control."""
    v_in = np.asarray(v_in, dtype=np.float64)
    lse_in = np.asarray(lse_in, dtype=np.float64)
    M = len(o_indptr) - 1
    out = np.zeros((M, lse_in.shape[1], v_in.shape[2]))
    for r in range(M):
        lo, hi = int(o_indptr[r]), int(o_indptr[r + 1])
        l = lse_in[lo:hi]
        w = np.exp(l - l.max(axis=0))
        out[r] = (w[:, :, None] * v_in[lo:hi]).sum(axis=0) / w.sum(axis=0)[:, None]
    return out
