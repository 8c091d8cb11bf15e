"""RoPE + KV append into the paged pool (oracle; test infrastructure only).

Source: ROCm ATOM PR #1701.
  * Sections 1 and 3.3 (the fused RoPE kernel that also ropes every query): one
    fused kernel applies RoPE to every query and to the new token's rope part of K,
    joins the non-rope latent with the roped part, and writes the row into the KV
    cache only for the slots this rank owns.
  * Section 3.2: fp8 KV is stored as codes that dequantise as code * k_scale.
mlxcel PR #1004, Left out / unsure: fused RoPE + KV-append decode kernels (#905) are
the step before this path.

The pages fix no formula beyond that, so these are the readings (each listed in the
design notes):
  * RoPE rotates pairs of elements by position * theta_i, with cos and sin taken from a
    caller table cos_sin[pos] = [cos theta_0 .. cos theta_{r/2-1}, sin theta_0 ..
    sin theta_{r/2-1}] (so the frequency base and any scaling are the caller's), on
    the first `rot_dim` columns of the rope part.  Pairs are (i, i + r/2) ("neox") or
    (2i, 2i + 1) (interleaved); both are supported.
  * The rotation runs in float32 with each product rounded: x' = x c - y s and
    y' = y c + x s.  Outputs are rounded to nearest even: bf16 for q and bf16 pools,
    OCP E4M3FN for fp8 pools with saturation to +-448 of x / scale.  Those roundings
    decide integers (bit patterns), so the oracle takes them in the same float32
    precision as the kernel; tests pin the float32 rotation to the exact float64
    rotation separately.
  * slot_mapping[t] = page * page_size + slot; a negative slot skips token t's KV
    write (a slot owned by another rank, or padding); queries are roped for every t.
"""
from __future__ import annotations

import numpy as np

from .attention import e4m3_to_f64

E4M3_MAX = 448.0


# ---------------------------------------------------------------- rounding steps
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bit patterns, to nearest with ties to even.

    bf16 keeps the top 16 bits of the float32 pattern; the discarded low half is
    compared with its midpoint 0x8000, and a tie keeps the even top half.  NaN stays
    a quiet NaN with its sign."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    top, low = u >> 16, u & 0xFFFF
    up = (low > 0x8000) | ((low == 0x8000) & ((top & 1) == 1))
    r = (top + up.astype(np.uint64)) & 0xFFFF
    nan = np.isnan(x)
    r = np.where(nan, (top & 0x8000) | 0x7FC0, r)
    return r.astype(np.uint16)


def _e4m3_table():
    codes = np.arange(0x80, dtype=np.int64)            # non-negative codes
    vals = e4m3_to_f64(codes)
    finite = ~np.isnan(vals)
    return codes[finite], vals[finite]                # ascending values 0 .. 448


_E4M3_CODES, _E4M3_VALS = _e4m3_table()


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """OCP E4M3FN codes of x: nearest representable value, ties to the even code
    (even mantissa), magnitudes above 448 saturate to 448, NaN -> 0x7F with the
    sign bit of x.  The sign is kept for zero and for values that round to zero."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64) << 7
    a = np.minimum(np.abs(x), E4M3_MAX)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    hi = np.searchsorted(_E4M3_VALS, a, side="left")       # first value >= a
    hi = np.clip(hi, 0, len(_E4M3_VALS) - 1)
    lo = np.clip(hi - 1, 0, len(_E4M3_VALS) - 1)
    vh, vl = _E4M3_VALS[hi], _E4M3_VALS[lo]
    ch, cl = _E4M3_CODES[hi], _E4M3_CODES[lo]
    dh, dl = vh - a, a - vl
    pick_hi = (dh < dl) | ((dh == dl) & ((ch & 1) == 0))
    exact = vh == a
    code = np.where(exact | pick_hi, ch, cl)
    code = np.where(nan, 0x7F, code)
    return (code | sign).astype(np.uint8)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ------------------------------------------------------------------------ RoPE
def rope_pair_index(rot_dim: int, neox: bool):
    """(first, second) element index of each of the rot_dim/2 pairs; pair i uses
    frequency i."""
    h = rot_dim // 2
    i = np.arange(h)
    return (i, i + h) if neox else (2 * i, 2 * i + 1)


def rope_f32(v: np.ndarray, pos: np.ndarray, cos_sin: np.ndarray, rot_dim: int, neox: bool) -> np.ndarray:
    """Rotate the first rot_dim columns of v [..., n, D] (float32) by the angles of
    positions pos [...] (one per leading index), in float32 with each product
    rounded; columns from rot_dim on are returned unchanged."""
    v = np.array(v, dtype=np.float32, copy=True)
    h = rot_dim // 2
    a, b = rope_pair_index(rot_dim, neox)
    cs = cos_sin[pos].astype(np.float32)                 # [..., rot_dim]
    c = cs[..., None, :h]
    s = cs[..., None, h:rot_dim]
    x = v[..., a].copy()
    y = v[..., b].copy()
    xc = (x * c).astype(np.float32)
    ys = (y * s).astype(np.float32)
    yc = (y * c).astype(np.float32)
    xs = (x * s).astype(np.float32)
    v[..., a] = (xc - ys).astype(np.float32)
    v[..., b] = (yc + xs).astype(np.float32)
    return v


def rope_f64(v: np.ndarray, angles: np.ndarray, rot_dim: int, neox: bool) -> np.ndarray:
    """The exact rotation in float64: pair i of v turned by angles[..., i]."""
    v = np.array(v, dtype=np.float64, copy=True)
    a, b = rope_pair_index(rot_dim, neox)
    c, s = np.cos(angles)[..., None, :], np.sin(angles)[..., None, :]
    x, y = v[..., a].copy(), v[..., b].copy()
    v[..., a] = x * c - y * s
    v[..., b] = y * c + x * s
    return v


# ---------------------------------------------------------------- the full op
def store(values_f32: np.ndarray, kv_dtype: str, scale: float) -> np.ndarray:
    """Pool codes of float32 values: bf16 bits, or E4M3 codes of x / scale (the
    division rounded to float32 first, as the kernel does)."""
    if kv_dtype == "bf16":
        return f32_to_bf16_bits(values_f32)
    if kv_dtype == "fp8_e4m3":
        q = (np.asarray(values_f32, dtype=np.float32) / np.float32(scale)).astype(np.float32)
        return encode_e4m3(q.astype(np.float64))
    raise ValueError(kv_dtype)


def rope_append(q_bits, k_nope_bits, k_rope_bits, v_bits, cos_sin, positions, slot_mapping, *,
                rot_dim: int, neox: bool, q_rope_col: int, k_pool, v_pool, page_size: int,
                kv_dtype: str, k_scale: float = 1.0, v_scale: float = 1.0):
    """The fused step for T new tokens.

    q_bits [T, Hq, Dq] bf16: columns [q_rope_col, q_rope_col + rot_dim) of every head
    are roped (every token).  For each token with slot_mapping[t] >= 0, the K row
    [k_nope | rope(k_rope)] of every KV head and (when given) the V row are stored at
    k_pool[page, slot] / v_pool[page, slot].  Returns new (q_bits, k_pool, v_pool)."""
    pos = np.asarray(positions, dtype=np.int64)
    q = bf16_bits_to_f32(q_bits)
    qr = rope_f32(q[..., q_rope_col:q_rope_col + rot_dim], pos, cos_sin, rot_dim, neox)
    q_out = np.array(q_bits, copy=True)
    q_out[..., q_rope_col:q_rope_col + rot_dim] = f32_to_bf16_bits(qr)

    kr = rope_f32(bf16_bits_to_f32(k_rope_bits), pos, cos_sin, rot_dim, neox)
    parts = [kr] if k_nope_bits is None else [bf16_bits_to_f32(k_nope_bits), kr]
    k_row = np.concatenate(parts, axis=-1)                # [T, Hkv, Dn + Dr] float32
    k_codes = store(k_row, kv_dtype, k_scale)
    k_out = np.array(k_pool, copy=True)
    v_out = None if v_pool is None else np.array(v_pool, copy=True)
    v_codes = None if v_bits is None else store(bf16_bits_to_f32(v_bits), kv_dtype, v_scale)
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0:
            continue
        page, slot = divmod(int(s), page_size)
        k_out[page, slot] = k_codes[t]
        if v_out is not None:
            v_out[page, slot] = v_codes[t]
    return q_out, k_out, v_out
