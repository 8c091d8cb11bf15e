"""Seeded synthetic inputs for paged split-KV decode.

This module only *makes inputs*: random query/key/value values, request lengths,
page tables over a permuted page pool, and merge-kernel partial rows.  It holds no
step of the attention, merge or cascade-planning arithmetic, so the float64 oracle
and the CUDA library can both be fed from it without sharing any of the method.

Every generator takes an integer seed and uses ``numpy.random.default_rng(seed)``.
Value tensors are returned as torch CPU tensors (bf16, or uint8 fp8-e4m3 codes);
page tables are int32 numpy arrays.

Workload shapes follow the decode settings described on the mlxcel PR #1004 page
("compute shared prompt prefixes once per decode batch", sections Summary and
Decomposition) and the MLA shape of the ROCm ATOM PR #1701 page (section 3.2):

* tiny cascade   - 4 requests, Hq=8, Hkv=2, D=64, page 16; requests 0-2 share a
                   4-page prefix, request 3 stands alone; split tile 32 tokens
* flat decode    - 32 requests, Hq=32, Hkv=8, D=128, page 16, lengths U[512,4096]
                   with a partial last page, 16384-page pool; tile 512 tokens
* cascade decode - 64 requests, 16 of them share an 8192-token prefix with private
                   suffixes U[64,1024]; 48 independent requests U[512,4096]
* merge sweep    - H=32, D=128 partial rows, log2 LSE ~ U(-5,20), groups U[1,16]
* MLA decode     - 128 requests, 128 query heads, 1 latent head of 576 (V = first
                   512 columns), page 64, fp8-e4m3 pool with a per-tensor scale,
                   lengths U[4096,32768]; tile 2048 tokens
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0
FP8_E4M3_NAN_CODE = 0x7F


@dataclasses.dataclass
class Workload:
    """One decode batch over a paged KV pool.

    q            [B, Hq, Dqk] bf16
    k_pool       [num_pages, page_size, Hkv, Dqk]  bf16, or uint8 fp8-e4m3 codes
    v_pool       [num_pages, page_size, Hkv, Dv]   bf16 / uint8, or None when V is the
                 first Dv columns of the K rows (a shared MLA latent)
    page_indptr  [B+1] int32, page_indices [nnz] int32, last_page_len [B] int32
    """

    name: str
    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: Optional[torch.Tensor]
    kv_dtype: str  # "bf16" or "fp8_e4m3"
    k_scale: float
    v_scale: float
    page_indptr: np.ndarray
    page_indices: np.ndarray
    last_page_len: np.ndarray
    page_size: int
    num_pages: int
    Hq: int
    Hkv: int
    Dqk: int
    Dv: int
    sm_scale: float
    tile_tokens: int
    lengths: np.ndarray
    min_shared_pages: int = 16
    min_members: int = 2

    @property
    def batch(self) -> int:
        return int(self.page_indptr.shape[0] - 1)

    @property
    def latent_v(self) -> bool:
        return self.v_pool is None

    def kv_bytes_per_token(self) -> int:
        """Bytes of K and V one token carries for all KV heads (unique reads)."""
        esz = 2 if self.kv_dtype == "bf16" else 1
        if self.latent_v:
            return self.Hkv * self.Dqk * esz
        return self.Hkv * (self.Dqk + self.Dv) * esz


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def lengths_with_partial_last_page(rng, n, lo, hi, page_size) -> np.ndarray:
    """Integers uniform in [lo, hi] that are not multiples of page_size."""
    out = np.empty(n, dtype=np.int64)
    for i in range(n):
        while True:
            v = int(rng.integers(lo, hi + 1))
            if v % page_size != 0:
                out[i] = v
                break
    return out


def page_table(lengths: Sequence[int], page_size: int, num_pages: int, rng,
               shared: Optional[tuple] = None):
    """CSR page table for requests of the given token lengths.

    Page ids are handed out request by request from one random permutation of the
    pool.  ``shared = (members, shared_pages)`` makes every listed request reference
    the same first ``shared_pages`` page ids (allocated once), as a refcounted prompt
    prefix would.  Returns (page_indptr, page_indices, last_page_len) as int32.
    """
    lengths = [int(x) for x in lengths]
    B = len(lengths)
    perm = rng.permutation(num_pages).astype(np.int64)
    cursor = 0
    shared_ids = np.empty(0, dtype=np.int64)
    members = set()
    if shared is not None:
        members = set(int(m) for m in shared[0])
        sp = int(shared[1])
        shared_ids = perm[cursor:cursor + sp]
        cursor += sp
    indptr = [0]
    indices = []
    last = []
    for b, L in enumerate(lengths):
        assert L >= 1
        n = (L + page_size - 1) // page_size
        if b in members:
            sp = shared_ids.shape[0]
            assert n > sp
            own = perm[cursor:cursor + (n - sp)]
            cursor += n - sp
            ids = np.concatenate([shared_ids, own])
        else:
            ids = perm[cursor:cursor + n]
            cursor += n
        assert ids.shape[0] == n, "pool too small"
        indices.append(ids)
        indptr.append(indptr[-1] + n)
        last.append(L - (n - 1) * page_size)
    return (np.asarray(indptr, dtype=np.int32),
            np.concatenate(indices).astype(np.int32),
            np.asarray(last, dtype=np.int32))


def page_table_prefixes(lengths: Sequence[int], page_size: int, num_pages: int, rng, prefixes):
    """CSR page table where ``prefixes`` = [(members, n_pages), ...] are shared page
    blocks allocated once each: a request's page list is the blocks of every prefix
    it belongs to, in list order, then its own pages (a system prompt followed by a
    per-tenant sub-prefix, as refcounted prompt blocks would be)."""
    lengths = [int(x) for x in lengths]
    perm = rng.permutation(num_pages).astype(np.int64)
    cursor = 0
    blocks = []
    for members, n in prefixes:
        blocks.append((set(int(m) for m in members), perm[cursor:cursor + int(n)]))
        cursor += int(n)
    indptr, indices, last = [0], [], []
    for b, L in enumerate(lengths):
        n = (L + page_size - 1) // page_size
        pre = [ids for mem, ids in blocks if b in mem]
        pre = np.concatenate(pre) if pre else np.empty(0, dtype=np.int64)
        assert n > pre.shape[0]
        own = perm[cursor:cursor + (n - pre.shape[0])]
        cursor += n - pre.shape[0]
        ids = np.concatenate([pre, own])
        assert ids.shape[0] == n, "pool too small"
        indices.append(ids)
        indptr.append(indptr[-1] + n)
        last.append(L - (n - 1) * page_size)
    return (np.asarray(indptr, dtype=np.int32), np.concatenate(indices).astype(np.int32),
            np.asarray(last, dtype=np.int32))


def _valid_slots(indptr, indices, last, num_pages, page_size) -> np.ndarray:
    """Per pool page: number of leading slots that hold a token (0 if unreferenced)."""
    valid = np.zeros(num_pages, dtype=np.int64)
    B = indptr.shape[0] - 1
    for b in range(B):
        ids = indices[indptr[b]:indptr[b + 1]]
        valid[ids[:-1]] = page_size
        valid[ids[-1]] = max(valid[ids[-1]], int(last[b]))
    return valid


def fill_pool_bf16(rng, num_pages, page_size, Hkv, D, valid, canary: bool) -> torch.Tensor:
    """bf16 pool with N(0,1) values in referenced slots; NaN (or 0) elsewhere."""
    pool = torch.full((num_pages, page_size, Hkv, D),
                      float("nan") if canary else 0.0, dtype=torch.bfloat16)
    mask = torch.from_numpy(np.arange(page_size)[None, :] < valid[:, None])
    count = int(mask.sum())
    vals = rng.standard_normal((count, Hkv, D), dtype=np.float32)
    pool[mask] = _bf16(vals)
    return pool


def fill_pool_fp8(rng, num_pages, page_size, Hkv, D, valid, canary: bool):
    """fp8-e4m3 pool from N(0,1) with one per-tensor scale = amax / 448.

    Codes are produced by torch's round-to-nearest-even float8_e4m3fn cast of
    value / scale.  Returns (uint8 code tensor, scale).
    """
    mask_np = np.arange(page_size)[None, :] < valid[:, None]
    count = int(mask_np.sum())
    vals = rng.standard_normal((count, Hkv, D), dtype=np.float32)
    amax = float(np.abs(vals).max()) if count else 1.0
    scale = amax / 448.0
    codes = torch.from_numpy(vals / np.float32(scale)).to(torch.float8_e4m3fn).view(torch.uint8)
    pool = torch.full((num_pages, page_size, Hkv, D),
                      FP8_E4M3_NAN_CODE if canary else 0, dtype=torch.uint8)
    pool[torch.from_numpy(mask_np)] = codes
    return pool, float(np.float32(scale))


def _make(name, rng, lengths, *, Hq, Hkv, Dqk, Dv, page_size, num_pages, tile_tokens,
          kv_dtype="bf16", latent_v=False, shared=None, canary=True,
          min_shared_pages=16, min_members=2, sm_scale=None, prefixes=None) -> Workload:
    if prefixes is not None:
        indptr, indices, last = page_table_prefixes(lengths, page_size, num_pages, rng, prefixes)
    else:
        indptr, indices, last = page_table(lengths, page_size, num_pages, rng, shared)
    valid = _valid_slots(indptr, indices, last, num_pages, page_size)
    B = len(lengths)
    if kv_dtype == "bf16":
        k_pool = fill_pool_bf16(rng, num_pages, page_size, Hkv, Dqk, valid, canary)
        v_pool = None if latent_v else fill_pool_bf16(rng, num_pages, page_size, Hkv, Dv,
                                                      valid, canary)
        k_scale = v_scale = 1.0
    else:
        k_pool, k_scale = fill_pool_fp8(rng, num_pages, page_size, Hkv, Dqk, valid, canary)
        if latent_v:
            v_pool, v_scale = None, k_scale
        else:
            v_pool, v_scale = fill_pool_fp8(rng, num_pages, page_size, Hkv, Dv, valid, canary)
    q = _bf16(rng.standard_normal((B, Hq, Dqk), dtype=np.float32))
    return Workload(
        name=name, q=q, k_pool=k_pool, v_pool=v_pool, kv_dtype=kv_dtype,
        k_scale=k_scale, v_scale=v_scale, page_indptr=indptr, page_indices=indices,
        last_page_len=last, page_size=page_size, num_pages=num_pages, Hq=Hq, Hkv=Hkv,
        Dqk=Dqk, Dv=Dv,
        sm_scale=float(1.0 / math.sqrt(Dqk)) if sm_scale is None else float(sm_scale),
        tile_tokens=tile_tokens, lengths=np.asarray(lengths, dtype=np.int64),
        min_shared_pages=min_shared_pages, min_members=min_members)


def tiny_cascade(seed: int = 0, canary: bool = True) -> Workload:
    """4 requests; 0-2 share a 64-token (4-page) prefix plus private suffixes of
    32-80 tokens; request 3 is a standalone 96 tokens.  Hq=8, Hkv=2, D=64."""
    rng = np.random.default_rng(seed)
    P, shared_pages = 16, 4
    suffix = [int(rng.integers(32, 81)) for _ in range(3)]
    lengths = [shared_pages * P + s for s in suffix] + [96]
    return _make("tiny_cascade", rng, lengths, Hq=8, Hkv=2, Dqk=64, Dv=64, page_size=P,
                 num_pages=64, tile_tokens=2 * P, shared=([0, 1, 2], shared_pages),
                 canary=canary, min_shared_pages=4, min_members=2)


def flat_decode(seed: int = 0, canary: bool = True, batch: int = 32, num_pages: int = 16384) -> Workload:
    """32 requests, Hq=32, Hkv=8, D=128, page 16, lengths U[512,4096] with a partial
    last page, random permutation of a 16384-page pool, tile 512 tokens."""
    rng = np.random.default_rng(seed)
    P = 16
    lengths = lengths_with_partial_last_page(rng, batch, 512, 4096, P)
    return _make("flat_decode", rng, lengths, Hq=32, Hkv=8, Dqk=128, Dv=128, page_size=P,
                 num_pages=num_pages, tile_tokens=512, canary=canary)


def cascade_decode(seed: int = 0, canary: bool = True, members: int = 16,
                   others: int = 48, shared_tokens: int = 8192) -> Workload:
    """64 requests, Hq=32, Hkv=8, D=128, page 16.  The first ``members`` requests
    share an 8192-token (512-page) prefix and add private suffixes U[64,1024];
    the other 48 have independent lengths U[512,4096].  16384-page pool."""
    rng = np.random.default_rng(seed)
    P = 16
    shared_pages = shared_tokens // P
    suffix = rng.integers(64, 1025, size=members)
    own = rng.integers(512, 4097, size=others)
    lengths = [shared_tokens + int(s) for s in suffix] + [int(x) for x in own]
    # interleave members and non-members by a seeded shuffle of batch positions
    order = rng.permutation(len(lengths))
    lengths = [lengths[i] for i in order]
    member_ids = sorted(int(np.where(order == i)[0][0]) for i in range(members))
    return _make("cascade_decode", rng, lengths, Hq=32, Hkv=8, Dqk=128, Dv=128,
                 page_size=P, num_pages=16384, tile_tokens=512,
                 shared=(member_ids, shared_pages), canary=canary)


def nested_decode(seed: int = 0, canary: bool = True, tenants: Sequence[int] = (8, 8),
                  system_tokens: int = 4096, tenant_tokens: int = 2048, others: int = 16,
                  page_size: int = 16, num_pages: int = 16384) -> Workload:
    """A system prompt shared by every tenant's requests, one sub-prefix per tenant,
    private suffixes U[64,1024]; plus independent requests U[512,4096].  Hq=32,
    Hkv=8, D=128, tile 512 (the flat-decode heads).  Batch positions are shuffled."""
    rng = np.random.default_rng(seed)
    P = page_size
    n_mem = int(sum(tenants))
    suffix = rng.integers(64, 1025, size=n_mem)
    own = rng.integers(512, 4097, size=others)
    lengths = [system_tokens + tenant_tokens + int(x) for x in suffix] + [int(x) for x in own]
    order = rng.permutation(len(lengths))
    lengths = [lengths[i] for i in order]
    pos = {int(order[j]): j for j in range(len(order))}           # original index -> batch slot
    members = [pos[i] for i in range(n_mem)]
    groups, k = [], 0
    for t in tenants:
        groups.append(members[k:k + int(t)])
        k += int(t)
    prefixes = [(members, system_tokens // P)] + [(g, tenant_tokens // P) for g in groups]
    return _make("nested_decode", rng, lengths, Hq=32, Hkv=8, Dqk=128, Dv=128, page_size=P,
                 num_pages=num_pages, tile_tokens=512, canary=canary, prefixes=prefixes)


def mla_decode(seed: int = 0, canary: bool = True, batch: int = 128,
               lo: int = 4096, hi: int = 32768, num_pages: int = 65536) -> Workload:
    """128 requests, 128 query heads over 1 latent KV head of 576 columns
    (512 + 64); V is the first 512 columns of the same rows.  Page 64, fp8-e4m3
    pool with a per-tensor scale, lengths U[4096,32768], tile 2048 tokens."""
    rng = np.random.default_rng(seed)
    P = 64
    lengths = rng.integers(lo, hi + 1, size=batch)
    return _make("mla_decode", rng, lengths, Hq=128, Hkv=1, Dqk=576, Dv=512, page_size=P,
                 num_pages=num_pages, tile_tokens=2048, kv_dtype="fp8_e4m3",
                 latent_v=True, canary=canary)


def merge_groups(rng, num_out: int, lo: int = 1, hi: int = 16) -> np.ndarray:
    """o_indptr [num_out+1] with group sizes uniform in [lo, hi]; group 0 is forced
    to a single row so every sweep holds a group of one."""
    sizes = rng.integers(lo, hi + 1, size=num_out)
    if num_out:
        sizes[0] = 1
    indptr = np.zeros(num_out + 1, dtype=np.int64)
    np.cumsum(sizes, out=indptr[1:])
    assert indptr[-1] < 2 ** 31
    return indptr.astype(np.int32)


def merge_inputs(seed: int, num_out: int, H: int = 32, D: int = 128):
    """Host merge inputs: v_in f32 N(0,1) [N,H,D], lse_in log2 ~ U(-5,20) [N,H]."""
    rng = np.random.default_rng(seed)
    o_indptr = merge_groups(rng, num_out)
    N = int(o_indptr[-1])
    v_in = torch.from_numpy(rng.standard_normal((N, H, D), dtype=np.float32))
    lse_in = torch.from_numpy(rng.uniform(-5.0, 20.0, size=(N, H)).astype(np.float32))
    return v_in, lse_in, o_indptr


def merge_inputs_device(seed: int, num_out: int, H: int = 32, D: int = 128,
                        device="cuda"):
    """Large merge inputs drawn on the device by torch's seeded generator (host RAM
    cannot hold the 1M-row case).  Group sizes still come from numpy."""
    rng = np.random.default_rng(seed)
    o_indptr = merge_groups(rng, num_out)
    N = int(o_indptr[-1])
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    v_in = torch.randn((N, H, D), generator=g, device=device, dtype=torch.float32)
    lse_in = torch.rand((N, H), generator=g, device=device, dtype=torch.float32) * 25.0 - 5.0
    return v_in, lse_in, o_indptr


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU tensor as uint16."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def u8_codes(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy()


# ------------------------------------------------------------- RoPE + KV append
def rope_cos_sin_table(max_position: int, rot_dim: int, base: float = 10000.0) -> np.ndarray:
    """Caller data for the append step: cos_sin[p] = [cos p*theta_i .. , sin p*theta_i ..]
    with theta_i = base^(-2i/rot_dim), i < rot_dim/2 (the common rotary schedule; the
    append step itself only reads the table), float32 [max_position, rot_dim]."""
    i = np.arange(rot_dim // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / rot_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * theta[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


@dataclasses.dataclass
class AppendStep:
    """The new tokens of one decode step and the pool they are appended to.

    q [T, Hq, Dq] bf16; k_nope [T, Hkv, Dn] bf16 or None; k_rope [T, Hkv, Dr] bf16;
    v [T, Hkv, Dv] bf16 or None (latent: V lives in the K row); positions [T] int32;
    slot_mapping [T] int32 (page * page_size + slot, negative = skip); pools as in
    Workload (bf16, or uint8 fp8-e4m3 codes), filled with NaN canaries."""

    name: str
    q: torch.Tensor
    k_nope: Optional[torch.Tensor]
    k_rope: torch.Tensor
    v: Optional[torch.Tensor]
    positions: np.ndarray
    slot_mapping: np.ndarray
    cos_sin: np.ndarray
    rot_dim: int
    neox: bool
    q_rope_col: int
    k_pool: torch.Tensor
    v_pool: Optional[torch.Tensor]
    page_size: int
    kv_dtype: str
    k_scale: float
    v_scale: float


def append_step(seed: int = 0, kind: str = "gqa", T: int = 32, kv_dtype: str = "bf16", neox: bool = True,
                skip_every: int = 0, num_pages: int = 512, max_position: int = 32768) -> AppendStep:
    """One decode step's append for T requests.

    gqa: Hq=32, Hkv=8, D=128, full rotary (rot_dim 128), separate K and V pools,
         page 16 (the flat-decode shape).
    mla: 128 query heads of 576 whose last 64 columns are roped; the K row is the
         512-column latent followed by a 64-column roped part; no V pool, page 64
         (the MLA-decode shape).
    Each request appends one token at a random position at its own page slot (a
    permutation of the pool's slots); with skip_every > 0 every skip_every-th token
    has slot -1 (owned by another rank)."""
    rng = np.random.default_rng(seed)
    if kind == "gqa":
        Hq, Hkv, Dq, Dn, Dr, Dv, P, rot, qcol = 32, 8, 128, 0, 128, 128, 16, 128, 0
    elif kind == "mla":
        Hq, Hkv, Dq, Dn, Dr, Dv, P, rot, qcol = 128, 1, 576, 512, 64, 0, 64, 64, 512
    else:
        raise ValueError(kind)
    q = _bf16(rng.standard_normal((T, Hq, Dq)))
    k_nope = _bf16(rng.standard_normal((T, Hkv, Dn))) if Dn else None
    k_rope = _bf16(rng.standard_normal((T, Hkv, Dr)))
    v = _bf16(rng.standard_normal((T, Hkv, Dv))) if Dv else None
    positions = rng.integers(0, max_position, size=T).astype(np.int32)
    slots = rng.choice(num_pages * P, size=T, replace=False).astype(np.int32)
    if skip_every:
        slots[::skip_every] = -1
    Dk = Dn + Dr
    if kv_dtype == "bf16":
        k_pool = torch.full((num_pages, P, Hkv, Dk), 0, dtype=torch.int16).view(torch.bfloat16)
        k_pool.view(torch.int16).fill_(np.int16(BF16_NAN_BITS))
        v_pool = None
        if Dv:
            v_pool = torch.empty((num_pages, P, Hkv, Dv), dtype=torch.bfloat16)
            v_pool.view(torch.int16).fill_(np.int16(BF16_NAN_BITS))
    else:
        k_pool = torch.full((num_pages, P, Hkv, Dk), FP8_E4M3_NAN_CODE, dtype=torch.uint8)
        v_pool = torch.full((num_pages, P, Hkv, Dv), FP8_E4M3_NAN_CODE, dtype=torch.uint8) if Dv else None
    # per-tensor scales in the usual amax / 448 form over the new values
    ks = float(max(np.abs(k_rope.float().numpy()).max(),
                   np.abs(k_nope.float().numpy()).max() if k_nope is not None else 0.0) / 448.0 * 1.25)
    vs = float(np.abs(v.float().numpy()).max() / 448.0 * 1.25) if v is not None else 1.0
    return AppendStep(f"append_{kind}_{kv_dtype}", q, k_nope, k_rope, v, positions, slots,
                      rope_cos_sin_table(max_position, rot), rot, neox, qcol, k_pool, v_pool, P, kv_dtype,
                      ks if kv_dtype != "bf16" else 1.0, vs if kv_dtype != "bf16" else 1.0)
