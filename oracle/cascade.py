"""The two-level cascade evaluated level by level in float64 (oracle; test
infrastructure only).

Source: mlxcel PR #1004, "compute shared prompt prefixes once per decode batch",
Decomposition and Task item 2: level 0 attends the shared span once as one request
whose M*G query heads per KV head are stacked KV-head-major; level 1 attends every
request's remaining pages; each member's two states are merged by the log2-LSE
merge, and a non-member's single level-1 state passes through a group of one.

The cascade result is, by the page's own statement, the flat result up to
rounding; ``attention.decode_attention`` is the reference.  This module rebuilds the
levels independently so tests can check the invariants (disjoint-range merge,
conservation of pages, the stacking negative control) and localise a failure.
"""
from __future__ import annotations

import numpy as np

from . import attention as A
from . import planner as PL


def stack_queries(q: np.ndarray, members, Hkv: int, member_major: bool = False):
    """Level-0 query rows [Hkv*M*G, D] from q [B, Hq, D].

    KV-head-major (the page's rule): row kv*(M*G) + m*G + g = q[members[m], kv*G+g],
    a [M, Hkv, G, D] -> [Hkv, M, G, D] transpose.  ``member_major=True`` builds the
    wrong order m*(Hkv*G) + kv*G + g for the negative control.
    """
    B, Hq, D = q.shape
    G = Hq // Hkv
    M = len(members)
    q0 = np.empty((Hkv * M * G, D), dtype=q.dtype)
    for kv in range(Hkv):
        for m, b in enumerate(members):
            for g in range(G):
                h0 = (PL.member_major_head(kv, m, g, Hkv, G) if member_major
                      else PL.stacked_head(kv, m, g, M, G))
                q0[h0] = q[b, kv * G + g]
    return q0


def level0_partials(a: dict, members, shared_pages: int, tile_tokens: int,
                    member_major: bool = False):
    """Level-0 partials: the span's tokens of the first member (the same physical
    pages for every member) attended by the stacked queries, per T-token chunk.
    Returns v0 [C0, Hkv*M*G, Dv], lse0 [C0, Hkv*M*G]."""
    q = A.bf16_bits_to_f64(a["q_raw"])
    q0 = stack_queries(q, members, a["Hkv"], member_major)
    K, V = A.gather_kv(a, members[0])
    span_tokens = shared_pages * a["page_size"]
    ch = PL.chunks_of(span_tokens, tile_tokens)
    v0 = np.empty((len(ch), q0.shape[0], a["Dv"]))
    lse0 = np.empty((len(ch), q0.shape[0]))
    for c, (t0, t1) in enumerate(ch):
        v0[c], lse0[c] = A.attend(q0, K[t0:t1], V[t0:t1], a["sm_scale"])
    return v0, lse0


def unstack(v0: np.ndarray, lse0: np.ndarray, M: int, Hkv: int, G: int):
    """Inverse of the KV-head-major stacking: [C0, Hkv*M*G, .] -> [M, C0, Hq, .]."""
    C0 = v0.shape[0]
    Hq = Hkv * G
    vo = np.empty((M, C0, Hq, v0.shape[2]))
    lo = np.empty((M, C0, Hq))
    for kv in range(Hkv):
        for m in range(M):
            for g in range(G):
                h0 = PL.stacked_head(kv, m, g, M, G)
                vo[m, :, kv * G + g] = v0[:, h0]
                lo[m, :, kv * G + g] = lse0[:, h0]
    return vo, lo


def cascade_levels(a: dict, plan: dict, tile_tokens: int):
    """Run level 0, level 1 and the final merge from ``planner.plan_decode`` output.

    Returns (o [B, Hq, Dv], lse [B, Hq], v_part, lse_part) where the partial buffers
    are laid out by the plan's composite o_indptr.
    """
    q = A.bf16_bits_to_f64(a["q_raw"])
    B = len(a["page_indptr"]) - 1
    Hq, Dv, P = a["Hq"], a["Dv"], a["page_size"]
    G = Hq // a["Hkv"]
    members = plan["members"]
    N = plan["num_rows"]
    v_part = np.full((N, Hq, Dv), np.nan)
    lse_part = np.full((N, Hq), np.nan)
    if members:
        v0, lse0 = level0_partials(a, members, plan["shared_pages"], tile_tokens)
        vo, lo = unstack(v0, lse0, len(members), a["Hkv"], G)
        for m in range(len(members)):
            base = plan["member_row_base"][m]
            v_part[base:base + vo.shape[1]] = vo[m]
            lse_part[base:base + vo.shape[1]] = lo[m]
    cache = {}
    for b, page_off, n_tok, row in plan["l1_items"]:
        if b not in cache:
            cache = {b: A.gather_kv(a, b)}
        K, V = cache[b]
        t0 = (page_off - int(a["page_indptr"][b])) * P
        v_part[row], lse_part[row] = A.attend(q[b], K[t0:t0 + n_tok], V[t0:t0 + n_tok],
                                              a["sm_scale"])
    o, lse = A.merge_states(v_part, lse_part, plan["o_indptr"])
    return o, lse, v_part, lse_part
