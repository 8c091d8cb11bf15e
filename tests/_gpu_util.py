"""Shared helpers for the GPU parity tests: move a seeded workload to the device and
run the library's entry points on it."""
import numpy as np
import torch

import paged_split_kv_decode_gb300 as psd
from oracle import attention as A
from oracle import planner as PL

# Tolerances stated for this path: outputs max-abs 2e-3 (bf16 KV) or 1e-2 (fp8 KV),
# LSE 1e-3 in log2 units, all against the float64 oracle.
OUT_TOL = {"bf16": 2e-3, "fp8_e4m3": 1e-2}
LSE_TOL = 1e-3

_CTX = None


def ctx():
    global _CTX
    if _CTX is None:
        _CTX = psd.Context(0)
    return _CTX


class use_kernel:
    """Selects the partial kernel for few query rows per KV head ('auto' =
    small-group tensor cores, 'cuda_core' = the CUDA-core kernel) for a block."""

    def __init__(self, kind):
        self.kind = kind

    def __enter__(self):
        ctx().set_partial_kernel(self.kind)

    def __exit__(self, *exc):
        ctx().set_partial_kernel("auto")
        return False


class use_level0:
    """Selects the kernel for the stacked level-0 rows of a cascade ('auto',
    'mma_sync' = the 16-row-group tensor-core kernel in the fused launch, 'tcgen05' =
    one CTA per chunk, KV head and 128 rows on the 5th-generation tensor cores)."""

    def __init__(self, kind):
        self.kind = kind

    def __enter__(self):
        ctx().set_level0_kernel(self.kind)

    def __exit__(self, *exc):
        ctx().set_level0_kernel("auto")
        return False


class Dev:
    """Device copies of a synth.Workload."""

    def __init__(self, w, device="cuda"):
        self.w = w
        self.q = w.q.to(device)
        self.k = w.k_pool.to(device)
        self.v = self.k if w.v_pool is None else w.v_pool.to(device)
        self.indices = torch.from_numpy(np.ascontiguousarray(w.page_indices, dtype=np.int32)).to(device)
        self.table = psd.HostTable(w.page_indptr, w.page_indices, w.last_page_len, w.page_size)

    def args(self, q=None, Hkv=None):
        w = self.w
        return psd.decode_args(self.q if q is None else q, self.k, self.v, self.indices,
                               num_pages=w.num_pages, page_size=w.page_size,
                               Hkv=w.Hkv if Hkv is None else Hkv, Dv=w.Dv, sm_scale=w.sm_scale,
                               k_scale=w.k_scale, v_scale=w.v_scale)

    def decode(self, enable, min_shared_pages=None, min_members=None, with_stats=False):
        w = self.w
        plan = psd.plan_decode(self.table, w.tile_tokens, enable,
                               w.min_shared_pages if min_shared_pages is None else min_shared_pages,
                               w.min_members if min_members is None else min_members)
        o = torch.empty((w.batch, w.Hq, w.Dv), dtype=torch.float32, device="cuda")
        lse = torch.empty((w.batch, w.Hq), dtype=torch.float32, device="cuda")
        ws = psd.workspace_for(plan, w.Hq, w.Dv, "cuda")
        stats = psd.cascade_decode(ctx(), self.args(), plan, o, lse, ws)
        assert psd.check_device_error(ctx(), ws) == 0
        out = (o.cpu().double().numpy(), lse.cpu().double().numpy())
        return out + ((stats, plan) if with_stats else ())

    def partials(self):
        w = self.w
        items, o_indptr = psd.split_plan(self.table, w.tile_tokens)
        N = int(o_indptr[-1])
        v = torch.full((N, w.Hq, w.Dv), float("nan"), dtype=torch.float32, device="cuda")
        l = torch.full((N, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
        ws = torch.empty(psd.workspace_bytes(0, len(items), 0, w.Hq, w.Dv), dtype=torch.uint8,
                         device="cuda")
        psd.paged_decode_partial(ctx(), self.args(), items, v, l, ws)
        assert psd.check_device_error(ctx(), ws) == 0
        return v.cpu().double().numpy(), l.cpu().double().numpy(), items, o_indptr


def oracle_partials(w):
    a = A.workload_arrays(w)
    items, o_indptr = PL.split_plan(w.page_indptr, w.last_page_len, w.page_size, w.tile_tokens)
    chunks = [(b, (off - int(w.page_indptr[b])) * w.page_size,
               (off - int(w.page_indptr[b])) * w.page_size + n, row) for b, off, n, row in items]
    v, l = A.partial_attention(a, chunks)
    return v, l, o_indptr


def assert_close(got_o, got_l, ref_o, ref_l, kv_dtype, what=""):
    assert np.isfinite(got_o).all() and np.isfinite(got_l).all(), f"{what}: non-finite output"
    eo = np.abs(got_o - ref_o).max()
    el = np.abs(got_l - ref_l).max()
    assert eo <= OUT_TOL[kv_dtype], f"{what}: out max-abs {eo:.3g} > {OUT_TOL[kv_dtype]}"
    assert el <= LSE_TOL, f"{what}: lse max-abs {el:.3g} > {LSE_TOL}"
    return eo, el
