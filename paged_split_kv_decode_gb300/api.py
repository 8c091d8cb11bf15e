"""Thin Python binding over the C ABI (include/psd.h).

The functions keep the C names and only marshal arguments: torch tensors become
device pointers, numpy int32 arrays become host pointers, the current torch stream
becomes the CUDA stream.  Every step of the decode path (planning included) runs in
``libpsd.so``; nothing here computes any part of it.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np
import torch

from . import _lib as L


def _ptr_i32(a: np.ndarray):
    return a.ctypes.data_as(L.P_i32)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# The current stream's raw handle without building a torch.cuda.Stream object (that
# costs about 3 us a call on a Grace host, the getter below about 0.4 us).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> C.c_void_p:
    if stream is None:
        if _raw_stream is not None:
            return C.c_void_p(_raw_stream(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return C.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _dev_ptr(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _dev_or_pinned_ptr(t: torch.Tensor, name: str) -> int:
    """A CUDA tensor, or a pinned host tensor the kernels reach over the host link
    (the pointer is the same on both sides)."""
    if isinstance(t, torch.Tensor) and t.is_cuda:
        return _dev_ptr(t, name)
    if isinstance(t, torch.Tensor) and t.device.type == "cpu" and t.is_pinned():
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t.data_ptr()
    return _dev_ptr(t, name)


def _out_ptr(t: torch.Tensor, name: str) -> int:
    """Decode outputs may be pinned host tensors: the merge kernel then stores them
    into host memory directly."""
    return _dev_or_pinned_ptr(t, name)


def kv_dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return L.PSD_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return L.PSD_FP8_E4M3
    raise ValueError(f"unsupported KV dtype {t.dtype}")


class Context:
    """A psd_ctx bound to one CUDA device."""

    def __init__(self, device=None):
        lib = L.load()
        dev = torch.cuda.current_device() if device is None else int(device)
        self._h = C.c_void_p()
        L.check(lib.psd_create(C.byref(self._h), dev))
        self.device = dev

    @property
    def handle(self):
        return self._h

    def set_partial_kernel(self, kind: str):
        """psd_set_partial_kernel: 'auto', 'cuda_core' or 'tensor_core'."""
        code = {"auto": L.PSD_KERNEL_AUTO, "cuda_core": L.PSD_KERNEL_CUDA_CORE,
                "tensor_core": L.PSD_KERNEL_TENSOR_CORE}[kind]
        L.check(L.load().psd_set_partial_kernel(self._h, code))

    def set_level0_kernel(self, kind: str):
        """psd_set_level0_kernel: 'auto', 'mma_sync' or 'tcgen05' for the stacked
        level-0 rows of a cascade."""
        code = {"auto": 0, "mma_sync": 1, "tcgen05": 2}[kind]
        L.check(L.load().psd_set_level0_kernel(self._h, code))

    def test_withhold_loads(self, from_tile: int, wait_limit_cycles: int = 0):
        """psd_test_withhold_loads: a testing aid that makes the partial kernels' waits
        for an item's tiles from `from_tile` on run out, and the streaming merge's waits
        for a CTA's input rows from that index on (from_tile < 0 switches it off)."""
        L.check(L.load().psd_test_withhold_loads(self._h, int(from_tile), int(wait_limit_cycles)))

    def set_timing(self, enable: bool = True):
        """psd_set_timing: CUDA events around every kernel the library launches."""
        L.check(L.load().psd_set_timing(self._h, int(bool(enable))))

    def kernel_times(self) -> dict:
        """psd_get_kernel_times of the most recent call, in milliseconds."""
        a, b, c = C.c_float(), C.c_float(), C.c_float()
        L.check(L.load().psd_get_kernel_times(self._h, C.byref(a), C.byref(b), C.byref(c)))
        return {"level0_ms": a.value, "partial_ms": b.value, "merge_ms": c.value}

    def autotune_tile(self, args: L.DecodeArgs, table: "HostTable", tiles, o: torch.Tensor, lse: torch.Tensor,
                      workspace: torch.Tensor, enable: int = 1, min_shared_pages: int = 16, min_members: int = 2,
                      reps: int = 5, stream=None):
        """psd_autotune_tile: times cascade_decode per candidate tile (cold L2) and
        records the fastest for this shape bucket.  Returns (best_tile, [mean ms])."""
        t = np.ascontiguousarray(tiles, dtype=np.int32)
        ms = (C.c_float * len(t))()
        best = C.c_int32()
        L.check(L.load().psd_autotune_tile(
            self._h, C.byref(args), C.byref(table.c), t.ctypes.data_as(L.P_i32), len(t), int(enable),
            int(min_shared_pages), int(min_members), int(reps), _dev_ptr(o, "o"), _dev_ptr(lse, "lse"),
            _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream),
            C.byref(best), ms))
        return best.value, [float(x) for x in ms]

    def tuned_tile(self, args: L.DecodeArgs, table: "HostTable", default_tile: int, enable: int = 1,
                   min_shared_pages: int = 16, min_members: int = 2) -> int:
        """psd_tuned_tile: the tile recorded for this batch's shape bucket, else default_tile."""
        return int(L.load().psd_tuned_tile(self._h, C.byref(args), C.byref(table.c), int(enable),
                                           int(min_shared_pages), int(min_members), int(default_tile)))

    def counters(self) -> dict:
        c = L.Counters()
        L.check(L.load().psd_get_counters(self._h, C.byref(c)))
        return {k: getattr(c, k) for k, _ in L.Counters._fields_}

    def close(self):
        if self._h:
            L.load().psd_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostTable:
    """A host CSR page table kept alive for the C ABI."""

    def __init__(self, page_indptr, page_indices, last_page_len, page_size: int):
        self.indptr = _i32(page_indptr)
        self.indices = _i32(page_indices)
        self.last = _i32(last_page_len)
        self.page_size = int(page_size)
        self.c = L.PageTable(_ptr_i32(self.indptr), _ptr_i32(self.indices), _ptr_i32(self.last),
                             int(self.indptr.shape[0] - 1), self.page_size)

    @property
    def batch(self):
        return int(self.indptr.shape[0] - 1)

    @property
    def nnz(self):
        return int(self.indptr[-1])


def split_plan(table: HostTable, tile_tokens: int):
    """psd_split_plan: flat work list -> (items [n, 4] int32, o_indptr [B+1])."""
    lib = L.load()
    cap = max(table.nnz, 1)
    items = (L.WorkItem * cap)()
    n = C.c_int32()
    o_indptr = np.zeros(table.batch + 1, dtype=np.int32)
    L.check(lib.psd_split_plan(C.byref(table.c), int(tile_tokens), items, cap, C.byref(n),
                               _ptr_i32(o_indptr)))
    arr = np.ctypeslib.as_array(C.cast(items, L.P_i32), shape=(cap * 4,)).reshape(cap, 4)
    return arr[: n.value].copy(), o_indptr


def detect_shared_prefix(table: HostTable, min_shared_pages: int = 16, min_members: int = 2):
    """detect_shared_prefix -> (members list, shared_pages, decline_reason)."""
    lib = L.load()
    members = np.zeros(max(table.batch, 1), dtype=np.int32)
    nm, sp, reason = C.c_int32(), C.c_int32(), C.c_int32()
    L.check(lib.detect_shared_prefix(C.byref(table.c), int(min_shared_pages), int(min_members),
                                     _ptr_i32(members), C.byref(nm), C.byref(sp), C.byref(reason)))
    return [int(x) for x in members[: nm.value]], int(sp.value), int(reason.value)


class Plan:
    """A psd_cascade_plan with caller-owned (numpy) arrays."""

    def __init__(self, table: HostTable):
        self.table = table
        bc, ic = C.c_int32(), C.c_int32()
        L.check(L.load().psd_plan_capacity(C.byref(table.c), C.byref(bc), C.byref(ic)))
        self.members_a = np.zeros(bc.value, dtype=np.int32)
        self.row_base_a = np.zeros(bc.value, dtype=np.int32)
        self.o_indptr_a = np.zeros(bc.value + 1, dtype=np.int32)
        self.l0 = (L.WorkItem * ic.value)()
        self.l1 = (L.WorkItem * ic.value)()
        self.c = L.CascadePlan()
        self.c.batch_capacity = bc.value
        self.c.item_capacity = ic.value
        self.c.members = _ptr_i32(self.members_a)
        self.c.member_row_base = _ptr_i32(self.row_base_a)
        self.c.l0_items = self.l0
        self.c.l1_items = self.l1
        self.c.o_indptr = _ptr_i32(self.o_indptr_a)

    def _items(self, arr, n):
        cap = self.c.item_capacity
        a = np.ctypeslib.as_array(C.cast(arr, L.P_i32), shape=(cap * 4,)).reshape(cap, 4)
        return a[:n].copy()

    @property
    def members(self):
        return [int(x) for x in self.members_a[: self.c.num_members]]

    @property
    def member_row_base(self):
        return [int(x) for x in self.row_base_a[: self.c.num_members]]

    @property
    def o_indptr(self):
        return [int(x) for x in self.o_indptr_a[: self.c.batch + 1]]

    @property
    def l0_items(self):
        return self._items(self.l0, self.c.l0_num_items)

    @property
    def l1_items(self):
        return self._items(self.l1, self.c.l1_num_items)

    @property
    def num_items(self):
        return self.c.l0_num_items + self.c.l1_num_items

    def __getattr__(self, name):
        if name in ("num_members", "shared_pages", "decline_reason", "num_rows", "tile_tokens",
                    "batch", "page_size", "l0_num_items", "l1_num_items"):
            return getattr(self.c, name)
        raise AttributeError(name)


class CachedPlan:
    """A plan owned by a PlanCache (a view of its psd_cascade_plan); valid until the
    next lookup on that cache.  Same read accessors as Plan."""

    def __init__(self, ptr, hit: bool):
        self.c = ptr.contents
        self.hit = hit

    def _i32(self, p, n):
        return [int(x) for x in np.ctypeslib.as_array(C.cast(p, L.P_i32), shape=(max(n, 1),))[:n]]

    @property
    def members(self):
        return self._i32(self.c.members, self.c.num_members)

    @property
    def member_row_base(self):
        return self._i32(self.c.member_row_base, self.c.num_members)

    @property
    def o_indptr(self):
        return self._i32(self.c.o_indptr, self.c.batch + 1)

    def _items(self, arr, n):
        if n == 0:
            return np.zeros((0, 4), dtype=np.int32)
        return np.ctypeslib.as_array(C.cast(arr, L.P_i32), shape=(n * 4,)).reshape(n, 4).copy()

    @property
    def l0_items(self):
        return self._items(self.c.l0_items, self.c.l0_num_items)

    @property
    def l1_items(self):
        return self._items(self.c.l1_items, self.c.l1_num_items)

    @property
    def num_items(self):
        return self.c.l0_num_items + self.c.l1_num_items

    def __getattr__(self, name):
        if name in ("num_members", "shared_pages", "decline_reason", "num_rows", "tile_tokens",
                    "batch", "page_size", "l0_num_items", "l1_num_items"):
            return getattr(self.c, name)
        raise AttributeError(name)


class PlanCache:
    """psd_plan_cache: plans memoised by page-table contents and KV lengths."""

    def __init__(self, capacity: int = 8):
        self._h = C.c_void_p()
        L.check(L.load().psd_plan_cache_create(C.byref(self._h), int(capacity)))

    def lookup(self, table: HostTable, tile_tokens: int, enable: int = 1, min_shared_pages: int = 16,
               min_members: int = 2, generation: int = -1) -> CachedPlan:
        """psd_plan_cache_lookup, or psd_plan_cache_lookup_gen when generation >= 0."""
        ptr = C.POINTER(L.CascadePlan)()
        hit = C.c_int32()
        L.check(L.load().psd_plan_cache_lookup_gen(self._h, int(generation), C.byref(table.c),
                                                   int(tile_tokens), int(enable), int(min_shared_pages),
                                                   int(min_members), C.byref(ptr), C.byref(hit)))
        return CachedPlan(ptr, bool(hit.value))

    def stats(self) -> dict:
        h, m, n = C.c_int64(), C.c_int64(), C.c_int32()
        L.check(L.load().psd_plan_cache_stats(self._h, C.byref(h), C.byref(m), C.byref(n)))
        return {"hits": h.value, "misses": m.value, "entries": n.value}

    def close(self):
        if self._h:
            L.load().psd_plan_cache_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def rope_append_kv(ctx: Context, q, k_nope, k_rope, v, cos_sin, positions, slot_mapping, k_pool, v_pool, *,
                   rot_dim: int, neox: bool, q_rope_col: int, page_size: int, k_scale: float = 1.0,
                   v_scale: float = 1.0, fault=None, stream=None):
    """rope_append_kv: rope q in place and write the new tokens' K/V rows into the pools.

    q [T, Hq, Dq] bf16, k_nope [T, Hkv, Dn] bf16 or None, k_rope [T, Hkv, Dr] bf16,
    v [T, Hkv, Dv] bf16 or None, cos_sin [max_position, rot_dim] f32, positions and
    slot_mapping [T] int32, pools bf16 (or uint8 fp8-e4m3 codes) [pages, page_size,
    Hkv, D].  Returns the int32 fault word tensor (the one given, or a new zero one)."""
    T = int(positions.numel())
    if fault is None:
        fault = torch.zeros(1, dtype=torch.int32, device=k_pool.device)
    for name, t in (("positions", positions), ("slot_mapping", slot_mapping)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    if cos_sin.dtype != torch.float32:
        raise TypeError("cos_sin must be float32")
    a = L.RopeAppendArgs()
    Hq = int(q.shape[1]) if q is not None else 0
    a.q = _dev_ptr(q, "q") if q is not None else None
    a.Hq, a.Dq, a.q_rope_col = Hq, (int(q.shape[2]) if q is not None else 0), int(q_rope_col)
    a.k_nope = _dev_ptr(k_nope, "k_nope") if k_nope is not None else None
    a.k_rope = _dev_ptr(k_rope, "k_rope")
    a.Hkv, a.Dk_nope, a.Dk_rope = int(k_rope.shape[1]), (int(k_nope.shape[2]) if k_nope is not None else 0), \
        int(k_rope.shape[2])
    a.v = _dev_ptr(v, "v") if v is not None else None
    a.Dv = int(v.shape[2]) if v is not None else 0
    a.rot_dim, a.neox = int(rot_dim), int(bool(neox))
    a.cos_sin = _dev_ptr(cos_sin, "cos_sin")
    a.max_position = int(cos_sin.shape[0])
    a.positions = _dev_ptr(positions, "positions")
    a.slot_mapping = _dev_ptr(slot_mapping, "slot_mapping")
    a.num_tokens = T
    a.k_pool = _dev_ptr(k_pool, "k_pool")
    a.v_pool = _dev_ptr(v_pool, "v_pool") if v_pool is not None else None
    a.num_pages, a.page_size = int(k_pool.shape[0]), int(page_size)
    a.kv_dtype = kv_dtype_code(k_pool)
    a.k_scale, a.v_scale = float(k_scale), float(v_scale)
    a.fault_dev = _dev_ptr(fault, "fault")
    L.check(L.load().rope_append_kv(ctx.handle, C.byref(a), _stream(stream)))
    return fault


def build_cascade_plan(table: HostTable, members, shared_pages: int, tile_tokens: int) -> Plan:
    plan = Plan(table)
    m = _i32(list(members) if len(members) else [0])
    L.check(L.load().build_cascade_plan(C.byref(table.c), _ptr_i32(m), len(members),
                                        int(shared_pages), int(tile_tokens), C.byref(plan.c)))
    return plan


def plan_decode(table: HostTable, tile_tokens: int, enable: int = 1, min_shared_pages: int = 16,
                min_members: int = 2, plan: Plan = None) -> Plan:
    """psd_plan_decode: detection + cascade plan, or the flat plan with a reason."""
    plan = plan if plan is not None else Plan(table)
    L.check(L.load().psd_plan_decode(C.byref(table.c), int(tile_tokens), int(enable),
                                     int(min_shared_pages), int(min_members), C.byref(plan.c)))
    return plan


def cascade_env_enabled(fallback: int = 0) -> int:
    return int(L.load().psd_cascade_env_enabled(int(fallback)))


def workspace_bytes(batch: int, num_items: int, num_rows: int, Hq: int, Dv: int) -> int:
    return int(L.load().psd_workspace_bytes(int(batch), int(num_items), int(num_rows), int(Hq), int(Dv)))


def decode_args(q, k_pool, v_pool, page_indices_dev, *, num_pages: int, page_size: int,
                Hkv: int, Dv: int, sm_scale: float, k_scale: float = 1.0,
                v_scale: float = 1.0) -> L.DecodeArgs:
    """psd_decode_args from device tensors (v_pool is k_pool for a shared latent).
    q and page_indices may instead be pinned host tensors, read by the partial kernels
    over the host link (not by the MLA latent kernel, which takes device q)."""
    a = L.DecodeArgs()
    a.q = _dev_or_pinned_ptr(q, "q")
    a.k_pool = _dev_ptr(k_pool, "k_pool")
    a.v_pool = _dev_ptr(v_pool, "v_pool")
    if page_indices_dev.dtype != torch.int32:
        raise ValueError("page_indices must be int32")
    a.page_indices_dev = _dev_or_pinned_ptr(page_indices_dev, "page_indices")
    a.num_page_indices = int(page_indices_dev.numel())
    a.num_pages = int(num_pages)
    a.batch, a.Hq, a.Dqk = (int(x) for x in q.shape)
    a.Hkv = int(Hkv)
    a.Dv = int(Dv)
    a.page_size = int(page_size)
    a.kv_dtype = kv_dtype_code(k_pool)
    a.k_scale, a.v_scale, a.sm_scale = float(k_scale), float(v_scale), float(sm_scale)
    return a


def paged_decode_partial(ctx: Context, args: L.DecodeArgs, items: np.ndarray, v_out: torch.Tensor,
                         lse_out: torch.Tensor, workspace: torch.Tensor, stream=None):
    """paged_decode_partial over a host work list ([n, 4] int32 rows
    (q_index, page_off, n_tokens, out_row))."""
    it = _i32(items).reshape(-1, 4)
    n = it.shape[0]
    arr = (L.WorkItem * max(n, 1)).from_buffer_copy(it.tobytes() or bytes(16))
    L.check(L.load().paged_decode_partial(
        ctx.handle, C.byref(args), arr, n, _dev_ptr(v_out, "v_out"), _dev_ptr(lse_out, "lse_out"),
        int(v_out.shape[0]), _dev_ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def merge_states(ctx: Context, v_in: torch.Tensor, lse_in: torch.Tensor, o_indptr_dev: torch.Tensor,
                 v_out: torch.Tensor, lse_out: torch.Tensor = None, stream=None):
    """merge_states: v_in [N, H, D] f32, lse_in [N, H] f32, o_indptr [M+1] int32 (device)."""
    M = int(o_indptr_dev.numel()) - 1
    H, D = int(v_in.shape[1]), int(v_in.shape[2])
    L.check(L.load().merge_states(
        ctx.handle, _dev_ptr(v_in, "v_in"), _dev_ptr(lse_in, "lse_in"),
        _dev_ptr(o_indptr_dev, "o_indptr"), M, H, D, _dev_ptr(v_out, "v_out"),
        None if lse_out is None else _dev_ptr(lse_out, "lse_out"), _stream(stream)))


def cascade_decode(ctx: Context, args: L.DecodeArgs, plan: Plan, o: torch.Tensor,
                   lse: torch.Tensor = None, workspace: torch.Tensor = None, stream=None) -> dict:
    """cascade_decode (flat when the plan has no members); returns the path stats."""
    stats = L.CascadeStats()
    L.check(L.load().cascade_decode(
        ctx.handle, C.byref(args), C.byref(plan.c), _out_ptr(o, "o"),
        None if lse is None else _out_ptr(lse, "lse"), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), C.byref(stats), _stream(stream)))
    return {k: getattr(stats, k) for k, _ in L.CascadeStats._fields_}


def cascade_decode_no_alloc(ctx: Context, args: L.DecodeArgs, plan: Plan, o: torch.Tensor,
                            lse: torch.Tensor = None, fault_bits: torch.Tensor = None,
                            stream=None) -> dict:
    """cascade_decode_no_alloc: cascade_decode without a workspace, for callers that
    cannot allocate device memory (scratch lives in the library's fixed 16 MiB
    device array; see include/psd.h).  fault_bits: optional device int32[1]."""
    stats = L.CascadeStats()
    L.check(L.load().cascade_decode_no_alloc(
        ctx.handle, C.byref(args), C.byref(plan.c), _dev_ptr(o, "o"),
        None if lse is None else _dev_ptr(lse, "lse"),
        None if fault_bits is None else _dev_ptr(fault_bits, "fault_bits"),
        C.byref(stats), _stream(stream)))
    return {k: getattr(stats, k) for k, _ in L.CascadeStats._fields_}


def check_device_error(ctx: Context, workspace: torch.Tensor, stream=None) -> int:
    """psd_check_device_error: raises PsdError on a flagged device fault."""
    bits = C.c_int32()
    st = L.load().psd_check_device_error(ctx.handle, _dev_ptr(workspace, "workspace"), _stream(stream),
                                         C.byref(bits))
    if st != L.PSD_OK:
        err = L.PsdError(st, L.load().psd_last_error().decode(errors="replace"))
        err.fault_bits = int(bits.value)
        raise err
    return int(bits.value)


class NestedPlan:
    """A psd_nested_plan with caller-owned (numpy) arrays."""

    def __init__(self, table: HostTable, max_levels: int):
        self.table = table
        bc, ec, sc, ic = C.c_int32(), C.c_int32(), C.c_int32(), C.c_int32()
        L.check(L.load().psd_plan_nested_capacity(C.byref(table.c), int(max_levels), C.byref(bc), C.byref(ec),
                                                  C.byref(sc), C.byref(ic)))
        self.segments_a = (L.Segment * sc.value)()
        self.members_a = np.zeros(ec.value, dtype=np.int32)
        self.row_base_a = np.zeros(ec.value, dtype=np.int32)
        self.o_indptr_a = np.zeros(bc.value + 1, dtype=np.int32)
        self.l0 = (L.WorkItem * ic.value)()
        self.l1 = (L.WorkItem * ic.value)()
        self.c = L.NestedPlan()
        self.c.batch_capacity, self.c.entry_capacity = bc.value, ec.value
        self.c.segment_capacity, self.c.item_capacity = sc.value, ic.value
        self.c.segments = self.segments_a
        self.c.members = _ptr_i32(self.members_a)
        self.c.member_row_base = _ptr_i32(self.row_base_a)
        self.c.l0_items = self.l0
        self.c.l1_items = self.l1
        self.c.o_indptr = _ptr_i32(self.o_indptr_a)

    def _items(self, arr, n):
        cap = self.c.item_capacity
        a = np.ctypeslib.as_array(C.cast(arr, L.P_i32), shape=(cap * 4,)).reshape(cap, 4)
        return a[:n].copy()

    @property
    def segments(self):
        return [(s.first_member, s.num_members, s.start_page, s.shared_pages, s.first_item, s.num_items)
                for s in self.segments_a[: self.c.num_segments]]

    @property
    def members(self):
        return [int(x) for x in self.members_a[: self.c.num_entries]]

    @property
    def member_row_base(self):
        return [int(x) for x in self.row_base_a[: self.c.num_entries]]

    @property
    def o_indptr(self):
        return [int(x) for x in self.o_indptr_a[: self.c.batch + 1]]

    @property
    def l0_items(self):
        return self._items(self.l0, self.c.l0_num_items)

    @property
    def l1_items(self):
        return self._items(self.l1, self.c.l1_num_items)

    @property
    def num_items(self):
        return self.c.l0_num_items + self.c.l1_num_items

    def __getattr__(self, name):
        if name in ("num_segments", "num_entries", "decline_reason", "num_rows", "tile_tokens", "batch",
                    "page_size", "max_levels", "l0_num_items", "l1_num_items"):
            return getattr(self.c, name)
        raise AttributeError(name)


def plan_nested(table: HostTable, tile_tokens: int, enable: int = 1, min_shared_pages: int = 16,
                min_members: int = 2, max_levels: int = 2) -> NestedPlan:
    """psd_plan_nested: several disjoint and nested shared spans (see include/psd.h)."""
    plan = NestedPlan(table, max_levels)
    L.check(L.load().psd_plan_nested(C.byref(table.c), int(tile_tokens), int(enable), int(min_shared_pages),
                                     int(min_members), int(max_levels), C.byref(plan.c)))
    return plan


def nested_workspace_for(plan: NestedPlan, Hq: int, Dv: int, device) -> torch.Tensor:
    n = int(L.load().psd_nested_workspace_bytes(C.byref(plan.c), int(Hq), int(Dv)))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def cascade_decode_nested(ctx: Context, args: L.DecodeArgs, plan: NestedPlan, o: torch.Tensor,
                          lse: torch.Tensor = None, workspace: torch.Tensor = None, stream=None) -> dict:
    """cascade_decode_nested: one stacked level-0 launch per segment, level 1, one merge."""
    stats = L.CascadeStats()
    L.check(L.load().cascade_decode_nested(
        ctx.handle, C.byref(args), C.byref(plan.c), _dev_ptr(o, "o"),
        None if lse is None else _dev_ptr(lse, "lse"), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), C.byref(stats), _stream(stream)))
    return {k: getattr(stats, k) for k, _ in L.CascadeStats._fields_}


def workspace_for(plan: Plan, Hq: int, Dv: int, device) -> torch.Tensor:
    n = workspace_bytes(plan.batch, max(plan.num_items, 1), plan.num_rows, Hq, Dv)
    return torch.empty(n, dtype=torch.uint8, device=device)
