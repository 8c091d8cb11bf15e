"""ctypes view of the C ABI in ``include/psd.h`` (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

i32 = C.c_int32
i64 = C.c_int64
P_i32 = C.POINTER(C.c_int32)

PSD_OK = 0
STATUS_NAMES = {0: "PSD_OK", 1: "PSD_ERR_INVALID_ARG", 2: "PSD_ERR_UNSUPPORTED", 3: "PSD_ERR_CUDA",
                4: "PSD_ERR_DEVICE_FAULT", 5: "PSD_ERR_WORKSPACE_TOO_SMALL"}
PSD_BF16, PSD_FP8_E4M3 = 0, 1
PSD_KERNEL_AUTO, PSD_KERNEL_CUDA_CORE, PSD_KERNEL_TENSOR_CORE = 0, 1, 2

# Every symbol include/psd.h declares.
EXPORTS = [
    "psd_create", "psd_destroy", "psd_last_error", "psd_get_counters", "psd_cascade_env_enabled",
    "psd_set_partial_kernel", "psd_set_level0_kernel", "psd_set_timing", "psd_get_kernel_times", "psd_test_withhold_loads",
    "psd_split_plan", "detect_shared_prefix", "build_cascade_plan", "psd_plan_decode",
    "psd_plan_capacity", "psd_workspace_bytes", "paged_decode_partial", "merge_states",
    "cascade_decode", "psd_check_device_error", "cascade_decode_no_alloc",
    "psd_plan_cache_create", "psd_plan_cache_destroy", "psd_plan_cache_lookup", "psd_plan_cache_lookup_gen",
    "psd_plan_cache_stats", "rope_append_kv", "psd_plan_nested_capacity", "psd_plan_nested",
    "psd_nested_workspace_bytes", "cascade_decode_nested", "psd_autotune_tile", "psd_tuned_tile",
]


class PageTable(C.Structure):
    _fields_ = [("page_indptr", P_i32), ("page_indices", P_i32), ("last_page_len", P_i32),
                ("batch", i32), ("page_size", i32)]


class RopeAppendArgs(C.Structure):
    _fields_ = [("q", C.c_void_p), ("Hq", i32), ("Dq", i32), ("q_rope_col", i32),
                ("k_nope", C.c_void_p), ("k_rope", C.c_void_p), ("Hkv", i32), ("Dk_nope", i32),
                ("Dk_rope", i32), ("v", C.c_void_p), ("Dv", i32), ("rot_dim", i32), ("neox", i32),
                ("cos_sin", C.c_void_p), ("max_position", i32), ("positions", C.c_void_p),
                ("slot_mapping", C.c_void_p), ("num_tokens", i32), ("k_pool", C.c_void_p),
                ("v_pool", C.c_void_p), ("num_pages", i64), ("page_size", i32), ("kv_dtype", i32),
                ("k_scale", C.c_float), ("v_scale", C.c_float), ("fault_dev", C.c_void_p)]


class WorkItem(C.Structure):
    _fields_ = [("q_index", i32), ("page_off", i32), ("n_tokens", i32), ("out_row", i32)]


class DecodeArgs(C.Structure):
    _fields_ = [("q", C.c_void_p), ("k_pool", C.c_void_p), ("v_pool", C.c_void_p),
                ("page_indices_dev", C.c_void_p), ("num_page_indices", i64), ("num_pages", i64),
                ("batch", i32), ("Hq", i32), ("Hkv", i32), ("Dqk", i32), ("Dv", i32),
                ("page_size", i32), ("kv_dtype", i32), ("k_scale", C.c_float),
                ("v_scale", C.c_float), ("sm_scale", C.c_float)]


class CascadePlan(C.Structure):
    _fields_ = [("batch_capacity", i32), ("item_capacity", i32), ("members", P_i32),
                ("member_row_base", P_i32), ("l0_items", C.POINTER(WorkItem)),
                ("l1_items", C.POINTER(WorkItem)), ("o_indptr", P_i32), ("batch", i32),
                ("page_size", i32), ("tile_tokens", i32), ("num_members", i32),
                ("shared_pages", i32), ("decline_reason", i32), ("l0_num_items", i32),
                ("l1_num_items", i32), ("num_rows", i32)]


class Segment(C.Structure):
    _fields_ = [("first_member", i32), ("num_members", i32), ("start_page", i32), ("shared_pages", i32),
                ("first_item", i32), ("num_items", i32)]


class NestedPlan(C.Structure):
    _fields_ = [("batch_capacity", i32), ("entry_capacity", i32), ("segment_capacity", i32),
                ("item_capacity", i32), ("segments", C.POINTER(Segment)), ("members", P_i32),
                ("member_row_base", P_i32), ("l0_items", C.POINTER(WorkItem)),
                ("l1_items", C.POINTER(WorkItem)), ("o_indptr", P_i32), ("batch", i32), ("page_size", i32),
                ("tile_tokens", i32), ("max_levels", i32), ("num_segments", i32), ("num_entries", i32),
                ("decline_reason", i32), ("l0_num_items", i32), ("l1_num_items", i32), ("num_rows", i32)]


class CascadeStats(C.Structure):
    _fields_ = [("path", i32), ("decline_reason", i32), ("batch", i32), ("members", i32),
                ("shared_pages", i32), ("shared_tokens", i32), ("prefix_chunks", i32),
                ("suffix_chunks", i32)]


class Counters(C.Structure):
    _fields_ = [("launches_flat", i64), ("launches_cascade", i64), ("cascade_shared_tokens", i64),
                ("cascade_member_sequences", i64), ("cascade_failures", i64),
                ("lists_inline", i64), ("lists_uploaded", i64)]


_LIB = None


class PsdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.fault_bits = 0  # PSD_FAULT_* bits, for PSD_ERR_DEVICE_FAULT


def _sig(lib):
    V = C.c_void_p
    lib.psd_create.argtypes = [C.POINTER(V), C.c_int]
    lib.psd_destroy.argtypes = [V]
    lib.psd_last_error.restype = C.c_char_p
    lib.psd_last_error.argtypes = []
    lib.psd_get_counters.argtypes = [V, C.POINTER(Counters)]
    lib.psd_set_partial_kernel.argtypes = [V, i32]
    lib.psd_set_level0_kernel.argtypes = [V, i32]
    lib.psd_set_timing.argtypes = [V, i32]
    lib.psd_test_withhold_loads.argtypes = [V, i32, C.c_int64]
    lib.psd_get_kernel_times.argtypes = [V, C.POINTER(C.c_float), C.POINTER(C.c_float),
                                         C.POINTER(C.c_float)]
    lib.psd_cascade_env_enabled.argtypes = [i32]
    lib.psd_cascade_env_enabled.restype = i32
    lib.psd_split_plan.argtypes = [C.POINTER(PageTable), i32, C.POINTER(WorkItem), i32, P_i32, P_i32]
    lib.detect_shared_prefix.argtypes = [C.POINTER(PageTable), i32, i32, P_i32, P_i32, P_i32, P_i32]
    lib.build_cascade_plan.argtypes = [C.POINTER(PageTable), P_i32, i32, i32, i32,
                                       C.POINTER(CascadePlan)]
    lib.psd_plan_decode.argtypes = [C.POINTER(PageTable), i32, i32, i32, i32, C.POINTER(CascadePlan)]
    lib.psd_plan_capacity.argtypes = [C.POINTER(PageTable), P_i32, P_i32]
    lib.psd_plan_cache_create.argtypes = [C.POINTER(V), i32]
    lib.psd_plan_cache_destroy.argtypes = [V]
    lib.psd_plan_cache_lookup.argtypes = [V, C.POINTER(PageTable), i32, i32, i32, i32,
                                          C.POINTER(C.POINTER(CascadePlan)), P_i32]
    lib.psd_plan_cache_lookup_gen.argtypes = [V, i64, C.POINTER(PageTable), i32, i32, i32, i32,
                                              C.POINTER(C.POINTER(CascadePlan)), P_i32]
    lib.psd_plan_cache_stats.argtypes = [V, C.POINTER(i64), C.POINTER(i64), P_i32]
    lib.rope_append_kv.argtypes = [V, C.POINTER(RopeAppendArgs), V]
    lib.psd_autotune_tile.argtypes = [V, C.POINTER(DecodeArgs), C.POINTER(PageTable), P_i32, i32, i32, i32, i32,
                                      i32, V, V, V, C.c_size_t, V, P_i32, C.POINTER(C.c_float)]
    lib.psd_tuned_tile.argtypes = [V, C.POINTER(DecodeArgs), C.POINTER(PageTable), i32, i32, i32, i32]
    lib.psd_tuned_tile.restype = i32
    lib.psd_plan_nested_capacity.argtypes = [C.POINTER(PageTable), i32, P_i32, P_i32, P_i32, P_i32]
    lib.psd_plan_nested.argtypes = [C.POINTER(PageTable), i32, i32, i32, i32, i32, C.POINTER(NestedPlan)]
    lib.psd_nested_workspace_bytes.argtypes = [C.POINTER(NestedPlan), i32, i32]
    lib.psd_nested_workspace_bytes.restype = C.c_size_t
    lib.cascade_decode_nested.argtypes = [V, C.POINTER(DecodeArgs), C.POINTER(NestedPlan), V, V, V, C.c_size_t,
                                          C.POINTER(CascadeStats), V]
    lib.psd_workspace_bytes.argtypes = [i32, i32, i64, i32, i32]
    lib.psd_workspace_bytes.restype = C.c_size_t
    lib.paged_decode_partial.argtypes = [V, C.POINTER(DecodeArgs), C.POINTER(WorkItem), i32, V, V,
                                         i64, V, C.c_size_t, V]
    lib.merge_states.argtypes = [V, V, V, V, i64, i32, i32, V, V, V]
    lib.cascade_decode.argtypes = [V, C.POINTER(DecodeArgs), C.POINTER(CascadePlan), V, V, V,
                                   C.c_size_t, C.POINTER(CascadeStats), V]
    lib.psd_check_device_error.argtypes = [V, V, V, P_i32]
    lib.cascade_decode_no_alloc.argtypes = [V, C.POINTER(DecodeArgs), C.POINTER(CascadePlan), V, V, V,
                                            C.POINTER(CascadeStats), V]
    for name in EXPORTS:
        f = getattr(lib, name)
        if f.restype is C.c_int or f.restype is None:
            if name not in ("psd_last_error", "psd_cascade_env_enabled", "psd_workspace_bytes",
                            "psd_nested_workspace_bytes", "psd_tuned_tile"):
                f.restype = C.c_int


def load(build: bool = True):
    """Load libpsd.so (building it in-tree first when missing or stale)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.build() if build else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; build it with __graft_entry__.build()")
    lib = C.CDLL(path)
    _sig(lib)
    _LIB = lib
    return lib


def check(status: int):
    if status != PSD_OK:
        raise PsdError(status, load().psd_last_error().decode(errors="replace"))
