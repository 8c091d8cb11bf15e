"""Paged split-KV decode for one NVIDIA GB300 (sm_103a).

The compute lives in ``libpsd.so`` (hand-written CUDA behind the C ABI declared in
``include/psd.h``); ``api`` is a thin ctypes binding with the same names.
"""
from .api import (CachedPlan, Context, HostTable, NestedPlan, Plan, PlanCache,  # noqa: F401
                  build_cascade_plan, cascade_decode, cascade_decode_nested, nested_workspace_for,
                  plan_nested,
                  cascade_decode_no_alloc,
                  cascade_env_enabled, check_device_error, decode_args, detect_shared_prefix,
                  merge_states, paged_decode_partial, plan_decode, rope_append_kv, split_plan,
                  workspace_bytes, workspace_for)
from ._lib import PsdError, load  # noqa: F401
