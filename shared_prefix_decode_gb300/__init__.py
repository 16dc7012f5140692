"""Shared-prefix (cascade) decode attention for GB300 (sm_103a).

The compute path is the CUDA library ``_lib/libhp.so`` (C ABI in
``include/hp.h``); ``binding`` is its ctypes binding and ``workloads`` the
seeded synthetic input generator.  Importing the package does not load the
library; the first call does, and raises if it has not been built.
"""
from .binding import (  # noqa: F401
    CascadePlan,
    HpError,
    LoopPlan,
    hp_cascade_append_kv,
    hp_cascade_contexts,
    hp_cascade_decode,
    hp_cascade_decode_append,
    hp_cascade_decode_loop,
    hp_cascade_loop_plan_bytes,
    hp_cascade_plan,
    hp_cascade_plan_bytes,
    hp_cascade_plan_stats,
    hp_merge_states,
    hp_prefix_attn,
    hp_read_device_status,
    hp_suffix_decode_paged,
    library,
)

__all__ = [
    "CascadePlan", "HpError", "LoopPlan", "hp_cascade_append_kv", "hp_cascade_contexts", "hp_cascade_decode",
    "hp_cascade_decode_append", "hp_cascade_decode_loop", "hp_cascade_loop_plan_bytes", "hp_cascade_plan",
    "hp_cascade_plan_bytes", "hp_cascade_plan_stats", "hp_merge_states", "hp_prefix_attn",
    "hp_read_device_status", "hp_suffix_decode_paged", "library",
]
