"""Jagged Flash Attention for GB300 (sm_103a).

The compute path is libjfa.so (hand-written CUDA; C ABI in include/jfa.h);
``jfa`` is its thin ctypes binding and ``workloads`` draws seeded inputs.
"""
from . import jfa, workloads  # noqa: F401
from .jfa import (block_attn_bwd, block_attn_fwd, block_plan, jfa_bwd, jfa_device_status, jfa_fwd,  # noqa: F401
                  jfa_get_block_schedule, jfa_get_bwd_schedule, jfa_get_schedule, jfa_plan_bwd, jfa_plan_fwd,
                  jfa_plan_window,
                  jfa_profile_enable, jfa_profile_read, jfa_profile_select, jfa_selftest_wait_timeout,
                  jfa_set_block_schedule, jfa_set_bwd_schedule, jfa_set_schedule, jfa_status_string,
                  jfa_fwd_topk, jfa_topk_rows, jfa_topk_select, jfa_workspace_size)
