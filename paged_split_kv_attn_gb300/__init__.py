"""Paged split-KV GQA attention for single-token decode on GB300 (sm_103a).

The work runs in ``libpskv.so`` (hand-written CUDA kernels behind the C ABI of
``include/pskv.h``); this package is its thin Python binding, with the same
entry-point names.  PyTorch provides device memory and streams only.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import (EXPORTS, Layout, PskvError, decode_attn_multirow, decode_attn_splitkv,
                       decode_attn_tree,
                       decode_attn_splitkv_static, decode_attn_windowed,
                       decode_attn_workspace_bytes, kv_append_rows, kv_prep_append, load_library,
                       merge_partials, merge_partials_workspace_bytes, paged_kv_layout_create,
                       pskv_check_flags, pskv_kernel_launches, pskv_partial_scratch_bytes,
                       pskv_plan_splits,
                       prefill_attn_paged, prefill_attn_workspace_bytes,
                       decode_attn_multirow_workspace_bytes,
                       pskv_strerror, pskv_version, workspace)

__all__ = ["EXPORTS", "Layout", "PskvError", "decode_attn_multirow", "decode_attn_splitkv",
           "decode_attn_tree",
           "decode_attn_splitkv_static", "decode_attn_windowed",
           "decode_attn_workspace_bytes", "kv_append_rows", "kv_prep_append", "load_library",
           "merge_partials",
           "merge_partials_workspace_bytes", "paged_kv_layout_create", "pskv_check_flags",
           "pskv_kernel_launches",
           "pskv_partial_scratch_bytes", "pskv_plan_splits", "pskv_strerror", "pskv_version",
           "prefill_attn_paged", "prefill_attn_workspace_bytes",
           "decode_attn_multirow_workspace_bytes",
           "workspace"]
