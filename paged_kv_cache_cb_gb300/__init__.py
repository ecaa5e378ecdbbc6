"""GB300-native paged-KV continuous-batching attention step.

A C-ABI CUDA library for sm_103a (``libcbattn.so``, declared in
``include/cbattn.h``) and this thin Python binding with the same entry-point
names.  PyTorch only supplies device memory and streams.
"""
from ._lib import (CB_EDEVICE, CB_EINVAL, CB_ETIMEOUT, CB_EWORKSPACE, CB_MAX_REQS, CB_OK, CBError, Graph, Scheduler,
                   cb_build_slot_mapping, cb_copy_blocks, cb_hbm_copy, cb_kv_append, cb_kv_append_paged_attention,
                   cb_kv_append_paged_attention_window, cb_last_error, cb_last_launch_count, cb_paged_attention,
                   cb_paged_attention_noalloc, cb_paged_attention_window, cb_paged_attention_workspace_size,
                   cb_strerror, lib)

__all__ = [
    "CB_OK", "CB_EINVAL", "CB_EWORKSPACE", "CB_EDEVICE", "CB_ETIMEOUT", "CB_MAX_REQS", "CBError", "Graph", "Scheduler",
    "cb_build_slot_mapping", "cb_copy_blocks", "cb_hbm_copy", "cb_kv_append", "cb_kv_append_paged_attention",
    "cb_kv_append_paged_attention_window", "cb_last_error", "cb_last_launch_count", "cb_paged_attention",
    "cb_paged_attention_noalloc", "cb_paged_attention_window", "cb_paged_attention_workspace_size", "cb_strerror",
    "lib",
]
