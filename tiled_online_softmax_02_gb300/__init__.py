"""GB300-native tiled online-softmax attention forward (sm_103a).

Also the DSA indexer's sparse index selection (dsa_index_select).

The compute lives in libattn.so (C ABI in include/attn.h), built from csrc/
by ``tiled_online_softmax_02_gb300.build.build()``.  This package only
marshals torch tensors into that library.
"""
from ._binding import (ATTN_BF16, ATTN_ERR_CUDA, ATTN_ERR_INVALID_ARG, ATTN_ERR_TIMEOUT,
                       ATTN_ERR_UNSUPPORTED, ATTN_F16, ATTN_F32, ATTN_OK, AttnError, attn_fwd,
                       attn_fwd_f32_split, attn_fwd_splitkv, dsa_index_select,
                       get_device_status, host_copy_bytes, library_path, load_library,
                       selftest_bounded_wait,
                       set_wait_timeout_ns, status_string)

__all__ = ["attn_fwd", "attn_fwd_f32_split", "attn_fwd_splitkv", "dsa_index_select", "get_device_status",
           "host_copy_bytes", "set_wait_timeout_ns", "selftest_bounded_wait",
           "load_library", "library_path", "status_string", "AttnError", "ATTN_OK",
           "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT",
           "ATTN_F32", "ATTN_F16", "ATTN_BF16"]
