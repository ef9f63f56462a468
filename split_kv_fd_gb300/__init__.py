"""split_kv_fd_gb300: split-KV decode attention (FlashDecoding) for GB300.

The compute path is the CUDA library ``libfd.so`` (C ABI in include/fd.h,
kernels in csrc/); ``fd`` is its Python binding.  ``workloads`` and
``inputs`` hold the synthetic workload shapes and the seeded input drawing.
"""
from .fd import (FDError, auto_num_splits, combine_lse, combine_mlo, decode,  # noqa: F401
                 decode_fp8, decode_gqa, decode_gqa_fp8, decode_gqa_paged, decode_gqa_paged_fp8, decode_noalloc, decode_paged, decode_split,
                 device_status, load,
                 merge_lse, new_workspace, num_sms, selftest_wait_timeout, workspace_size,
                 workspace_size_gqa)

__all__ = ["FDError", "auto_num_splits", "combine_lse", "combine_mlo", "decode", "decode_fp8",
           "decode_gqa", "decode_gqa_fp8", "decode_gqa_paged", "decode_gqa_paged_fp8", "decode_noalloc", "workspace_size_gqa",
           "decode_paged", "decode_split", "device_status", "load", "merge_lse", "new_workspace",
           "num_sms", "selftest_wait_timeout",
           "workspace_size"]
