"""MLA tree-verify attention for GB300 (sm_103a).

The computation runs in ``libmla_tree_verify.so`` (CUDA kernels behind the C ABIs of
``include/mla_tree_verify.h`` and ``include/causal_conv1d_dedup.h``); ``binding`` marshals
torch tensors to it.  Build the
library with ``mla_tree_verify_gb300.build.build()``.
"""
from .binding import (CONV1D_BAD_ACCEPT, CONV1D_BAD_SLOT, CONV1D_DTYPE_BF16,  # noqa: F401
                      CONV1D_DTYPE_F32, CONV1D_PAD_SLOT,
                      DEV_BAD_INDPTR, DEV_BAD_MASK, DEV_BAD_SLOT, DEV_TIMEOUT,
                      GATHER_BAD_ARGS, GATHER_BAD_SLOT, MERGE_AUTO, MERGE_NO_TMEM,
                      MERGE_PREFER_TMEM, MlaTreeVerifyError, conv1d_update, kv_gather,
                      mla_tree_verify, mla_tree_verify_debug, mla_tree_verify_debug_ex,
                      plan_header, prepare, read_device_status, split_grid, workspace_bytes)
