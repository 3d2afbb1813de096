"""Exact, IO-aware softmax attention for NVIDIA GB300 (sm_103a).

The compute lives in ``libfa_gb300.so`` (hand-written CUDA, C-ABI in
``include/fa.h``); this package is its Python binding. Importing it does not
load the library; the first call does, and raises if it has not been built.
"""
from ._build import build  # noqa: F401
from .api import (FAError, FlashAttention, Session, alloc_workspace, fa_backward,  # noqa: F401
                  fa_backward_dkdv, fa_backward_dq, fa_backward_grads, fa_backward_noalloc,
                  fa_backward_preprocess,
                  fa_backward_workspace_size, fa_forward, fa_get_device_status,
                  fa_online_softmax_stats, fa_standard_forward, fa_standard_matrix_bytes,
                  fa_selftest_mma, fa_selftest_wait_timeout, flash_attention, lib, status_string, version)
