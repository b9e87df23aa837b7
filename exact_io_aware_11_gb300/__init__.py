"""Exact IO-aware attention (FlashAttention method) for one GB300 GPU.

The computation lives in libfa.so (hand-written sm_103a CUDA kernels behind
the C-ABI of include/fa.h); this package is its thin Python binding.
"""
from ._lib import (FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED,
                   FA_OK, AttentionOptions, FaError, attention_backward, attention_forward,
                   backward, blocksparse_backward, blocksparse_forward,
                   bwd_split_workspace_bytes, bwd_workspace_bytes, dropout_backward, dropout_forward, dropout_mask,
                   device_status, forward, fwd_workspace_bytes, lib, library_path, selftest_wait_timeout,
                   status_string)

__all__ = ["FA_ERR_CUDA", "FA_ERR_DEVICE_TIMEOUT", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED",
           "FA_OK", "AttentionOptions", "FaError", "attention_backward", "attention_forward",
           "backward", "blocksparse_backward", "blocksparse_forward",
           "bwd_split_workspace_bytes", "bwd_workspace_bytes", "dropout_backward", "dropout_forward", "dropout_mask",
           "device_status", "forward", "fwd_workspace_bytes", "lib", "library_path", "selftest_wait_timeout",
           "status_string"]
