"""Context-parallel causal attention on one GB300 (sm_103a).

Python face of libcpattn.so: block attention with global offsets and per-row
LSE, the LSE merge, the Ring-Attention schedule of P virtual ranks
(contiguous / zigzag / striped), the Ulysses seq<->head permutation, and
the backward pass of block and ring attention.  The functions
marshal torch tensors into the C ABI declared in include/cpattn.h; all
computation happens in the library's CUDA kernels.
"""

from ._lib import (CP_BF16, CP_CONTIGUOUS, CP_ERR_BOUNDS, CP_ERR_TIMEOUT, CP_F32, CP_MAX_RANKS, CP_STRIPED,
                   CP_ZIGZAG, CpError, cp_attn_block, cp_attn_block_backward,
                   cp_attn_block_backward_workspace_size, cp_check_device_error, cp_debug_bounds,
                   cp_head_to_seq, cp_last_error, cp_lse_merge, cp_ring_backward, cp_ring_backward_host,
                   cp_ring_backward_host_workspace_size, cp_ring_backward_step,
                   cp_ring_backward_workspace_size, cp_ring_copy_workspace_size, cp_ring_forward,
                   cp_ring_forward_copy, cp_ring_forward_fused, cp_ring_forward_host,
                   cp_ring_forward_steps, ring_runs_fused, ring_backward_runs_fused,
                   cp_ring_backward_fused_step,
                   cp_ring_forward_noalloc, cp_ring_host_workspace_size, cp_ring_step, cp_ring_step_blocks,
                   cp_ring_workspace_size, cp_selftest_wait_timeout, cp_seq_to_head,
                   cp_ulysses_forward, cp_ulysses_forward_host, cp_ulysses_host_workspace_size,
                   cp_ulysses_stage, cp_ulysses_workspace_size, cp_usp_forward,
                   cp_usp_forward_host, cp_usp_host_workspace_size, cp_usp_stage,
                   cp_usp_workspace_size, cp_version, lib, library_path)

__all__ = [
    "CP_BF16", "CP_CONTIGUOUS", "CP_ERR_BOUNDS", "CP_ERR_TIMEOUT", "CP_F32", "CP_MAX_RANKS",
    "CP_STRIPED",
    "CP_ZIGZAG", "CpError", "cp_attn_block", "cp_attn_block_backward",
    "cp_attn_block_backward_workspace_size", "cp_check_device_error", "cp_debug_bounds",
    "cp_head_to_seq",
    "cp_last_error", "cp_lse_merge", "cp_ring_backward", "cp_ring_backward_host",
    "cp_ring_backward_host_workspace_size", "cp_ring_backward_step",
    "cp_ring_backward_workspace_size", "cp_ring_copy_workspace_size", "cp_ring_forward",
    "cp_ring_forward_copy", "cp_ring_forward_fused", "cp_ring_forward_host",
    "cp_ring_forward_steps", "ring_runs_fused", "ring_backward_runs_fused",
    "cp_ring_backward_fused_step",
    "cp_ring_forward_noalloc",
    "cp_ring_host_workspace_size", "cp_ring_step", "cp_ring_step_blocks",
    "cp_ring_workspace_size", "cp_selftest_wait_timeout", "cp_seq_to_head",
    "cp_ulysses_forward", "cp_ulysses_forward_host", "cp_ulysses_host_workspace_size",
    "cp_ulysses_stage", "cp_ulysses_workspace_size", "cp_usp_forward", "cp_usp_forward_host",
    "cp_usp_host_workspace_size", "cp_usp_stage", "cp_usp_workspace_size", "cp_version", "lib",
    "library_path",
]
