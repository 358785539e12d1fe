"""Chunkwise-parallel forward of linear attention with a diagonal-plus-low-rank decay,
as hand-written CUDA for GB300 (sm_103a) behind the C ABI of libdplr (include/dplr.h).

``forward`` / ``Forward`` marshal torch device tensors into ``dplr_la_forward``;
``ForwardHost`` and ``ForwardHostSeq`` marshal host tensors into ``dplr_la_forward_host``
(heads split into groups) and ``dplr_la_forward_host_seq`` (the sequence split into segments),
with the transfers overlapped with the kernels; the C-ABI mirrors (``dplr_la_forward``,
``dplr_la_chunk_maps``, ...) take raw pointers. There is no CPU fallback: without
libdplr.so the calls raise.
"""

from .dplr import (  # noqa: F401
    DPLR_BF16, DPLR_F32, DPLR_GDN, DPLR_GENERIC, DPLR_HDLA, DPLR_OK, DplrError, Forward, ForwardHost, ForwardHostSeq, LIB_PATH,
    default_groups, default_segments, dplr_desc, dplr_la_check, dplr_la_chunk_maps, dplr_la_forward, dplr_la_forward_host,
    dplr_la_forward_noalloc, dplr_la_host_workspace_size, dplr_la_forward_host_seq, dplr_la_host_seq_workspace_size, dplr_la_noalloc_status, dplr_la_read_status, dplr_la_set_wait_limit, dplr_la_path, dplr_la_decode_step, Decode, dplr_la_backward, dplr_la_backward_workspace_size, Backward, dplr_hla_forward, dplr_hla_workspace_size, dplr_hla_path, HLA, dplr_gdp_forward, dplr_gdp_workspace_size, dplr_gdp_path, GDP, dplr_la_kernel_count, dplr_la_stage_workspace_size,
    dplr_la_state_scan, dplr_la_workspace_size, forward, library, make_desc, status_string,
)
