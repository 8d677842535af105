"""GB300 (sm_103a) Gated DeltaNet chunked prefill: forward and backward.

The compute runs in ``libgdr.so`` (hand-written CUDA, C ABI in
``include/gdr.h``); this package is its thin ctypes binding plus the seeded
synthetic input generators.
"""
from .binding import (KernelTimer, GDR_BF16, GDR_F32, GDR_PATH_AUTO, GDR_PATH_SIMT, GDR_PATH_TC, GdrError, Problem,
                      alloc_workspace, bwd_workspace_size, check_status, fwd_workspace_size, gdr_bwd, gdr_fwd,
                      get_plan, load, make_opts, tc_available, version)
from .api import chunk_gated_delta_rule, chunk_gated_delta_rule_bwd, chunk_gated_delta_rule_fwd

__all__ = ["KernelTimer", "gdr_fwd", "gdr_bwd", "check_status", "version", "load", "Problem", "make_opts", "GdrError",
           "fwd_workspace_size", "bwd_workspace_size", "alloc_workspace", "get_plan", "GDR_BF16", "GDR_F32",
           "GDR_PATH_AUTO", "GDR_PATH_SIMT", "GDR_PATH_TC", "tc_available", "chunk_gated_delta_rule",
           "chunk_gated_delta_rule_fwd", "chunk_gated_delta_rule_bwd"]
