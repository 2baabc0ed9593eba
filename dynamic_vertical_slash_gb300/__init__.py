"""GB300 (sm_103a) Vertical-Slash sparse attention: the hot path of MTraining's
dynamic sparse attention as a C-ABI CUDA library (``libvs.so``) with a thin
Python binding of the same names.

    vs_estimate           online vertical / slash selection (Algorithm 1)
    vs_estimate_topp      the same with top-p budgets per head (topp, Pool)
    vs_select_topp        top-p budgets and selection on given scores
    vs_build_block_index  sparse index arena (sparseformat / convert_index)
    vs_attn_fwd           sparse attention forward (O, LSE; merge mode)
    vs_attn_bwd           sparse attention backward (dQ, dK, dV)
    striped_permute       64-token block-level striping
    ring_permute          striped or ZigZag ring layout
    vs_ring_work          mask entries per worker pair of a striped / ZigZag ring
    vs_check_status       device status word of a workspace or arena
    vs_selftest_wait_timeout  failure-detection self-test (a bounded wait runs out)
"""
from ._binding import (VSError, make_shape, make_stripe, make_window, ring_permute, striped_permute, trace_enable,
                       trace_report, trace_reset,
                       vs_attn_bwd, vs_attn_fwd,
                       vs_build_block_index, vs_check_status, vs_estimate, vs_estimate_topp, vs_index_counts,
                       vs_select_topp, vs_selftest_wait_timeout, vs_ring_work, lib, launch_count, status_string)
from .pipeline import StripedWorker, VSAttention, ZigZagWorker, flop_counts

__all__ = ["VSError", "make_shape", "make_stripe", "striped_permute", "vs_attn_bwd", "vs_attn_fwd",
           "vs_build_block_index", "vs_check_status", "vs_estimate", "vs_index_counts", "lib", "launch_count",
           "status_string", "VSAttention", "StripedWorker", "flop_counts", "vs_selftest_wait_timeout",
           "vs_estimate_topp", "vs_select_topp", "vs_ring_work", "make_window", "ring_permute", "ZigZagWorker"]
