"""Chunk-centric fused AllGather-GEMM, GEMM-ReduceScatter, GEMM-AllReduce and GEMM-AllToAll
for one GB300 (sm_103a).

The compute path is the CUDA library ``libdt.so`` (sources in ``csrc/``, C ABI in
``include/dt.h``); ``capi`` is its ctypes binding.  Importing this package loads nothing;
the library is loaded on first use and every call fails loudly if it is not built.
"""
from .capi import (BACKENDS, OP_A2A, OP_AG, OP_AR, OP_RS, DtArgs, DtError,  # noqa: F401
                   a2a_chunks, allgather, a2a_signals, ag_gemm, ag_gemm_kernel_overlap,
                   ag_gemm_static_scratch, check, col_band, debug_drop_transfer, ffn_ag_rs, gemm_a2a,
                   gemm_a2a_kernel_overlap, gemm_ar, gemm_ar_kernel_overlap, gemm_rs,
                   gemm_rs_kernel_overlap, make_args, static_scratch_check, swizzle_plan,
                   swizzle_plan_device, tile_count, tile_rows, trace_attach, trace_bytes,
                   trace_decode, tune_ag_gemm, tune_reduce, workspace_init, workspace_size)
