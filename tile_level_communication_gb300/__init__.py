"""Chunk-centric fused AllGather-GEMM and GEMM-ReduceScatter for one GB300 (sm_103a).

The compute path is the CUDA library ``libdt.so`` (sources in ``csrc/``, C ABI in
``include/dt.h``); ``capi`` is its ctypes binding.  Importing this package loads nothing;
the library is loaded on first use and every call fails loudly if it is not built.
"""
from .capi import (BACKENDS, OP_AG, OP_AR, OP_RS, DtArgs, DtError, ag_gemm,  # noqa: F401
                   ag_gemm_static_scratch,
                   ag_gemm_kernel_overlap, check, debug_drop_transfer, ffn_ag_rs, gemm_ar,
                   gemm_ar_kernel_overlap, gemm_rs, gemm_rs_kernel_overlap, make_args,
                   swizzle_plan, swizzle_plan_device, tile_count, tune_ag_gemm, tune_reduce,
                   workspace_init, workspace_size)
