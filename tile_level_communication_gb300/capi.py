"""ctypes binding of libdt.so (include/dt.h): argument marshalling only.

Every step of the fused AllGather-GEMM / GEMM-ReduceScatter / GEMM-AllReduce /
GEMM-AllToAll runs in the library's CUDA
kernels; this module converts Python arguments into the C structs and pointers, calls the
C entry point with the same name, and raises ``DtError`` on a non-OK status.  Tensors may be
anything with ``data_ptr()`` (torch tensors) or plain integer addresses.  When the library
is not built, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdt.so")

DT_OK, DT_ERR_INVALID, DT_ERR_UNSUPPORTED, DT_ERR_TIMEOUT, DT_ERR_CUDA, DT_ERR_WORKSPACE = range(6)
BACKENDS = {"auto": 0, "copy_engine": 1, "tma": 2, "ldst": 3, "tma_tile": 4}
DTYPES = {"bf16": 0, "f32": 1}
ACTS = {"none": 0, "gelu_tanh": 1, "silu": 2}
OP_AG, OP_RS, OP_AR, OP_A2A = 0, 1, 2, 3
MAX_WORLD = 16

# every function include/dt.h declares: name -> (restype, argtypes)
_P = ctypes.c_void_p
_SIGS = {
    "dt_args_default": (None, [_P]),
    "dt_version": (ctypes.c_int, []),
    "dt_sizeof_args": (ctypes.c_size_t, []),
    "dt_sizeof_tune_point": (ctypes.c_size_t, []),
    "dt_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dt_last_error": (ctypes.c_char_p, []),
    "dt_workspace_size": (ctypes.c_size_t, [_P, ctypes.c_int]),
    "dt_workspace_init": (ctypes.c_int, [_P, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "dt_ag_gemm": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_gemm_rs": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_allgather": (ctypes.c_int, [_P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_ag_gemm_kernel_overlap": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_gemm_rs_kernel_overlap": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_gemm_ar": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_gemm_ar_kernel_overlap": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_gemm_a2a": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_gemm_a2a_kernel_overlap": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "dt_a2a_signals": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int64, _P]),
    "dt_tile_count": (ctypes.c_int64, [_P, ctypes.c_int]),
    "dt_tile_rows": (ctypes.c_int32, [_P, ctypes.c_int]),
    "dt_col_band": (ctypes.c_int32, [_P, ctypes.c_int]),
    "dt_swizzle_plan": (ctypes.c_int, [_P, ctypes.c_int, _P, ctypes.c_int64]),
    "dt_swizzle_plan_device": (ctypes.c_int, [_P, ctypes.c_int, _P, ctypes.c_int64, _P]),
    "dt_check": (ctypes.c_int, [_P, _P, _P]),
    "dt_debug_drop_transfer": (ctypes.c_int, [ctypes.c_int32]),
    "dt_trace_bytes": (ctypes.c_size_t, [_P]),
    "dt_trace_attach": (ctypes.c_int, [_P, ctypes.c_size_t]),
    "dt_ag_gemm_static_scratch": (ctypes.c_int, [_P, _P, _P, _P, _P]),
    "dt_static_scratch_check": (ctypes.c_int, [_P, _P]),
    "dt_ffn_ag_rs": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, ctypes.c_size_t,
                                    _P, _P, _P]),
    "dt_tune_ag_gemm": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_size_t, _P, ctypes.c_int32, _P,
                                       ctypes.c_int32, _P, _P]),
    "dt_tune_reduce": (ctypes.c_int, [ctypes.c_int, _P, _P, _P, _P, ctypes.c_size_t, _P,
                                      ctypes.c_int32, _P, ctypes.c_int32, _P, _P]),
}
STATIC_SCRATCH_BYTES = 32 * 1024 * 1024


class DtArgs(ctypes.Structure):
    """Mirror of ``dt_args``."""
    _fields_ = [
        ("world_size", ctypes.c_int32), ("rank", ctypes.c_int32),
        ("m", ctypes.c_int64), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
        ("chunk_rows", ctypes.c_int64),
        ("swizzle", ctypes.c_int32), ("backend", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
        ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("group", ctypes.c_int32),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64),
        ("timeout_us", ctypes.c_int64),
        ("num_sms", ctypes.c_int32), ("copy_ctas", ctypes.c_int32),
        ("act", ctypes.c_int32), ("col_band", ctypes.c_int32),
    ]


class DtTunePoint(ctypes.Structure):
    """Mirror of ``dt_tune_point``."""
    _fields_ = [("chunk_rows", ctypes.c_int64), ("backend", ctypes.c_int32),
                ("copy_ctas", ctypes.c_int32), ("swizzle", ctypes.c_int32),
                ("group", ctypes.c_int32), ("tile_m", ctypes.c_int32),
                ("col_band", ctypes.c_int32), ("ms", ctypes.c_float), ("status", ctypes.c_int32)]


class DtError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status
        self.message = message


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m tile_level_communication_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, argt) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = argt
        if h.dt_sizeof_args() != ctypes.sizeof(DtArgs):
            raise RuntimeError("dt_args layout mismatch between libdt.so and the binding")
        if h.dt_sizeof_tune_point() != ctypes.sizeof(DtTunePoint):
            raise RuntimeError("dt_tune_point layout mismatch between libdt.so and the binding")
        _lib = h
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().dt_status_string(status).decode()
    except Exception:  # library missing: still format the error
        return f"status {status}"


def _raise(status: int):
    if status != DT_OK:
        raise DtError(status, lib().dt_last_error().decode())


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _ptr_array(xs):
    arr = (ctypes.c_void_p * len(xs))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def make_args(world_size: int, m: int, n: int, k: int, *, rank: int = 0, chunk_rows: int = 128,
              swizzle: bool = True, backend: str = "auto", out_dtype: str = "bf16",
              lda: int = 0, ldb: int = 0, ldc: int = 0, timeout_us: int = 0, num_sms: int = 0,
              group: int = 8, copy_ctas: int = 0, act: str = "none", tile_m: int = 0,
              col_band: int = 0) -> DtArgs:
    a = DtArgs()
    lib().dt_args_default(ctypes.byref(a))
    a.world_size, a.rank, a.m, a.n, a.k = world_size, rank, m, n, k
    a.chunk_rows = chunk_rows
    a.swizzle = 1 if swizzle else 0
    a.backend = BACKENDS[backend]
    a.out_dtype = DTYPES[out_dtype]
    a.lda, a.ldb, a.ldc = lda, ldb, ldc
    a.timeout_us = timeout_us
    a.num_sms = num_sms
    a.group = group
    a.copy_ctas = copy_ctas
    a.act = ACTS[act]
    a.tile_m = tile_m
    a.col_band = col_band
    return a


def workspace_size(args: DtArgs, op: int) -> int:
    n = lib().dt_workspace_size(ctypes.byref(args), op)
    if n == 0:
        raise DtError(DT_ERR_INVALID, lib().dt_last_error().decode())
    return int(n)


def workspace_init(args: DtArgs, op: int, workspace, nbytes: int, stream=None):
    _raise(lib().dt_workspace_init(ctypes.byref(args), op, _ptr(workspace), nbytes, _stream(stream)))


def _nbytes(workspace, nbytes):
    if nbytes is not None:
        return nbytes
    return int(workspace.numel() * workspace.element_size())


def ag_gemm(shards, b, c, workspace, args: DtArgs, stream=None, ws_bytes=None):
    _raise(lib().dt_ag_gemm(_ptr_array(shards), _ptr(b), _ptr(c), _ptr(workspace),
                            _nbytes(workspace, ws_bytes), ctypes.byref(args), _stream(stream)))


def allgather(shards, out, workspace, args: DtArgs, stream=None, ws_bytes=None):
    """AllGather alone (the fused op's chunk transfer): out ([M, K], ld args.ldc or K)
    receives every shard's rows in rank order."""
    _raise(lib().dt_allgather(_ptr_array(shards), _ptr(out), _ptr(workspace),
                              _nbytes(workspace, ws_bytes), ctypes.byref(args), _stream(stream)))


def gemm_rs(a_list, b_list, out_list, workspace, args: DtArgs, stream=None, ws_bytes=None):
    _raise(lib().dt_gemm_rs(_ptr_array(a_list), _ptr_array(b_list), _ptr_array(out_list),
                            _ptr(workspace), _nbytes(workspace, ws_bytes), ctypes.byref(args),
                            _stream(stream)))


def ag_gemm_static_scratch(shards, b, c, args: DtArgs, stream=None):
    """dt_ag_gemm on the library's fixed device scratch: for callers that cannot allocate
    device memory.  Problems needing more than STATIC_SCRATCH_BYTES are rejected."""
    _raise(lib().dt_ag_gemm_static_scratch(_ptr_array(shards), _ptr(b), _ptr(c),
                                           ctypes.byref(args), _stream(stream)))


def gemm_ar(a_list, b_list, out_list, workspace, args: DtArgs, stream=None, ws_bytes=None):
    """Fused GEMM-AllReduce: out_list[r] ([M, N]) receives sum_q A_q @ B_q for every r."""
    _raise(lib().dt_gemm_ar(_ptr_array(a_list), _ptr_array(b_list), _ptr_array(out_list),
                            _ptr(workspace), _nbytes(workspace, ws_bytes), ctypes.byref(args),
                            _stream(stream)))


def gemm_ar_kernel_overlap(a_list, b_list, out_list, workspace, args: DtArgs, stream=None,
                           ws_bytes=None):
    _raise(lib().dt_gemm_ar_kernel_overlap(_ptr_array(a_list), _ptr_array(b_list),
                                           _ptr_array(out_list), _ptr(workspace),
                                           _nbytes(workspace, ws_bytes), ctypes.byref(args),
                                           _stream(stream)))


def ag_gemm_kernel_overlap(shards, b, c, workspace, args: DtArgs, stream=None, ws_bytes=None):
    _raise(lib().dt_ag_gemm_kernel_overlap(_ptr_array(shards), _ptr(b), _ptr(c), _ptr(workspace),
                                           _nbytes(workspace, ws_bytes), ctypes.byref(args),
                                           _stream(stream)))


def gemm_rs_kernel_overlap(a_list, b_list, out_list, workspace, args: DtArgs, stream=None,
                           ws_bytes=None):
    _raise(lib().dt_gemm_rs_kernel_overlap(_ptr_array(a_list), _ptr_array(b_list),
                                           _ptr_array(out_list), _ptr(workspace),
                                           _nbytes(workspace, ws_bytes), ctypes.byref(args),
                                           _stream(stream)))


def gemm_a2a(a_list, b_list, out_list, workspace, args: DtArgs, stream=None, ws_bytes=None):
    """Fused GEMM-AllToAll: out_list[h] ([M, N/W]) receives columns h*N/W .. of every
    A_q @ B_q, rows stacked by source rank q."""
    _raise(lib().dt_gemm_a2a(_ptr_array(a_list), _ptr_array(b_list), _ptr_array(out_list),
                             _ptr(workspace), _nbytes(workspace, ws_bytes), ctypes.byref(args),
                             _stream(stream)))


def gemm_a2a_kernel_overlap(a_list, b_list, y_list, out_list, workspace, args: DtArgs,
                            stream=None, ws_bytes=None):
    """Baseline: per-step GEMMs into the ranks' own y_q ([M/W, N]) and copy-engine copies."""
    _raise(lib().dt_gemm_a2a_kernel_overlap(_ptr_array(a_list), _ptr_array(b_list),
                                            _ptr_array(y_list), _ptr_array(out_list),
                                            _ptr(workspace), _nbytes(workspace, ws_bytes),
                                            ctypes.byref(args), _stream(stream)))


def a2a_chunks(args: DtArgs) -> int:
    ms = args.m // args.world_size
    nc = -(-ms // args.chunk_rows) if ms > 0 else 0
    return args.world_size * args.world_size * nc


def a2a_signals(args: DtArgs, workspace, stream=None):
    """(flags, counts, epoch) of the last GEMM-AllToAll call on ``workspace``: uint32 arrays
    indexed (h * W + q) * nC + j (synchronises ``stream``)."""
    n = a2a_chunks(args)
    flags = np.zeros(n, dtype=np.uint32)
    counts = np.zeros(n, dtype=np.uint32)
    epoch = ctypes.c_uint32(0)
    _raise(lib().dt_a2a_signals(ctypes.byref(args), _ptr(workspace), _stream(stream),
                                flags.ctypes.data, counts.ctypes.data, n, ctypes.byref(epoch)))
    return flags, counts, int(epoch.value)


def tile_count(args: DtArgs, op: int) -> int:
    """Tiles of the execution order (the library's count, tile rows resolved)."""
    t = lib().dt_tile_count(ctypes.byref(args), op)
    if t < 0:
        _raise(DT_ERR_INVALID)
    return int(t)


def tile_rows(args: DtArgs, op: int) -> int:
    """Rows of one tile of the order: 128 (one CTA) or 256 (a CTA pair)."""
    r = lib().dt_tile_rows(ctypes.byref(args), op)
    if r < 0:
        _raise(DT_ERR_INVALID)
    return int(r)


def col_band(args: DtArgs, op: int) -> int:
    """Column tiles per column band of the ReduceScatter / AllReduce order (Tn: one band)."""
    r = lib().dt_col_band(ctypes.byref(args), op)
    if r < 0:
        _raise(DT_ERR_INVALID)
    return int(r)


def swizzle_plan(args: DtArgs, op: int) -> np.ndarray:
    """Host evaluation of the tile order (order[p] = tile run at position p)."""
    t = tile_count(args, op)
    out = np.zeros(t, dtype=np.int32)
    _raise(lib().dt_swizzle_plan(ctypes.byref(args), op, out.ctypes.data, t))
    return out


def swizzle_plan_device(args: DtArgs, op: int, order_dev, stream=None):
    """Device evaluation into ``order_dev`` (int32 device buffer of tile_count entries)."""
    _raise(lib().dt_swizzle_plan_device(ctypes.byref(args), op, _ptr(order_dev),
                                        tile_count(args, op), _stream(stream)))


_BACKEND_NAMES = {v: k for k, v in BACKENDS.items()}


def _points(buf, n):
    return [dict(chunk_rows=int(p.chunk_rows), backend=_BACKEND_NAMES.get(p.backend, p.backend),
                 copy_ctas=int(p.copy_ctas), swizzle=bool(p.swizzle), group=int(p.group),
                 tile_m=int(p.tile_m), col_band=int(p.col_band), ms=float(p.ms),
                 status=int(p.status)) for p in buf[:n]]


def tune_ag_gemm(shards, b, c, workspace, args: DtArgs, reps: int = 3, stream=None,
                 ws_bytes=None, max_points: int = 128):
    """Enumerate-and-measure tuner; writes the fastest knobs into `args`, returns the points."""
    buf = (DtTunePoint * max_points)()
    n = ctypes.c_int32(0)
    _raise(lib().dt_tune_ag_gemm(_ptr_array(shards), _ptr(b), _ptr(c), _ptr(workspace),
                                 _nbytes(workspace, ws_bytes), ctypes.byref(args), reps, buf,
                                 max_points, ctypes.byref(n), _stream(stream)))
    return _points(buf, min(n.value, max_points))


def tune_reduce(op: int, a_list, b_list, out_list, workspace, args: DtArgs, reps: int = 3,
                stream=None, ws_bytes=None, max_points: int = 128):
    """Tuner of dt_gemm_rs (op OP_RS), dt_gemm_ar (OP_AR) or dt_gemm_a2a (OP_A2A); writes the
    best into `args`."""
    buf = (DtTunePoint * max_points)()
    n = ctypes.c_int32(0)
    _raise(lib().dt_tune_reduce(op, _ptr_array(a_list), _ptr_array(b_list), _ptr_array(out_list),
                                _ptr(workspace), _nbytes(workspace, ws_bytes), ctypes.byref(args),
                                reps, buf, max_points, ctypes.byref(n), _stream(stream)))
    return _points(buf, min(n.value, max_points))


def ffn_ag_rs(x_shards, w1, w2_list, h, out_list, ws_ag, ws_rs, ag: DtArgs, rs: DtArgs,
              stream=None, ws_ag_bytes=None, ws_rs_bytes=None):
    """Tensor-parallel feed-forward block: h = act(AllGather(x) W1), out = ReduceScatter(h W2)."""
    _raise(lib().dt_ffn_ag_rs(_ptr_array(x_shards), _ptr(w1), _ptr_array(w2_list), _ptr(h),
                              _ptr_array(out_list), _ptr(ws_ag), _nbytes(ws_ag, ws_ag_bytes),
                              _ptr(ws_rs), _nbytes(ws_rs, ws_rs_bytes), ctypes.byref(ag),
                              ctypes.byref(rs), _stream(stream)))


def debug_drop_transfer(step: int):
    """Host-side fault injection: the next AllGather-GEMM call (any backend) leaves out the
    copy and the ready flag of transfer step `step`."""
    _raise(lib().dt_debug_drop_transfer(step))


def check(workspace, stream=None):
    """Synchronise, read and clear the device error word; returns (status, info[4])."""
    info = (ctypes.c_uint32 * 4)()
    st = lib().dt_check(_ptr(workspace), _stream(stream), info)
    return st, list(info)


def trace_bytes(args: DtArgs) -> int:
    n = lib().dt_trace_bytes(ctypes.byref(args))
    if n == 0:
        raise DtError(DT_ERR_INVALID, lib().dt_last_error().decode())
    return int(n)


def trace_attach(buf, nbytes=None):
    """Attach a device buffer (int64 / uint8 tensor or pointer) for the AllGather-GEMM's debug
    timeline; None detaches."""
    if buf is None:
        _raise(lib().dt_trace_attach(None, 0))
    else:
        _raise(lib().dt_trace_attach(_ptr(buf), _nbytes(buf, nbytes)))


def trace_decode(words, args: DtArgs) -> dict:
    """The timeline read back (a sequence of uint64 words) as times in microseconds from the
    first CTA's start; None where nothing was recorded."""
    none = (1 << 64) - 1
    w = [int(x) & none for x in words]
    t0 = w[0]

    def rel(x):
        return None if x == none else (x - t0) / 1e3

    ms = args.m // args.world_size
    nc = -(-ms // args.chunk_rows) if ms else 0
    chunks = {}
    for s in range(args.world_size):
        for j in range(nc):
            c = s * nc + j
            chunks[(s, j)] = {"released_us": rel(w[4 + 3 * c]), "first_miss_us": rel(w[5 + 3 * c]),
                              "first_read_us": rel(w[6 + 3 * c])}
    return {"kernel_us": rel(w[1]), "stall_us_total": w[2] / 1e3, "stalled_waits": w[3],
            "chunks": chunks}


def static_scratch_check(stream=None):
    """check() for the fixed scratch of the current device; returns (status, info[4])."""
    info = (ctypes.c_uint32 * 4)()
    st = lib().dt_static_scratch_check(_stream(stream), info)
    return st, list(info)
