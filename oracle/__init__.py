"""CPU oracle for the virtual-rank ring AllReduce -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline and
reference arm may import this package. The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

Two independent implementations live here:

* `allreduce` (C, `vr_oracle.c`): the closed-form ring-order fold. Chunk c of
  each loop starts at rank c+1 and visits ranks c+2, ..., c; the chunk map
  follows NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程, ch.2 §2.2 (channel
  split) and §2.3 (RingARAlgorithm::getNextSendAddr).
* `simulate.simulate` (Python): a literal stage-by-stage execution of the ring
  with one FIFO queue per edge, using library arithmetic (numpy, torch) for the
  element type. It must equal the fold on every input.

Element types are given by name: int8 uint8 int32 uint32 int64 uint64 float16
bfloat16 float32 float64 float8_e4m3 float8_e5m2. bfloat16 buffers are numpy
uint16 arrays of raw codes, the 8-bit floating types numpy uint8 arrays of raw
codes; float16 buffers may be numpy float16 or uint16 (same bits).
"""
import ctypes
import os

import numpy as np

from . import build as _build

DTYPES = {"int8": 0, "uint8": 1, "int32": 2, "uint32": 3, "int64": 4, "uint64": 5,
          "float16": 6, "bfloat16": 7, "float32": 8, "float64": 9,
          "float8_e4m3": 10, "float8_e5m2": 11}
ELEM_SIZE = {"int8": 1, "uint8": 1, "int32": 4, "uint32": 4, "int64": 8, "uint64": 8,
             "float16": 2, "bfloat16": 2, "float32": 4, "float64": 8,
             "float8_e4m3": 1, "float8_e5m2": 1}
NP_DTYPE = {"int8": np.int8, "uint8": np.uint8, "int32": np.int32, "uint32": np.uint32,
            "int64": np.int64, "uint64": np.uint64, "float16": np.float16,
            "bfloat16": np.uint16, "float32": np.float32, "float64": np.float64,
            "float8_e4m3": np.uint8, "float8_e5m2": np.uint8}
OPS = {"sum": 0, "prod": 1, "max": 2, "min": 3}
FLOAT_TYPES = ("float16", "bfloat16", "float32", "float64", "float8_e4m3", "float8_e5m2")

_u64 = ctypes.c_uint64
_libs = {}


def load(path=None):
    """Load (building first if needed) the oracle library at `path`."""
    if path is None:
        path = _build.build()
    if path not in _libs:
        lib = ctypes.CDLL(path)
        lib.oracle_allreduce.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _u64,
                                         ctypes.c_int, _u64, ctypes.POINTER(ctypes.c_void_p),
                                         ctypes.c_void_p, ctypes.c_int]
        lib.oracle_allreduce.restype = ctypes.c_int
        lib.oracle_allreduce_at.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _u64,
                                            ctypes.c_int, _u64, ctypes.c_void_p,
                                            ctypes.c_void_p, _u64, ctypes.c_void_p]
        lib.oracle_allreduce_at.restype = ctypes.c_int
        lib.oracle_reduce_scatter.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _u64,
                                              ctypes.POINTER(ctypes.c_void_p),
                                              ctypes.POINTER(ctypes.c_void_p)]
        lib.oracle_reduce_scatter.restype = ctypes.c_int
        lib.oracle_all_gather.argtypes = [ctypes.c_int, ctypes.c_int, _u64,
                                          ctypes.POINTER(ctypes.c_void_p),
                                          ctypes.POINTER(ctypes.c_void_p)]
        lib.oracle_all_gather.restype = ctypes.c_int
        lib.oracle_allreduce_scaled.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int64, ctypes.c_int,
            ctypes.c_int, _u64, ctypes.c_int, _u64, ctypes.POINTER(ctypes.c_void_p),
            ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
        lib.oracle_allreduce_scaled.restype = ctypes.c_int
        lib.oracle_tree_node.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int)]
        lib.oracle_tree_node.restype = None
        lib.oracle_tree_split.argtypes = [_u64, ctypes.c_int]
        lib.oracle_tree_split.restype = _u64
        lib.oracle_tree_allreduce.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _u64,
                                              ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p]
        lib.oracle_tree_allreduce.restype = ctypes.c_int
        lib.oracle_tree_allreduce_scaled.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int64, ctypes.c_int, _u64,
            ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p]
        lib.oracle_tree_allreduce_scaled.restype = ctypes.c_int
        lib.oracle_channel_range.argtypes = [_u64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.POINTER(_u64), ctypes.POINTER(_u64)]
        lib.oracle_channel_range.restype = None
        lib.oracle_num_chunk_ranges.argtypes = [_u64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                _u64]
        lib.oracle_num_chunk_ranges.restype = _u64
        lib.oracle_chunk_ranges.argtypes = [_u64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u64,
                                            _u64] + [ctypes.c_void_p] * 5
        lib.oracle_chunk_ranges.restype = _u64
        lib.oracle_round_to_format.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int]
        lib.oracle_round_to_format.restype = ctypes.c_double
        for name in ("oracle_f16_decode", "oracle_bf16_decode"):
            getattr(lib, name).argtypes = [ctypes.c_uint16]
            getattr(lib, name).restype = ctypes.c_double
        for name in ("oracle_f16_from_double", "oracle_bf16_from_double"):
            getattr(lib, name).argtypes = [ctypes.c_double]
            getattr(lib, name).restype = ctypes.c_uint16
        for name in ("oracle_fp8e4m3_decode", "oracle_fp8e5m2_decode"):
            getattr(lib, name).argtypes = [ctypes.c_uint8]
            getattr(lib, name).restype = ctypes.c_double
        for name in ("oracle_fp8e4m3_from_double", "oracle_fp8e5m2_from_double"):
            getattr(lib, name).argtypes = [ctypes.c_double]
            getattr(lib, name).restype = ctypes.c_uint8
        _libs[path] = lib
    return _libs[path]


def _check_buffers(xs, dtype):
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    es = ELEM_SIZE[dtype]
    count = len(xs[0])
    out = []
    for x in xs:
        x = np.ascontiguousarray(x)
        if x.itemsize != es or len(x) != count or x.ndim != 1:
            raise ValueError("every rank buffer must be 1-D, same length, element size "
                             f"{es} for {dtype}")
        out.append(x)
    return out, count


def allreduce(xs, dtype, op, n_channels, chunk_bytes, nthreads=1, lib=None):
    """Ring-order AllReduce of the rank buffers `xs` (a list of N 1-D arrays).

    Returns one array: the value every rank's receive buffer must hold.
    """
    xs, count = _check_buffers(xs, dtype)
    L = lib if lib is not None else load()
    out = np.empty_like(xs[0])
    ptrs = (ctypes.c_void_p * len(xs))(*[x.ctypes.data for x in xs])
    rc = L.oracle_allreduce(DTYPES[dtype], OPS[op], len(xs), count, n_channels, chunk_bytes,
                            ptrs, out.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError("oracle_allreduce rejected its arguments")
    return out


def allreduce_at(vals, idx, count, dtype, op, n_channels, chunk_bytes, lib=None):
    """The reduced value of selected elements only.

    vals: array [N, m] of the N ranks' values at the m element indices `idx`
    of buffers of `count` elements. Returns an array of m values.
    """
    L = lib if lib is not None else load()
    vals = np.ascontiguousarray(vals)
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    n, m = vals.shape
    if vals.itemsize != ELEM_SIZE[dtype] or len(idx) != m:
        raise ValueError("vals must be [N, m] of the element size; idx of length m")
    out = np.empty(m, vals.dtype)
    rc = L.oracle_allreduce_at(DTYPES[dtype], OPS[op], n, count, n_channels, chunk_bytes,
                               vals.ctypes.data, idx.ctypes.data, m, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_allreduce_at rejected its arguments")
    return out


def allreduce_scaled(xs, dtype, kind, scalar, n_channels, chunk_bytes, nthreads=1, lib=None):
    """AllReduce with the average (kind "avg") or the pre-multiplied sum
    (kind "premulsum", by `scalar`: a float for floating types, an int for
    integer types) in the ring's order; returns the result."""
    xs, count = _check_buffers(xs, dtype)
    L = lib if lib is not None else load()
    out = np.empty(count, xs[0].dtype)
    xp = (ctypes.c_void_p * len(xs))(*[x.ctypes.data for x in xs])
    op_ = (ctypes.c_void_p * 1)(out.ctypes.data)
    k = {"premulsum": 0, "avg": 1}[kind]
    fs = float(scalar) if kind == "premulsum" and dtype in FLOAT_TYPES else 0.0
    is_ = int(scalar) if kind == "premulsum" and dtype not in FLOAT_TYPES else 0
    if L.oracle_allreduce_scaled(DTYPES[dtype], k, fs, is_, 0, len(xs), count, n_channels,
                                 chunk_bytes, xp, op_, nthreads) != 0:
        raise ValueError("oracle_allreduce_scaled rejected its arguments")
    return out


def reduce_scatter_scaled(xs, dtype, kind, scalar, lib=None):
    """ReduceScatter with the average or the pre-multiplied sum."""
    xs, count = _check_buffers(xs, dtype)
    n = len(xs)
    L = lib if lib is not None else load()
    outs = [np.empty(count // n, xs[0].dtype) for _ in range(n)]
    xp = (ctypes.c_void_p * n)(*[x.ctypes.data for x in xs])
    op_ = (ctypes.c_void_p * n)(*[o.ctypes.data for o in outs])
    k = {"premulsum": 0, "avg": 1}[kind]
    fs = float(scalar) if kind == "premulsum" and dtype in FLOAT_TYPES else 0.0
    is_ = int(scalar) if kind == "premulsum" and dtype not in FLOAT_TYPES else 0
    if L.oracle_allreduce_scaled(DTYPES[dtype], k, fs, is_, 1, n, count, 1, 16, xp, op_,
                                 1) != 0:
        raise ValueError("oracle_allreduce_scaled rejected its arguments")
    return outs


def tree_node(n, rank, tree, lib=None):
    """(parent, child0, child1) of `rank` in double-binary-tree `tree` (0 or
    1) of n ranks; -1 where there is none."""
    L = lib if lib is not None else load()
    u, a, b = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    L.oracle_tree_node(n, rank, tree, ctypes.byref(u), ctypes.byref(a), ctypes.byref(b))
    return u.value, a.value, b.value


def tree_split(count, elem_size, lib=None):
    """First element reduced by the second tree."""
    L = lib if lib is not None else load()
    return L.oracle_tree_split(count, elem_size)


def tree_allreduce(xs, dtype, op, lib=None):
    """Double-binary-tree AllReduce of the N buffers `xs`: the first half of
    the elements reduced by tree 0, the rest by tree 1; returns the result
    (every rank's output)."""
    xs, count = _check_buffers(xs, dtype)
    L = lib if lib is not None else load()
    out = np.empty(count, xs[0].dtype)
    xp = (ctypes.c_void_p * len(xs))(*[x.ctypes.data for x in xs])
    if L.oracle_tree_allreduce(DTYPES[dtype], OPS[op], len(xs), count, xp,
                               out.ctypes.data) != 0:
        raise ValueError("oracle_tree_allreduce rejected its arguments")
    return out


def tree_allreduce_scaled(xs, dtype, kind, scalar, lib=None):
    """Double-binary-tree AllReduce with the average (kind "avg") or the
    pre-multiplied sum (kind "premulsum", by `scalar`)."""
    xs, count = _check_buffers(xs, dtype)
    L = lib if lib is not None else load()
    out = np.empty(count, xs[0].dtype)
    xp = (ctypes.c_void_p * len(xs))(*[x.ctypes.data for x in xs])
    k = {"premulsum": 0, "avg": 1}[kind]
    fs = float(scalar) if kind == "premulsum" and dtype in FLOAT_TYPES else 0.0
    is_ = int(scalar) if kind == "premulsum" and dtype not in FLOAT_TYPES else 0
    if L.oracle_tree_allreduce_scaled(DTYPES[dtype], k, fs, is_, len(xs), count, xp,
                                      out.ctypes.data) != 0:
        raise ValueError("oracle_tree_allreduce_scaled rejected its arguments")
    return out


def reduce_scatter(xs, dtype, op, lib=None):
    """Ring ReduceScatter: xs are N buffers of N * recvcount elements; returns
    the N outputs (rank b: the ring-order reduction of block b)."""
    xs, count = _check_buffers(xs, dtype)
    n = len(xs)
    if count % n:
        raise ValueError("each send buffer holds N blocks")
    recvcount = count // n
    L = lib if lib is not None else load()
    outs = [np.empty(recvcount, xs[0].dtype) for _ in range(n)]
    xp = (ctypes.c_void_p * n)(*[x.ctypes.data for x in xs])
    op_ = (ctypes.c_void_p * n)(*[o.ctypes.data for o in outs])
    if L.oracle_reduce_scatter(DTYPES[dtype], OPS[op], n, recvcount, xp, op_) != 0:
        raise ValueError("oracle_reduce_scatter rejected its arguments")
    return outs


def all_gather(xs, dtype, lib=None):
    """AllGather: returns the N outputs, each the concatenation of xs."""
    xs, count = _check_buffers(xs, dtype)
    n = len(xs)
    L = lib if lib is not None else load()
    outs = [np.empty(n * count, xs[0].dtype) for _ in range(n)]
    xp = (ctypes.c_void_p * n)(*[x.ctypes.data for x in xs])
    op_ = (ctypes.c_void_p * n)(*[o.ctypes.data for o in outs])
    if L.oracle_all_gather(ELEM_SIZE[dtype], n, count, xp, op_) != 0:
        raise ValueError("oracle_all_gather rejected its arguments")
    return outs


def channel_range(count, n_channels, elem_size, ch, lib=None):
    """[begin, end) of channel `ch`."""
    L = lib if lib is not None else load()
    b, e = _u64(), _u64()
    L.oracle_channel_range(count, n_channels, elem_size, ch, ctypes.byref(b), ctypes.byref(e))
    return b.value, e.value


def chunk_ranges(count, n_ranks, n_channels, elem_size, chunk_bytes, lib=None):
    """Every non-empty chunk in schedule order, as a dict of numpy arrays with keys
    channel, loop, chunk, begin, end (absolute element offsets)."""
    L = lib if lib is not None else load()
    n = L.oracle_num_chunk_ranges(count, n_ranks, n_channels, elem_size, chunk_bytes)
    ch = np.zeros(n, np.int32)
    lp = np.zeros(n, np.int64)
    ck = np.zeros(n, np.int32)
    b = np.zeros(n, np.uint64)
    e = np.zeros(n, np.uint64)
    L.oracle_chunk_ranges(count, n_ranks, n_channels, elem_size, chunk_bytes, n,
                          ch.ctypes.data, lp.ctypes.data, ck.ctypes.data, b.ctypes.data,
                          e.ctypes.data)
    return {"channel": ch, "loop": lp, "chunk": ck, "begin": b, "end": e}


def round_to_format(x, p, emin, emax, lib=None):
    L = lib if lib is not None else load()
    return L.oracle_round_to_format(float(x), p, emin, emax)


def f16_from_double(x, lib=None):
    return (lib or load()).oracle_f16_from_double(float(x))


def bf16_from_double(x, lib=None):
    return (lib or load()).oracle_bf16_from_double(float(x))


def f16_decode(h, lib=None):
    return (lib or load()).oracle_f16_decode(int(h))


def bf16_decode(h, lib=None):
    return (lib or load()).oracle_bf16_decode(int(h))


def fp8_decode(h, fmt, lib=None):
    """Value of the 8-bit code `h` of format "e4m3" or "e5m2"."""
    return getattr(lib or load(), f"oracle_fp8{fmt}_decode")(int(h))


def fp8_from_double(x, fmt, lib=None):
    """Code of x rounded to format "e4m3" or "e5m2" (nearest even, saturating)."""
    return getattr(lib or load(), f"oracle_fp8{fmt}_from_double")(float(x))
