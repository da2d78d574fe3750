"""Virtual-rank ring AllReduce on one GPU: Python binding of libvr.so.

The functions named like the C ABI (include/vr.h) only marshal arguments;
every step of the AllReduce runs in the library's CUDA kernels. There is no
CPU fallback: if libvr.so has not been built, every call raises ImportError.

    import ring_allreduce_virtual_gb300 as vr
    comm = vr.Communicator(n_ranks=8, n_channels=16, proto="simple",
                           chunk_bytes=512 << 10)
    comm.all_reduce(send_tensors, recv_tensors, op="sum")   # on the current stream

Build the library with `python -m ring_allreduce_virtual_gb300.build`.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvr.so")

PROTOS = {"simple": 0, "ll": 1, "ll128": 2}
DTYPES = {"int8": 0, "uint8": 1, "int32": 2, "uint32": 3, "int64": 4, "uint64": 5,
          "float16": 6, "bfloat16": 7, "float32": 8, "float64": 9, "float8_e4m3": 10,
          "float8_e5m2": 11}
OPS = {"sum": 0, "prod": 1, "max": 2, "min": 3, "avg": 4}
RESULTS = {0: "vrSuccess", 1: "vrInvalidArgument", 2: "vrInvalidUsage", 3: "vrCudaError",
           4: "vrInternalError", 5: "vrTimeout"}
vrSuccess, vrInvalidArgument, vrInvalidUsage, vrCudaError, vrInternalError, vrTimeout = range(6)
TRANSPORTS = {0: "global", 2: "warp", 3: "warpcluster"}
MAX_RANKS = 128


class VrError(RuntimeError):
    """A non-success vrResult_t; `.code` holds the raw value."""

    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {RESULTS.get(code, code)} ({vrGetErrorString(code)})")


_lib_handle = None


def lib():
    """The loaded libvr.so (ctypes). Raises ImportError if it was not built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m ring_allreduce_virtual_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
        L.vrCommCreate.argtypes = [ctypes.POINTER(vp), i32, i32, i32, sz]
        L.vrAllReduce.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i32, i32, vp]
        L.vrCommDestroy.argtypes = [vp]
        L.vrCommGetAsyncError.argtypes = [vp, ctypes.POINTER(i32)]
        L.vrCommSetTimeout.argtypes = [vp, u64]
        L.vrCommGetInfo.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                    ctypes.POINTER(i32), ctypes.POINTER(sz)]
        L.vrGetErrorString.argtypes = [i32]
        L.vrGetErrorString.restype = ctypes.c_char_p
        L.vrReduceScatter.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i32, i32, vp]
        L.vrAllGather.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i32, vp]
        L.vrRingWalk.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i32, i32, vp]
        L.vrAllReduceTree.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i32, i32,
                                      vp]
        L.vrCommGetPlan.argtypes = [vp, sz, i32, ctypes.POINTER(sz), ctypes.POINTER(i32)]
        L.vrAllReduceNoAlloc.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), sz, i32, i32,
                                         i32, sz, i32, i32, vp]
        L.vrAllReduceNoAllocGetStatus.argtypes = [ctypes.POINTER(i32)]
        L.vrRedOpCreatePreMulSum.argtypes = [ctypes.POINTER(i32), ctypes.c_char_p, i32, vp]
        L.vrRedOpDestroy.argtypes = [i32, vp]
        for name in ("vrCommCreate", "vrAllReduce", "vrCommDestroy", "vrCommGetAsyncError",
                     "vrCommSetTimeout", "vrCommGetInfo", "vrAllReduceNoAlloc",
                     "vrAllReduceNoAllocGetStatus",
                     "vrReduceScatter", "vrAllGather", "vrRingWalk", "vrCommGetPlan",
                     "vrAllReduceTree", "vrRedOpCreatePreMulSum", "vrRedOpDestroy"):
            getattr(L, name).restype = i32
        _lib_handle = L
    return _lib_handle


def _code(table, v, what):
    if isinstance(v, str):
        if v not in table:
            raise ValueError(f"unknown {what} {v!r}")
        return table[v]
    return int(v)


def _check(rc, where):
    if rc != vrSuccess:
        raise VrError(rc, where)


# --------------------------------------------------------------- C ABI names
def vrGetErrorString(result):
    return lib().vrGetErrorString(int(result)).decode()


def vrCommCreate(nRanks, nChannels, proto, chunkBytes):
    """Returns the communicator handle (an int)."""
    h = ctypes.c_void_p()
    _check(lib().vrCommCreate(ctypes.byref(h), int(nRanks), int(nChannels),
                              _code(PROTOS, proto, "protocol"), int(chunkBytes)), "vrCommCreate")
    return h.value


def vrAllReduce(comm, sendbufs, recvbufs, count, dtype, op, stream=0):
    """sendbufs / recvbufs: sequences of device addresses (ints)."""
    n = len(sendbufs)
    sb = (ctypes.c_void_p * n)(*[int(p) for p in sendbufs])
    rb = (ctypes.c_void_p * len(recvbufs))(*[int(p) for p in recvbufs])
    _check(lib().vrAllReduce(comm, sb, rb, int(count), _code(DTYPES, dtype, "dtype"),
                             _code(OPS, op, "op"), int(stream) or None), "vrAllReduce")


def vrReduceScatter(comm, sendbufs, recvbufs, recvcount, dtype, op, stream=0):
    sb = (ctypes.c_void_p * len(sendbufs))(*[int(p) for p in sendbufs])
    rb = (ctypes.c_void_p * len(recvbufs))(*[int(p) for p in recvbufs])
    _check(lib().vrReduceScatter(comm, sb, rb, int(recvcount), _code(DTYPES, dtype, "dtype"),
                                 _code(OPS, op, "op"), int(stream) or None), "vrReduceScatter")


def vrAllGather(comm, sendbufs, recvbufs, sendcount, dtype, stream=0):
    sb = (ctypes.c_void_p * len(sendbufs))(*[int(p) for p in sendbufs])
    rb = (ctypes.c_void_p * len(recvbufs))(*[int(p) for p in recvbufs])
    _check(lib().vrAllGather(comm, sb, rb, int(sendcount), _code(DTYPES, dtype, "dtype"),
                             int(stream) or None), "vrAllGather")


def vrAllReduceTree(comm, sendbufs, recvbufs, count, dtype, op, stream=0):
    sb = (ctypes.c_void_p * len(sendbufs))(*[int(p) for p in sendbufs])
    rb = (ctypes.c_void_p * len(recvbufs))(*[int(p) for p in recvbufs])
    _check(lib().vrAllReduceTree(comm, sb, rb, int(count), _code(DTYPES, dtype, "dtype"),
                                 _code(OPS, op, "op"), int(stream) or None), "vrAllReduceTree")


def vrRingWalk(comm, sendbufs, recvbufs, count, dtype, op, stream=0):
    sb = (ctypes.c_void_p * len(sendbufs))(*[int(p) for p in sendbufs])
    rb = (ctypes.c_void_p * len(recvbufs))(*[int(p) for p in recvbufs])
    _check(lib().vrRingWalk(comm, sb, rb, int(count), _code(DTYPES, dtype, "dtype"),
                            _code(OPS, op, "op"), int(stream) or None), "vrRingWalk")


def vrCommGetPlan(comm, count, dtype):
    """(parts, rings) of one AllReduce of `count` elements: ring passes and
    rings running at once."""
    parts, rings = ctypes.c_size_t(), ctypes.c_int()
    _check(lib().vrCommGetPlan(comm, int(count), _code(DTYPES, dtype, "dtype"),
                               ctypes.byref(parts), ctypes.byref(rings)), "vrCommGetPlan")
    return parts.value, rings.value


_ELEM_SIZE = {"int8": 1, "uint8": 1, "int32": 4, "uint32": 4, "int64": 8, "uint64": 8,
              "float16": 2, "bfloat16": 2, "float32": 4, "float64": 8, "float8_e4m3": 1,
              "float8_e5m2": 1}


def _scalar_bytes(scalar, dtype):
    """One element of `dtype` as little-endian bytes: a bytes object is taken
    as it is; an integer type takes int(scalar) modulo 2^bits (wrapping, like
    the C cast); float16/32/64 round float(scalar) to nearest even (numpy);
    bfloat16 rounds it to float32 and then to bfloat16 (torch's conversions,
    both to nearest even; exact for any value that a float32 holds); the 8-bit floating types round
    it to float32, clamp it to the largest finite value and round it with
    torch's conversion (nearest even)."""
    import numpy as np
    es = _ELEM_SIZE[dtype]
    if isinstance(scalar, (bytes, bytearray)):
        if len(scalar) != es:
            raise ValueError(f"scalar bytes must be {es} long for {dtype}")
        return bytes(scalar)
    if dtype in ("float16", "float32", "float64"):
        return np.array(float(scalar), {"float16": np.float16, "float32": np.float32,
                                        "float64": np.float64}[dtype]).tobytes()
    if dtype in ("float8_e4m3", "float8_e5m2"):
        import torch
        tdt, top = ((torch.float8_e4m3fn, 448.0) if dtype == "float8_e4m3"
                    else (torch.float8_e5m2, 57344.0))
        f = np.clip(np.array([float(scalar)], np.float32), -top, top)
        return torch.from_numpy(f).to(tdt).view(torch.uint8).numpy().tobytes()
    if dtype == "bfloat16":
        import torch
        f = torch.tensor([float(scalar)], dtype=torch.float32)
        return f.to(torch.bfloat16).view(torch.int16).numpy().tobytes()
    return (int(scalar) & ((1 << (8 * es)) - 1)).to_bytes(es, "little")


def vrRedOpCreatePreMulSum(comm, scalar, dtype):
    """A pre-multiplied sum by `scalar` for `dtype` on `comm`; returns the op
    (an int >= vrNumOps, usable wherever an op name is)."""
    op = ctypes.c_int()
    _check(lib().vrRedOpCreatePreMulSum(ctypes.byref(op), _scalar_bytes(scalar, dtype),
                                        _code(DTYPES, dtype, "dtype"), comm),
           "vrRedOpCreatePreMulSum")
    return op.value


def vrRedOpDestroy(op, comm):
    _check(lib().vrRedOpDestroy(int(op), comm), "vrRedOpDestroy")


def vrCommDestroy(comm):
    _check(lib().vrCommDestroy(comm), "vrCommDestroy")


def vrCommGetAsyncError(comm):
    """Returns the vrResult_t of errors found after enqueue (vrSuccess or vrTimeout)."""
    e = ctypes.c_int()
    _check(lib().vrCommGetAsyncError(comm, ctypes.byref(e)), "vrCommGetAsyncError")
    return e.value


def vrCommSetTimeout(comm, timeoutMs):
    _check(lib().vrCommSetTimeout(comm, int(timeoutMs)), "vrCommSetTimeout")


def vrCommGetInfo(comm):
    t, s, d, b = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    _check(lib().vrCommGetInfo(comm, ctypes.byref(t), ctypes.byref(s), ctypes.byref(d),
                               ctypes.byref(b)), "vrCommGetInfo")
    return {"transport": TRANSPORTS.get(t.value, t.value), "slot_bytes": s.value,
            "depth": d.value, "device_bytes": b.value}


def vrAllReduceNoAlloc(sendbufs, recvbufs, count, nRanks, nChannels, proto, chunkBytes, dtype,
                       op, stream=0):
    """AllReduce without a communicator and without allocating: for callers
    that cannot allocate device memory where they need it (see include/vr.h).
    sendbufs / recvbufs: sequences of nRanks device addresses (ints); with
    count 0 they may be empty (the call then only sets the device up)."""
    if int(count) != 0 and (len(sendbufs) != int(nRanks) or len(recvbufs) != int(nRanks)):
        raise ValueError(f"need {int(nRanks)} send and receive addresses, got "
                         f"{len(sendbufs)} and {len(recvbufs)}")
    sb = (ctypes.c_void_p * max(1, len(sendbufs)))(*[int(p) for p in sendbufs])
    rb = (ctypes.c_void_p * max(1, len(recvbufs)))(*[int(p) for p in recvbufs])
    _check(lib().vrAllReduceNoAlloc(sb, rb, int(count), int(nRanks), int(nChannels),
                                    _code(PROTOS, proto, "protocol"), int(chunkBytes),
                                    _code(DTYPES, dtype, "dtype"), _code(OPS, op, "op"),
                                    int(stream) or None), "vrAllReduceNoAlloc")


def vrAllReduceNoAllocGetStatus():
    """vrSuccess, or vrTimeout if a device wait of the last vrAllReduceNoAlloc
    call on the current device gave up (read after synchronising its stream,
    before the next call)."""
    e = ctypes.c_int()
    _check(lib().vrAllReduceNoAllocGetStatus(ctypes.byref(e)), "vrAllReduceNoAllocGetStatus")
    return e.value


# ------------------------------------------------------------ torch helper
_TORCH_NAMES = {"torch.int8": "int8", "torch.uint8": "uint8", "torch.int32": "int32",
                "torch.uint32": "uint32", "torch.int64": "int64", "torch.uint64": "uint64",
                "torch.float16": "float16", "torch.bfloat16": "bfloat16",
                "torch.float32": "float32", "torch.float64": "float64",
                "torch.float8_e4m3fn": "float8_e4m3", "torch.float8_e5m2": "float8_e5m2"}


class Communicator:
    """A communicator over `n_ranks` virtual ranks on the current CUDA device."""

    def __init__(self, n_ranks, n_channels, proto="simple", chunk_bytes=512 << 10):
        self.n_ranks, self.n_channels = n_ranks, n_channels
        self.proto, self.chunk_bytes = proto, chunk_bytes
        self.handle = vrCommCreate(n_ranks, n_channels, proto, chunk_bytes)

    def info(self):
        return vrCommGetInfo(self.handle)

    def set_timeout(self, ms):
        vrCommSetTimeout(self.handle, ms)

    def async_error(self):
        return vrCommGetAsyncError(self.handle)

    def all_reduce(self, sends, recvs, op="sum", stream=None, dtype=None):
        """Enqueue the AllReduce of the N CUDA tensors `sends` into `recvs`
        (same dtype, same element count, contiguous) on `stream` (default: the
        current torch stream). `dtype` (a name) overrides the element type
        taken from the tensors, e.g. "uint32" for int32 tensors holding
        unsigned values."""
        import torch
        if len(sends) != self.n_ranks or len(recvs) != self.n_ranks:
            raise ValueError("need one send and one receive tensor per rank")
        t0 = sends[0]
        if dtype is None:
            dtype = _TORCH_NAMES.get(str(t0.dtype))
        elif torch.empty(0, dtype=t0.dtype).element_size() != _ELEM_SIZE.get(dtype, 0):
            raise ValueError(f"dtype {dtype} does not match the tensors' element size")
        if dtype is None:
            raise ValueError(f"unsupported dtype {t0.dtype}")
        for t in list(sends) + list(recvs):
            if not t.is_cuda or t.dtype != t0.dtype or t.numel() != t0.numel() or \
                    not t.is_contiguous():
                raise ValueError("tensors must be contiguous CUDA tensors of one dtype and size")
        if stream is None:
            stream = torch.cuda.current_stream()
        vrAllReduce(self.handle, [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs],
                    t0.numel(), dtype, op, stream.cuda_stream)

    def _marshal(self, sends, recvs, dtype, send_numel=None, recv_numel=None):
        import torch
        if len(sends) != self.n_ranks or len(recvs) != self.n_ranks:
            raise ValueError("need one send and one receive tensor per rank")
        t0 = sends[0]
        if dtype is None:
            dtype = _TORCH_NAMES.get(str(t0.dtype))
        if dtype is None:
            raise ValueError(f"unsupported dtype {t0.dtype}")
        for t, n in [(t, send_numel) for t in sends] + [(t, recv_numel) for t in recvs]:
            if not t.is_cuda or t.dtype != t0.dtype or t.numel() != n or not t.is_contiguous():
                raise ValueError("tensors must be contiguous CUDA tensors of one dtype and the "
                                 "collective's sizes")
        return dtype, torch.cuda.current_stream()

    def reduce_scatter(self, sends, recvs, op="sum", stream=None, dtype=None):
        """recvs[r] (n elements) = ring reduction of block r of every sends[k]
        (N * n elements)."""
        n = recvs[0].numel()
        dtype, cur = self._marshal(sends, recvs, dtype, self.n_ranks * n, n)
        vrReduceScatter(self.handle, [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs],
                        n, dtype, op, (stream or cur).cuda_stream)

    def all_gather(self, sends, recvs, stream=None, dtype=None):
        """recvs[r] (N * n elements) = concatenation of sends (n elements each)."""
        n = sends[0].numel()
        dtype, cur = self._marshal(sends, recvs, dtype, n, self.n_ranks * n)
        vrAllGather(self.handle, [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs],
                    n, dtype, (stream or cur).cuda_stream)

    def premul_sum(self, scalar, dtype):
        """A reduction op: the sum of every rank's element times `scalar`
        (rounded to `dtype`); valid on this communicator for `dtype` only."""
        return vrRedOpCreatePreMulSum(self.handle, scalar, dtype)

    def destroy_op(self, op):
        vrRedOpDestroy(op, self.handle)

    def plan(self, count, dtype):
        """(parts, rings) of one AllReduce of `count` elements of `dtype`."""
        return vrCommGetPlan(self.handle, count, dtype)

    def all_reduce_tree(self, sends, recvs, op="sum", stream=None, dtype=None):
        """The AllReduce by the double binary tree (another reduction order)."""
        n = sends[0].numel()
        dtype, cur = self._marshal(sends, recvs, dtype, n, n)
        vrAllReduceTree(self.handle, [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs],
                        n, dtype, op, (stream or cur).cuda_stream)

    def ring_walk(self, sends, recvs, op="sum", stream=None, dtype=None):
        """The calibration fold: the AllReduce's result computed without the
        ring (every input read once, every output written once)."""
        n = sends[0].numel()
        dtype, cur = self._marshal(sends, recvs, dtype, n, n)
        vrRingWalk(self.handle, [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs],
                   n, dtype, op, (stream or cur).cuda_stream)

    def destroy(self):
        if self.handle is not None:
            h, self.handle = self.handle, None
            vrCommDestroy(h)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()
