"""Literal stage-by-stage simulation of the ring AllReduce -- TEST INFRASTRUCTURE.

A second oracle, independent of the C fold in `vr_oracle.c`: it shares no code
with it (its own chunk map, its own arithmetic via numpy / torch CPU ops) and
executes the schedule instead of evaluating a closed form. Small inputs only.

The schedule, from NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程:
  * ch.2 §2.2 (channel walkthrough, step 3): each channel owns a contiguous
    count/nChannels slice (reading: rounded up to 16 bytes of elements).
  * ch.2 §2.3 (RingARAlgorithm fields and getNextSendAddr): a loop has
    nStepsPerLoop = 2 (N - 1) sends; at loop stage s a rank sends chunk
    (ringIndex + N - 1 - (s mod N)) mod N; the last loop's chunk size is
    alignUp(divUp(rem, N), 16 / elemSize); a chunk's size is
    min(rem - chunkOffset, curChunkSize).
  * ch.2 §2.3 (same passage): each rank receives from its ring predecessor and
    sends to its successor; the reduce-scatter half adds the incoming partial to
    the rank's own chunk, the all-gather half forwards finished chunks.

Every message carries, as metadata, the chunk id and the set of ranks already
folded in, so the simulation also checks the ring invariants: the chunk a rank
receives is the one the formula says it sends next, and a finished chunk holds
every rank exactly once.
"""
from collections import deque

import numpy as np


def _ceil_div(a, b):
    return -(-a // b)


def _align_up(a, b):
    return _ceil_div(a, b) * b


# The 8-bit floating types: torch's formats and their largest finite values.
_FP8 = {"float8_e4m3": ("float8_e4m3fn", 448.0), "float8_e5m2": ("float8_e5m2", 57344.0)}


class _Arith:
    """Elementwise op in the element type, rounded after every op (library
    arithmetic: numpy for ints / float16 / float32 / float64, torch CPU for
    bfloat16; the 8-bit floating types compute in numpy float32 and round
    through torch's conversion after clamping to the largest finite value,
    which is how saturating round-to-nearest-even ends)."""

    def __init__(self, dtype, op):
        self.dtype, self.op = dtype, op

    def _fp8_round(self, w):
        import torch
        name, maxf = _FP8[self.dtype]
        with np.errstate(invalid="ignore"):
            c = np.clip(np.asarray(w, np.float32), -maxf, maxf)
        return torch.from_numpy(np.ascontiguousarray(c)).to(getattr(torch, name))

    def to_work(self, x):
        if self.dtype in _FP8:
            import torch
            t = torch.from_numpy(np.ascontiguousarray(x).view(np.uint8))
            return t.view(getattr(torch, _FP8[self.dtype][0])).to(torch.float32).numpy()
        if self.dtype == "bfloat16":
            import torch
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
        if self.dtype == "float16":
            return np.ascontiguousarray(x).view(np.float16)
        return np.ascontiguousarray(x)

    def from_work(self, w):
        if self.dtype in _FP8:
            import torch
            return self._fp8_round(w).view(torch.uint8).numpy()
        if self.dtype == "bfloat16":
            import torch
            return w.contiguous().view(torch.int16).numpy().view(np.uint16)
        return w

    def __call__(self, a, b):
        op = self.op
        if self.dtype == "bfloat16":
            import torch
            if op == "sum":
                return a + b
            if op == "prod":
                return a * b
            if op == "max":
                return torch.where(a > b, a, b)
            return torch.where(a < b, a, b)
        with np.errstate(over="ignore", invalid="ignore"):
            if op == "sum":
                r = a + b
            elif op == "prod":
                r = a * b
            elif op == "max":
                r = np.where(a > b, a, b)
            else:
                r = np.where(a < b, a, b)
        if self.dtype in _FP8:
            import torch
            return self._fp8_round(r).to(torch.float32).numpy()
        return r


def simulate(xs, dtype, op, n_channels, chunk_bytes):
    """Run the ring on the N rank buffers `xs`; return the N receive buffers."""
    N = len(xs)
    count = len(xs[0])
    e = np.dtype(xs[0].dtype).itemsize
    ar = _Arith(dtype, op)
    own = [ar.to_work(x) for x in xs]
    recv = [ar.to_work(np.zeros_like(x)) for x in xs]
    align = 16 // e
    chunk_elems = chunk_bytes // e
    per = _align_up(_ceil_div(count, n_channels), align)
    for ch in range(n_channels):
        cb = min(count, ch * per)
        ce = min(count, cb + per)
        size = ce - cb
        loop_size = N * chunk_elems
        n_steps_per_loop = 2 * (N - 1)
        for loop_off in range(0, size, loop_size):
            rem = size - loop_off
            cur = _align_up(_ceil_div(rem, N), align) if rem < loop_size else chunk_elems

            def chunk_span(cid):
                lo = cid * cur
                nelem = min(rem - lo, cur)
                if nelem <= 0:
                    return cb + loop_off, cb + loop_off  # empty chunk
                return cb + loop_off + lo, cb + loop_off + lo + nelem

            def send_chunk(ring_index, stage):
                return (ring_index + N - 1 - (stage % N)) % N

            if N == 1:
                b, t = chunk_span(0)
                recv[0][b:t] = own[0][b:t]
                continue
            fifo = [deque() for _ in range(N)]   # fifo[r]: edge r -> r+1
            # Stage s = 0 .. nStepsPerLoop: send at stages < nStepsPerLoop,
            # receive at stages >= 1.
            for s in range(n_steps_per_loop + 1):
                outgoing = []
                for r in range(N):
                    msg = None
                    if s >= 1:
                        cid, ranks, data = fifo[(r - 1) % N].popleft()
                        b, t = chunk_span(cid)
                        if s <= N - 1:                       # reduce-scatter: add own
                            assert r not in ranks
                            data = ar(data, own[r][b:t])
                            ranks = ranks + (r,)
                        if s >= N - 1:                       # finished: keep a copy
                            assert sorted(ranks) == list(range(N))
                            recv[r][b:t] = data
                        msg = (cid, ranks, data)
                    if s < n_steps_per_loop:
                        cid = send_chunk(r, s)
                        if msg is None:                      # stage 0: own chunk
                            b, t = chunk_span(cid)
                            msg = (cid, (r,), own[r][b:t].clone()
                                   if hasattr(own[r], "clone") else own[r][b:t].copy())
                        else:
                            assert msg[0] == cid, "ring invariant: forward what arrived"
                        outgoing.append((r, msg))
                for r, msg in outgoing:
                    fifo[r].append(msg)
            assert all(len(q) == 0 for q in fifo)
    return [ar.from_work(w) for w in recv]


def simulate_reduce_scatter(xs, dtype, op):
    """Literal ring reduce-scatter over the N blocks (one block per message):
    at stage s rank r sends block (r + N - 1 - s) mod N, the receiver adds its
    own copy of the block; after N - 1 transfers rank r holds block r."""
    N = len(xs)
    ar = _Arith(dtype, op)
    count = len(xs[0]) // N
    own = [ar.to_work(x) for x in xs]
    blk = lambda r, b: own[r][b * count:(b + 1) * count]
    if N == 1:
        return [ar.from_work(blk(0, 0))]
    fifo = [deque() for _ in range(N)]
    result = [None] * N
    for s in range(N):
        outgoing = []
        for r in range(N):
            if s == 0:
                b = (r + N - 1) % N
                outgoing.append((r, (b, (r,), blk(r, b))))
                continue
            b, ranks, data = fifo[(r - 1) % N].popleft()
            assert r not in ranks
            data = ar(data, blk(r, b))
            ranks = ranks + (r,)
            if s == N - 1:
                assert b == r and sorted(ranks) == list(range(N))
                result[r] = data
            else:
                assert b == (r + N - 1 - s) % N, "ring invariant"
                outgoing.append((r, (b, ranks, data)))
        for r, msg in outgoing:
            fifo[r].append(msg)
    return [ar.from_work(v) for v in result]


def simulate_all_gather(xs):
    """Literal ring all-gather: at stage s rank r forwards block (r - s) mod N."""
    N = len(xs)
    count = len(xs[0])
    outs = [np.zeros(N * count, xs[0].dtype) for _ in range(N)]
    for r in range(N):
        outs[r][r * count:(r + 1) * count] = xs[r]
    if N == 1:
        return outs
    fifo = [deque() for _ in range(N)]
    for s in range(N):
        outgoing = []
        for r in range(N):
            if s == 0:
                outgoing.append((r, (r, xs[r])))
                continue
            b, data = fifo[(r - 1) % N].popleft()
            assert b == (r - s) % N, "ring invariant"
            outs[r][b * count:(b + 1) * count] = data
            if s < N - 1:
                outgoing.append((r, (b, data)))
        for r, msg in outgoing:
            fifo[r].append(msg)
    assert all(len(q) == 0 for q in fifo)
    return outs
