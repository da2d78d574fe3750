"""Helpers of the GPU parity tests: run the CUDA path through the binding on
seeded inputs and compare every rank's output with the CPU oracle."""
import numpy as np
import torch

import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic

GUARD = 64          # guard elements before and after every output buffer
GUARD_BYTE = 0xA5


def guarded(count, tdtype, dev, offset=0, fill=None):
    """A buffer of `count` elements inside guard regions; `offset` extra
    elements in front shift its address (to test unaligned pointers)."""
    base = torch.empty(count + 2 * GUARD + offset, dtype=tdtype, device=dev)
    base.view(torch.uint8).fill_(GUARD_BYTE)
    view = base[GUARD + offset: GUARD + offset + count]
    if fill is not None:
        view.copy_(fill)
    return base, view


def guards_intact(base, count, offset=0):
    b = base.view(torch.uint8)
    es = base.element_size()
    head = b[: (GUARD + offset) * es]
    tail = b[(GUARD + offset + count) * es:]
    return bool((head == GUARD_BYTE).all()) and bool((tail == GUARD_BYTE).all())


def bytes_equal(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8),
                          np.ascontiguousarray(b).view(np.uint8))


def make_comm(n, nch, proto, chunk):
    """A communicator; a protocol name with a suffix "-global", "-warp" or
    "-warpcluster" forces that FIFO transport (VR_TRANSPORT) instead of letting the
    library pick."""
    import os
    transport = None
    if "-" in proto:
        proto, transport = proto.split("-", 1)
    old = os.environ.get("VR_TRANSPORT")
    if transport:
        os.environ["VR_TRANSPORT"] = transport
    try:
        return vr.Communicator(n, nch, proto, chunk)
    finally:
        if transport:
            if old is None:
                del os.environ["VR_TRANSPORT"]
            else:
                os.environ["VR_TRANSPORT"] = old


def run_case(n, count, dtype, op, proto, nch, chunk, dist=None, seed=0, inplace=False,
             offset=0, comm=None, xs=None, method="all_reduce"):
    """Run one AllReduce on the GPU and check it against the oracle, element
    by element, on every rank; also check guard regions and untouched inputs.
    `method` names the Communicator call: all_reduce (the ring) or ring_walk
    (the calibration fold)."""
    dev = torch.device("cuda")
    dist = dist or synthetic.default_recipe(dtype)
    if xs is None:
        xs = synthetic.rank_buffers(n, count, dtype, dist, seed, "cpu")
    tdt = synthetic.TORCH_DTYPE[dtype]
    own = comm is None
    if own:
        comm = make_comm(n, nch, proto, chunk)
    try:
        sends, recvs, bases = [], [], []
        for x in xs:
            sb, sv = guarded(count, tdt, dev, offset, fill=x)
            if inplace:
                sends.append(sv)
                recvs.append(sv)
                bases.append(sb)
            else:
                rb, rv = guarded(count, tdt, dev, offset)
                sends.append(sv)
                recvs.append(rv)
                bases.append((sb, rb))
        getattr(comm, method)(sends, recvs, op, dtype=dtype)
        torch.cuda.synchronize()
        assert comm.async_error() == vr.vrSuccess
        host = [synthetic.to_numpy(x) for x in xs]
        want = oracle.allreduce(host, dtype, op, nch, chunk, nthreads=8)
        for r in range(n):
            got = synthetic.to_numpy(recvs[r])
            if not bytes_equal(got, want):
                bad = np.nonzero(got.view(np.uint8) != want.view(np.uint8))[0]
                raise AssertionError(f"rank {r}: {len(bad)} bytes differ, first at byte "
                                     f"{bad[0]} (n={n} count={count} {dtype} {op} {proto} "
                                     f"nch={nch} chunk={chunk})")
            if inplace:
                assert guards_intact(bases[r], count, offset), f"guard overwritten, rank {r}"
            else:
                sb, rb = bases[r]
                assert guards_intact(rb, count, offset), f"guard overwritten, rank {r}"
                assert guards_intact(sb, count, offset), f"send guard overwritten, rank {r}"
                assert bytes_equal(synthetic.to_numpy(sends[r]), host[r]), f"input {r} modified"
        return want
    finally:
        if own:
            comm.destroy()


def sample_indices(count, n, nch, es, chunk, rng, m=20000):
    """Random element indices plus the first, second and last element of every
    chunk of the schedule (where chunk and channel boundaries fall)."""
    idx = [rng.integers(0, count, min(m, count), dtype=np.uint64)]
    ranges = oracle.chunk_ranges(count, n, nch, es, chunk)
    b, e = ranges["begin"], ranges["end"]
    idx += [b, np.minimum(b + 1, e - 1), e - 1]
    idx.append(np.array([0, count - 1], np.uint64))
    return np.unique(np.concatenate(idx).astype(np.uint64))


def check_sampled(xs, recvs, dtype, op, nch, chunk, rng, m=20000):
    """Full-size check: every output equals rank 0's (whole buffers, on the
    device) and sampled elements equal the oracle's per-element value.
    Returns (number of sampled elements, sampled oracle values, sampled inputs)."""
    n = len(xs)
    count = xs[0].numel()
    for r in range(1, n):
        assert torch.equal(recvs[r].view(torch.uint8), recvs[0].view(torch.uint8)), \
            f"rank {r} output differs from rank 0"
    es = xs[0].element_size()
    idx = sample_indices(count, n, nch, es, chunk, rng, m)
    it = torch.from_numpy(idx.astype(np.int64)).to(xs[0].device)
    vals = np.stack([synthetic.to_numpy(x[it]) for x in xs])
    want = oracle.allreduce_at(vals, idx, count, dtype, op, nch, chunk)
    got = synthetic.to_numpy(recvs[0][it])
    if not bytes_equal(got, want):
        g = got.view(np.uint8).reshape(len(idx), -1)
        w = want.view(np.uint8).reshape(len(idx), -1)
        diff = idx[np.nonzero((g != w).any(axis=1))[0]].tolist()
        raise AssertionError(f"{len(diff)} of {len(idx)} sampled elements differ, "
                             f"first at index {diff[:5]}")
    return len(idx), want, vals
