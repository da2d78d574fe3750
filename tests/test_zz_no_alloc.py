"""vrAllReduceNoAlloc (GPU): the AllReduce for callers that cannot allocate
device memory where they need it -- code under a framework's caching
allocator that must account for every device byte, or a latency-critical path
where cudaMalloc would stall the device. Its scratch is a fixed array the
library defines in device memory, shared by every call.

Called through the C ABI (the binding only marshals arguments), its outputs
must equal, bit for bit, those of the communicator entry point on the
global-memory FIFO transport with the same ring parameters, and the oracle's,
on two calls in a row (the second call must not be disturbed by what the
first left in the shared scratch). A call with count 0 is the warm-up that
sets a device up; the geometry limit (nChannels * nRanks <= 496) is checked
on both sides. This file is collected last on purpose."""
import os

import pytest
import torch

import gpu_helpers as H
import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


def _reference(xs, n, nch, proto, chunk, dtype, op):
    """The same AllReduce through vrCommCreate / vrAllReduce, global FIFOs."""
    old = os.environ.get("VR_TRANSPORT")
    os.environ["VR_TRANSPORT"] = "global"
    try:
        comm = vr.Communicator(n, nch, proto, chunk)
    finally:
        if old is None:
            del os.environ["VR_TRANSPORT"]
        else:
            os.environ["VR_TRANSPORT"] = old
    outs = [torch.empty_like(x) for x in xs]
    try:
        comm.all_reduce(xs, outs, op, dtype=dtype)
        torch.cuda.synchronize()
        assert comm.async_error() == vr.vrSuccess
    finally:
        comm.destroy()
    return outs


def _no_alloc(xs, outs, count, n, nch, proto, chunk, dtype, op):
    vr.vrAllReduceNoAlloc([x.data_ptr() for x in xs], [o.data_ptr() for o in outs], count, n, nch,
                          proto, chunk, dtype, op, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert vr.vrAllReduceNoAllocGetStatus() == vr.vrSuccess


def test_zero_count_call_is_the_warm_up():
    stream = torch.cuda.current_stream().cuda_stream
    for proto in ("simple", "ll", "ll128"):
        vr.vrAllReduceNoAlloc([], [], 0, 8, 4, proto, 16384, "float32", "sum", stream)
    torch.cuda.synchronize()
    xs = synthetic.rank_buffers(8, 5000, "float32", "uniform", 5, torch.device("cuda"))
    outs = [torch.empty_like(x) for x in xs]
    _no_alloc(xs, outs, 5000, 8, 4, "simple", 16384, "float32", "sum")
    want = oracle.allreduce([synthetic.to_numpy(x) for x in xs], "float32", "sum", 4, 16384,
                            nthreads=8)
    for o in outs:
        assert H.bytes_equal(synthetic.to_numpy(o), want)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_no_alloc_matches_the_communicator_twice_in_a_row(proto):
    dev = torch.device("cuda")
    cases = [(8, 100003, 4, 16384, "float32", "sum", 11),
             (5, 77777, 3, 4096, "bfloat16", "sum", 12)]
    for n, count, nch, chunk, dtype, op, seed in cases:
        for call in range(2):
            xs = synthetic.rank_buffers(n, count, dtype, synthetic.default_recipe(dtype),
                                        seed + call, dev)
            want = _reference(xs, n, nch, proto, chunk, dtype, op)
            outs = [torch.full_like(x, 7) for x in xs]
            _no_alloc(xs, outs, count, n, nch, proto, chunk, dtype, op)
            exact = oracle.allreduce([synthetic.to_numpy(x) for x in xs], dtype, op, nch, chunk,
                                     nthreads=8)
            for r in range(n):
                assert torch.equal(outs[r].view(torch.uint8), want[r].view(torch.uint8)), \
                    (proto, n, dtype, call, r)
                assert H.bytes_equal(synthetic.to_numpy(outs[r]), exact), (proto, n, dtype, r)


def test_no_alloc_geometry_limit_both_sides():
    dev = torch.device("cuda")
    # 16 ranks x 31 channels = 496 edges: the largest geometry that fits.
    n, nch, count = 16, 31, 40000
    xs = synthetic.rank_buffers(n, count, "int32", "int:-1048576:1048576", 3, dev)
    outs = [torch.empty_like(x) for x in xs]
    _no_alloc(xs, outs, count, n, nch, "simple", 4096, "int32", "sum")
    want = oracle.allreduce([synthetic.to_numpy(x) for x in xs], "int32", "sum", nch, 4096,
                            nthreads=8)
    for o in outs:
        assert H.bytes_equal(synthetic.to_numpy(o), want)
    # 71 ranks x 7 channels = 497 edges, and 16 x 32 = 512: rejected.
    for n_, nch_ in ((71, 7), (16, 32)):
        with pytest.raises(vr.VrError) as e:
            vr.vrAllReduceNoAlloc([1] * n_, [1] * n_, 1024, n_, nch_, "simple", 4096, "float32",
                                  "sum")
        assert e.value.code == vr.vrInvalidUsage


def test_no_alloc_one_rank_copies_and_zero_count_writes_nothing():
    dev = torch.device("cuda")
    x = synthetic.rank_buffers(1, 3001, "float32", "uniform", 4, dev)[0]
    out = torch.full_like(x, 7)
    _no_alloc([x], [out], 3001, 1, 2, "simple", 4096, "float32", "sum")
    assert torch.equal(out, x)
    xs = synthetic.rank_buffers(4, 100, "float32", "uniform", 6, dev)
    outs = [torch.full_like(v, 7) for v in xs]
    _no_alloc(xs, outs, 0, 4, 2, "simple", 4096, "float32", "sum")
    for o in outs:
        assert bool((o == 7).all())
