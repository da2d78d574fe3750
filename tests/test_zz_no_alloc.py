"""vrAllReduceNoAlloc (GPU): the AllReduce for callers that cannot allocate
device memory where they need it -- code under a framework's caching
allocator that must account for every device byte, or a latency-critical path
where cudaMalloc would stall the device. Its scratch is a fixed array the
library defines in device memory, shared by every call.

Called through the C ABI (the binding only marshals arguments), its outputs
must equal, bit for bit, those of the communicator entry point on the
global-memory FIFO transport with the same ring parameters, on two calls in a
row (the second call must not be disturbed by what the first left in the
shared scratch). This file is collected last on purpose."""
import os

import pytest
import torch

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


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_no_alloc_matches_the_communicator_twice_in_a_row(proto):
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    cases = [(8, 100003, 4, 16384, "float32", "sum", 11),
             (5, 77777, 3, 4096, "bfloat16", "sum", 12)]
    for n, count, nch, chunk, dtype, op, seed in cases:
        for call in range(2):
            xs = synthetic.rank_buffers(n, count, dtype, synthetic.default_recipe(dtype),
                                        seed + call, dev)
            want = _reference(xs, n, nch, proto, chunk, dtype, op)
            outs = [torch.full_like(x, 7) for x in xs]
            vr.vrAllReduceNoAlloc([x.data_ptr() for x in xs], [o.data_ptr() for o in outs],
                                  count, n, nch, proto, chunk, dtype, op, stream.cuda_stream)
            torch.cuda.synchronize()
            for r in range(n):
                assert torch.equal(outs[r].view(torch.uint8), want[r].view(torch.uint8)), \
                    (proto, n, dtype, call, r)


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    with pytest.raises(vr.VrError) as e:
        vr.vrAllReduceNoAlloc([1] * 16, [1] * 16, 1024, 16, 32, "simple", 4096, "float32", "sum")
    assert e.value.code == vr.vrInvalidUsage
