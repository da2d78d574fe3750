"""The ring-walk calibration fold (vrRingWalk) vs the CPU oracle, bit for bit,
and vs the ring itself (GPU).

The fold reads every rank's chunk in ring order from rank c+1, so it must
reproduce the ring's result exactly: every element type x reduction, ragged
tails, several loops and channels, in place, unaligned pointers, rings beyond
one SM (N = 72, 128), and the full-size bandwidth workload on sampled
elements."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic, workloads

pytestmark = pytest.mark.gpu

# (n ranks, count, channels, chunk bytes)
SHAPES = [
    (1, 1000, 1, 16), (2, 1, 1, 16), (2, 3, 2, 16), (3, 7, 1, 16), (4, 65536, 1, 512 << 10),
    (4, 65539, 3, 4096), (5, 4097, 4, 48), (8, 100003, 7, 64 << 10), (16, 33333, 2, 1 << 10),
    (7, 50000, 16, 16), (12, 2 ** 18 + 1, 4, 1 << 20), (72, 40000, 8, 64 << 10),
    (128, 5000, 3, 256), (9, 2 ** 20 + 3, 2, 16 << 10),
]


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "n{}_c{}_ch{}_k{}".format(*s))
def test_float32_sum_shapes(shape):
    n, count, nch, chunk = shape
    H.run_case(n, count, "float32", "sum", "simple", nch, chunk, seed=hash(shape) & 0xffff,
               method="ring_walk")


@pytest.mark.parametrize("dtype", list(vr.DTYPES))
def test_every_dtype_and_op(dtype):
    with H.make_comm(5, 3, "simple", 4096) as comm:
        for i, op in enumerate(oracle.OPS):
            for count in (1003, 40961):
                H.run_case(5, count, dtype, op, "simple", 3, 4096, seed=31 * i + count,
                           comm=comm, method="ring_walk")


def test_in_place_and_unaligned():
    H.run_case(4, 70001, "float32", "sum", "simple", 3, 8192, inplace=True, seed=5,
               method="ring_walk")
    H.run_case(3, 12345, "bfloat16", "sum", "simple", 2, 256, offset=1, seed=6,
               method="ring_walk")
    H.run_case(6, 9999, "int8", "max", "simple", 2, 64, offset=3, seed=7, method="ring_walk")


def test_equals_ring():
    """The fold and the ring, on the same inputs, give the same bytes."""
    dev = torch.device("cuda")
    for proto in ("simple", "ll", "ll128"):
        xs = synthetic.rank_buffers(8, 300007, "bfloat16", "normal:0.01", 3, dev)
        a = [torch.empty_like(x) for x in xs]
        b = [torch.empty_like(x) for x in xs]
        with vr.Communicator(8, 16, proto, 64 << 10) as comm:
            comm.all_reduce(xs, a, "sum")
            comm.ring_walk(xs, b, "sum")
            torch.cuda.synchronize()
        for r in range(8):
            assert torch.equal(a[r].view(torch.uint8), b[r].view(torch.uint8)), (proto, r)


def test_zero_count():
    with vr.Communicator(4, 1, "simple", 4096) as comm:
        vr.vrRingWalk(comm.handle, [0] * 4, [0] * 4, 0, "float32", "sum")


def test_full_size_headline_sampled():
    """The 16 x 1 GiB fp32 workload: sampled elements equal the oracle's."""
    w = workloads.HEADLINE
    dev = torch.device("cuda")
    xs = synthetic.rank_buffers(w.n_ranks, w.count, w.dtype, w.dist, w.seed, dev)
    outs = [torch.empty_like(x) for x in xs]
    with vr.Communicator(w.n_ranks, w.n_channels, w.proto, w.chunk_bytes) as comm:
        comm.ring_walk(xs, outs, w.op)
        torch.cuda.synchronize()
    H.check_sampled(xs, outs, w.dtype, w.op, w.n_channels, w.chunk_bytes,
                    np.random.default_rng(9))
