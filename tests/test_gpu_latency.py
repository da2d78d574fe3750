"""The latency kernel against the oracle (GPU).

A warp-ring call whose parts all run at once (one part per ring, one FIFO
step per stage) takes the latency kernel, and so does a Simple call of
several passes on rings inside one CTA; VR_LATENCY_KERNEL=0 keeps both on the
general kernel. Both kernels must equal the oracle element by element on every
rank, for every element type and reduction, both protocols it serves (Simple,
LL), rings in one CTA and over a cluster, all three collectives, the scaled
sums, ragged tails, stages whose chunk slice is empty, and rings that run
several parts one after another (the own-data prefetch crossing from one part
into the next)."""
import pytest
import torch

import gpu_helpers as H
import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic

pytestmark = pytest.mark.gpu

PROTOS = ["simple", "ll", "simple-warpcluster", "ll-warpcluster"]
# (n ranks, count of float32, channels, chunk bytes): one pass on every
# transport above; ragged tails, empty last chunks, 8 B to 2 MiB per rank.
SHAPES = [(2, 1, 1, 16), (2, 5, 1, 16), (3, 7, 1, 16), (3, 1000, 2, 256), (4, 65539, 3, 4096),
          (5, 4097, 4, 48), (8, 2, 16, 512 << 10), (8, 262144, 16, 512 << 10),
          (8, 524288, 16, 512 << 10), (16, 33333, 2, 1 << 10), (7, 5000, 16, 16),
          (13, 100003, 5, 16384)]


# Several passes of rings inside one CTA, Simple: (n ranks, count of float32,
# channels, chunk bytes), ragged tails and partial last loops.
# Each needs more than three passes, so that no one-pass or one-own-slot
# geometry takes it.
MULTI = [(2, 4_000_003, 1, 4096), (4, 8_000_003, 2, 4096), (5, 7_777_777, 3, 8192),
         (8, 12_000_017, 16, 128 << 10), (16, 8 << 20, 4, 65536)]


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


@pytest.fixture(params=["1", "0"], ids=["latency", "general"])
def kernel(request, monkeypatch):
    monkeypatch.setenv("VR_LATENCY_KERNEL", request.param)
    return request.param


def _one_pass(comm, count, dtype):
    parts, rings = comm.plan(count, dtype)
    return parts <= rings


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "n{}_c{}_ch{}_k{}".format(*s))
def test_one_pass_shapes(proto, shape, kernel):
    n, count, nch, chunk = shape
    with H.make_comm(n, nch, proto, chunk) as comm:
        assert _one_pass(comm, count, "float32"), (shape, comm.plan(count, "float32"))
        H.run_case(n, count, "float32", "sum", proto, nch, chunk, seed=n * 7 + count,
                   comm=comm)


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("dtype", list(vr.DTYPES))
def test_every_dtype_and_op(proto, dtype, kernel):
    with H.make_comm(6, 3, proto, 4096) as comm:
        for i, op in enumerate(oracle.OPS):
            for count in (999, 30001):
                H.run_case(6, count, dtype, op, proto, 3, 4096, seed=13 * i + count, comm=comm)


@pytest.mark.parametrize("proto", PROTOS)
def test_in_place_and_repeated(proto, kernel):
    with H.make_comm(5, 2, proto, 2048) as comm:
        for i in range(6):
            H.run_case(5, 20011 + 13 * i, "bfloat16", "sum", proto, 2, 2048, seed=i,
                       inplace=bool(i & 1), comm=comm)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll-warpcluster"])
def test_halves(proto, kernel):
    dev = torch.device("cuda")
    n, m = 6, 3001
    xs = synthetic.rank_buffers(n, n * m, "float32", "uniform", 21, dev)
    outs = [torch.empty(m, device=dev) for _ in range(n)]
    with H.make_comm(n, 2, proto, 4096) as comm:
        comm.reduce_scatter(xs, outs, "sum")
        torch.cuda.synchronize()
        want = oracle.reduce_scatter([synthetic.to_numpy(x) for x in xs], "float32", "sum")
        for r in range(n):
            assert H.bytes_equal(synthetic.to_numpy(outs[r]), want[r]), r
        ys = synthetic.rank_buffers(n, m, "float16", "uniform", 22, dev)
        gs = [torch.empty(n * m, dtype=torch.float16, device=dev) for _ in range(n)]
        comm.all_gather(ys, gs)
        torch.cuda.synchronize()
        want = oracle.all_gather([synthetic.to_numpy(y) for y in ys], "float16")
        for r in range(n):
            assert H.bytes_equal(synthetic.to_numpy(gs[r]), want[r]), r


@pytest.mark.parametrize("proto", ["simple", "ll-warpcluster"])
def test_scaled_sums(proto, kernel):
    dev = torch.device("cuda")
    n, count = 7, 12345
    for dtype in ("float32", "bfloat16", "int32"):
        xs = synthetic.rank_buffers(n, count, dtype, synthetic.default_recipe(dtype), 31, dev)
        outs = [torch.empty_like(x) for x in xs]
        with H.make_comm(n, 3, proto, 4096) as comm:
            comm.all_reduce(xs, outs, "avg", dtype=dtype)
            torch.cuda.synchronize()
            want = oracle.allreduce_scaled([synthetic.to_numpy(x) for x in xs], dtype, "avg",
                                           None, 3, 4096)
            for o in outs:
                assert H.bytes_equal(synthetic.to_numpy(o), want), dtype


@pytest.mark.parametrize("shape", MULTI, ids=lambda s: "n{}_c{}_ch{}_k{}".format(*s))
def test_several_passes_simple(shape, kernel):
    n, count, nch, chunk = shape
    with H.make_comm(n, nch, "simple", chunk) as comm:
        assert comm.info()["transport"] == "warp"
        parts, rings = comm.plan(count, "float32")
        assert parts > rings, (shape, parts, rings)
        for i, (dtype, op) in enumerate((("float32", "sum"), ("int32", "max"),
                                         ("bfloat16", "sum"), ("float64", "min"))):
            H.run_case(n, count, dtype, op, "simple", nch, chunk, seed=n + 31 * i, comm=comm,
                       inplace=i == 2)


def test_several_passes_halves_and_scaled(kernel):
    dev = torch.device("cuda")
    n, m = 4, 2_000_003  # blocks of ~2 x 977 chunks per channel: many passes
    xs = synthetic.rank_buffers(n, n * m, "float32", "uniform", 41, dev)
    outs = [torch.empty(m, device=dev) for _ in range(n)]
    with H.make_comm(n, 2, "simple", 4096) as comm:
        comm.reduce_scatter(xs, outs, "sum")
        torch.cuda.synchronize()
        want = oracle.reduce_scatter([synthetic.to_numpy(x) for x in xs], "float32", "sum")
        for r in range(n):
            assert H.bytes_equal(synthetic.to_numpy(outs[r]), want[r]), r
        ys = synthetic.rank_buffers(n, m, "int8", "int:-128:127", 42, dev)
        gs = [torch.empty(n * m, dtype=torch.int8, device=dev) for _ in range(n)]
        comm.all_gather(ys, gs)
        torch.cuda.synchronize()
        want = oracle.all_gather([synthetic.to_numpy(y) for y in ys], "int8")
        for r in range(n):
            assert H.bytes_equal(synthetic.to_numpy(gs[r]), want[r]), r
        for dtype in ("float32", "int32"):
            zs = synthetic.rank_buffers(n, 8_000_003, dtype, synthetic.default_recipe(dtype), 43,
                                        dev)
            os_ = [torch.empty_like(z) for z in zs]
            comm.all_reduce(zs, os_, "avg", dtype=dtype)
            torch.cuda.synchronize()
            want = oracle.allreduce_scaled([synthetic.to_numpy(z) for z in zs], dtype, "avg",
                                           None, 2, 4096)
            for o in os_:
                assert H.bytes_equal(synthetic.to_numpy(o), want), dtype
