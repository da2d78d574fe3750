"""Rings and trees of any size over a cluster (GPU).

A ring of N > 16 ranks whose size no cluster divides evenly (17, 19, 23, 31,
34, 37, 71, ...) spans C CTAs holding ceil(N / C) or floor(N / C) ranks each.
Every collective on it -- the AllReduce in each protocol, ReduceScatter,
AllGather, the average and the pre-multiplied sum, and the double binary tree
-- must equal the oracle element by element on every rank, in both the
general and the latency kernel."""
import pytest
import torch

import gpu_helpers as H
import oracle
from ring_allreduce_virtual_gb300 import synthetic

pytestmark = pytest.mark.gpu

SIZES = [17, 19, 23, 31, 34, 37, 71]


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
@pytest.mark.parametrize("n", SIZES)
def test_allreduce(proto, n):
    with H.make_comm(n, 3, proto, 8192) as comm:
        assert comm.info()["transport"] == "warpcluster", n
        # one pass (the latency kernel for Simple and LL) and several passes
        H.run_case(n, 7777, "int32", "max", proto, 3, 8192, seed=n + 1, comm=comm)
        H.run_case(n, 100003, "float16", "sum", proto, 3, 8192, seed=n, comm=comm)
        H.run_case(n, 3_000_017, "float32", "sum", proto, 3, 8192, seed=n + 2, comm=comm)


@pytest.mark.parametrize("n", SIZES)
def test_halves(n):
    dev = torch.device("cuda")
    m = 5003
    xs = synthetic.rank_buffers(n, n * m, "bfloat16", "uniform", n, dev)
    outs = [torch.empty(m, dtype=torch.bfloat16, device=dev) for _ in range(n)]
    with H.make_comm(n, 2, "simple", 4096) as comm:
        comm.reduce_scatter(xs, outs, "sum")
        torch.cuda.synchronize()
        want = oracle.reduce_scatter([synthetic.to_numpy(x) for x in xs], "bfloat16", "sum")
        for r in range(n):
            assert H.bytes_equal(synthetic.to_numpy(outs[r]), want[r]), r
        ys = synthetic.rank_buffers(n, m, "int8", "int:-128:127", n + 1, dev)
        gs = [torch.empty(n * m, dtype=torch.int8, device=dev) for _ in range(n)]
        comm.all_gather(ys, gs)
        torch.cuda.synchronize()
        want = oracle.all_gather([synthetic.to_numpy(y) for y in ys], "int8")
        for r in range(n):
            assert H.bytes_equal(synthetic.to_numpy(gs[r]), want[r]), r


@pytest.mark.parametrize("n", SIZES)
def test_scaled_sums(n):
    dev = torch.device("cuda")
    count = 60013
    for dtype, kind, scalar in (("float32", "avg", None), ("bfloat16", "premulsum", 0.375),
                                ("int32", "avg", None), ("int32", "premulsum", -3)):
        xs = synthetic.rank_buffers(n, count, dtype, synthetic.default_recipe(dtype), n, dev)
        outs = [torch.empty_like(x) for x in xs]
        with H.make_comm(n, 2, "ll", 4096) as comm:
            op = "avg" if kind == "avg" else comm.premul_sum(scalar, dtype)
            comm.all_reduce(xs, outs, op, dtype=dtype)
            torch.cuda.synchronize()
            want = oracle.allreduce_scaled([synthetic.to_numpy(x) for x in xs], dtype, kind,
                                           scalar, 2, 4096)
            for o in outs:
                assert H.bytes_equal(synthetic.to_numpy(o), want), (dtype, kind)


@pytest.mark.parametrize("n", SIZES)
def test_tree(n):
    dev = torch.device("cuda")
    for dtype, op, count in (("float32", "sum", 200003), ("int32", "min", 9999)):
        xs = synthetic.rank_buffers(n, count, dtype, synthetic.default_recipe(dtype), n, dev)
        outs = [torch.empty_like(x) for x in xs]
        with H.make_comm(n, 2, "simple", 4096) as comm:
            comm.all_reduce_tree(xs, outs, op, dtype=dtype)
            torch.cuda.synchronize()
            want = oracle.tree_allreduce([synthetic.to_numpy(x) for x in xs], dtype, op)
            for o in outs:
                assert H.bytes_equal(synthetic.to_numpy(o), want), (dtype, op)


@pytest.mark.parametrize("ctas", [5, 7, 9, 10, 11, 13, 16])
def test_uneven_splits_of_a_24_rank_ring(ctas, monkeypatch):
    """Splits of a 24-rank ring that leave CTAs of different sizes give the
    oracle's bytes, like the even ones."""
    monkeypatch.setenv("VR_CLUSTER_CTAS", str(ctas))
    for proto in ("simple-warpcluster", "ll-warpcluster", "ll128-warpcluster"):
        H.run_case(24, 50021, "bfloat16", "sum", proto, 2, 4096, seed=ctas)
        H.run_case(24, 2_000_003, "float32", "sum", proto, 5, 65536, seed=ctas + 1)
    xs = synthetic.rank_buffers(24, 30011, "float32", "uniform", ctas, torch.device("cuda"))
    outs = [torch.empty_like(x) for x in xs]
    with H.make_comm(24, 2, "simple", 4096) as comm:
        comm.all_reduce_tree(xs, outs, "sum")
        torch.cuda.synchronize()
    want = oracle.tree_allreduce([synthetic.to_numpy(x) for x in xs], "float32", "sum")
    for o in outs:
        assert H.bytes_equal(synthetic.to_numpy(o), want)
