"""The 8-bit floating types (GPU) against the oracle, bit for bit, on inputs
that reach every finite code: subnormals, exact ties and sums and products
past the largest finite value (which saturate), on every protocol and
transport, the tree, the calibration fold and ReduceScatter."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic

pytestmark = pytest.mark.gpu
FP8 = ["float8_e4m3", "float8_e5m2"]
PROTOS = ["simple", "ll", "ll128", "simple-global", "ll-global", "ll128-global",
          "simple-warpcluster", "ll-warpcluster", "ll128-warpcluster"]


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


def _finite_codes(dtype, n, count, seed):
    """Random codes over every finite value of the format (NaN and, for E5M2,
    the infinities left out)."""
    rng = np.random.default_rng(seed)
    if dtype == "float8_e4m3":
        pool = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    else:
        pool = np.array([c for c in range(256) if c & 0x7C != 0x7C], np.uint8)
    return [torch.from_numpy(rng.choice(pool, count)).view(synthetic.TORCH_DTYPE[dtype])
            for _ in range(n)]


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("dtype", FP8)
def test_every_code_every_op(proto, dtype):
    n = 6 if proto.endswith("warpcluster") else 5
    with H.make_comm(n, 3, proto, 4096) as comm:
        for i, op in enumerate(oracle.OPS):
            xs = _finite_codes(dtype, n, 40961, seed=i)
            H.run_case(n, 40961, dtype, op, proto, 3, 4096, comm=comm, xs=xs)


@pytest.mark.parametrize("dtype", FP8)
def test_tree_and_walk(dtype):
    dev = torch.device("cuda")
    with vr.Communicator(7, 2, "simple", 8192) as comm:
        for i, op in enumerate(oracle.OPS):
            xs = _finite_codes(dtype, 7, 30011, seed=10 + i)
            H.run_case(7, 30011, dtype, op, "simple", 2, 8192, comm=comm, xs=xs,
                       method="ring_walk")
            ins = [x.to(dev) for x in xs]
            outs = [torch.empty_like(x) for x in ins]
            comm.all_reduce_tree(ins, outs, op, dtype=dtype)
            torch.cuda.synchronize()
            want = oracle.tree_allreduce([synthetic.to_numpy(x) for x in xs], dtype, op)
            for o in outs:
                assert H.bytes_equal(synthetic.to_numpy(o), want), (dtype, op)


@pytest.mark.parametrize("dtype", FP8)
def test_reduce_scatter(dtype):
    dev = torch.device("cuda")
    n, rc = 4, 10007
    with vr.Communicator(n, 2, "ll128", 4096) as comm:
        for i, op in enumerate(oracle.OPS):
            xs = _finite_codes(dtype, n, n * rc, seed=20 + i)
            outs = [torch.empty(rc, dtype=xs[0].dtype, device=dev) for _ in range(n)]
            comm.reduce_scatter([x.to(dev) for x in xs], outs, op, dtype=dtype)
            torch.cuda.synchronize()
            want = oracle.reduce_scatter([synthetic.to_numpy(x) for x in xs], dtype, op)
            for r in range(n):
                assert H.bytes_equal(synthetic.to_numpy(outs[r]), want[r]), (dtype, op, r)


@pytest.mark.parametrize("dtype,top", [("float8_e4m3", 448.0), ("float8_e5m2", 57344.0)])
def test_saturation(dtype, top):
    """Every rank holds the largest finite value: the sum saturates to it, a
    pre-multiplied sum by -2 to its negative; the average equals the
    oracle's (sums of top/8 that round on the way)."""
    dev = torch.device("cuda")
    tdt = synthetic.TORCH_DTYPE[dtype]
    x = torch.full((4099,), top, dtype=torch.float32, device=dev).to(tdt)
    xs = [x.clone() for _ in range(8)]
    outs = [torch.empty_like(x) for _ in range(8)]
    with vr.Communicator(8, 2, "ll", 4096) as comm:
        comm.all_reduce(xs, outs, "sum")
        torch.cuda.synchronize()
        assert all(bool((o.float() == top).all()) for o in outs)
        comm.all_reduce(xs, outs, "avg")
        torch.cuda.synchronize()
        want = oracle.allreduce_scaled([synthetic.to_numpy(v) for v in xs], dtype, "avg", None,
                                       2, 4096)
        assert all(H.bytes_equal(synthetic.to_numpy(o), want) for o in outs)
        op = comm.premul_sum(-2.0, dtype)
        comm.all_reduce(xs, outs, op)
        torch.cuda.synchronize()
        comm.destroy_op(op)
        assert all(bool((o.float() == -top).all()) for o in outs)
