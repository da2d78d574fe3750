"""The average and the pre-multiplied sum (GPU) against the oracle, bit for
bit, on every rank: the ring AllReduce on every protocol and both on-chip
transports, ReduceScatter, the tree, the calibration fold, one rank; every
element type; and the calls that refuse them (other transports, the no-alloc
entry, an op of another type or communicator, a released op)."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic

pytestmark = pytest.mark.gpu
PROTOS = ["simple", "ll", "ll128", "simple-warpcluster", "ll-warpcluster", "ll128-warpcluster"]
# Scalars that a float32 holds exactly (so every rounding of them to a
# narrower type is a single one), and integer scalars, negative ones wrapping
# for the unsigned types.
FLOAT_SCALARS = (float(np.float32(0.1)), -2.5)
INT_SCALARS = (3, -7)


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


def _scalars(dtype):
    return FLOAT_SCALARS if dtype in oracle.FLOAT_TYPES else INT_SCALARS


def scaled_case(comm, n, count, dtype, kind, scalar, nch, chunk, seed, method="all_reduce",
                inplace=False, offset=0):
    dev = torch.device("cuda")
    xs = synthetic.rank_buffers(n, count, dtype, synthetic.default_recipe(dtype), seed, "cpu")
    tdt = synthetic.TORCH_DTYPE[dtype]
    op = "avg" if kind == "avg" else comm.premul_sum(scalar, dtype)
    try:
        sends, recvs, bases = [], [], []
        for x in xs:
            sb, sv = H.guarded(count, tdt, dev, offset, fill=x)
            if inplace:
                rb, rv = sb, sv
            else:
                rb, rv = H.guarded(count, tdt, dev, offset)
            sends.append(sv)
            recvs.append(rv)
            bases.append(rb)
        getattr(comm, method)(sends, recvs, op, dtype=dtype)
        torch.cuda.synchronize()
        assert comm.async_error() == vr.vrSuccess
        host = [synthetic.to_numpy(x) for x in xs]
        want = oracle.allreduce_scaled(host, dtype, kind, scalar, nch, chunk, nthreads=8)
        for r in range(n):
            got = synthetic.to_numpy(recvs[r])
            if not H.bytes_equal(got, want):
                bad = np.nonzero(got.view(np.uint8) != want.view(np.uint8))[0]
                raise AssertionError(f"rank {r}: {len(bad)} bytes differ, first at byte {bad[0]} "
                                     f"(n={n} count={count} {dtype} {kind} {scalar} {method})")
            assert H.guards_intact(bases[r], count, offset), f"guard overwritten, rank {r}"
            if not inplace:
                assert H.bytes_equal(synthetic.to_numpy(sends[r]), host[r]), f"input {r} modified"
    finally:
        if kind != "avg":
            comm.destroy_op(op)


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("dtype", list(vr.DTYPES))
def test_allreduce_avg_and_premulsum(proto, dtype):
    n = 6 if proto.endswith("warpcluster") else 5
    with H.make_comm(n, 3, proto, 4096) as comm:
        for i, count in enumerate((1, 1003, 70001)):
            scaled_case(comm, n, count, dtype, "avg", None, 3, 4096, seed=i)
            for j, s in enumerate(_scalars(dtype)):
                scaled_case(comm, n, count, dtype, "premulsum", s, 3, 4096, seed=10 * i + j)


@pytest.mark.parametrize("n,proto", [(2, "simple"), (16, "ll"), (16, "ll128"), (7, "simple"),
                                     (24, "simple"), (72, "ll"), (32, "ll128")])
def test_ring_sizes_and_cluster_rings(n, proto):
    """Every rank count the warp ring takes, and rings over a cluster's CTAs."""
    with vr.Communicator(n, 4, proto, 64 << 10) as comm:
        for dtype in ("float32", "bfloat16", "int32"):
            scaled_case(comm, n, 300007, dtype, "avg", None, 4, 64 << 10, seed=n)
            scaled_case(comm, n, 65539, dtype, "premulsum", _scalars(dtype)[1], 4, 64 << 10,
                        seed=n + 1)


def test_in_place_unaligned_and_large_chunks():
    with vr.Communicator(8, 2, "simple", 1 << 20) as comm:
        scaled_case(comm, 8, 3 * 2 ** 20 + 5, "float16", "avg", None, 2, 1 << 20, seed=1,
                    inplace=True)
        scaled_case(comm, 8, 1234567, "float32", "premulsum", -2.5, 2, 1 << 20, seed=2,
                    offset=1)
        scaled_case(comm, 8, 777777, "int64", "avg", None, 2, 1 << 20, seed=3, offset=3)


@pytest.mark.parametrize("dtype", list(vr.DTYPES))
def test_ring_walk_scaled(dtype):
    """The calibration fold scales as the ring does: the same result."""
    with vr.Communicator(9, 5, "simple", 16 << 10) as comm:
        scaled_case(comm, 9, 200003, dtype, "avg", None, 5, 16 << 10, seed=4, method="ring_walk")
        scaled_case(comm, 9, 200003, dtype, "premulsum", _scalars(dtype)[0], 5, 16 << 10,
                    seed=5, method="ring_walk")


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int8", "uint64"])
def test_one_rank(dtype):
    """One rank: the average is the input; the pre-multiplied sum scales it."""
    with vr.Communicator(1, 1, "simple", 4096) as comm:
        scaled_case(comm, 1, 10007, dtype, "avg", None, 1, 4096, seed=6)
        scaled_case(comm, 1, 10007, dtype, "premulsum", _scalars(dtype)[1], 1, 4096, seed=7)
        scaled_case(comm, 1, 10007, dtype, "premulsum", _scalars(dtype)[0], 1, 4096, seed=8,
                    inplace=True)


def _rs_scaled(comm, n, rc, dtype, kind, scalar, seed, inplace=False):
    dev = torch.device("cuda")
    xs = synthetic.rank_buffers(n, n * rc, dtype, synthetic.default_recipe(dtype), seed, dev)
    host = [synthetic.to_numpy(x) for x in xs]
    op = "avg" if kind == "avg" else comm.premul_sum(scalar, dtype)
    try:
        if inplace:
            sends = [x.clone() for x in xs]
            outs = [s[r * rc:(r + 1) * rc] for r, s in enumerate(sends)]
        else:
            sends = xs
            outs = [torch.empty(rc, dtype=xs[0].dtype, device=dev) for _ in range(n)]
            for o in outs:
                o.view(torch.uint8).fill_(3)
        comm.reduce_scatter(sends, outs, op, dtype=dtype)
        torch.cuda.synchronize()
        assert comm.async_error() == vr.vrSuccess
        want = oracle.reduce_scatter_scaled(host, dtype, kind, scalar)
        for r in range(n):
            assert H.bytes_equal(synthetic.to_numpy(outs[r]), want[r]), (n, rc, dtype, kind, r)
    finally:
        if kind != "avg":
            comm.destroy_op(op)


@pytest.mark.parametrize("proto", PROTOS)
def test_reduce_scatter_scaled(proto):
    # a ring over a cluster needs two ranks at least
    for n in ((3, 8) if proto.endswith("warpcluster") else (1, 3, 8)):
        with H.make_comm(n, 2, proto, 16 << 10) as comm:
            for dtype in ("float32", "float16", "int32", "uint8"):
                _rs_scaled(comm, n, 50001, dtype, "avg", None, seed=n)
                _rs_scaled(comm, n, 4099, dtype, "premulsum", _scalars(dtype)[1], seed=n + 1,
                           inplace=True)


def test_avg_of_equal_inputs_is_the_input_for_integers():
    """Integer average of N equal buffers: the wrapped sum N x divided by N
    gives x back wherever N x does not wrap."""
    dev = torch.device("cuda")
    x = torch.randint(-1000, 1000, (100003,), dtype=torch.int32, device=dev)
    xs = [x.clone() for _ in range(12)]
    outs = [torch.empty_like(x) for _ in range(12)]
    with vr.Communicator(12, 2, "ll", 16 << 10) as comm:
        comm.all_reduce(xs, outs, "avg")
        torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, x)


def test_refusals():
    dev = torch.device("cuda")
    x = [torch.ones(64, device=dev) for _ in range(4)]
    y = [torch.empty(64, device=dev) for _ in range(4)]
    # The global-FIFO transport and the tree reduce with the plain ops only.
    with H.make_comm(4, 1, "simple-global", 4096) as comm:
        with pytest.raises(vr.VrError) as e:
            comm.all_reduce(x, y, "avg")
        assert e.value.code == vr.vrInvalidUsage
        op = comm.premul_sum(2.0, "float32")
        with pytest.raises(vr.VrError) as e:
            comm.all_reduce(x, y, op)
        assert e.value.code == vr.vrInvalidUsage
        comm.destroy_op(op)
    with vr.Communicator(4, 1, "simple", 4096) as comm, \
            vr.Communicator(4, 1, "simple", 4096) as other:
        op = comm.premul_sum(2.0, "float32")
        # an op made for float32: another dtype, another communicator
        with pytest.raises(vr.VrError) as e:
            comm.all_reduce([t.half() for t in x], [t.half() for t in y], op)
        assert e.value.code == vr.vrInvalidArgument
        with pytest.raises(vr.VrError) as e:
            other.all_reduce(x, y, op)
        assert e.value.code == vr.vrInvalidArgument
        comm.all_reduce(x, y, op)
        torch.cuda.synchronize()
        assert all(torch.equal(t, torch.full_like(t, 8.0)) for t in y)
        comm.destroy_op(op)
        with pytest.raises(vr.VrError) as e:
            comm.all_reduce(x, y, op)
        assert e.value.code == vr.vrInvalidArgument
        with pytest.raises(vr.VrError) as e:
            comm.destroy_op(op)
        assert e.value.code == vr.vrInvalidArgument
        # sixteen live ops at most
        ops = [comm.premul_sum(float(i), "float32") for i in range(16)]
        with pytest.raises(vr.VrError) as e:
            comm.premul_sum(1.0, "float32")
        assert e.value.code == vr.vrInvalidUsage
        for o in ops:
            comm.destroy_op(o)
    # The no-alloc entry takes the plain ops only.
    with pytest.raises(vr.VrError) as e:
        vr.vrAllReduceNoAlloc([t.data_ptr() for t in x], [t.data_ptr() for t in y], 64, 4, 1,
                              "simple", 4096, "float32", "avg")
    assert e.value.code == vr.vrInvalidArgument


def _tree_scaled(comm, n, count, dtype, kind, scalar, seed):
    dev = torch.device("cuda")
    xs = synthetic.rank_buffers(n, count, dtype, synthetic.default_recipe(dtype), seed, dev)
    outs = [torch.empty_like(x) for x in xs]
    op = "avg" if kind == "avg" else comm.premul_sum(scalar, dtype)
    try:
        comm.all_reduce_tree(xs, outs, op, dtype=dtype)
        torch.cuda.synchronize()
        assert comm.async_error() == vr.vrSuccess
        want = oracle.tree_allreduce_scaled([synthetic.to_numpy(x) for x in xs], dtype, kind,
                                            scalar)
        for r in range(n):
            assert H.bytes_equal(synthetic.to_numpy(outs[r]), want), (n, dtype, kind, r)
    finally:
        if kind != "avg":
            comm.destroy_op(op)


@pytest.mark.parametrize("dtype", list(vr.DTYPES))
def test_tree_scaled(dtype):
    with vr.Communicator(7, 1, "simple", 4096) as comm:
        for i, count in enumerate((1, 1003, 100003)):
            _tree_scaled(comm, 7, count, dtype, "avg", None, seed=i)
            _tree_scaled(comm, 7, count, dtype, "premulsum", _scalars(dtype)[1], seed=10 + i)


@pytest.mark.parametrize("n", [1, 2, 16, 24, 72])
def test_tree_scaled_sizes(n):
    """Every tree shape up to one CTA, trees over a cluster, one rank."""
    with vr.Communicator(n, 1, "simple", 4096) as comm:
        for dtype in ("float32", "bfloat16", "int32", "int8"):
            _tree_scaled(comm, n, 65539, dtype, "avg", None, seed=n)
            _tree_scaled(comm, n, 4099, dtype, "premulsum", _scalars(dtype)[0], seed=n + 1)
