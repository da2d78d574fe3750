"""ReduceScatter and AllGather on the ring (GPU), against the oracle, bit for
bit, on every rank: protocols, ring sizes, element types and ops, ragged
sizes, channels and chunk sizes, in place, one rank, zero elements."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic

pytestmark = pytest.mark.gpu
PROTOS = ["simple", "ll", "ll128", "simple-warpcluster", "ll-warpcluster", "ll128-warpcluster"]


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


def _filled(count, tdtype, dev, byte):
    """A buffer whose every byte is `byte` (any element type, 8-bit floats too)."""
    t = torch.empty(count, dtype=tdtype, device=dev)
    t.view(torch.uint8).fill_(byte)
    return t


def _rs_case(comm, n, rc, dtype, op, seed, inplace=False):
    dev = torch.device("cuda")
    dist = synthetic.default_recipe(dtype)
    xs = synthetic.rank_buffers(n, n * rc, dtype, dist, seed, dev)
    host = [synthetic.to_numpy(x) for x in xs]
    if inplace:
        sends = [x.clone() for x in xs]
        outs = [s[r * rc:(r + 1) * rc] for r, s in enumerate(sends)]
    else:
        sends = xs
        outs = [_filled(rc, xs[0].dtype, dev, 3) for _ in range(n)]
    comm.reduce_scatter(sends, outs, op, dtype=dtype)
    torch.cuda.synchronize()
    assert comm.async_error() == vr.vrSuccess
    want = oracle.reduce_scatter(host, dtype, op)
    for r in range(n):
        assert H.bytes_equal(synthetic.to_numpy(outs[r]), want[r]), (n, rc, dtype, op, r)
    if not inplace:
        for x, h in zip(xs, host):
            assert H.bytes_equal(synthetic.to_numpy(x), h)


def _ag_case(comm, n, sc, dtype, seed, inplace=False):
    dev = torch.device("cuda")
    xs = synthetic.rank_buffers(n, sc, dtype, synthetic.default_recipe(dtype), seed, dev)
    host = [synthetic.to_numpy(x) for x in xs]
    if inplace:
        outs = [torch.zeros(n * sc, dtype=xs[0].dtype, device=dev) for _ in range(n)]
        for r in range(n):
            outs[r][r * sc:(r + 1) * sc] = xs[r]
        sends = [outs[r][r * sc:(r + 1) * sc] for r in range(n)]
    else:
        sends = xs
        outs = [_filled(n * sc, xs[0].dtype, dev, 5) for _ in range(n)]
    comm.all_gather(sends, outs, dtype=dtype)
    torch.cuda.synchronize()
    assert comm.async_error() == vr.vrSuccess
    want = oracle.all_gather(host, dtype)
    for r in range(n):
        assert H.bytes_equal(synthetic.to_numpy(outs[r]), want[r]), (n, sc, dtype, r)


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("n", [2, 3, 5, 8, 16])
def test_reduce_scatter_shapes(proto, n):
    for nch, chunk, rc in ((1, 4096, 1), (3, 256, 1003), (2, 64 << 10, 50001), (5, 16, 777)):
        with H.make_comm(n, nch, proto, chunk) as comm:
            _rs_case(comm, n, rc, "float32", "sum", seed=rc + n)


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("n", [2, 3, 5, 8, 16])
def test_all_gather_shapes(proto, n):
    for nch, chunk, sc in ((1, 4096, 1), (3, 256, 1003), (2, 64 << 10, 50001), (5, 16, 777)):
        with H.make_comm(n, nch, proto, chunk) as comm:
            _ag_case(comm, n, sc, "float32", seed=sc + n)


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("dtype", list(vr.DTYPES))
def test_reduce_scatter_every_dtype_and_op(proto, dtype):
    with H.make_comm(4, 3, proto, 1024) as comm:
        for i, op in enumerate(oracle.OPS):
            _rs_case(comm, 4, 4099, dtype, op, seed=100 + i)
        _ag_case(comm, 4, 3001, dtype, seed=7)


@pytest.mark.parametrize("proto", PROTOS)
def test_in_place(proto):
    with H.make_comm(5, 2, proto, 2048) as comm:
        _rs_case(comm, 5, 12345, "bfloat16", "sum", seed=1, inplace=True)
        _ag_case(comm, 5, 12345, "float16", seed=2, inplace=True)


def test_one_rank_and_zero_elements():
    dev = torch.device("cuda")
    with vr.Communicator(1, 1, "simple", 4096) as comm:
        _rs_case(comm, 1, 999, "float32", "sum", seed=3)
        _ag_case(comm, 1, 999, "int32", seed=4)
    with vr.Communicator(4, 1, "simple", 4096) as comm:
        z = [torch.zeros(0, device=dev) for _ in range(4)]
        comm.reduce_scatter(z, [torch.zeros(0, device=dev) for _ in range(4)])
        comm.all_gather(z, [torch.zeros(0, device=dev) for _ in range(4)])
        torch.cuda.synchronize()


def test_halves_need_the_warp_transport():
    comm = H.make_comm(4, 1, "simple-global", 4096)
    try:
        x = torch.zeros(16, device="cuda")
        with pytest.raises(vr.VrError) as e:
            comm.reduce_scatter([x] * 4, [x[:4]] * 4)
        assert e.value.code == vr.vrInvalidUsage
    finally:
        comm.destroy()


def test_large_reduce_scatter_and_all_gather():
    """8 ranks, 16 Mi bf16 per block: every output checked on sampled
    elements against the oracle's per-block fold."""
    dev = torch.device("cuda")
    n, rc = 8, 16 << 20
    xs = synthetic.rank_buffers(n, n * rc, "bfloat16", "normal:0.01", 77, dev)
    outs = [torch.empty(rc, dtype=torch.bfloat16, device=dev) for _ in range(n)]
    with vr.Communicator(n, 16, "simple", 512 << 10) as comm:
        comm.reduce_scatter(xs, outs)
        torch.cuda.synchronize()
        rng = np.random.default_rng(0)
        idx = torch.from_numpy(rng.integers(0, rc, 4096)).to(dev)
        for b in range(n):
            vals = [synthetic.to_numpy(x[b * rc + idx]) for x in xs]
            # block b's fold over the sampled elements: ReduceScatter of the
            # sampled columns, one element per block
            cols = [np.concatenate([v if k == b else np.zeros_like(v) for k in range(n)])
                    for v in vals]
            want = oracle.reduce_scatter(cols, "bfloat16", "sum")[b]
            assert H.bytes_equal(synthetic.to_numpy(outs[b][idx]), want), b
        gath = [torch.empty(n * rc, dtype=torch.bfloat16, device=dev) for _ in range(n)]
        comm.all_gather(outs, gath)
        torch.cuda.synchronize()
        cat = torch.cat(outs)
        for g in gath:
            assert torch.equal(g.view(torch.int16), cat.view(torch.int16))


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_halves_on_rings_beyond_one_sm(proto):
    """72 ranks: the ring spans the CTAs of a cluster."""
    with vr.Communicator(72, 4, proto, 4096) as comm:
        assert comm.info()["transport"] == "warpcluster"
        _rs_case(comm, 72, 3001, "float16", "sum", seed=11)
        _ag_case(comm, 72, 2999, "int8", seed=12)
