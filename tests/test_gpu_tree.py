"""The double-binary-tree AllReduce (vrAllReduceTree) vs the CPU oracle's tree
fold, bit for bit, on every rank (GPU): every ring size 2..16, every element
type x reduction, ragged and unaligned buffers, in place, pieces spread over
many CTAs, and the full-size headline-shaped input on sampled elements."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


def tree_case(n, count, dtype, op, seed=0, inplace=False, offset=0, comm=None):
    dev = torch.device("cuda")
    xs = synthetic.rank_buffers(n, count, dtype, synthetic.default_recipe(dtype), seed, "cpu")
    tdt = synthetic.TORCH_DTYPE[dtype]
    own = comm is None
    if own:
        comm = vr.Communicator(n, 1, "simple", 4096)
    try:
        sends, recvs, bases = [], [], []
        for x in xs:
            sb, sv = H.guarded(count, tdt, dev, offset, fill=x)
            if inplace:
                sends.append(sv)
                recvs.append(sv)
                bases.append(sb)
            else:
                rb, rv = H.guarded(count, tdt, dev, offset)
                sends.append(sv)
                recvs.append(rv)
                bases.append(rb)
        comm.all_reduce_tree(sends, recvs, op, dtype=dtype)
        torch.cuda.synchronize()
        assert comm.async_error() == vr.vrSuccess
        want = oracle.tree_allreduce([synthetic.to_numpy(x) for x in xs], dtype, op)
        for r in range(n):
            got = synthetic.to_numpy(recvs[r])
            if not H.bytes_equal(got, want):
                bad = np.nonzero(got.view(np.uint8) != want.view(np.uint8))[0]
                raise AssertionError(f"rank {r}: {len(bad)} bytes differ, first at byte {bad[0]} "
                                     f"(n={n} count={count} {dtype} {op})")
            assert H.guards_intact(bases[r], count, offset), f"guard overwritten, rank {r}"
        return want
    finally:
        if own:
            comm.destroy()


@pytest.mark.parametrize("n", list(range(2, 17)))
def test_ring_sizes(n):
    for count in (1, 5, 1000, 65539, 300007):
        tree_case(n, count, "float32", "sum", seed=n * 7 + count)


@pytest.mark.parametrize("dtype", list(vr.DTYPES))
def test_every_dtype_and_op(dtype):
    with vr.Communicator(7, 1, "simple", 4096) as comm:
        for i, op in enumerate(oracle.OPS):
            for count in (1003, 40961):
                tree_case(7, count, dtype, op, seed=13 * i + count, comm=comm)


def test_in_place_and_unaligned():
    tree_case(6, 70001, "float32", "sum", inplace=True, seed=5)
    tree_case(5, 12345, "bfloat16", "sum", offset=1, seed=6)
    tree_case(8, 9999, "int8", "max", offset=3, seed=7)


def test_many_pieces_and_repeated_calls():
    with vr.Communicator(16, 1, "simple", 4096) as comm:
        for seed in range(3):
            tree_case(16, 3 * 2 ** 20 + 17, "float16", "sum", seed=seed, comm=comm)


def test_integer_result_equals_the_ring():
    """Integer sum does not depend on the order: tree and ring agree."""
    dev = torch.device("cuda")
    xs = synthetic.rank_buffers(9, 500001, "int32", "int:-1048576:1048576", 3, dev)
    a = [torch.empty_like(x) for x in xs]
    b = [torch.empty_like(x) for x in xs]
    with vr.Communicator(9, 4, "simple", 64 << 10) as comm:
        comm.all_reduce(xs, a, "sum")
        comm.all_reduce_tree(xs, b, "sum")
        torch.cuda.synchronize()
    for r in range(9):
        assert torch.equal(a[r], b[r])


@pytest.mark.parametrize("n", [18, 24, 32, 72, 128])
def test_trees_beyond_one_sm(n):
    """Trees of more than 16 ranks span the CTAs of a cluster."""
    with vr.Communicator(n, 1, "simple", 4096) as comm:
        tree_case(n, 100003, "float16", "sum", seed=n, comm=comm)
        tree_case(n, 7777, "int32", "max", seed=n + 1, comm=comm)
        tree_case(n, 4099, "float32", "sum", seed=n + 2, comm=comm)


@pytest.mark.parametrize("n,ctas", [(8, 2), (8, 4), (12, 3), (16, 8), (6, 6)])
def test_small_trees_split_over_a_cluster(n, ctas, monkeypatch):
    """Every tree edge between CTAs, on small trees split by hand."""
    monkeypatch.setenv("VR_CLUSTER_CTAS", str(ctas))
    tree_case(n, 300007, "bfloat16", "sum", seed=ctas)
    tree_case(n, 40961, "int64", "prod", seed=ctas + 1)


def test_rejects_unsplittable_rings_and_handles_edges(monkeypatch):
    dev = torch.device("cuda")
    # A cluster split that cannot hold the tree (more than 16 CTAs, or more
    # than 16 ranks in a CTA) is refused.
    with vr.Communicator(17, 1, "simple", 4096) as comm:
        x = [torch.zeros(8, device=dev) for _ in range(17)]
        for bad in ("17", "1"):
            monkeypatch.setenv("VR_CLUSTER_CTAS", bad)
            with pytest.raises(vr.VrError) as e:
                comm.all_reduce_tree(x, x)
            assert e.value.code == vr.vrInvalidUsage
        monkeypatch.delenv("VR_CLUSTER_CTAS")
    with vr.Communicator(1, 1, "simple", 4096) as comm:
        x, y = [torch.arange(10.0, device=dev)], [torch.zeros(10, device=dev)]
        comm.all_reduce_tree(x, y)
        torch.cuda.synchronize()
        assert torch.equal(x[0], y[0])
    with vr.Communicator(4, 1, "simple", 4096) as comm:
        vr.vrAllReduceTree(comm.handle, [0] * 4, [0] * 4, 0, "float32", "sum")


def test_full_size_sampled():
    """16 x 256 Mi fp32 (1 GiB per rank): sampled elements equal the oracle's
    tree fold; every rank's output is identical."""
    n, count = 16, 256 << 20
    dev = torch.device("cuda")
    xs = synthetic.rank_buffers(n, count, "float32", "uniform", 21, dev)
    outs = [torch.empty_like(x) for x in xs]
    with vr.Communicator(n, 1, "simple", 4096) as comm:
        comm.all_reduce_tree(xs, outs)
        torch.cuda.synchronize()
    for r in range(1, n):
        assert torch.equal(outs[r], outs[0])
    rng = np.random.default_rng(1)
    idx = np.unique(np.concatenate([rng.integers(0, count, 4000),
                                    [0, count // 2 - 1, count // 2, count - 1]]))
    it = torch.from_numpy(idx.astype(np.int64)).to(dev)
    vals = [synthetic.to_numpy(x[it]) for x in xs]
    # The oracle on the sampled elements: the split of the full buffer decides
    # each element's tree, so fold the samples of each half separately.
    split = oracle.tree_split(count, 4)
    got = synthetic.to_numpy(outs[0][it])
    for mask, tree in ((idx < split, 0), (idx >= split, 1)):
        sel = [v[mask] for v in vals]
        if len(sel[0]):
            assert H.bytes_equal(got[mask], _tree_fold_samples(sel, tree))


def _tree_fold_samples(vals, tree):
    """The oracle's tree `tree` fold of sampled elements: a buffer whose split
    falls after every sample (tree 0) or a two-part buffer whose second half
    holds them (tree 1)."""
    n, m = len(vals), len(vals[0])
    if tree == 0:
        pad = [np.concatenate([v, np.zeros(m + 8, v.dtype)]) for v in vals]
        return oracle.tree_allreduce(pad, "float32", "sum")[:m]
    # choose a length whose split is a multiple of 4 at or past m
    first = ((m + 3) // 4) * 4
    pad = [np.concatenate([np.zeros(first, v.dtype), v]) for v in vals]
    assert oracle.tree_split(len(pad[0]), 4) == first
    return oracle.tree_allreduce(pad, "float32", "sum")[first:]
