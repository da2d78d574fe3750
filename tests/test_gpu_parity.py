"""CUDA path vs the CPU oracle, element by element, on every rank (GPU).

Sizes span several FIFO slots, several loops and ragged tails; every element
type x reduction, every protocol, in place, unaligned pointers, one rank, zero
elements, repeated calls on one communicator and the FIFO-reset path."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import oracle
import ring_allreduce_virtual_gb300 as vr
from ring_allreduce_virtual_gb300 import synthetic

pytestmark = pytest.mark.gpu

# Plain protocol names run on the warp-ring transport wherever it fits (up to
# 16 ranks); a "-global" or "-warpcluster" suffix forces the other
# transports ("-warpcluster": the ring's warps spread over the CTAs of a
# cluster even when one CTA would hold them, to exercise those edges).
PROTOS = ["simple", "simple-global", "ll", "ll-global", "ll128",
          "ll128-global", "simple-warpcluster", "ll-warpcluster", "ll128-warpcluster"]
DTYPES = list(vr.DTYPES)
OPS = list(oracle.OPS)  # the plain reductions; avg and premulsum: test_gpu_scaled_ops

# (n ranks, count, channels, chunk bytes)
SHAPES = [
    (2, 1, 1, 16), (2, 2, 1, 16), (2, 3, 2, 16), (2, 17, 5, 32), (3, 7, 1, 16),
    (3, 1000, 2, 256), (4, 65536, 1, 512 << 10), (4, 65539, 3, 4096), (5, 4097, 4, 48),
    (8, 100003, 7, 64 << 10), (16, 33333, 2, 1 << 10), (7, 50000, 16, 16),
    (3, 3 * 2 ** 20 + 5, 3, 64 << 10), (6, 777777, 5, 24 << 10), (12, 2 ** 18 + 1, 4, 1 << 20),
]


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "n{}_c{}_ch{}_k{}".format(*s))
def test_float32_sum_shapes(proto, shape):
    n, count, nch, chunk = shape
    H.run_case(n, count, "float32", "sum", proto, nch, chunk, seed=hash(shape) & 0xffff)


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_every_dtype_and_op(proto, dtype):
    with H.make_comm(5, 3, proto, 4096) as comm:
        for i, op in enumerate(OPS):
            for count in (1003, 40961):
                H.run_case(5, count, dtype, op, proto, 3, 4096, seed=17 * i + count, comm=comm)


@pytest.mark.parametrize("proto", PROTOS)
def test_in_place(proto):
    H.run_case(4, 70001, "float32", "sum", proto, 3, 8192, inplace=True, seed=5)
    H.run_case(3, 12345, "bfloat16", "sum", proto, 2, 256, inplace=True, seed=6)


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_pointers(proto, offset):
    H.run_case(4, 9999, "float32", "sum", proto, 2, 1024, offset=offset, seed=offset)
    H.run_case(3, 5001, "int8", "max", proto, 2, 256, offset=offset, seed=offset)


def test_one_rank_is_a_copy():
    H.run_case(1, 12345, "float32", "sum", "simple", 1, 4096, seed=1)
    H.run_case(1, 777, "bfloat16", "sum", "ll", 3, 16, seed=2, inplace=True)


@pytest.mark.parametrize("proto", PROTOS)
def test_zero_count_launches_nothing(proto):
    with H.make_comm(4, 2, proto, 4096) as comm:
        xs = [torch.zeros(0, device="cuda") for _ in range(4)]
        comm.all_reduce(xs, [torch.zeros(0, device="cuda") for _ in range(4)])
        torch.cuda.synchronize()
        assert comm.async_error() == vr.vrSuccess


def test_worked_examples():
    """[r, r+1] over 4 ranks -> [6, 10]; element 0 = r over N ranks -> N(N-1)/2."""
    dev = torch.device("cuda")
    for proto in PROTOS:
        xs = synthetic.rank_buffers(4, 2, "float32", "pairs", 0, dev)
        outs = [torch.empty_like(x) for x in xs]
        with H.make_comm(4, 1, proto, 512 << 10) as comm:
            comm.all_reduce(xs, outs)
            torch.cuda.synchronize()
        assert all(o.tolist() == [6.0, 10.0] for o in outs)
        for n in (2, 4, 8):
            xs = synthetic.rank_buffers(n, 32 << 20, "float32", "first", 0, dev)
            outs = [torch.empty_like(x) for x in xs]
            with H.make_comm(n, 4, proto, 512 << 10) as comm:
                comm.all_reduce(xs, outs)
                torch.cuda.synchronize()
            for o in outs:
                assert o[0].item() == n * (n - 1) // 2
                assert int(torch.count_nonzero(o[1:])) == 0


@pytest.mark.parametrize("proto", PROTOS)
def test_repeated_calls_on_one_communicator(proto):
    """Flags carry a per-call step base, so the FIFO is never cleared between
    calls: back-to-back calls of different sizes and types must stay exact."""
    rng = np.random.default_rng(11)
    with H.make_comm(6, 4, proto, 2048) as comm:
        for i in range(40):
            dtype = DTYPES[int(rng.integers(len(DTYPES)))]
            count = int(rng.integers(1, 60000))
            op = OPS[int(rng.integers(len(OPS)))]
            H.run_case(6, count, dtype, op, proto, 4, 2048, seed=i, comm=comm)


@pytest.mark.parametrize("proto", PROTOS)
def test_fifo_reset_when_the_step_counter_wraps(proto, monkeypatch):
    monkeypatch.setenv("VR_DEBUG_STEP_WRAP", "300")
    with H.make_comm(4, 2, proto, 1024) as comm:
        for i in range(12):
            H.run_case(4, 30000 + 7 * i, "float32", "sum", proto, 2, 1024, seed=i, comm=comm)


@pytest.mark.parametrize("proto", PROTOS)
def test_fifo_geometry_does_not_change_results(proto, monkeypatch):
    """Slot size and depth are performance knobs only."""
    want = None
    for slot, depth in ((1024, 2), (4096, 3), (16384, 4), (65536, 8)):
        if "-" not in proto:
            if slot * depth > 32768:
                continue  # a shared-memory ring's FIFO must fit in one SM
        if proto.endswith("-warpcluster") and slot * depth > 8192:
            continue  # 16 one-rank ring parts per CTA: the FIFOs must fit in one SM
        monkeypatch.setenv("VR_FIFO_SLOT_BYTES", str(slot))
        monkeypatch.setenv("VR_FIFO_DEPTH", str(depth))
        got = H.run_case(5, 200003, "bfloat16", "sum", proto, 3, 16384, seed=3)
        if want is not None:
            assert H.bytes_equal(got, want)
        want = got


def test_stress_back_to_back():
    """Many small calls queued without synchronising, then all checked."""
    rng = np.random.default_rng(5)
    dev = torch.device("cuda")
    for proto in PROTOS:
        with H.make_comm(4, 3, proto, 1024) as comm:
            jobs = []
            for i in range(300):
                count = int(rng.integers(1, 5000))
                xs = synthetic.rank_buffers(4, count, "float32", "uniform", 1000 + i, dev)
                outs = [torch.empty_like(x) for x in xs]
                comm.all_reduce(xs, outs)
                jobs.append((xs, outs))
            torch.cuda.synchronize()
            assert comm.async_error() == vr.vrSuccess
            for xs, outs in jobs:
                want = oracle.allreduce([synthetic.to_numpy(x) for x in xs], "float32", "sum",
                                        3, 1024)
                for o in outs:
                    assert H.bytes_equal(synthetic.to_numpy(o), want)


def test_transport_choice():
    """Rings of 2..16 ranks run as warp rings in one SM's shared memory; every
    larger ring up to 128 ranks as warp rings over a cluster (CTAs of
    ceil(N / C) or floor(N / C) ranks); the other transports only when asked
    for."""
    for n in range(17, 129):
        with H.make_comm(n, 2, "simple", 4096) as comm:
            assert comm.info()["transport"] == "warpcluster", n
    for n, proto, want in ((2, "simple", "warp"), (16, "simple", "warp"),
                           (8, "ll", "warp"), (8, "ll128", "warp"),
                           (17, "simple", "warpcluster"), (17, "ll", "warpcluster"),
                           (71, "ll128", "warpcluster"), (127, "simple", "warpcluster"),
                           (72, "ll", "warpcluster"), (72, "simple", "warpcluster"),
                           (32, "ll128", "warpcluster"), (128, "simple", "warpcluster"),
                           (8, "simple-global", "global"), (8, "ll-global", "global"),
                           (8, "simple-warpcluster", "warpcluster")):
        with H.make_comm(n, 2, proto, 4096) as comm:
            assert comm.info()["transport"] == want, (n, proto)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128",
                                   "simple-warpcluster", "ll-warpcluster"])
@pytest.mark.parametrize("n", [2, 3, 5, 8, 13, 16])
def test_ring_sizes(proto, n):
    H.run_case(n, 300007, "float32", "sum", proto, 5, 16384, seed=n)
    H.run_case(n, 4099, "bfloat16", "max", proto, 2, 64, seed=n + 1)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128",
                                   "ll-warpcluster"])
@pytest.mark.parametrize("depth,in_depth,slot", [(2, 1, 1024), (3, 2, 4096), (4, 4, 8192),
                                                 (6, 3, 1024)])
def test_fifo_geometry_of_shared_memory_rings(proto, depth, in_depth, slot, monkeypatch):
    monkeypatch.setenv("VR_FIFO_DEPTH", str(depth))
    monkeypatch.setenv("VR_FIFO_IN_DEPTH", str(in_depth))
    monkeypatch.setenv("VR_FIFO_SLOT_BYTES", str(slot))
    H.run_case(6, 500009, "float32", "sum", proto, 3, 65536, seed=depth)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
@pytest.mark.parametrize("n", [18, 24, 32, 48, 72, 96, 128])
def test_rings_beyond_one_sm(proto, n):
    """Rings of more than 16 ranks: warps over the CTAs of a cluster."""
    with H.make_comm(n, 3, proto, 8192) as comm:
        assert comm.info()["transport"] == "warpcluster", n
        H.run_case(n, 100003, "float16", "sum", proto, 3, 8192, seed=n, comm=comm)
        H.run_case(n, 7777, "int32", "max", proto, 3, 8192, seed=n + 1, comm=comm)


@pytest.mark.parametrize("ctas", [2, 3, 4, 6, 8, 12])
def test_cluster_split_of_a_24_rank_ring(ctas, monkeypatch):
    """Every split of a 24-rank ring over a cluster gives the same bytes."""
    monkeypatch.setenv("VR_CLUSTER_CTAS", str(ctas))
    for proto in ("simple-warpcluster", "ll-warpcluster", "ll128-warpcluster"):
        H.run_case(24, 50021, "bfloat16", "sum", proto, 2, 4096, seed=ctas)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_stress_ten_thousand_calls(proto):
    """10^4 calls of random size, element type and reduction on one
    communicator, queued 500 at a time without synchronising (the latency
    kernel and the general kernel both take part), every output checked
    against the oracle."""
    rng = np.random.default_rng(17)
    dev = torch.device("cuda")
    kinds = [("float32", "sum"), ("bfloat16", "sum"), ("int32", "max"), ("int8", "min"),
             ("float16", "sum"), ("int64", "prod")]
    with H.make_comm(7, 3, proto, 4096) as comm:
        for batch in range(20):
            jobs = []
            for i in range(500):
                dtype, op = kinds[int(rng.integers(len(kinds)))]
                count = int(rng.integers(1, 3000)) if rng.random() < 0.9 else \
                    int(rng.integers(3000, 200000))
                xs = synthetic.rank_buffers(7, count, dtype, synthetic.default_recipe(dtype),
                                            batch * 1000 + i, dev)
                outs = [torch.empty_like(x) for x in xs]
                comm.all_reduce(xs, outs, op, dtype=dtype)
                jobs.append((xs, outs, dtype, op))
            torch.cuda.synchronize()
            assert comm.async_error() == vr.vrSuccess
            for xs, outs, dtype, op in jobs:
                want = oracle.allreduce([synthetic.to_numpy(x) for x in xs], dtype, op, 3, 4096)
                for o in outs:
                    assert H.bytes_equal(synthetic.to_numpy(o), want), (dtype, op, xs[0].numel())
