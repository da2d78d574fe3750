"""Failure detection without a GPU fault (GPU).

A virtual rank that never signals its neighbours (VR_DEBUG_SILENT_RANK, read
when the communicator is created) makes the other ranks' bounded waits run
out. Every wait of the kernels has a limit (here 200 ms, set with
vrCommSetTimeout); when one gives up it records vrTimeout in the status word,
every other wait sees the status and returns, and the kernel ends. The host
then reads the error without synchronising (vrCommGetAsyncError), and further
calls on that communicator fail fast with vrTimeout. Nothing traps, faults or
hangs: the context stays usable, which the last step checks."""
import time

import pytest
import torch

import gpu_helpers as H
import ring_allreduce_virtual_gb300 as vr

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _built():
    from ring_allreduce_virtual_gb300 import build
    build.build()


@pytest.mark.parametrize("proto", ["simple", "simple-global", "ll", "ll-global",
                                   "ll128", "ll128-global", "simple-warpcluster",
                                   "ll-warpcluster", "ll128-warpcluster"])
@pytest.mark.parametrize("kernel", ["1", "0"], ids=["latency", "general"])
def test_silent_rank_times_out_and_is_sticky(proto, kernel, monkeypatch):
    """With VR_LATENCY_KERNEL=1 the one-pass call below runs the latency
    kernel on the warp transports (Simple, LL); with 0, the general one."""
    monkeypatch.setenv("VR_LATENCY_KERNEL", kernel)
    monkeypatch.setenv("VR_DEBUG_SILENT_RANK", "1")
    dev = torch.device("cuda")
    comm = H.make_comm(4, 2, proto, 4096)
    monkeypatch.delenv("VR_DEBUG_SILENT_RANK")
    try:
        comm.set_timeout(200)
        xs = [torch.ones(100000, device=dev) for _ in range(4)]
        outs = [torch.empty_like(x) for x in xs]
        assert comm.async_error() == vr.vrSuccess
        t0 = time.time()
        comm.all_reduce(xs, outs)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        assert elapsed < 5.0, elapsed
        assert comm.async_error() == vr.vrTimeout
        with pytest.raises(vr.VrError) as e:
            comm.all_reduce(xs, outs)
        assert e.value.code == vr.vrTimeout
    finally:
        comm.destroy()
    # The device is still usable: a fresh communicator is exact.
    H.run_case(4, 10001, "float32", "sum", proto, 2, 4096, seed=9)


def test_destroyed_handle_is_rejected():
    comm = vr.Communicator(2, 1, "simple", 1024)
    h = comm.handle
    comm.destroy()
    with pytest.raises(vr.VrError) as e:
        vr.vrAllReduce(h, [1, 1], [1, 1], 1, "float32", "sum")
    assert e.value.code == vr.vrInvalidArgument
    with pytest.raises(vr.VrError):
        vr.vrCommDestroy(h)


def test_argument_errors():
    dev = torch.device("cuda")
    with vr.Communicator(2, 1, "simple", 1024) as comm:
        x = torch.zeros(16, dtype=torch.float32, device=dev)
        p = x.data_ptr()
        for args in (([p, 0], [p, p]), ([p, p + 2], [p, p]), ([p, p], [p + 1, p])):
            with pytest.raises(vr.VrError) as e:
                vr.vrAllReduce(comm.handle, args[0], args[1], 4, "float32", "sum")
            assert e.value.code == vr.vrInvalidArgument
        with pytest.raises(vr.VrError) as e:
            vr.vrAllReduce(comm.handle, [p, p], [p, p], 4, 99, "sum")
        assert e.value.code == vr.vrInvalidArgument
        with pytest.raises(vr.VrError) as e:
            vr.vrAllReduce(comm.handle, [p, p], [p, p], 4, "float32", 7)
        assert e.value.code == vr.vrInvalidArgument
        with pytest.raises(vr.VrError):
            comm.set_timeout(0)


def test_too_many_ranks_times_channels_is_invalid_usage():
    """Global-memory FIFOs need every (channel, rank) CTA resident at once;
    the warp rings over a cluster take any channel count."""
    with pytest.raises(vr.VrError) as e:
        H.make_comm(128, 128, "simple-global", 1024)
    assert e.value.code == vr.vrInvalidUsage
    with vr.Communicator(128, 128, "simple", 1024) as comm:
        assert comm.info()["transport"] == "warpcluster"


def test_no_alloc_silent_rank_times_out_and_is_reported(monkeypatch):
    """vrAllReduceNoAlloc with a rank that never signals: its waits give up
    after VR_TIMEOUT_MS, vrAllReduceNoAllocGetStatus reports vrTimeout, and
    the next call (which clears the status) is exact again."""
    dev = torch.device("cuda")
    n, count = 4, 100000
    xs = [torch.full((count,), float(r + 1), device=dev) for r in range(n)]
    outs = [torch.empty_like(x) for x in xs]
    args = ([x.data_ptr() for x in xs], [o.data_ptr() for o in outs], count, n, 2, "simple", 4096,
            "float32", "sum", torch.cuda.current_stream().cuda_stream)
    monkeypatch.setenv("VR_DEBUG_SILENT_RANK", "1")
    monkeypatch.setenv("VR_TIMEOUT_MS", "200")
    t0 = time.time()
    vr.vrAllReduceNoAlloc(*args)
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    assert vr.vrAllReduceNoAllocGetStatus() == vr.vrTimeout
    monkeypatch.delenv("VR_DEBUG_SILENT_RANK")
    monkeypatch.delenv("VR_TIMEOUT_MS")
    vr.vrAllReduceNoAlloc(*args)
    torch.cuda.synchronize()
    assert vr.vrAllReduceNoAllocGetStatus() == vr.vrSuccess
    for o in outs:
        assert bool((o == 10.0).all())
