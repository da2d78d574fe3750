"""vrCommGetPlan (GPU: a communicator needs a device): the parts and rings of
a call, worked out by hand from the chunk map and the FIFO geometry."""
import pytest
import torch

import ring_allreduce_virtual_gb300 as vr

pytestmark = pytest.mark.gpu


def _div_up(a, b):
    return -(-a // b)


def test_plan_of_the_headline_shape():
    # 16 ranks, 32 channels, 1 MiB chunks, 256 Mi fp32: per channel 8 Mi
    # elements = two loops of 16 chunks; each chunk moves in parts of one
    # Simple payload (a slot: depth 2, so half the FIFO).
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with vr.Communicator(16, 32, "simple", 1 << 20) as comm:
        slot = comm.info()["slot_bytes"]
        parts, rings = comm.plan(256 << 20, "float32")
        assert parts == 32 * 2 * _div_up(1 << 20, slot)
        assert rings == sms  # one 16-rank ring per CTA, one CTA per SM


def test_plan_of_a_tiny_call():
    # 8 ranks, 16 channels, 256 int32: channels of 16 elements, one last loop
    # with chunks of alignUp(divUp(16, 8), 4) = 4 elements: one part each;
    # two 8-rank rings per CTA, so 8 CTAs.
    with vr.Communicator(8, 16, "simple", 512 << 10) as comm:
        assert comm.plan(256, "int32") == (16, 16)
        assert comm.plan(0, "int32") == (0, 0)


def test_plan_of_global_fifos():
    import gpu_helpers as H
    with H.make_comm(72, 8, "ll-global", 64 << 10) as comm:
        parts, rings = comm.plan(2 << 20, "float16")
        assert rings == 8  # one ring per channel
        assert parts >= 8


def test_plan_of_a_ring_over_a_cluster():
    # 72 ranks over a cluster; 8 channels of 256 Ki fp16 = one last loop of
    # 72 chunks of 3648 elements (7296 B). Every chunk moves in the same
    # number of parts, so the parts are a multiple of 8, and the call takes
    # a FIFO geometry that runs it in one pass of the rings.
    with vr.Communicator(72, 8, "ll", 64 << 10) as comm:
        assert comm.info()["transport"] == "warpcluster"
        parts, rings = comm.plan(2 << 20, "float16")
        assert parts % 8 == 0 and parts <= rings, (parts, rings)
        # a small call: chunks of 64 elements, one part each
        assert comm.plan(72 * 8 * 64, "float16")[0] == 8


def test_one_own_slot_geometry_is_exact():
    """The 72-rank workload on the geometry it picks, bit for bit."""
    import gpu_helpers as H
    H.run_case(72, 2 << 20, "float16", "sum", "ll", 8, 64 << 10, seed=3)
    H.run_case(72, 2 << 20 | 13, "bfloat16", "sum", "simple", 8, 64 << 10, seed=4)
