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
    # 72 ranks: 6 CTAs of 12 ranks per ring, one ring part per CTA; 8 channels
    # of 256 Ki fp16 = one last loop of 72 chunks of 3648 elements (7296 B),
    # each moved in parts of one LL payload (half a slot).
    with vr.Communicator(72, 8, "ll", 64 << 10) as comm:
        assert comm.info()["transport"] == "warpcluster"
        payload = comm.info()["slot_bytes"] // 2
        parts, rings = comm.plan(2 << 20, "float16")
        assert parts == 8 * _div_up(7296, payload)
        assert 1 <= rings <= torch.cuda.get_device_properties(0).multi_processor_count // 6
