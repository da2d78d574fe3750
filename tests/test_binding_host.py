"""Host-side logic of the Python binding (CPU): the scalar of a
pre-multiplied sum as bytes of its element type, and the name tables."""
import numpy as np
import pytest
import torch

import ring_allreduce_virtual_gb300 as vr


def test_integer_scalars_wrap_like_a_c_cast():
    assert vr._scalar_bytes(3, "int8") == b"\x03"
    assert vr._scalar_bytes(-7, "int8") == (-7 & 0xFF).to_bytes(1, "little")
    assert vr._scalar_bytes(-7, "uint32") == (2 ** 32 - 7).to_bytes(4, "little")
    assert vr._scalar_bytes(2 ** 40 + 5, "int32") == (5).to_bytes(4, "little")
    assert vr._scalar_bytes(-1, "uint64") == b"\xff" * 8


@pytest.mark.parametrize("x", [0.1, -2.5, 1e-8, 65519.0, 3.0e38, float("inf")])
def test_float_scalars_round_to_nearest_even(x):
    with np.errstate(over="ignore"):
        assert vr._scalar_bytes(x, "float16") == np.array(x, np.float16).tobytes()
        assert vr._scalar_bytes(x, "float32") == np.array(x, np.float32).tobytes()
    assert vr._scalar_bytes(x, "float64") == np.array(x, np.float64).tobytes()
    want = torch.tensor([x], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()
    assert vr._scalar_bytes(x, "bfloat16") == (want & 0xFFFF).to_bytes(2, "little")


def test_bfloat16_ties_and_nan():
    # 1 + 2^-8 lies halfway between two bfloat16 values: ties to even (1.0)
    assert vr._scalar_bytes(1 + 2.0 ** -8, "bfloat16") == (0x3F80).to_bytes(2, "little")
    assert vr._scalar_bytes(1 + 3 * 2.0 ** -8, "bfloat16") == (0x3F82).to_bytes(2, "little")
    b = int.from_bytes(vr._scalar_bytes(float("nan"), "bfloat16"), "little")
    assert (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0


@pytest.mark.parametrize("dtype,top,code", [("float8_e4m3", 448.0, 0x7E),
                                            ("float8_e5m2", 57344.0, 0x7B)])
def test_fp8_scalars_saturate(dtype, top, code):
    assert vr._scalar_bytes(1.0, dtype) == bytes([0x38 if dtype == "float8_e4m3" else 0x3C])
    assert vr._scalar_bytes(top * 3, dtype) == bytes([code])
    assert vr._scalar_bytes(-top * 3, dtype) == bytes([code | 0x80])


def test_bytes_pass_through_and_sizes():
    assert vr._scalar_bytes(b"\x01\x02", "float16") == b"\x01\x02"
    with pytest.raises(ValueError):
        vr._scalar_bytes(b"\x01", "float16")
    for name, code in vr.DTYPES.items():
        assert len(vr._scalar_bytes(1, name)) == vr._ELEM_SIZE[name], name
    assert vr.OPS["avg"] == 4 and sorted(vr.DTYPES.values()) == list(range(12))


def test_no_alloc_wrapper_checks_the_address_lists():
    # A host-only check: a list shorter or longer than nRanks never reaches
    # the library (which would read past the array).
    with pytest.raises(ValueError):
        vr.vrAllReduceNoAlloc([1, 2, 3], [1, 2, 3, 4], 16, 4, 1, "simple", 4096, "float32", "sum")
    with pytest.raises(ValueError):
        vr.vrAllReduceNoAlloc([1] * 5, [1] * 5, 16, 4, 1, "simple", 4096, "float32", "sum")
