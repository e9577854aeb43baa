"""The oracle against its pins (CPU only)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_page_facts_consistent():
    """The transcribed page facts agree with one another."""
    f = oracle_pins.read_facts()
    ein = [int(v) for v in f["epilogue_in_shape"].split(",")]
    eout = [int(v) for v in f["epilogue_out_shape"].split(",")]
    assert eout == [ein[0]] + ein[2:]
    assert int(f["epilogue_slice_len"]) == ein[2] * ein[3] * ein[4]
    b = [int(v) for v in f["bn_in_shape"].split(",")]
    assert int(f["bn_channel_count"]) == b[0] * b[2] * b[3]
    i = [int(v) for v in f["in2d_shape"].split(",")]
    assert int(f["in2d_slices"]) == i[0] * i[1] and int(f["in2d_slice_len"]) == i[2] * i[3]
