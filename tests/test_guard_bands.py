"""The guard bands that the GPU tests put around every output (gpu_util.guarded): checked here on
host tensors, so that the mechanism itself needs no GPU. A write past either end of an output must
be reported, a write inside it must not, and long runs must check (and let go of) their outputs
before they hold too much memory."""

import pytest
import torch

import gpu_util as gu


def _raw(i=-1):
    """The whole buffer (band, output, band) of the i-th output allocated since the last check."""
    return gu._guarded[i][0]


def test_guarded_output_has_the_shape_dtype_and_offset_asked_for():
    t = gu.guarded((3, 8), torch.bfloat16, device="cpu")
    assert t.shape == (3, 8) and t.dtype == torch.bfloat16 and t.is_contiguous()
    assert t.data_ptr() - _raw().data_ptr() == gu.GUARD_BYTES
    assert t.data_ptr() % 16 == 0
    z = gu.guarded((0, 16), torch.float32, device="cpu")
    assert z.shape == (0, 16) and z.numel() == 0
    t.fill_(1.0)  # the whole output may be written
    gu.check_guards()
    assert gu._guarded == [] and gu._guarded_bytes == 0


@pytest.mark.parametrize("side,offset", [("before", gu.GUARD_BYTES - 1), ("before", 0), ("after", 0),
                                         ("after", gu.GUARD_BYTES - 1)])
def test_a_write_into_either_band_is_reported(side, offset):
    t = gu.guarded((4, 4), torch.float32, device="cpu")
    buf = _raw()
    nbytes = t.numel() * 4
    buf[offset if side == "before" else gu.GUARD_BYTES + nbytes + offset] = 0
    with pytest.raises(AssertionError, match="guard band %s" % side):
        gu.check_guards()
    gu.check_guards()  # the failed check let go of its outputs: nothing is left to check


def test_long_runs_check_before_they_hold_too_much(monkeypatch):
    monkeypatch.setattr(gu, "_GUARD_CHECK_BYTES", 1024)
    gu.guarded((128,), torch.float32, device="cpu")  # 512 bytes held
    _raw()[0] = 0                                       # its leading band written
    with pytest.raises(AssertionError, match="guard band before"):
        gu.guarded((160,), torch.float32, device="cpu")  # 640 more would pass 1024: the check runs first
    assert gu._guarded == []
