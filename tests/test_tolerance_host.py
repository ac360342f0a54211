"""The bf16 output bound used by the GPU parity tests, checked on the CPU.

Below |ref| = 8 the bound is the stated max-abs 2e-2.  At and above it a stored
bf16 value is an fp32 result within 2e-2 rounded once, so it may differ from
the real value by 2e-2 plus half the bf16 spacing at its magnitude: 0.05125 on
[8, 16), 0.0825 on [16, 32).  A value a whole spacing away must fail.
"""
import numpy as np
import pytest

from tests.gpu_helpers import assert_close, bf16_ulp


def test_bf16_spacing():
    assert bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert bf16_ulp(np.array([8.0, 15.9]))[0] == 0.0625
    assert bf16_ulp(np.array([-20.0]))[0] == 0.125


@pytest.mark.parametrize("ref,err,ok", [
    (0.5, 0.0199, True), (0.5, 0.0201, False),
    (7.9, 0.0199, True), (7.9, 0.0201, False),
    (9.0, 0.0512, True), (9.0, 0.0520, False), (9.0, 0.0625, False),
    (-12.0, -0.0512, True), (-12.0, 0.0626, False),
    (15.99, 0.0820, True),                      # may round into [16, 32): half of 0.125 plus 2e-2
    (20.0, 0.0824, True), (20.0, 0.0830, False),
])
def test_bf16_bound(ref, err, ok):
    # many exact points keep the relative-L2 part of the check out of the way
    refs = np.concatenate([[ref], np.full(10000, 1.0)])
    got = refs.copy()
    got[0] += err
    if ok:
        assert_close(got, refs, "bf16")
    else:
        with pytest.raises(AssertionError):
            assert_close(got, refs, "bf16")
