"""Property checks of the oracle's q8_0 blocks (reading Q1) over many random blocks of
F16-representable values (what the ring stores: F16 inputs, or float32 values of the same
range): the round trip stays within half a quantisation step plus the F16 scale's
rounding, the largest magnitude of a block maps to code +-127, codes stay in [-127, 127],
and scaling a block by a power of two scales its scale and keeps its codes (while the
scale stays a normal F16 value).  CPU only."""

import numpy as np
import pytest

from oracle import ring_oracle as orc

hypothesis = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
hnp = pytest.importorskip("hypothesis.extra.numpy")

blocks = hnp.arrays(np.float32, (3, orc.Q8_BLOCK),
                    elements=st.floats(-60.0, 60.0, allow_nan=False, width=16))


def _f16_ulp(x):
    a = np.abs(np.asarray(x, np.float64))
    return np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -14))) - 10)


@hypothesis.settings(max_examples=300, deadline=None)
@hypothesis.given(blocks)
def test_round_trip_within_half_a_step(x):
    codes, scales = orc.q8_0_quantize(x)
    back = orc.q8_0_dequantize(codes, scales)
    amax = np.abs(x.astype(np.float64)).max(axis=-1)
    d = amax / 127.0
    d16 = scales.astype(np.float64)[:, 0]
    bound = 0.5 * d * (1 + 1e-4) + 127 * np.abs(d16 - d) + 1e-30
    assert np.all(np.abs(back - x.astype(np.float64)) <= np.repeat(bound, orc.Q8_BLOCK).reshape(x.shape))
    assert np.all(np.abs(codes.astype(np.int32)) <= 127)
    nz = amax > 0
    peak = np.abs(codes.astype(np.int32)).max(axis=-1)
    assert np.all(peak[nz] == 127) and np.all(peak[~nz] == 0)
    assert np.all(np.abs(d16 - d) <= 0.5 * _f16_ulp(d) + 1e-30)


@hypothesis.settings(max_examples=200, deadline=None)
@hypothesis.given(blocks, st.integers(-6, 6))
def test_power_of_two_scaling_keeps_codes(x, k):
    c0, s0 = orc.q8_0_quantize(x)
    c1, s1 = orc.q8_0_quantize(x * np.float32(2.0 ** k))
    d0 = np.abs(x.astype(np.float64)).max(axis=-1) / 127.0
    normal = (d0 >= 2.0 ** -13) & (d0 * 2.0 ** k >= 2.0 ** -13)
    np.testing.assert_array_equal(c1[normal], c0[normal])
    np.testing.assert_array_equal(s1.astype(np.float64)[:, 0][normal],
                                  s0.astype(np.float64)[:, 0][normal] * 2.0 ** k)
