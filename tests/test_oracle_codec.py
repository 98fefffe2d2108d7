"""Pins for the oracle's IEEE binary16 codec, against numpy's float16 (an
independent implementation of the same IEEE 754 format)."""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore:overflow encountered in cast")


def test_decode_exhaustive(oracle_lib):
    # every one of the 65,536 bit patterns decodes as numpy decodes it
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle_lib.half_to_double(0x8000)) == -1.0


def _np_round(x: float) -> int:
    return int(np.array(x, dtype=np.float64).astype(np.float16).view(np.uint16))


def _targeted_values():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e300, -1e300,
            math.inf, -math.inf, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26,
            2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 2.0 ** -14 - 2.0 ** -26, 3 * 2.0 ** -25,
            5 * 2.0 ** -25, 1e-10, 2047.0, 2049.0, 2051.0, 4097.0, 4098.0, 4099.0]
    # midpoints (ties) and near-ties at every normal exponent, both parities
    for e in range(-14, 16):
        ulp = 2.0 ** (e - 10)
        for m in (0, 1, 2, 3, 1021, 1022, 1023):
            base = 2.0 ** e + m * ulp
            for off in (0.5 * ulp, 0.5 * ulp * (1 - 2 ** -40), 0.5 * ulp * (1 + 2 ** -40)):
                vals.append(base + off)
                vals.append(-(base + off))
    # ties in the subnormal range
    for m in range(0, 1024, 37):
        vals.append((m + 0.5) * 2.0 ** -24)
    return vals


def test_encode_targeted(oracle_lib):
    for x in _targeted_values():
        assert oracle_lib.double_to_half(x) == _np_round(x), x


def test_encode_random(oracle_lib):
    rng = np.random.default_rng(1234)
    # log-uniform magnitudes across the whole binary16 range and beyond
    mags = np.exp2(rng.uniform(-30, 17, size=200_000))
    xs = mags * rng.choice([-1.0, 1.0], size=mags.size)
    ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle_lib.double_to_half(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_encode_nan(oracle_lib):
    h = oracle_lib.double_to_half(math.nan)
    assert (h & 0x7C00) == 0x7C00 and (h & 0x3FF) != 0


def test_round_trip_all_finite(oracle_lib):
    for b in range(0, 65536, 7):
        if (b & 0x7C00) == 0x7C00:
            continue
        assert oracle_lib.double_to_half(oracle_lib.half_to_double(b)) == b
