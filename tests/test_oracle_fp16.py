"""Pins the oracle's binary16 conversions to numpy's (a library routine that
rounds fp64 -> fp16 directly, to nearest even)."""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_decode_all_bit_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])
    # signed zero survives
    assert np.signbit(orc.f16_to_f64(0x8000))


def test_encode_matches_numpy(orc):
    rng = np.random.default_rng(123)
    xs = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.uniform(-9, 5, 4000),
        # every exact midpoint between adjacent finite fp16 values (ties -> even)
        (np.arange(0, 0x7bff, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
         + np.arange(1, 0x7c00, 7, dtype=np.uint16).view(np.float16).astype(np.float64)) / 2,
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
         3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1 / 127.0, 127 / 127.0],
    ])
    for x in xs:
        ref = int(np.array(x).astype(np.float16).view(np.uint16))
        assert orc.f64_to_f16(x) == ref, (x, hex(ref))
    assert orc.f64_to_f16(float("nan")) & 0x7c00 == 0x7c00
