"""Number-format helpers of the oracle against library routines (numpy binary16, struct)."""
import struct

import numpy as np

import oracle


def test_f16_decode_all_patterns(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode(oracle_lib):
    rng = np.random.default_rng(0)
    for b in list(rng.integers(0, 65536, 2000)) + [0, 0x8000, 0x3F80, 0x7F7F, 0x0001]:
        (f,) = struct.unpack("<f", struct.pack("<I", int(b) << 16))
        g = oracle.bf16_to_f64(int(b))
        if np.isnan(f):
            assert np.isnan(g)
        else:
            assert g == f


def test_f16_rne_matches_numpy(oracle_lib):
    rng = np.random.default_rng(1)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.uniform(-9, 5, 3000))
    # halfway cases, subnormals, overflow boundary, signed zeros
    h = np.arange(0, 65504, 1.0 / 3)
    xs += [0.0, -0.0, 65504.0, 65519.99, 65520.0, 70000.0, -65520.0, 2.0 ** -24,
           2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11,
           1.0 + 3 * 2.0 ** -11, 2048.0 + 1.0, 2048.0 + 3.0]
    xs += list(h[:500])
    for x in xs:
        ref = int(np.array([x], np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.f64_to_f16_rne(float(x)) == ref, x
