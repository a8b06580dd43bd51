"""Pins of the oracle's E4M3 codec against something other than itself.

* PyTorch's float8_e4m3fn type (an independent library implementation of OCP E4M3):
  decode of all 256 codes, and round-to-nearest-even encode of every finite FP16 value
  below the saturation knee plus random float32 values.
* Values the OCP OFP8 v1.0 specification states for E4M3: max normal 448 (0x7E),
  min normal 2**-6 (0x08), min subnormal 2**-9 (0x01), NaN S.1111.111, no infinity.
"""

import numpy as np
import pytest
import torch

from oracle import e4m3


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_table_matches_torch_float8():
    ours = e4m3.decode_table()
    ref = torch_decode_all()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    # signed zero
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_decode_spec_values():
    t = e4m3.decode_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x08] == 2.0 ** -6
    assert t[0x01] == 2.0 ** -9
    assert t[0x07] == 7 * 2.0 ** -9
    assert t[0x38] == 1.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.all(np.isfinite(np.delete(t, [0x7F, 0xFF])))
    assert np.all(np.diff(t[:0x7F]) > 0)            # monotone non-negative codes


def test_encode_matches_torch_on_all_fp16_values():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    vals = vals[np.isfinite(vals) & (np.abs(vals) < 464.0)]
    ours = e4m3.encode_rne_satfinite(vals)
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encode_matches_torch_on_random_fp32():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(200000) * np.exp2(rng.uniform(-14, 9, size=200000))
    x = x.astype(np.float32)
    x = x[np.abs(x) < 464.0].astype(np.float64)
    ours = e4m3.encode_rne_satfinite(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encode_ties_to_even():
    # midpoint of 0 and 2**-9 -> 0 (even); midpoint of 2**-9 and 2**-8 -> 2**-8 (code 2)
    assert e4m3.encode_rne_satfinite(np.array([2.0 ** -10]))[0] == 0x00
    assert e4m3.encode_rne_satfinite(np.array([1.5 * 2.0 ** -9]))[0] == 0x02
    # between 1.0 (0x38) and 1.125 (0x39): midpoint 1.0625 -> 1.0 (even)
    assert e4m3.encode_rne_satfinite(np.array([1.0625]))[0] == 0x38
    # between 1.125 (0x39) and 1.25 (0x3A): midpoint -> 1.25 (even)
    assert e4m3.encode_rne_satfinite(np.array([1.1875]))[0] == 0x3A


def test_encode_saturates_and_keeps_sign():
    y = np.array([448.0, 449.0, 464.0, 500.0, 1e30, -1e30, -448.5, -0.0, -1e-9, 1e-9])
    c = e4m3.encode_rne_satfinite(y)
    assert list(c) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80, 0x80, 0x00]


def test_encode_rejects_nonfinite():
    with pytest.raises(ValueError):
        e4m3.encode_rne_satfinite(np.array([np.nan]))


def test_round_trip_all_finite_codes():
    t = e4m3.decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], dtype=np.uint8)
    assert np.array_equal(e4m3.encode_rne_satfinite(t[codes]), codes)
