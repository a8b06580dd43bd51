"""Pins of the BASE oracle (oracle/base.py) to facts other than its own formula.

* Truncation characterisation: keeping the high byte of an FP16 word and zeroing the
  low byte is truncation toward zero of the value to the grid of its binade with two
  fraction bits (1 implicit + 2 stored significand bits; the subnormal range keeps
  multiples of 2^-16). Checked for every finite FP16 value with exact rational
  arithmetic (``fractions``), which shares nothing with the bit manipulation.
* Exact round trip TARGET -> BASE -> TARGET (ElasticKV App. B.2: promotion restores
  TARGET exactly from the low bytes), bit for bit, and the skip rules.
* Decode over BASE pages equals ordinary softmax attention (torch SDPA in float64) over
  the truncated values, and the gather writes those same truncated values.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import base, decode, gather

torch = pytest.importorskip("torch")


def _truncate_fraction(x: Fraction) -> Fraction:
    """|x| truncated to its binade's grid with 2 fraction bits, sign kept."""
    if x == 0:
        return Fraction(0)
    sgn = -1 if x < 0 else 1
    a = abs(x)
    e = math.floor(math.log2(a))               # binade [2^e, 2^(e+1)), exact for dyadics
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    unit = Fraction(2) ** (e - 2) if e >= -14 else Fraction(1, 2 ** 16)   # fp16 min normal 2^-14
    return sgn * (a // unit) * unit


def test_base_value_is_truncation_for_every_finite_fp16():
    words = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = words.view(np.float16)
    finite = np.isfinite(vals)
    got = base.base_value((words[finite] >> 8).astype(np.uint8))
    xs = vals[finite].astype(np.float64)
    for x, g in zip(xs[::7], got[::7]):          # every 7th value: ~9,000 exact checks
        want = _truncate_fraction(Fraction(float(x)))
        assert Fraction(float(g)) == want, (x, g, want)
    # and the full set against the same rule through float64 (exact: dyadic values)
    e = np.floor(np.log2(np.where(xs == 0, 1.0, np.abs(xs))))
    unit = np.where(e >= -14, np.exp2(e - 2), 2.0 ** -16)
    want = np.sign(xs) * np.floor(np.abs(xs) / unit) * unit
    assert np.array_equal(got, want)


def test_base_value_special_codes():
    assert base.base_value([0x00])[0] == 0.0
    assert math.copysign(1.0, base.base_value([0x80])[0]) == -1.0      # -0
    assert base.base_value([0x3c])[0] == 1.0
    assert base.base_value([0x7b])[0] == 57344.0                        # largest finite BASE
    assert np.isinf(base.base_value([0x7c])[0])


def test_round_trip_is_exact_and_skips():
    rng = np.random.default_rng(11)
    P, H, D = 10, 2, 64
    n = 16 * H * D
    x = (rng.standard_normal((P, 16, H, D)) * 3).astype(np.float16)
    x[4, 0, 0, 0] = np.inf
    v = x.reshape(P, -1).view(np.uint8).copy()
    mode = np.zeros(P, np.uint8)
    mode[2] = 1                                      # compact: skipped
    ids = [0, 2, 3, 4, 7]
    v2, m2, low, bad = base.demote_to_base(v, ids, mode, H, D)
    assert bad == [4] and m2[4] == 0 and np.array_equal(v2[4], v[4])
    assert m2[2] == 1 and np.array_equal(v2[2], v[2])
    for p in (0, 3, 7):
        assert m2[p] == base.MODE_BASE
        assert np.array_equal(v2[p, n:], v[p, n:])           # second half untouched
    back, m3 = base.promote(v2, [0, 3, 7], m2, low[[0, 3, 7]], H, D)
    assert np.array_equal(back, v) and np.array_equal(m3[[0, 3, 7]], [0, 0, 0])


def test_decode_over_base_pages_is_sdpa_over_truncated_values():
    rng = np.random.default_rng(12)
    P, H, G, D = 12, 2, 3, 64
    lens = np.array([40, 100], np.int32)
    k = rng.standard_normal((P, 16, H, D)).astype(np.float16)
    x = rng.standard_normal((P, 16, H, D)).astype(np.float16)
    v = x.reshape(P, -1).view(np.uint8).copy()
    mode = np.zeros(P, np.uint8)
    v, mode, _, _ = base.demote_to_base(v, np.arange(0, P, 2), mode, H, D)   # half the pages BASE
    perm = rng.permutation(P).astype(np.int32)
    bt = np.zeros((2, 7), np.int32)
    bt[0, :3], bt[1, :7] = perm[:3], perm[3:10]
    q = rng.standard_normal((2, H * G, D)).astype(np.float16)
    out, lse = decode.paged_decode(q, k, v, None, 0, mode, 0, bt, lens)
    # truncated values by the arithmetic rule, not by the byte layout
    xf = x.astype(np.float64)
    e = np.floor(np.log2(np.where(xf == 0, 1.0, np.abs(xf))))
    unit = np.where(e >= -14, np.exp2(e - 2), 2.0 ** -16)
    trunc = np.sign(xf) * np.floor(np.abs(xf) / unit) * unit
    vals = np.where((mode == base.MODE_BASE)[:, None, None, None], trunc, xf)
    for b in range(2):
        L = int(lens[b])
        pages = bt[b, : (L + 15) // 16]
        K = torch.from_numpy(k[pages].astype(np.float64).reshape(-1, H, D)[:L])
        V = torch.from_numpy(vals[pages].reshape(-1, H, D)[:L])
        Q = torch.from_numpy(q[b].astype(np.float64)).reshape(H, G, 1, D)
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, K.permute(1, 0, 2)[:, None], V.permute(1, 0, 2)[:, None], scale=1 / math.sqrt(D))
        assert np.allclose(out[b], ref.reshape(H * G, D).numpy(), rtol=0, atol=1e-12)


def test_gather_writes_truncated_values_for_base_pages():
    rng = np.random.default_rng(13)
    P, H, D = 6, 2, 64
    k = rng.standard_normal((P, 16, H, D)).astype(np.float16)
    x = rng.standard_normal((P, 16, H, D)).astype(np.float16)
    v = x.reshape(P, -1).view(np.uint8).copy()
    v, mode, _, _ = base.demote_to_base(v, [1, 4], np.zeros(P, np.uint8), H, D)
    bt = np.arange(P, dtype=np.int32)[None, :]
    ws_k, ws_v, idx = gather.gather_prefill(k, v, None, 0, mode, 0, bt, np.array([[0, 0, P]]))
    for p in range(P):
        w = ws_v[p].view(np.uint16)
        if p in (1, 4):
            assert np.array_equal(w, x[p].view(np.uint16) & np.uint16(0xFF00))
        else:
            assert np.array_equal(w, x[p].view(np.uint16))
