"""Pins of the cache-writer oracle (oracle/writer.py).

* Layout, by brute force on tiny pools: exactly the row (page, t % 16) of each written
  token changes, in K and in V, and nothing else; t < 0 writes nothing.
* K and TARGET V are the input bits (knlp.io: "K bit-exact").
* E4M3 V: the codes equal torch's float8_e4m3fn cast of the fp32 quotient (a library
  routine; inputs kept below 448 in magnitude, where that cast is RNE), and decode back
  to within half an E4M3 step of v / s ("V within FP8 noise").
* BASE V: the stored byte is the value truncated to 2 fraction bits (the BASE rule).
* Written pages read back through the decode oracle: a one-token sequence whose only
  token is the appended one returns that token's dequantised value.
"""

import numpy as np
import pytest

from oracle import decode, e4m3, writer

torch = pytest.importorskip("torch")

H, D = 2, 64


def _pools(P, mode_list, seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((P, 16, H, D)).astype(np.float16)
    v = rng.integers(0, 256, size=(P, 2 * 16 * H * D), dtype=np.uint8)
    v[:, :] = np.where(v == 0x7F, 0x11, v)              # no E4M3 NaN codes in the filler
    return k, v, np.array(mode_list, dtype=np.uint8)


def test_only_the_new_rows_change():
    P = 6
    k, v, modes = _pools(P, [0, 1, 2, 0, 1, 2], 1)
    scales = np.full((P, H), 0.01, np.float32)
    bt = np.array([[0, 1, 2], [3, 4, 5], [1, 2, 0]], np.int32)
    pos = np.array([5, 33, -1], np.int32)               # page 0 row 5, page 5 row 1, none
    rng = np.random.default_rng(2)
    kn = rng.standard_normal((3, H, D)).astype(np.float16)
    vn = (rng.standard_normal((3, H, D)) * 0.5).astype(np.float16)
    k2, v2 = writer.append_token(k, v, scales, 1, modes, 0, bt, pos, kn, vn)
    changed_k = {(p, r) for p in range(P) for r in range(16) if not np.array_equal(k2[p, r], k[p, r])}
    assert changed_k == {(0, 5), (5, 1)}
    assert np.array_equal(k2[0, 5].view(np.uint16), kn[0].view(np.uint16))
    assert np.array_equal(k2[5, 1].view(np.uint16), kn[1].view(np.uint16))
    diff = np.nonzero(np.any(v2 != v, axis=1))[0].tolist()
    assert diff == [0, 5]
    # TARGET page 0: bytes of row 5 only, equal to the input bits
    row = H * D * 2
    assert np.array_equal(v2[0, 5 * row: 6 * row], vn[0].reshape(-1).view(np.uint8))
    assert np.array_equal(np.delete(v2[0], np.s_[5 * row: 6 * row]), np.delete(v[0], np.s_[5 * row: 6 * row]))
    # BASE page 5, row 1: one byte per value
    rb = H * D
    assert np.array_equal(np.delete(v2[5], np.s_[rb: 2 * rb]), np.delete(v[5], np.s_[rb: 2 * rb]))


def test_e4m3_row_is_the_library_cast_and_within_half_a_step():
    P = 3
    k, v, modes = _pools(P, [1, 1, 1], 3)
    rng = np.random.default_rng(4)
    s = np.array([[0.003, 0.02], [0.5, 1e-4], [1.0, 2.0]], np.float32)
    bt = np.array([[0], [1], [2]], np.int32)
    pos = np.array([0, 7, 15], np.int32)
    vn = (rng.standard_normal((3, H, D)) * 0.4).astype(np.float16)
    for b in range(3):                                  # keep |v / s| < 448
        vn[b] = np.clip(vn[b].astype(np.float32), -400 * s[b][:, None], 400 * s[b][:, None]).astype(np.float16)
    kn = rng.standard_normal((3, H, D)).astype(np.float16)
    _, v2 = writer.append_token(k, v, s, 1, modes, 0, bt, pos, kn, vn)
    for b in range(3):
        t = pos[b]
        codes = v2[b, t * H * D: (t + 1) * H * D].reshape(H, D)
        q32 = torch.from_numpy(vn[b].astype(np.float32)) / torch.from_numpy(s[b]).reshape(H, 1)
        lib = q32.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes, lib)
        back = e4m3.decode(codes) * s[b].astype(np.float64).reshape(H, 1)
        y = vn[b].astype(np.float64)
        # half a step of the E4M3 grid around y/s: step = 2^(floor(log2|y/s|) - 3), >= 2^-9
        ys = np.abs(y / s[b].astype(np.float64).reshape(H, 1))
        step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(ys, 2.0 ** -9))), -6) - 3)
        assert np.all(np.abs(back - y) <= 0.5 * step * s[b].reshape(H, 1) * (1 + 1e-6))


def test_base_row_is_truncation():
    P = 2
    k, v, modes = _pools(P, [2, 2], 5)
    rng = np.random.default_rng(6)
    vn = (rng.standard_normal((2, H, D)) * 3).astype(np.float16)
    kn = rng.standard_normal((2, H, D)).astype(np.float16)
    bt = np.array([[0], [1]], np.int32)
    _, v2 = writer.append_token(k, v, None, 0, modes, 0, bt, np.array([3, 9], np.int32), kn, vn)
    for b, t in ((0, 3), (1, 9)):
        hb = v2[b, t * H * D: (t + 1) * H * D].astype(np.uint16) << 8
        got = hb.view(np.float16).astype(np.float64).reshape(H, D)
        x = vn[b].astype(np.float64)
        e = np.floor(np.log2(np.where(x == 0, 1.0, np.abs(x))))
        unit = np.where(e >= -14, np.exp2(e - 2), 2.0 ** -16)
        assert np.array_equal(got, np.sign(x) * np.floor(np.abs(x) / unit) * unit)


def test_appended_token_reads_back_through_decode():
    P = 4
    k, v, modes = _pools(P, [0, 1, 2, 0], 7)
    s = np.full((P, H), 0.01, np.float32)
    rng = np.random.default_rng(8)
    kn = rng.standard_normal((3, H, D)).astype(np.float16)
    vn = (rng.standard_normal((3, H, D)) * 0.5).astype(np.float16)
    bt = np.array([[0], [1], [2]], np.int32)
    k2, v2 = writer.append_token(k, v, s, 1, modes, 0, bt, np.zeros(3, np.int32), kn, vn)
    q = rng.standard_normal((3, 2 * H, D)).astype(np.float16)
    out, _ = decode.paged_decode(q, k2, v2, s, 1, modes, 0, bt, np.ones(3, np.int32))
    # one token: softmax weight 1, out = its dequantised value
    want = [vn[0].astype(np.float64),
            e4m3.decode(v2[1, : H * D].reshape(H, D)) * s[1].astype(np.float64).reshape(H, 1),
            (v2[2, : H * D].astype(np.uint16) << 8).view(np.float16).astype(np.float64).reshape(H, D)]
    for b in range(3):
        assert np.allclose(out[b], np.repeat(want[b], 2, axis=0), rtol=0, atol=1e-12)
