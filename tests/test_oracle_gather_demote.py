"""Pins of the gather and demotion oracles.

Gather is pinned against PyTorch's float8_e4m3fn -> float32 cast followed by a torch
float32 multiply and float16 cast (independent IEEE arithmetic), against bit copies
for K and TARGET pages, and against the page table. Demotion is pinned against torch
float32 division plus the torch float8 cast, and against invariants: +-absmax encodes
to +-448, reconstruction error is within half an E4M3 step times the scale, an
all-zero page gets scale 1, and demote -> gather reproduces the dequantised values.
"""

import numpy as np
import pytest
import torch

from mixed_precision_paged_gb300 import workloads as wl
from oracle import demote as odm
from oracle import e4m3
from oracle import gather as og


def gather_case(fmt, scale_mode, seed):
    return wl.make_decode_case([40, 64, 17], 8, 4, 64, v_format=fmt, scale_mode=scale_mode,
                               pool_pages=14, seed=seed, poison=False)


def torch_dequant_fp16(codes, s):
    f = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32)
    return (f * torch.from_numpy(s.astype(np.float32))).to(torch.float16).numpy()


@pytest.mark.parametrize("fmt,scale_mode", [("e4m3", 0), ("e4m3", 1), ("mixed", 1), ("fp16", 0)])
def test_gather_matches_independent_cast(fmt, scale_mode):
    c = gather_case(fmt, scale_mode, 21)
    pr = np.array([[1, 1, 3], [0, 0, 2], [2, 0, 2]])
    ws_k, ws_v, idx = og.gather_prefill(c.k_pages, c.v_pages, c.v_scales, scale_mode,
                                        c.page_mode, c.uniform_mode, c.block_table, pr)
    pages = [c.block_table[1][1], c.block_table[1][2], c.block_table[1][3],
             c.block_table[0][0], c.block_table[0][1], c.block_table[2][0], c.block_table[2][1]]
    assert ws_k.shape[0] == 7 and np.array_equal(idx, np.arange(7))
    S, H, D = 16, 4, 64
    n = S * H * D
    for w, p in enumerate(pages):
        assert np.array_equal(ws_k[w].view(np.uint16), c.k_pages[p].view(np.uint16))
        mode = c.uniform_mode if c.page_mode is None else c.page_mode[p]
        if mode == 0:
            assert np.array_equal(ws_v[w].reshape(-1).view(np.uint8), c.v_pages[p][: 2 * n])
        else:
            s = (np.full(H, c.v_scales[0]) if scale_mode == 0 else c.v_scales[p])
            s = np.broadcast_to(s.reshape(1, H, 1), (S, H, D))
            ref = torch_dequant_fp16(c.v_pages[p][:n].reshape(S, H, D), s)
            assert np.array_equal(ws_v[w].view(np.uint16), ref.view(np.uint16))


def test_gather_without_scale_is_plain_cast():
    c = gather_case("e4m3", 1, 22)
    pr = np.array([[0, 0, 3]])
    _, ws_v, _ = og.gather_prefill(c.k_pages, c.v_pages, c.v_scales, 1, None, 1,
                                   c.block_table, pr, apply_scale=False)
    for w in range(3):
        p = c.block_table[0][w]
        ref = torch.from_numpy(c.v_pages[p].copy()).view(torch.float8_e4m3fn).to(torch.float16)
        assert np.array_equal(ws_v[w].reshape(-1).view(np.uint16), ref.numpy().view(np.uint16))


def test_gather_empty_range():
    c = gather_case("e4m3", 0, 23)
    ws_k, ws_v, idx = og.gather_prefill(c.k_pages, c.v_pages, c.v_scales, 0, None, 1,
                                        c.block_table, np.zeros((0, 3), dtype=np.int64))
    assert ws_k.shape[0] == 0 and idx.size == 0


def fp16_pool(P, H, D, std, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((P, 16, H, D)) * std).astype(np.float16)
    return x, x.reshape(P, -1).view(np.uint8).copy()


def test_demote_matches_torch_division_and_cast():
    P, H, D = 6, 4, 64
    x, vb = fp16_pool(P, H, D, np.sqrt(2.0), 31)
    mode = np.zeros(P, dtype=np.uint8)
    sc = np.zeros((P, H), dtype=np.float32)
    ids = np.array([4, 1, 2])
    v2, m2, s2 = odm.demote_pages(vb, ids, mode, sc, H, D)
    n = 16 * H * D
    for p in range(P):
        if p not in ids:
            assert np.array_equal(v2[p], vb[p]) and m2[p] == 0
            continue
        xt = torch.from_numpy(x[p].astype(np.float32))
        a = xt.abs().amax(dim=(0, 2))
        s_ref = a / torch.tensor(448.0, dtype=torch.float32)            # IEEE fp32 divide
        assert np.array_equal(s2[p], s_ref.numpy())
        y = xt / s_ref.reshape(1, H, 1)
        codes = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(v2[p][:n].reshape(16, H, D), codes)
        assert np.array_equal(v2[p][n:], vb[p][n:])          # second half untouched
        assert m2[p] == 1


def test_demote_invariants():
    P, H, D = 3, 2, 128
    x, vb = fp16_pool(P, H, D, 1.0, 32)
    x[1] = 0
    x[2, 3, 1, 7] = -np.abs(x[2]).max() * 2                   # unique absmax, negative
    vb = x.reshape(P, -1).view(np.uint8).copy()
    v2, m2, s2 = odm.demote_pages(vb, [0, 1, 2], np.zeros(P, np.uint8),
                                  np.zeros((P, H), np.float32), H, D)
    n = 16 * H * D
    codes = v2[:, :n].reshape(P, 16, H, D)
    assert codes[2, 3, 1, 7] == 0xFE
    assert np.all(s2[1] == 1.0) and np.all((codes[1] & 0x7F) == 0)
    for p in (0, 2):
        deq = e4m3.decode(codes[p]) * s2[p].reshape(1, H, 1).astype(np.float64)
        y = np.abs(x[p].astype(np.float64)) / s2[p].reshape(1, H, 1)
        # half an E4M3 step at |y|: steps are 2**-9 below 2**-6, else 2**(e-3)
        e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
        half_step = 0.5 * np.exp2(e - 3) * s2[p].reshape(1, H, 1)
        assert np.all(np.abs(deq - x[p]) <= half_step * (1 + 1e-6) + 1e-12)


def test_demote_skips_non_target_and_nonfinite():
    P, H, D = 3, 2, 64
    x, vb = fp16_pool(P, H, D, 1.0, 33)
    x[2, 0, 0, 0] = np.inf
    vb = x.reshape(P, -1).view(np.uint8).copy()
    mode = np.array([1, 0, 0], dtype=np.uint8)
    v2, m2, s2 = odm.demote_pages(vb, [0, 1, 2], mode, np.zeros((P, H), np.float32), H, D)
    assert np.array_equal(v2[0], vb[0]) and m2[0] == 1
    assert m2[1] == 1
    assert np.array_equal(v2[2], vb[2]) and m2[2] == 0


def test_demote_then_gather_round_trip():
    P, H, D = 4, 4, 64
    x, vb = fp16_pool(P, H, D, np.sqrt(2.0), 34)
    v2, m2, s2 = odm.demote_pages(vb, [0, 2], np.zeros(P, np.uint8),
                                  np.zeros((P, H), np.float32), H, D)
    k = np.zeros((P, 16, H, D), np.float16)
    bt = np.arange(P, dtype=np.int32)[None, :]
    _, ws_v, _ = og.gather_prefill(k, v2, s2, 1, m2, 0, bt, np.array([[0, 0, 4]]))
    n = 16 * H * D
    for p in range(P):
        if m2[p] == 0:
            assert np.array_equal(ws_v[p], x[p])
        else:
            deq = e4m3.decode(v2[p][:n].reshape(16, H, D)) * s2[p].reshape(1, H, 1)
            assert np.array_equal(ws_v[p], deq.astype(np.float32).astype(np.float16))
            err = np.abs(ws_v[p].astype(np.float64) - x[p].astype(np.float64))
            # E4M3 keeps 3 mantissa bits: relative error <= 2**-4, plus fp16 rounding
            assert np.all(err <= np.abs(x[p].astype(np.float64)) * (2.0 ** -4 + 2.0 ** -10) + 1e-3)
