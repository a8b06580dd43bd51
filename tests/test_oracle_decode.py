"""Pins of the decode oracle against closed forms, a library routine and brute force.

Each pin is chosen so that a plausible mistake in ``oracle.decode`` fails one of them:
a wrong GQA mapping, a dropped or misplaced scale, a wrong page/row index, a missing
softmax scale, a transposed operand or a wrong log-normaliser. ``test_planted_*``
plant such mistakes in a copy of the oracle and check that the pins catch them.
"""

import math

import numpy as np
import pytest
import torch

from mixed_precision_paged_gb300 import workloads as wl
from oracle import decode as od
from oracle import e4m3


def run(case, **kw):
    return od.paged_decode(case.q, case.k_pages, case.v_pages, case.v_scales, case.scale_mode,
                           case.page_mode, case.uniform_mode, case.block_table, case.seq_lens, **kw)


def dequant_token(case, b, t):
    """Float64 V of token t of sequence b, through the page table (all KV heads)."""
    S = wl.PAGE_SIZE
    p = int(case.block_table[b][t // S])
    r = t % S
    H, D = case.num_kv_heads, case.head_dim
    mode = case.uniform_mode if case.page_mode is None else int(case.page_mode[p])
    n = S * H * D
    if mode == wl.MODE_TARGET_FP16:
        return case.v_pages[p][: 2 * n].view("<f2").reshape(S, H, D)[r].astype(np.float64)
    codes = case.v_pages[p][:n].reshape(S, H, D)[r]
    s = (np.full(H, case.v_scales[0]) if case.scale_mode == wl.SCALE_PER_TENSOR
         else case.v_scales[p]).astype(np.float64)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return ref * s[:, None]


@pytest.mark.parametrize("fmt,scale_mode", [("e4m3", 0), ("e4m3", 1), ("fp16", 0), ("mixed", 1)])
def test_single_token_returns_value_times_scale(fmt, scale_mode):
    case = wl.make_decode_case([1, 1], 8, 2, 64, v_format=fmt, scale_mode=scale_mode,
                               pool_pages=5, seed=3)
    out, lse = run(case)
    G = 4
    for b in range(2):
        v = dequant_token(case, b, 0)
        for hq in range(8):
            assert np.array_equal(out[b, hq], v[hq // G])
        z = (case.k_pages[case.block_table[b][0], 0].astype(np.float64)
             @ case.q[b].astype(np.float64).T) / math.sqrt(64)
        assert np.allclose(lse[b], [z[hq // G, hq] for hq in range(8)], rtol=0, atol=1e-12)


def test_uniform_values_are_returned():
    case = wl.make_decode_case([37, 100], 4, 2, 64, v_format="fp16", pool_pages=12,
                               seed=4, uniform_v=0.75)
    out, _ = run(case)
    assert np.allclose(out, 0.75, rtol=0, atol=1e-12)


def test_zero_query_gives_mean_of_values():
    case = wl.make_decode_case([37, 100], 4, 2, 64, v_format="mixed", scale_mode=1,
                               pool_pages=12, seed=5, q_zero=True)
    out, lse = run(case)
    for b, L in enumerate([37, 100]):
        V = np.stack([dequant_token(case, b, t) for t in range(L)])     # [L][H][D]
        for hq in range(4):
            assert np.allclose(out[b, hq], V[:, hq // 2].mean(axis=0), rtol=0, atol=1e-12)
        assert np.allclose(lse[b], math.log(L), atol=1e-12)


def test_all_fp16_matches_torch_sdpa_float64():
    lens = [1, 16, 17, 100]
    case = wl.make_decode_case(lens, 8, 2, 128, v_format="fp16", pool_pages=16, seed=6)
    out, _ = run(case)
    S = wl.PAGE_SIZE
    for b, L in enumerate(lens):
        pages = case.block_table[b][: (L + S - 1) // S]
        K = np.concatenate([case.k_pages[p] for p in pages])[:L]           # [L][H][D]
        V = np.concatenate([case.v_pages[p].view("<f2").reshape(S, 2, 128) for p in pages])[:L]
        q = torch.from_numpy(case.q[b].astype(np.float64))[:, None, :]    # [Hq][1][D]
        k = torch.from_numpy(K.astype(np.float64)).permute(1, 0, 2)        # [H][L][D]
        v = torch.from_numpy(V.astype(np.float64)).permute(1, 0, 2)
        k = k.repeat_interleave(4, dim=0)
        v = v.repeat_interleave(4, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v)[:, 0].numpy()
        assert np.allclose(out[b], ref, rtol=0, atol=1e-12)


def test_block_table_permutation_invariance():
    case = wl.make_decode_case([37, 100, 5], 4, 2, 64, v_format="mixed", scale_mode=1,
                               pool_pages=20, seed=8)
    out0, lse0 = run(case)
    rng = np.random.default_rng(9)
    P = case.num_pages
    perm = rng.permutation(P)                 # new position of old page p is perm[p]
    k2 = np.empty_like(case.k_pages); k2[perm] = case.k_pages
    v2 = np.empty_like(case.v_pages); v2[perm] = case.v_pages
    s2 = np.empty_like(case.v_scales); s2[perm] = case.v_scales
    m2 = np.empty_like(case.page_mode); m2[perm] = case.page_mode
    bt2 = perm[case.block_table].astype(np.int32)
    out1, lse1 = od.paged_decode(case.q, k2, v2, s2, 1, m2, 0, bt2, case.seq_lens)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_gqa_mapping_is_contiguous_groups():
    # KV head h holds the constant value h + 1; q head hq must read head hq // G.
    H, G = 4, 2
    case = wl.make_decode_case([20], H * G, H, 64, v_format="fp16", pool_pages=2, seed=10)
    S = wl.PAGE_SIZE
    for p in range(2):
        vals = np.broadcast_to((np.arange(H) + 1.0)[None, :, None], (S, H, 64)).astype(np.float16)
        case.v_pages[p][:] = vals.reshape(-1).view(np.uint8)
    out, _ = run(case)
    for hq in range(H * G):
        assert np.allclose(out[0, hq], hq // G + 1.0, atol=1e-12)


def brute_force(case, sm_scale):
    """Token-by-token pure-Python attention (math.exp, explicit loops)."""
    B, Hq, D = case.q.shape
    H = case.num_kv_heads
    G = Hq // H
    outs = np.zeros((B, Hq, D))
    lses = np.zeros((B, Hq))
    for b in range(B):
        L = int(case.seq_lens[b])
        vs = [dequant_token(case, b, t) for t in range(L)]
        for hq in range(Hq):
            h = hq // G
            zs = []
            for t in range(L):
                p = int(case.block_table[b][t // 16])
                k = case.k_pages[p][t % 16][h]
                zs.append(sum(float(case.q[b, hq, d]) * float(k[d]) for d in range(D)) * sm_scale)
            m = max(zs)
            ws = [math.exp(z - m) for z in zs]
            tot = sum(ws)
            for d in range(D):
                outs[b, hq, d] = sum(w * vs[t][h][d] for t, w in enumerate(ws)) / tot
            lses[b, hq] = m + math.log(tot)
    return outs, lses


@pytest.mark.parametrize("fmt,scale_mode,seed", [("e4m3", 0, 11), ("mixed", 1, 12), ("fp16", 0, 13)])
def test_brute_force_tiny(fmt, scale_mode, seed):
    case = wl.make_decode_case([3, 18, 33], 4, 2, 16, v_format=fmt, scale_mode=scale_mode,
                               pool_pages=9, seed=seed)
    out, lse = run(case)
    ref_out, ref_lse = brute_force(case, 1.0 / 4.0)
    assert np.allclose(out, ref_out, rtol=0, atol=1e-11)
    assert np.allclose(lse, ref_lse, rtol=0, atol=1e-11)


def test_explicit_sm_scale_and_default():
    case = wl.make_decode_case([21], 2, 1, 64, v_format="fp16", pool_pages=2, seed=14)
    a, _ = run(case)
    b, _ = run(case, sm_scale=1.0 / 8.0)
    c, _ = run(case, sm_scale=0.5)
    assert np.array_equal(a, b) and not np.allclose(a, c)


def test_empty_sequence():
    case = wl.make_decode_case([0, 5], 2, 1, 64, v_format="e4m3", pool_pages=2, seed=15)
    out, lse = run(case)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1]))


def test_poisoned_tail_is_not_read():
    case = wl.make_decode_case([37, 100], 4, 2, 64, v_format="mixed", scale_mode=1,
                               pool_pages=32, seed=16)
    out, lse = run(case)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


# ------------------------------------------------------------------ planted mistakes

def _mutant_attend(kind):
    def attend(q_b, K, V, sm_scale):
        H_q, D = q_b.shape
        L, H_kv, _ = K.shape
        G = H_q // H_kv
        out = np.zeros((H_q, D)); lse = np.full(H_q, -np.inf)
        for hq in range(H_q):
            h = hq % H_kv if kind == "gqa" else hq // G
            s = 1.0 if kind == "no_scale" else sm_scale
            z = (K[:, h, :] @ q_b[hq].astype(np.float64)) * s
            m = z.max(); w = np.exp(z - m)
            out[hq] = (w @ V[:, h, :]) / (w.sum() if kind != "no_norm" else 1.0)
            lse[hq] = m + math.log(w.sum())
        return out, lse
    return attend


@pytest.mark.parametrize("kind,pin", [
    ("gqa", test_gqa_mapping_is_contiguous_groups),
    ("no_scale", test_all_fp16_matches_torch_sdpa_float64),
    ("no_norm", test_uniform_values_are_returned),
])
def test_planted_mistake_is_caught(monkeypatch, kind, pin):
    monkeypatch.setattr(od, "attend", _mutant_attend(kind))
    with pytest.raises(AssertionError):
        pin()


def test_planted_scale_drop_is_caught(monkeypatch):
    orig = od.dequant_value_page

    def no_scale(v_page_bytes, mode, scale_row, H_kv, D, S=16):
        return orig(v_page_bytes, mode, np.ones_like(scale_row), H_kv, D, S)
    monkeypatch.setattr(od, "dequant_value_page", no_scale)
    with pytest.raises(AssertionError):
        test_single_token_returns_value_times_scale("e4m3", 1)


def test_planted_row_index_mistake_is_caught(monkeypatch):
    orig = od.sequence_kv

    def shifted(b, *a):
        K, V = orig(b, *a)
        return K, np.roll(V, 1, axis=0)
    monkeypatch.setattr(od, "sequence_kv", shifted)
    with pytest.raises(AssertionError):
        test_brute_force_tiny("e4m3", 0, 11)
