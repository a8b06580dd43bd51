"""Pins of the prefill oracle (oracle/prefill.py) to things other than its own formula:

* torch's scaled_dot_product_attention with is_causal=True in float64 (a library routine)
  on the same prompt laid out contiguously, GQA by repeating the KV heads;
* the first query row of every prompt returns its first value row exactly (one key);
* with identical keys, row s returns the mean of values 0..s (uniform causal weights);
* the workspace layout: shuffling which pages a prompt owns, with page_off following,
  changes nothing.
"""

import math

import numpy as np
import pytest

from oracle import prefill

torch = pytest.importorskip("torch")


def _case(lens, H_q, H_kv, D, seed, slack=3):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    npages = [(l + 15) // 16 for l in lens]
    page_off = np.concatenate([[0], np.cumsum(npages)[:-1]]).astype(np.int32)
    W = sum(npages) + slack
    q = rng.standard_normal((int(cu[-1]), H_q, D)).astype(np.float16)
    ws_k = rng.standard_normal((W, 16, H_kv, D)).astype(np.float16)
    ws_v = rng.standard_normal((W, 16, H_kv, D)).astype(np.float16)
    return q, ws_k, ws_v, cu, page_off


def test_matches_torch_sdpa_causal():
    lens = [1, 17, 40, 100]
    H_q, H_kv, D = 8, 2, 64
    q, k, v, cu, po = _case(lens, H_q, H_kv, D, 1)
    out, lse = prefill.prefill_attention(q, k, v, cu, po)
    for i, L in enumerate(lens):
        pages = po[i] + np.arange((L + 15) // 16)
        K = torch.from_numpy(k[pages].astype(np.float64).reshape(-1, H_kv, D)[:L]).permute(1, 0, 2)
        V = torch.from_numpy(v[pages].astype(np.float64).reshape(-1, H_kv, D)[:L]).permute(1, 0, 2)
        Q = torch.from_numpy(q[cu[i]: cu[i + 1]].astype(np.float64)).permute(1, 0, 2)
        K = K.repeat_interleave(H_q // H_kv, dim=0)
        V = V.repeat_interleave(H_q // H_kv, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=1 / math.sqrt(D))
        assert np.allclose(out[cu[i]: cu[i + 1]], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_first_row_is_first_value_and_uniform_keys_average():
    lens = [33, 20]
    H_q, H_kv, D = 4, 4, 64
    q, k, v, cu, po = _case(lens, H_q, H_kv, D, 2)
    k[:] = k[0, 0, 0]                                   # every key identical
    out, _ = prefill.prefill_attention(q, k, v, cu, po)
    for i, L in enumerate(lens):
        V = v[po[i] + np.arange((L + 15) // 16)].astype(np.float64).reshape(-1, H_kv, D)[:L]
        assert np.array_equal(out[cu[i]], V[0])         # one key: its value exactly
        for s in (1, 7, L - 1):
            assert np.allclose(out[cu[i] + s], V[: s + 1].mean(axis=0), rtol=0, atol=1e-12)


def test_page_placement_is_irrelevant():
    lens = [50, 31]
    q, k, v, cu, po = _case(lens, 4, 2, 64, 3, slack=0)
    out, lse = prefill.prefill_attention(q, k, v, cu, po)
    # give prompt 1 the first pages and prompt 0 the last ones
    n0, n1 = (lens[0] + 15) // 16, (lens[1] + 15) // 16
    perm = np.concatenate([np.arange(n0, n0 + n1), np.arange(n0)])
    k2, v2 = k[perm], v[perm]
    po2 = np.array([n1, 0], np.int32)
    out2, lse2 = prefill.prefill_attention(q, k2, v2, cu, po2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
