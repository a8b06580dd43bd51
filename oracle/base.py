"""ElasticKV BASE value pages, in exact integer / float64 arithmetic. Oracle only.

ElasticKV ("Does Execution Require Target KV Fidelity?"), Sec. 3 opening, Sec. 3.2 and
App. B.2-B.3: BASE keeps the high-order 8 bits of each 16-bit TARGET value; the
low-order 8 bits refine it exactly back to TARGET. There is no scale and no
dequantisation transform: attention places the stored byte in the high half of the
native 16-bit word, zero-fills the low half and reinterprets the word as FP16.

* ``base_value``     -- float64 value of BASE bytes (high byte, low byte zero).
* ``demote_to_base`` -- TARGET -> BASE in place: the page's first S*H_kv*D bytes
                        become the high bytes, the low bytes are returned (the
                        "CPU backing" that exact promotion restores from).
* ``promote``        -- BASE -> TARGET in place from those low bytes (App. B.2:
                        promotion re-attaches the low byte in one step).

A page holding NaN/inf is not demoted (reported, left TARGET), as for the E4M3
demotion. Pins: ``tests/test_oracle_base.py``.
"""

import numpy as np

PAGE_SIZE = 16
MODE_TARGET_FP16 = 0
MODE_COMPACT_E4M3 = 1
MODE_BASE = 2


def base_value(codes):
    """Float64 values of BASE bytes: the FP16 whose high byte is the code and whose
    low byte is zero."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.uint16)
    words = (c << np.uint16(8)).astype("<u2")
    return words.view("<f2").astype(np.float64)


def demote_to_base(v_pages, page_ids, page_mode, H_kv, D, S=PAGE_SIZE):
    """TARGET -> BASE for each listed TARGET page. Returns (v_pages', page_mode',
    low [P][S*H_kv*D] uint8 (zeros for pages not demoted), nonfinite page list)."""
    v = np.array(v_pages, dtype=np.uint8, copy=True)
    m = np.array(page_mode, dtype=np.uint8, copy=True)
    n = S * H_kv * D
    low = np.zeros((v.shape[0], n), dtype=np.uint8)
    bad = []
    for p in np.asarray(page_ids).reshape(-1):
        p = int(p)
        if m[p] != MODE_TARGET_FP16:
            continue
        words = np.ascontiguousarray(v[p, : 2 * n]).view("<u2")
        if not np.all(np.isfinite(words.view("<f2"))):
            bad.append(p)
            continue
        high = (words >> np.uint16(8)).astype(np.uint8)
        low[p] = (words & np.uint16(0xFF)).astype(np.uint8)
        v[p, :n] = high
        m[p] = MODE_BASE
    return v, m, low, bad


def promote(v_pages, page_ids, page_mode, low, H_kv, D, S=PAGE_SIZE):
    """BASE -> TARGET for each listed BASE page, from its low bytes ``low[i]`` (one row
    per listed page, in list order). Returns (v_pages', page_mode')."""
    v = np.array(v_pages, dtype=np.uint8, copy=True)
    m = np.array(page_mode, dtype=np.uint8, copy=True)
    n = S * H_kv * D
    for i, p in enumerate(np.asarray(page_ids).reshape(-1)):
        p = int(p)
        if m[p] != MODE_BASE:
            continue
        high = v[p, :n].astype(np.uint16)
        words = (high << np.uint16(8)) | np.asarray(low[i], dtype=np.uint8).astype(np.uint16)
        v[p, : 2 * n] = words.astype("<u2").view(np.uint8)
        m[p] = MODE_TARGET_FP16
    return v, m
