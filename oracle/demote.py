"""TARGET -> compact demotion of FP16 value pages. Oracle only, exact.

ElasticKV Sec. 3.4 "Transition protocols": demotion is a synchronous, in-place
transition on the GPU; a page changes state only once the transition has completed.
The compact format is the scaled FP8 E4M3 of the knlp.io page (not ElasticKV's FP16
high byte). The pages do not say how scales are calibrated; the plain absmax reading
is taken, one scale per (page, KV head):

1. a_h = max |x| over the page's 16 x D values of KV head h (exact).
2. s_h = fp32_RN(a_h / 448); s_h = 1.0 when a_h == 0.
3. y = fp32_RN(x / s_h).
4. code = E4M3 round-to-nearest-even of y, saturating to +-448, sign kept.

Steps 2 and 3 compute the quotient in float64 and round it to float32. Double rounding
is innocuous for division when the wide format has at least 2p+2 bits (53 >= 2*24+2;
S. A. Figueroa, "When is double rounding innocuous?", SIGNUM Newsletter 30(3), 1995),
so the result is the IEEE float32 quotient.

The codes overwrite the first S*H_kv*D bytes of the page's value slot; the page mode
becomes compact and the scales are stored. Pages that are not TARGET are skipped.
"""

import numpy as np

from . import e4m3

PAGE_SIZE = 16
MODE_TARGET_FP16 = 0
MODE_COMPACT_E4M3 = 1


def page_scales(x):
    """Scales float32 [H_kv] of one FP16 page ``x`` [S][H_kv][D]."""
    a = np.abs(x.astype(np.float64)).max(axis=(0, 2))
    s = (a / 448.0).astype(np.float32)
    s[a == 0] = np.float32(1.0)
    return s


def quantise_page(x, s):
    """E4M3 codes uint8 [S][H_kv][D] of FP16 page ``x`` with scales ``s`` [H_kv]."""
    y = (x.astype(np.float64) / s.astype(np.float64).reshape(1, -1, 1)).astype(np.float32)
    return e4m3.encode_rne_satfinite(y.astype(np.float64))


def demote_pages(v_pages, page_ids, page_mode, scale_out, H_kv, D, S=PAGE_SIZE):
    """Oracle of ``ekv_demote_pages``; returns updated copies (inputs untouched).

    v_pages: uint8 [P][v_page_stride_bytes] with FP16 TARGET pages;
    page_mode: uint8 [P]; scale_out: float32 [P][H_kv].
    """
    v = v_pages.copy()
    mode = page_mode.copy()
    scales = scale_out.copy()
    n = S * H_kv * D
    for p in np.asarray(page_ids).reshape(-1):
        p = int(p)
        if mode[p] != MODE_TARGET_FP16:
            continue
        x = np.ascontiguousarray(v[p][: 2 * n]).view("<f2").reshape(S, H_kv, D)
        if not np.all(np.isfinite(x)):
            continue          # a page holding NaN/inf is reported and left TARGET
        s = page_scales(x)
        codes = quantise_page(x, s)
        v[p][:n] = codes.reshape(-1)
        scales[p] = s
        mode[p] = MODE_COMPACT_E4M3
    return v, mode, scales
